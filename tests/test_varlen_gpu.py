"""Parity of the variable-length packed entry points (attn_fwd_varlen, attn_bwd_varlen)
with the FP64 oracle, through the C ABI, with guard zones around every output (the
kernels write packed rows one by one, so a stray row would land in a neighbour's
sequence or outside the buffer)."""
import math

import numpy as np
import pytest
import torch

import oracle
import tiled_online_softmax_attention_gb300 as attn
from gpu_util import GRAD_REL_L2, LSE_REL, O_MAX_ABS, Guarded, f64, grad_err, half_ulp, sample_rows

pytestmark = pytest.mark.gpu


def packed(lens_q, lens_k, H, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    t = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    Tq, Tk = sum(lens_q), sum(lens_k)
    x = {"q": torch.randn((Tq, H, d), generator=g), "k": torch.randn((Tk, H, d), generator=g),
         "v": torch.randn((Tk, H, d), generator=g), "dout": torch.randn((Tq, H, d), generator=g)}
    x = {n: a.to(t) for n, a in x.items()}
    x["cu_q"] = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32)
    x["cu_k"] = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32)
    return x


def run_varlen(x, causal, scale, backward=True):
    Tq, H, d = x["q"].shape
    Tk = x["k"].shape[0]
    B = x["cu_q"].numel() - 1
    lq = np.diff(x["cu_q"].numpy())
    lk = np.diff(x["cu_k"].numpy())
    max_q, max_k = max(1, int(lq.max())), max(1, int(lk.max()))
    q, k, v, do, cu_q, cu_k = (x[n].cuda() for n in ("q", "k", "v", "dout", "cu_q", "cu_k"))
    o = Guarded((Tq, H, d), q.dtype)
    lse = Guarded((H, Tq), torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = attn.attn_fwd_varlen(q, k, v, o.t, lse.t, cu_q, cu_k, B, H, max_q, max_k, Tq, Tk, d, q.dtype, causal, scale,
                              status)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and o.intact() and lse.intact(), "forward wrote outside its outputs"
    if not backward:
        return o.t, lse.t
    dq, dk, dv = Guarded((Tq, H, d), q.dtype), Guarded((Tk, H, d), q.dtype), Guarded((Tk, H, d), q.dtype)
    nb = attn.attn_bwd_workspace_bytes(B, H, max_q, d)
    ws = Guarded((nb // 4,), torch.float32)
    rc = attn.attn_bwd_varlen(q, k, v, o.t, do, lse.t, dq.t, dk.t, dv.t, ws.t, nb, cu_q, cu_k, B, H, max_q, max_k, Tq,
                              Tk, d, q.dtype, causal, scale, status)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and dq.intact() and dk.intact() and dv.intact() and ws.intact()
    return o.t, lse.t, dq.t, dk.t, dv.t


LENS = [1, 127, 300, 0, 129, 513, 64]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("extra_keys", [False, True])
def test_varlen_fwd_bwd(extra_keys, causal, d, dtype):
    lens_k = [n + e for n, e in zip(LENS, [0, 5, 100, 3, 0, 7, 200])] if extra_keys else LENS
    lens_k = [max(n, 1) if q > 0 else n for n, q in zip(lens_k, LENS)]
    x = packed(LENS, lens_k, 3, d, dtype, seed=41 + d + causal)
    scale = 1.0 / math.sqrt(d)
    o, lse, dq, dk, dv = run_varlen(x, causal, scale)
    ro, rl = oracle.attn_fwd_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], causal, scale)
    go = f64(o)
    assert float(np.max(np.abs(go - ro) - half_ulp(ro, o.dtype))) <= O_MAX_ABS
    gl = f64(lse)
    assert float(np.max(np.abs(gl - rl) / np.maximum(np.abs(rl), 1))) <= LSE_REL
    rq, rk, rv = oracle.attn_bwd_varlen(x["q"], x["k"], x["v"], x["dout"], x["cu_q"], x["cu_k"], causal, scale)
    for name, g, r in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        e = grad_err(g, r)
        assert e <= GRAD_REL_L2, f"{name} relative L2 {e:.3e} (causal={causal} d={d} {dtype} extra={extra_keys})"


@pytest.mark.parametrize("d", [128, 256])
def test_varlen_single_sequence_equals_attn_fwd(d):
    N, H = 700, 4
    x = packed([N], [N], H, d, "bf16", seed=5)
    o, lse, dq, dk, dv = run_varlen(x, True, 0.1)
    q, k, v, do = (x[n].permute(1, 0, 2).unsqueeze(0).contiguous().cuda() for n in ("q", "k", "v", "dout"))
    o2, l2 = attn.forward(q, k, v, True, 0.1)
    assert torch.equal(o.permute(1, 0, 2), o2[0]) and torch.equal(lse, l2[0])
    g2 = attn.backward(q, k, v, o2, l2, do, True, 0.1)
    for a, b in zip((dq, dk, dv), g2):
        assert torch.equal(a.permute(1, 0, 2), b[0])


@pytest.mark.parametrize("d", [64, 256])
def test_varlen_degenerate_sequences(d):
    """A sequence without keys, and causal with fewer keys than queries: O = 0, lse = -inf,
    zero gradients; their neighbours are unaffected."""
    lens_q, lens_k = [200, 150, 300], [200, 0, 100]
    x = packed(lens_q, lens_k, 2, d, "bf16", seed=6)
    o, lse, dq, dk, dv = run_varlen(x, True, 0.125)
    cq, ck = x["cu_q"].tolist(), x["cu_k"].tolist()
    go, gl = f64(o), f64(lse)
    for b in (1, 2):
        assert np.all(go[cq[b]:cq[b + 1]] == 0) and np.all(np.isneginf(gl[:, cq[b]:cq[b + 1]]))
        assert np.all(f64(dq)[cq[b]:cq[b + 1]] == 0)
        assert np.all(f64(dk)[ck[b]:ck[b + 1]] == 0) and np.all(f64(dv)[ck[b]:ck[b + 1]] == 0)
    ro, rl = oracle.attn_fwd(x["q"][:200].permute(1, 0, 2), x["k"][:200].permute(1, 0, 2),
                             x["v"][:200].permute(1, 0, 2), True, 0.125)
    assert float(np.max(np.abs(go[:200] - ro.transpose(1, 0, 2)))) <= O_MAX_ABS


def test_varlen_long_batch_sampled():
    """Four sequences of 4000, 1000, 2500 and 8192 tokens, H=16, d=128, causal: sampled
    rows of every sequence against the oracle (forward rows, dQ rows, dK/dV rows)."""
    lens = [4000, 1000, 2500, 8192]
    H, d = 16, 128
    x = packed(lens, lens, H, d, "bf16", seed=7)
    scale = 1.0 / math.sqrt(d)
    o, lse, dq, dk, dv = run_varlen(x, True, scale)
    o, lse, dq, dk, dv = (f64(t) for t in (o, lse, dq, dk, dv))
    cu = x["cu_q"].tolist()
    for b, n in enumerate(lens):
        rows = sample_rows(n, extra=6, seed=b)
        for h in (0, H - 1):
            sl = slice(cu[b], cu[b + 1])
            qh, kh, vh, dh = (x[nm][sl, h] for nm in ("q", "k", "v", "dout"))
            ro, rl = oracle.attn_fwd(qh, kh, vh, True, scale, rows=rows)
            assert float(np.max(np.abs(o[cu[b] + rows, h] - ro))) <= O_MAX_ABS + 2 ** -8 * float(np.abs(ro).max())
            assert float(np.max(np.abs(lse[h, cu[b] + rows] - rl) / np.maximum(np.abs(rl), 1))) <= LSE_REL
            rq, rk, rv = oracle.attn_bwd(qh, kh, vh, dh, True, scale, qrows=rows, kcols=rows)
            for name, g, r in (("dQ", dq[cu[b] + rows, h], rq), ("dK", dk[cu[b] + rows, h], rk),
                               ("dV", dv[cu[b] + rows, h], rv)):
                e = grad_err(g, r)
                assert e <= GRAD_REL_L2, f"sequence {b} head {h} {name} relative L2 {e:.3e}"


def random_batches(n, seed=77):
    import random

    rnd = random.Random(seed)
    out = []
    for i in range(n):
        B = rnd.randint(1, 6)
        causal = rnd.random() < 0.5
        d = rnd.choice([64, 128, 256])
        dtype = rnd.choice(["bf16", "fp16"])
        lq, lk = [], []
        for _ in range(B):
            q = rnd.choice([0, 1, 63, 127, 128, 129, 200, 300, 513])
            if causal:
                k = q + rnd.choice([0, 1, 50, 200])
            else:
                k = rnd.choice([1, 5, 128, 257, 600]) if q > 0 else rnd.choice([0, 7])
            lq.append(q)
            lk.append(k)
        if sum(lq) == 0:
            lq[0], lk[0] = 5, max(lk[0], 5)
        out.append((i, tuple(lq), tuple(lk), causal, d, dtype))
    return out


@pytest.mark.parametrize("i,lens_q,lens_k,causal,d,dtype", random_batches(40))
def test_varlen_random_batches(i, lens_q, lens_k, causal, d, dtype):
    """Seeded random batches of 1-6 sequences (empty ones included), forward and backward."""
    x = packed(list(lens_q), list(lens_k), 2, d, dtype, seed=600 + i)
    scale = 1.0 / math.sqrt(d)
    o, lse, dq, dk, dv = run_varlen(x, causal, scale)
    ro, rl = oracle.attn_fwd_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], causal, scale)
    assert float(np.max(np.abs(f64(o) - ro) - half_ulp(ro, o.dtype))) <= O_MAX_ABS
    assert float(np.max(np.abs(f64(lse) - rl) / np.maximum(np.abs(rl), 1))) <= LSE_REL
    rq, rk, rv = oracle.attn_bwd_varlen(x["q"], x["k"], x["v"], x["dout"], x["cu_q"], x["cu_k"], causal, scale)
    for name, g, r in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        e = grad_err(g, r)
        assert e <= GRAD_REL_L2, f"{name} relative L2 {e:.3e}"
