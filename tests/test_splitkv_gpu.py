"""Split-KV forward (key ranges in separate CTAs, merged by the two-block rule) against
the FP64 oracle, element by element, and against attn_fwd."""
import math

import numpy as np
import pytest
import torch

import oracle
import tiled_online_softmax_attention_gb300 as attn
import workloads
from gpu_util import LSE_REL, O_MAX_ABS, Guarded, f64, lse_err, o_err, run_fwd

pytestmark = pytest.mark.gpu


def run_split(q, k, v, causal, n_splits, scale=None):
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = Guarded((B, H, N, d), q.dtype)
    lse = Guarded((B, H, N), torch.float32)
    nbytes = attn.attn_fwd_splitkv_workspace_bytes(B, H, N, d, n_splits)
    ws = Guarded((nbytes // 4,), torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = attn.attn_fwd_splitkv(q, k, v, o.t, lse.t, ws.t, nbytes, B, H, N, d, q.dtype, causal, scale, n_splits,
                               status)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert o.intact() and lse.intact() and ws.intact(), "split-KV wrote outside its buffers"
    return o.t, lse.t


@pytest.mark.parametrize("n_splits", [1, 2, 3, 8])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("N", [1, 129, 300, 1000])
def test_splitkv_vs_oracle(N, d, causal, n_splits):
    x = workloads.draw(1, 3, N, d, "bf16", seed=3000 + N + d + n_splits)
    o, lse = run_split(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal, n_splits)
    o_ref, lse_ref = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, 1.0 / math.sqrt(d))
    assert o_err(o, o_ref) <= O_MAX_ABS
    assert lse_err(lse, lse_ref) <= LSE_REL


@pytest.mark.parametrize("causal", [False, True])
def test_splitkv_long_single_head_matches_fwd(causal):
    """One head of 16384 tokens, 4 ranges: sampled rows against the oracle, all rows
    against attn_fwd."""
    x = workloads.draw(1, 1, 16384, 128, "bf16", seed=77)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = run_split(q, k, v, causal, 4)
    o1, l1 = run_fwd(q, k, v, causal)
    assert float((o.float() - o1.float()).abs().max()) <= O_MAX_ABS
    assert float(((lse - l1).abs() / l1.abs().clamp_min(1)).max()) <= LSE_REL
    rows = np.array([0, 1, 127, 128, 8191, 8192, 16383])
    o_ref, lse_ref = oracle.attn_fwd(x["q"][0, 0], x["k"][0, 0], x["v"][0, 0], causal, 1 / math.sqrt(128), rows=rows)
    assert float(np.max(np.abs(f64(o)[0, 0, rows] - o_ref))) <= O_MAX_ABS
    assert float(np.max(np.abs(f64(lse)[0, 0, rows] - lse_ref) / np.maximum(np.abs(lse_ref), 1))) <= LSE_REL


def test_splitkv_stress_fp16():
    """The numerics-stress workload (scores near +-1000, one-hot rows, uniform rows) through 3 ranges."""
    x = workloads.inputs("c4")
    o, lse = run_split(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), False, 3)
    o_ref, lse_ref = oracle.attn_fwd(x["q"], x["k"], x["v"], False, 1 / math.sqrt(128))
    assert o_err(o, o_ref) <= O_MAX_ABS
    assert lse_err(lse, lse_ref) <= LSE_REL


def run_split_rect(q, k, v, causal, n_splits, scale=None):
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = Guarded((B, H, Nq, d), q.dtype)
    lse = Guarded((B, H, Nq), torch.float32)
    nbytes = attn.attn_fwd_splitkv_workspace_bytes(B, H, Nq, d, n_splits)
    ws = Guarded((nbytes // 4,), torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = attn.attn_fwd_splitkv_rect(q, k, v, o.t, lse.t, ws.t, nbytes, B, H, Nq, Nk, d, q.dtype, causal, scale,
                                    n_splits, status)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert o.intact() and lse.intact() and ws.intact(), "split-KV wrote outside its buffers"
    return o.t, lse.t


def draw_rect(B, H, Nq, Nk, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, H, Nq, d), generator=g).to(torch.bfloat16)
    k = torch.randn((B, H, Nk, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, H, Nk, d), generator=g).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("n_splits", [2, 5])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("Nq,Nk", [(1, 1000), (64, 4097), (128, 3000), (200, 2000), (300, 300), (513, 700)])
def test_splitkv_rect_vs_oracle(Nq, Nk, d, causal, n_splits):
    """Few queries against many keys (causal: the queries are the last Nq of Nk positions)."""
    q, k, v = draw_rect(1, 2, Nq, Nk, d, seed=Nq * 31 + Nk + d + n_splits)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_split_rect(q.cuda(), k.cuda(), v.cuda(), causal, n_splits, scale)
    ro, rl = oracle.attn_fwd(q, k, v, causal, scale)
    assert o_err(o, ro) <= O_MAX_ABS, f"O error {o_err(o, ro):.3e}"
    assert lse_err(lse, rl) <= LSE_REL


@pytest.mark.parametrize("causal", [False, True])
def test_splitkv_rect_decode_shape_sampled(causal):
    """B=1, H=8, 128 new queries after 32640 earlier positions (Nk = 32768), 16 ranges:
    sampled rows of three heads against the oracle."""
    B, H, Nq, Nk, d = 1, 8, 128, 32768, 128
    q, k, v = draw_rect(B, H, Nq, Nk, d, seed=91)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_split_rect(q.cuda(), k.cuda(), v.cuda(), causal, 16, scale)
    rows = [0, 1, 17, 63, 64, 100, 126, 127]
    for h in (0, 4, 7):
        ro, rl = oracle.attn_fwd(q[0, h], k[0, h], v[0, h], causal, scale, rows=rows)
        assert o_err(o[0, h], ro, rows) <= O_MAX_ABS
        assert float(np.max(np.abs(f64(lse[0, h])[rows] - rl) / np.maximum(np.abs(rl), 1))) <= LSE_REL


@pytest.mark.parametrize("causal", [False, True])
def test_splitkv_d256_decode_shape(causal):
    """d = 256, B=1, H=4, 128 new queries against Nk = 16384 keys, 8 and 16 ranges: all rows
    against the unsplit attn_fwd_rect, sampled rows of two heads against the oracle."""
    B, H, Nq, Nk, d = 1, 4, 128, 16384, 256
    q, k, v = draw_rect(B, H, Nq, Nk, d, seed=92)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1 = torch.empty_like(qd)
    l1 = torch.empty((B, H, Nq), device="cuda", dtype=torch.float32)
    assert attn.attn_fwd_rect(qd, kd, vd, o1, l1, B, H, Nq, Nk, d, qd.dtype, causal, scale) == attn.ATTN_OK
    rows = [0, 1, 17, 63, 64, 100, 126, 127]
    for ns in (8, 16):
        o, lse = run_split_rect(qd, kd, vd, causal, ns, scale)
        assert float((o.float() - o1.float()).abs().max()) <= O_MAX_ABS
        assert float(((lse - l1).abs() / l1.abs().clamp_min(1)).max()) <= LSE_REL
        for h in (0, 3):
            ro, rl = oracle.attn_fwd(q[0, h], k[0, h], v[0, h], causal, scale, rows=rows)
            assert o_err(o[0, h], ro, rows) <= O_MAX_ABS
            assert float(np.max(np.abs(f64(lse[0, h])[rows] - rl) / np.maximum(np.abs(rl), 1))) <= LSE_REL


# ---------------------------------------------------------------- packed variable-length batches


def run_split_varlen(x, causal, n_splits, scale, Tq_pad=0):
    """attn_fwd_varlen_splitkv through the C ABI, guarded outputs; Tq_pad extra query tokens
    after cu_q[B] belong to no sequence and must stay as they were (NaN here)."""
    Tq0, H, d = x["q"].shape
    Tq = Tq0 + Tq_pad
    Tk = x["k"].shape[0]
    B = x["cu_q"].numel() - 1
    max_q = max(1, int(np.diff(x["cu_q"].numpy()).max()))
    max_k = max(1, int(np.diff(x["cu_k"].numpy()).max()))
    q = torch.cat([x["q"], torch.zeros((Tq_pad, H, d), dtype=x["q"].dtype)]).cuda()
    k, v, cu_q, cu_k = (x[n].cuda() for n in ("k", "v", "cu_q", "cu_k"))
    o = Guarded((Tq, H, d), q.dtype)
    lse = Guarded((H, Tq), torch.float32)
    o.t.fill_(float("nan"))
    lse.t.fill_(float("nan"))
    nb = attn.attn_fwd_varlen_splitkv_workspace_bytes(H, Tq, d, n_splits)
    assert nb == n_splits * Tq * H * (d + 1) * 4
    ws = Guarded((nb // 4,), torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = attn.attn_fwd_varlen_splitkv(q, k, v, o.t, lse.t, ws.t, nb, cu_q, cu_k, B, H, max_q, max_k, Tq, Tk, d,
                                      q.dtype, causal, scale, n_splits, status)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and o.intact() and lse.intact() and ws.intact(), "wrote outside its buffers"
    return o.t, lse.t


VARLEN_LENS = [1, 127, 300, 0, 129, 513, 64]


@pytest.mark.parametrize("n_splits", [2, 5])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("extra_keys", [False, True])
def test_splitkv_varlen_vs_oracle(extra_keys, causal, d, n_splits):
    """Packed batches (an empty sequence included; with extra_keys, up to 2000 more keys than
    queries, the decode-like case) against the oracle, and against attn_fwd_varlen."""
    from test_varlen_gpu import packed, run_varlen
    lens_k = [n + e for n, e in zip(VARLEN_LENS, [0, 2000, 100, 3, 700, 7, 1500])] if extra_keys else VARLEN_LENS
    lens_k = [max(n, 1) if q > 0 else n for n, q in zip(lens_k, VARLEN_LENS)]
    x = packed(VARLEN_LENS, lens_k, 3, d, "bf16", seed=301 + d + causal + n_splits)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_split_varlen(x, causal, n_splits, scale)
    ro, rl = oracle.attn_fwd_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], causal, scale)
    assert o_err(o, ro) <= O_MAX_ABS, f"O error {o_err(o, ro):.3e}"
    assert lse_err(lse, rl) <= LSE_REL
    o1, l1 = run_varlen(x, causal, scale, backward=False)
    assert float((o.float() - o1.float()).abs().max()) <= O_MAX_ABS
    assert float(((lse - l1).abs() / l1.abs().clamp_min(1)).max()) <= LSE_REL


@pytest.mark.parametrize("d", [64, 256])
def test_splitkv_varlen_degenerate_and_unowned_rows(d):
    """A sequence without keys and a causal one with fewer keys than queries get O = 0,
    lse = -inf through the merge; query tokens after cu_q[B] are left untouched."""
    from test_varlen_gpu import packed
    lens_q, lens_k = [200, 150, 300], [2000, 0, 100]
    x = packed(lens_q, lens_k, 2, d, "bf16", seed=16)
    o, lse = run_split_varlen(x, True, 4, 0.125, Tq_pad=37)
    go, gl = f64(o), f64(lse)
    cq = x["cu_q"].tolist()
    for b in (1, 2):
        assert np.all(go[cq[b]:cq[b + 1]] == 0) and np.all(np.isneginf(gl[:, cq[b]:cq[b + 1]]))
    assert np.all(np.isnan(go[cq[3]:])) and np.all(np.isnan(gl[:, cq[3]:])), "a row outside every sequence was written"
    ro, rl = oracle.attn_fwd(x["q"][:200].permute(1, 0, 2), x["k"][:2000].permute(1, 0, 2),
                             x["v"][:2000].permute(1, 0, 2), True, 0.125)
    assert float(np.max(np.abs(go[:200] - ro.transpose(1, 0, 2)))) <= O_MAX_ABS
    assert float(np.max(np.abs(gl[:, :200] - rl) / np.maximum(np.abs(rl), 1))) <= LSE_REL


def _random_batches(n, seed):
    from test_varlen_gpu import random_batches
    return random_batches(n, seed=seed)


@pytest.mark.parametrize("i,lens_q,lens_k,causal,d,dtype", _random_batches(20, seed=92))
def test_splitkv_varlen_random_batches(i, lens_q, lens_k, causal, d, dtype):
    """Seeded random packed batches (1-6 sequences, empty ones included, bf16 and fp16)
    through split-KV with 1, 2, 3 or 7 ranges."""
    from test_varlen_gpu import packed
    x = packed(list(lens_q), list(lens_k), 2, d, dtype, seed=950 + i)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_split_varlen(x, causal, (1, 2, 3, 7)[i % 4], scale)
    ro, rl = oracle.attn_fwd_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], causal, scale)
    assert o_err(o, ro) <= O_MAX_ABS, f"O error {o_err(o, ro):.3e}"
    assert lse_err(lse, rl) <= LSE_REL
