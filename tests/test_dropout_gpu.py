"""Dropout (attn_fwd_dropout / attn_bwd_dropout) against the FP64 oracle with the same
keep mask (Philox4x32-10, definition in include/attn.h), through the C ABI.

Tolerances: dropout scales the kept probabilities by Z = 256 / (256 - t), so output
magnitudes, and the rounding errors that scale with them, grow by Z; the O bound is
O_MAX_ABS * Z plus the output type's half-ulp.  The logsumexp is the undropped one and
keeps its bound; gradients keep their relative-L2 bound."""
import math

import numpy as np
import pytest
import torch

import oracle
import tiled_online_softmax_attention_gb300 as attn
import workloads
from gpu_util import (GRAD_REL_L2, LSE_REL, O_MAX_ABS, Guarded, assert_same_grads, f64, grad_err, half_ulp, lse_err,
                      o_err, sample_rows)

pytestmark = pytest.mark.gpu


def t_of(p):
    return int(round(256 * p))


def run_fwd_drop(q, k, v, causal, scale, p, seed):
    B, H, N, d = q.shape
    o = Guarded((B, H, N, d), q.dtype)
    lse = Guarded((B, H, N), torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = attn.attn_fwd_dropout(q, k, v, o.t, lse.t, B, H, N, d, q.dtype, causal, scale, p, seed, status)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and o.intact() and lse.intact()
    return o.t, lse.t


def run_bwd_drop(q, k, v, o, lse, do, causal, scale, p, seed):
    B, H, N, d = q.shape
    outs = [Guarded((B, H, N, d), q.dtype) for _ in range(3)]
    nbytes = attn.attn_bwd_workspace_bytes(B, H, N, d)
    ws = Guarded((nbytes // 4,), torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = attn.attn_bwd_dropout(q, k, v, o, do, lse, outs[0].t, outs[1].t, outs[2].t, ws.t, nbytes, B, H, N, d,
                               q.dtype, causal, scale, p, seed, status)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and all(g.intact() for g in outs) and ws.intact()
    return tuple(g.t for g in outs)


@pytest.mark.parametrize("p", [0.1, 0.5])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 127, 128, 129, 300, 513])
def test_dropout_fwd_bwd(N, causal, d, p):
    x = workloads.draw(1, 2, N, d, "bf16", seed=3000 + N + d, with_dout=True)
    scale = 1.0 / math.sqrt(d)
    seed = 0x5EED0000 + N
    t = t_of(p)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = run_fwd_drop(q, k, v, causal, scale, p, seed)
    ro, rl = oracle.attn_fwd_dropout(x["q"], x["k"], x["v"], causal, scale, t, seed)
    z = 256.0 / (256 - t)
    assert o_err(o, ro) <= O_MAX_ABS * z, f"O error {o_err(o, ro):.3e}"
    assert lse_err(lse, rl) <= LSE_REL
    g = run_bwd_drop(q, k, v, o, lse, do, causal, scale, p, seed)
    r = oracle.attn_bwd_dropout(x["q"], x["k"], x["v"], x["dout"], causal, scale, t, seed)
    if N == 1:
        # One key: P = 1 and the exact dS = Z dP - D is 0, so dQ = dK = 0.  The GPU's D is
        # rowsum(dO o O) of the 16-bit O = round(Z V), off from Z dP by at most
        # sum_c |dO_c| half_ulp(O_c); dQ = scale dS K and dK = scale dS Q inherit that.
        o_ref = ro[..., 0, :]
        dsum = np.sum(np.abs(x["dout"].double().numpy()[..., 0, :]) * half_ulp(o_ref, torch.bfloat16), axis=-1)
        for gg, other in ((g[0], x["k"]), (g[1], x["q"])):
            bound = scale * (dsum[..., None] * 1.01 + 1e-6) * np.abs(other.double().numpy()[..., 0, :])
            assert np.all(np.abs(f64(gg)[..., 0, :]) <= bound + 1e-6), "N=1 gradient residue above its bound"
        assert grad_err(g[2], r[2]) <= GRAD_REL_L2
        return
    for name, gg, rr in zip(("dQ", "dK", "dV"), g, r):
        e = grad_err(gg, rr)
        assert e <= GRAD_REL_L2, f"{name} relative L2 {e:.3e} (N={N} d={d} causal={causal} p={p})"


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_dropout_fp16_and_bf16(dtype):
    x = workloads.draw(2, 3, 700, 128, dtype, seed=31, with_dout=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = run_fwd_drop(q, k, v, True, 0.09, 0.2, 77)
    ro, rl = oracle.attn_fwd_dropout(x["q"], x["k"], x["v"], True, 0.09, t_of(0.2), 77)
    assert o_err(o, ro) <= O_MAX_ABS * 256 / (256 - t_of(0.2)) and lse_err(lse, rl) <= LSE_REL
    g = run_bwd_drop(q, k, v, o, lse, do, True, 0.09, 0.2, 77)
    r = oracle.attn_bwd_dropout(x["q"], x["k"], x["v"], x["dout"], True, 0.09, t_of(0.2), 77)
    for gg, rr in zip(g, r):
        assert grad_err(gg, rr) <= GRAD_REL_L2


@pytest.mark.parametrize("d", [128, 256])
def test_dropout_mask_exact(d):
    """Q = 0 makes every visible probability 1/n; with V_j the unit vector e_j, O_ij * n is
    exactly the keep factor Z_ij of key j < d: the GPU's mask equals the oracle's, bit for bit
    of the keep decision."""
    B, H, N = 1, 3, d
    for causal in (False, True):
        q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
        k = torch.randn((B, H, N, d), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).cuda()
        v = torch.eye(d, dtype=torch.bfloat16).expand(B, H, N, d).contiguous().cuda()
        p, seed = 0.3, 0xABCDEF0123
        t = t_of(p)
        o, _ = run_fwd_drop(q, k, v, causal, 0.1, p, seed)
        o = f64(o)
        kept = 0
        for h in range(H):
            for i in range(N):
                n = i + 1 if causal else N
                for j in range(n):
                    zref = oracle.default().dropout_factor(h, i, j, t, seed)
                    got = o[0, h, i, j] * n
                    assert (got > 0) == (zref > 0), f"keep decision differs at head {h}, query {i}, key {j}"
                    kept += zref > 0
        total = H * (N * (N + 1) // 2 if causal else N * N)
        assert abs(1 - kept / total - t / 256) < 0.02


@pytest.mark.parametrize("d", [128, 256])
def test_dropout_dv_mask_exact(d):
    """The backward's keep mask, read through dV = (P o Z)^T dO: with Q = 0 every visible
    probability is 1/n_i, and with dO_i the unit vector e_i, dV_ji * n_i is the keep factor
    Z_ij.  The key-tile kernels hold the mask by key (a transposed draw), so this checks
    that transposition against the oracle's keep decisions."""
    B, H, N = 1, 2, d
    for causal in (False, True):
        q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
        k = torch.randn((B, H, N, d), generator=torch.Generator().manual_seed(6)).to(torch.bfloat16).cuda()
        v = torch.randn((B, H, N, d), generator=torch.Generator().manual_seed(7)).to(torch.bfloat16).cuda()
        do = torch.eye(d, dtype=torch.bfloat16).expand(B, H, N, d).contiguous().cuda()
        p, seed = 0.3, 0x1234567890
        t = t_of(p)
        o, lse = run_fwd_drop(q, k, v, causal, 0.1, p, seed)
        _, _, dv = run_bwd_drop(q, k, v, o, lse, do, causal, 0.1, p, seed)
        dv = f64(dv)
        for h in range(H):
            for i in range(N):
                n = i + 1 if causal else N
                for j in range(n):
                    zref = oracle.default().dropout_factor(h, i, j, t, seed)
                    assert (dv[0, h, j, i] * n > 0) == (zref > 0), \
                        f"backward keep decision differs at head {h}, query {i}, key {j}"
                for j in range(n, N):
                    assert dv[0, h, j, i] == 0, f"masked key {j} of query {i} has a dV entry"


def test_dropout_zero_is_plain_and_seeds_differ():
    x = workloads.draw(1, 2, 400, 128, "bf16", seed=8)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o0, l0 = run_fwd_drop(q, k, v, True, 0.088, 0.0, 1)
    o1, l1 = attn.forward(q, k, v, True, 0.088)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    oa, _ = run_fwd_drop(q, k, v, True, 0.088, 0.25, 1)
    ob, _ = run_fwd_drop(q, k, v, True, 0.088, 0.25, 1)
    oc, _ = run_fwd_drop(q, k, v, True, 0.088, 0.25, 2)
    assert torch.equal(oa, ob) and not torch.equal(oa, oc)


def test_dropout_training_step_sampled():
    """The training-step shape (B=2, H=16, N=8192, d=128, causal) with p = 0.1: sampled
    query rows (O, LSE, dQ) and key rows (dK, dV) of two heads."""
    w = workloads.WORKLOADS["c5"]
    x = workloads.inputs("c5")
    p, seed = 0.1, 20260101
    t = t_of(p)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = run_fwd_drop(q, k, v, True, w.scale, p, seed)
    dq, dk, dv = run_bwd_drop(q, k, v, o, lse, do, True, w.scale, p, seed)
    rows = sample_rows(w.N, extra=8, seed=9)
    for (b, h) in [(0, 0), (w.B - 1, w.H - 1)]:
        bh = b * w.H + h
        qb, kb, vb, dob = (x[n][b, h] for n in ("q", "k", "v", "dout"))
        ro, rl = oracle.attn_fwd_dropout(qb, kb, vb, True, w.scale, t, seed, rows=rows, bh0=bh)
        assert o_err(o[b, h], ro, rows) <= O_MAX_ABS * 256 / (256 - t)
        assert float(np.max(np.abs(f64(lse[b, h])[rows] - rl) / np.maximum(np.abs(rl), 1))) <= LSE_REL
        rq, rk, rv = oracle.attn_bwd_dropout(qb, kb, vb, dob, True, w.scale, t, seed, qrows=rows, kcols=rows, bh0=bh)
        for name, gg, rr in (("dQ", f64(dq[b, h])[rows], rq), ("dK", f64(dk[b, h])[rows], rk),
                             ("dV", f64(dv[b, h])[rows], rv)):
            e = grad_err(gg, rr)
            assert e <= GRAD_REL_L2, f"head ({b},{h}) {name} relative L2 {e:.3e}"


@pytest.mark.parametrize("causal", [False, True])
def test_dropout_d256_long_sampled(causal):
    """d = 256, B=1, H=4, N=4096, p = 0.1: sampled query rows (O, LSE, dQ) and key rows
    (dK, dV) of two heads."""
    B, H, N, d = 1, 4, 4096, 256
    x = workloads.draw(B, H, N, d, "bf16", seed=43, with_dout=True)
    scale = 1.0 / math.sqrt(d)
    p, seed = 0.1, 0xD256
    t = t_of(p)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = run_fwd_drop(q, k, v, causal, scale, p, seed)
    dq, dk, dv = run_bwd_drop(q, k, v, o, lse, do, causal, scale, p, seed)
    rows = sample_rows(N, extra=8, seed=4)
    for h in (0, 3):
        qb, kb, vb, dob = (x[n][0, h] for n in ("q", "k", "v", "dout"))
        ro, rl = oracle.attn_fwd_dropout(qb, kb, vb, causal, scale, t, seed, rows=rows, bh0=h)
        assert o_err(o[0, h], ro, rows) <= O_MAX_ABS * 256 / (256 - t)
        assert float(np.max(np.abs(f64(lse[0, h])[rows] - rl) / np.maximum(np.abs(rl), 1))) <= LSE_REL
        rq, rk, rv = oracle.attn_bwd_dropout(qb, kb, vb, dob, causal, scale, t, seed, qrows=rows, kcols=rows, bh0=h)
        for name, gg, rr in (("dQ", f64(dq[0, h])[rows], rq), ("dK", f64(dk[0, h])[rows], rk),
                             ("dV", f64(dv[0, h])[rows], rv)):
            e = grad_err(gg, rr)
            assert e <= GRAD_REL_L2, f"head {h} {name} relative L2 {e:.3e}"


# ---------------------------------------------------------------- packed variable-length batches


def run_varlen_drop(x, causal, scale, p, seed):
    """attn_fwd_varlen_dropout then attn_bwd_varlen_dropout through the C ABI, guarded outputs."""
    Tq, H, d = x["q"].shape
    Tk = x["k"].shape[0]
    B = x["cu_q"].numel() - 1
    max_q = max(1, int(np.diff(x["cu_q"].numpy()).max()))
    max_k = max(1, int(np.diff(x["cu_k"].numpy()).max()))
    q, k, v, do, cu_q, cu_k = (x[n].cuda() for n in ("q", "k", "v", "dout", "cu_q", "cu_k"))
    o = Guarded((Tq, H, d), q.dtype)
    lse = Guarded((H, Tq), torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = attn.attn_fwd_varlen_dropout(q, k, v, o.t, lse.t, cu_q, cu_k, B, H, max_q, max_k, Tq, Tk, d, q.dtype, causal,
                                      scale, p, seed, status)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and o.intact() and lse.intact(), "forward wrote outside its outputs"
    dq, dk, dv = Guarded((Tq, H, d), q.dtype), Guarded((Tk, H, d), q.dtype), Guarded((Tk, H, d), q.dtype)
    nb = attn.attn_bwd_workspace_bytes(B, H, max_q, d)
    ws = Guarded((nb // 4,), torch.float32)
    rc = attn.attn_bwd_varlen_dropout(q, k, v, o.t, do, lse.t, dq.t, dk.t, dv.t, ws.t, nb, cu_q, cu_k, B, H, max_q,
                                      max_k, Tq, Tk, d, q.dtype, causal, scale, p, seed, status)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and dq.intact() and dk.intact() and dv.intact() and ws.intact()
    return o.t, lse.t, dq.t, dk.t, dv.t


def oracle_varlen_dropout(x, causal, scale, t, seed):
    """The oracle's dropout forward and backward, one sequence at a time on its [H][n][d]
    slices as heads b*H .. b*H + H - 1 of the mask, written back in the packed layout."""
    Tq, H, d = x["q"].shape
    Tk = x["k"].shape[0]
    cq, ck = x["cu_q"].numpy(), x["cu_k"].numpy()
    ro, rl = np.zeros((Tq, H, d)), np.zeros((H, Tq))
    rq, rk, rv = np.zeros((Tq, H, d)), np.zeros((Tk, H, d)), np.zeros((Tk, H, d))
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
        if q1 == q0:
            continue
        sq, sk, sv, sd = (x[n][lo:hi].permute(1, 0, 2) for n, lo, hi in
                          (("q", q0, q1), ("k", k0, k1), ("v", k0, k1), ("dout", q0, q1)))
        o, l = oracle.attn_fwd_dropout(sq, sk, sv, causal, scale, t, seed, bh0=b * H)
        ro[q0:q1], rl[:, q0:q1] = np.transpose(o, (1, 0, 2)), l
        g = oracle.attn_bwd_dropout(sq, sk, sv, sd, causal, scale, t, seed, bh0=b * H)
        rq[q0:q1], rk[k0:k1], rv[k0:k1] = (np.transpose(a, (1, 0, 2)) for a in g)
    return ro, rl, rq, rk, rv


VARLEN_LENS = [1, 127, 300, 0, 129, 513, 64]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("extra_keys", [False, True])
def test_dropout_varlen_fwd_bwd(extra_keys, causal, d):
    """Packed batches (an empty sequence included; with extra_keys, more keys than
    queries) with p = 0.2 against the oracle's per-sequence dropout."""
    from test_varlen_gpu import packed
    lens_k = [n + e for n, e in zip(VARLEN_LENS, [0, 5, 100, 3, 0, 7, 200])] if extra_keys else VARLEN_LENS
    lens_k = [max(n, 1) if q > 0 else n for n, q in zip(lens_k, VARLEN_LENS)]
    x = packed(VARLEN_LENS, lens_k, 3, d, "bf16", seed=71 + d + causal)
    scale, p, seed = 1.0 / math.sqrt(d), 0.2, 0x7A51
    t = t_of(p)
    o, lse, dq, dk, dv = run_varlen_drop(x, causal, scale, p, seed)
    ro, rl, rq, rk, rv = oracle_varlen_dropout(x, causal, scale, t, seed)
    assert o_err(o, ro) <= O_MAX_ABS * 256 / (256 - t), f"O error {o_err(o, ro):.3e}"
    assert lse_err(lse, rl) <= LSE_REL
    for name, g, r in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        e = grad_err(g, r)
        assert e <= GRAD_REL_L2, f"{name} relative L2 {e:.3e} (causal={causal} d={d} extra={extra_keys})"


@pytest.mark.parametrize("d", [64, 128, 256])
def test_dropout_varlen_equals_padded(d):
    """Sequences of one length packed together give attn_fwd_dropout / attn_bwd_dropout's
    bytes on the [B][H][N][d] batch (dQ up to the order of the fused backward's float32
    additions at d <= 128): the packed mask is the padded batch's."""
    from test_varlen_gpu import packed
    B, H, N = 3, 2, 300
    x = packed([N] * B, [N] * B, H, d, "bf16", seed=9 + d)
    scale, p, seed = 0.07, 0.3, 12345
    o, lse, dq, dk, dv = run_varlen_drop(x, True, scale, p, seed)
    q, k, v, do = (x[n].reshape(B, N, H, d).permute(0, 2, 1, 3).contiguous().cuda() for n in ("q", "k", "v", "dout"))
    o2, l2 = run_fwd_drop(q, k, v, True, scale, p, seed)
    g2 = run_bwd_drop(q, k, v, o2, l2, do, True, scale, p, seed)
    unpack = lambda a: a.reshape(B, N, H, d).permute(0, 2, 1, 3)
    assert torch.equal(unpack(o), o2)
    assert torch.equal(lse.reshape(H, B, N).permute(1, 0, 2), l2)
    if d == 256:
        for name, a, b in zip(("dQ", "dK", "dV"), (dq, dk, dv), g2):
            assert torch.equal(unpack(a), b), f"{name} differs from the padded batch's"
    else:
        assert_same_grads(tuple(unpack(a) for a in (dq, dk, dv)), g2, "packed vs padded:")


# ---------------------------------------------------------------- rectangular shapes


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(1, 300), (100, 300), (129, 128), (200, 513), (513, 700)])
def test_dropout_rect_fwd_bwd(Nq, Nk, causal, d):
    """Nq queries against Nk keys (causal: the last Nq of Nk positions) with p = 0.15."""
    if causal and Nk < Nq:
        pytest.skip("causal needs Nk >= Nq")
    from test_rect_gpu import draw_rect
    x = draw_rect(1, 2, Nq, Nk, d, "bf16", seed=Nq * 7 + Nk + d)
    scale, p, seed = 1.0 / math.sqrt(d), 0.15, 0xC0FFEE
    t = t_of(p)
    B, H = 1, 2
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = Guarded((B, H, Nq, d), q.dtype), Guarded((B, H, Nq), torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = attn.attn_fwd_rect_dropout(q, k, v, o.t, lse.t, B, H, Nq, Nk, d, q.dtype, causal, scale, p, seed, status)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    dq = Guarded((B, H, Nq, d), q.dtype)
    dk, dv = Guarded((B, H, Nk, d), q.dtype), Guarded((B, H, Nk, d), q.dtype)
    nb = attn.attn_bwd_workspace_bytes(B, H, Nq, d)
    ws = Guarded((nb // 4,), torch.float32)
    rc = attn.attn_bwd_rect_dropout(q, k, v, o.t, do, lse.t, dq.t, dk.t, dv.t, ws.t, nb, B, H, Nq, Nk, d, q.dtype,
                                    causal, scale, p, seed, status)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and all(g.intact() for g in (o, lse, dq, dk, dv, ws))
    ro, rl = oracle.attn_fwd_dropout(x["q"], x["k"], x["v"], causal, scale, t, seed)
    assert o_err(o.t, ro) <= O_MAX_ABS * 256 / (256 - t), f"O error {o_err(o.t, ro):.3e}"
    assert lse_err(lse.t, rl) <= LSE_REL
    r = oracle.attn_bwd_dropout(x["q"], x["k"], x["v"], x["dout"], causal, scale, t, seed)
    for name, g, rr in zip(("dQ", "dK", "dV"), (dq.t, dk.t, dv.t), r):
        e = grad_err(g, rr)
        assert e <= GRAD_REL_L2, f"{name} relative L2 {e:.3e} ({Nq}x{Nk} causal={causal} d={d})"


def _random_batches(n, seed):
    from test_varlen_gpu import random_batches
    return random_batches(n, seed=seed)


@pytest.mark.parametrize("i,lens_q,lens_k,causal,d,dtype", _random_batches(20, seed=91))
def test_dropout_varlen_random_batches(i, lens_q, lens_k, causal, d, dtype):
    """Seeded random packed batches (1-6 sequences, empty ones included, bf16 and fp16)
    through the dropout entry points, p drawn from {0.05, 0.3}."""
    from test_varlen_gpu import packed
    x = packed(list(lens_q), list(lens_k), 2, d, dtype, seed=900 + i)
    scale, p, seed = 1.0 / math.sqrt(d), (0.05, 0.3)[i % 2], 4000 + i
    t = t_of(p)
    o, lse, dq, dk, dv = run_varlen_drop(x, causal, scale, p, seed)
    ro, rl, rq, rk, rv = oracle_varlen_dropout(x, causal, scale, t, seed)
    assert o_err(o, ro) <= O_MAX_ABS * 256 / (256 - t), f"O error {o_err(o, ro):.3e}"
    assert lse_err(lse, rl) <= LSE_REL
    for name, g, r in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        e = grad_err(g, r)
        assert e <= GRAD_REL_L2, f"{name} relative L2 {e:.3e}"


# ---------------------------------------------------------------- keep bits drawn once


def run_drop_bits(q, k, v, do, causal, scale, p, seed):
    """attn_fwd_dropout_bits then attn_bwd_dropout_bits, guarded outputs and keep bits."""
    B, H, N, d = q.shape
    o, lse = Guarded((B, H, N, d), q.dtype), Guarded((B, H, N), torch.float32)
    nbits = attn.attn_dropout_bits_bytes(B, H, N, N)
    bits = Guarded((nbits // 4,), torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = attn.attn_fwd_dropout_bits(q, k, v, o.t, lse.t, bits.t, nbits, B, H, N, d, q.dtype, causal, scale, p, seed,
                                    status)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and o.intact() and lse.intact() and bits.intact()
    outs = [Guarded((B, H, N, d), q.dtype) for _ in range(3)]
    nb = attn.attn_bwd_workspace_bytes(B, H, N, d)
    ws = Guarded((nb // 4,), torch.float32)
    rc = attn.attn_bwd_dropout_bits(q, k, v, o.t, do, lse.t, bits.t, nbits, outs[0].t, outs[1].t, outs[2].t, ws.t, nb,
                                    B, H, N, d, q.dtype, causal, scale, p, status)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and all(g.intact() for g in outs) and ws.intact() and bits.intact()
    return o.t, lse.t, bits.t, tuple(g.t for g in outs)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_dropout_bits_equal_drawing(causal, d):
    """The stored-bits path gives the drawing path's forward bytes and its dK, dV bytes (dQ
    up to the order of its float32 additions), matches the oracle, and every stored bit is
    the definition's keep decision."""
    B, H, N = 1, 2, 300
    x = workloads.draw(B, H, N, d, "bf16", seed=5100 + d + causal, with_dout=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    scale, p, seed = 1.0 / math.sqrt(d), 0.15, 0x1234ABCD5678
    o, lse, bits, g = run_drop_bits(q, k, v, do, causal, scale, p, seed)
    o2, l2 = run_fwd_drop(q, k, v, causal, scale, p, seed)
    assert torch.equal(o, o2) and torch.equal(lse, l2)
    g2 = run_bwd_drop(q, k, v, o2, l2, do, causal, scale, p, seed)
    assert_same_grads(g, g2, "stored bits vs drawing:")
    t = t_of(p)
    r = oracle.attn_bwd_dropout(x["q"], x["k"], x["v"], x["dout"], causal, scale, t, seed)
    for name, gg, rr in zip(("dQ", "dK", "dV"), g, r):
        assert grad_err(gg, rr) <= GRAD_REL_L2, name
    # every written word against the definition (word ((bh * ntk + j) * 4 + w) * Npad + i)
    words = bits.cpu().numpy().view(np.uint32)
    ntk, npad = (N + 127) // 128, (N + 127) // 128 * 128
    orc = oracle.default()
    for bh in range(B * H):
        for i in range(N):
            nk = i + 1 if causal else N
            for j0 in range(0, ((nk + 127) // 128) * 128, 32):
                word = int(words[((bh * ntk + j0 // 128) * 4 + (j0 % 128) // 32) * npad + i])
                for b in range(32):
                    j = j0 + b
                    if j >= N:
                        continue
                    want = orc.dropout_factor(bh, i, j, t, seed) > 0
                    assert bool((word >> b) & 1) == want, f"bit (bh {bh}, query {i}, key {j})"
