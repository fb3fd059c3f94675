"""Backward parity: dQ, dK, dV from the CUDA path (through the C ABI, from the CUDA
forward's O and logsumexp) against the FP64 oracle's chain rule."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import GRAD_REL_L2, assert_same_grads, f64, grad_err, run_bwd, run_bwd_fused, run_fwd, sample_rows

pytestmark = pytest.mark.gpu


def gpu_grads(x, causal, scale, fused=False):
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = run_fwd(q, k, v, causal, scale)
    if fused:
        return run_bwd_fused(q, k, v, o, lse, do, causal, scale)
    return run_bwd(q, k, v, o, lse, do, causal, scale)


@pytest.mark.parametrize("fused", [False, True], ids=["two_kernels", "fused"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 100, 128, 129, 256, 300, 640])
def test_bwd_small(N, d, causal, dtype, fused):
    x = workloads.draw(1, 2, N, d, dtype, seed=2000 + N + d, with_dout=True)
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv = gpu_grads(x, causal, scale, fused)
    rq, rk, rv = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], causal, scale)
    for name, g, r in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        assert np.all(np.isfinite(f64(g))), name + " non-finite"
        e = grad_err(g, r)
        assert e <= GRAD_REL_L2, f"{name} relative L2 {e:.3e} (N={N} d={d} causal={causal} {dtype})"


def test_bwd_training_step_sampled():
    """The full training-step workload; sampled query rows (dQ) and key rows (dK, dV)."""
    w = workloads.WORKLOADS["c5"]
    x = workloads.inputs("c5")
    dq, dk, dv = gpu_grads(x, True, w.scale)
    dq, dk, dv = f64(dq), f64(dk), f64(dv)
    for g in (dq, dk, dv):
        assert np.all(np.isfinite(g))
    rows = sample_rows(w.N, extra=16, seed=1)
    for (b, h) in [(0, 0), (w.B - 1, w.H - 1)]:
        rq, rk, rv = oracle.attn_bwd(x["q"][b, h], x["k"][b, h], x["v"][b, h], x["dout"][b, h], True, w.scale,
                                     qrows=rows, kcols=rows)
        for name, g, r in (("dQ", dq[b, h, rows], rq), ("dK", dk[b, h, rows], rk), ("dV", dv[b, h, rows], rv)):
            e = grad_err(g, r)
            assert e <= GRAD_REL_L2, f"c5 head ({b},{h}) {name} relative L2 {e:.3e}"


def test_bwd_deterministic():
    """attn_bwd without dropout and attn_bwd_deterministic: the same bytes on every call,
    and the same bytes as each other."""
    x = workloads.draw(1, 2, 400, 128, "bf16", seed=9, with_dout=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    scale = 1 / math.sqrt(128)
    o, lse = run_fwd(q, k, v, True, scale)
    g1 = run_bwd(q, k, v, o, lse, do, True, scale)
    g2 = run_bwd(q, k, v, o, lse, do, True, scale)
    g3 = run_bwd(q, k, v, o, lse, do, True, scale, deterministic=True)
    for a, b, c in zip(g1, g2, g3):
        assert torch.equal(a, b) and torch.equal(a, c)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_fused_matches_deterministic(causal, d):
    """The fused pass computes dV and dK with the deterministic dK/dV kernel's products in
    the same order (only the operand of dK moves from tensor to shared memory), so they are
    the same bytes.  Its dQ sums the same dS K products in another order (and the
    deterministic dQ kernel recomputes S, so a dS may round differently): close, not
    equal.  Two fused calls differ at most by the accumulator's summation order."""
    B, H, N = 2, 3, 1000
    x = workloads.draw(B, H, N, d, "bf16", seed=4100 + d + causal, with_dout=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    scale = 1.0 / math.sqrt(d)
    o, lse = run_fwd(q, k, v, causal, scale)
    g_det = run_bwd(q, k, v, o, lse, do, causal, scale, deterministic=True)
    g1 = run_bwd_fused(q, k, v, o, lse, do, causal, scale)
    g2 = run_bwd_fused(q, k, v, o, lse, do, causal, scale)
    assert torch.equal(g1[1], g_det[1]) and torch.equal(g1[2], g_det[2]), "fused dK/dV differ from deterministic"
    e = grad_err(g1[0], f64(g_det[0]))
    assert e <= 2e-3, f"fused dQ vs deterministic dQ relative L2 {e:.3e}"
    assert_same_grads(g2, g1, "two fused calls:")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [100, 300, 1000])
def test_bwd_one_grid_equals_stages(N, d, causal):
    """attn_bwd_deterministic runs dK/dV and dQ as one grid; the stage entry points launch
    them one by one.  Same kernels' arithmetic, so the same bytes."""
    from gpu_util import Guarded
    import tiled_online_softmax_attention_gb300 as attn

    B, H = 2, 3
    x = workloads.draw(B, H, N, d, "bf16", seed=4000 + N + d, with_dout=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    scale = 1.0 / math.sqrt(d)
    o, lse = run_fwd(q, k, v, causal, scale)
    g = run_bwd(q, k, v, o, lse, do, causal, scale, deterministic=True)
    nbytes = attn.attn_bwd_deterministic_workspace_bytes(B, H, N, d)
    ws = Guarded((nbytes // 4,), torch.float32)
    dq, dk, dv = (Guarded((B, H, N, d), q.dtype) for _ in range(3))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert attn.attn_bwd_prepare(o, do, lse, ws.t, nbytes, B, H, N, d, q.dtype) == attn.ATTN_OK
    assert attn.attn_bwd_dkdv(q, k, v, do, ws.t, nbytes, dk.t, dv.t, B, H, N, d, q.dtype, causal, scale,
                              status) == attn.ATTN_OK
    assert attn.attn_bwd_dq(q, k, v, do, ws.t, nbytes, dq.t, B, H, N, d, q.dtype, causal, scale,
                            status) == attn.ATTN_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and dq.intact() and dk.intact() and dv.intact() and ws.intact()
    for a, b in zip((dq.t, dk.t, dv.t), g):
        assert torch.equal(a, b)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_bwd_on_a_side_stream(d):
    """attn_bwd launched on a non-default stream (inputs produced on the default stream and
    ordered by an event) gives the default stream's bytes."""
    B, H, N = 1, 2, 700
    x = workloads.draw(B, H, N, d, "bf16", seed=4500 + d, with_dout=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    scale = 1.0 / math.sqrt(d)
    o, lse = run_fwd(q, k, v, True, scale)
    g0 = run_bwd(q, k, v, o, lse, do, True, scale)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g1 = run_bwd(q, k, v, o, lse, do, True, scale, stream=s)
    torch.cuda.synchronize()
    for a, b in zip(g0, g1):
        assert torch.equal(a, b)
