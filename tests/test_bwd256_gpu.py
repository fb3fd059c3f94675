"""Backward parity at head dimension 256 (three kernels, operands streamed in 128-column
halves): dQ, dK, dV through the C ABI against the FP64 oracle's chain rule, square and
rectangular, both masks, ragged tails; the stage entry points and attn_bwd_noalloc give
attn_bwd's bytes."""
import math

import numpy as np
import pytest
import torch

import oracle
import tiled_online_softmax_attention_gb300 as attn
import workloads
from gpu_util import GRAD_REL_L2, Guarded, f64, grad_err, run_bwd, run_fwd, sample_rows
from test_rect_gpu import draw_rect, run_bwd_rect, run_fwd_rect

pytestmark = pytest.mark.gpu

D = 256


def check(grads, refs, what):
    for name, g, r in zip(("dQ", "dK", "dV"), grads, refs):
        g = f64(g) if hasattr(g, "detach") else g
        assert np.all(np.isfinite(g)), f"{name} non-finite ({what})"
        e = grad_err(g, r)
        assert e <= GRAD_REL_L2, f"{name} relative L2 {e:.3e} ({what})"


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 100, 128, 129, 256, 300, 640])
def test_bwd256_small(N, causal, dtype):
    x = workloads.draw(1, 2, N, D, dtype, seed=3000 + N, with_dout=True)
    scale = 1.0 / math.sqrt(D)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = run_fwd(q, k, v, causal, scale)
    grads = run_bwd(q, k, v, o, lse, do, causal, scale)
    refs = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], causal, scale)
    check(grads, refs, f"N={N} causal={causal} {dtype}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(1, 300), (100, 300), (128, 129), (129, 128), (200, 513), (513, 700)])
def test_bwd256_rect(Nq, Nk, causal):
    if causal and Nk < Nq:
        pytest.skip("causal needs Nk >= Nq")
    x = draw_rect(1, 2, Nq, Nk, D, "bf16", seed=Nq * 13 + Nk)
    scale = 1.0 / math.sqrt(D)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = run_fwd_rect(q, k, v, causal, scale)
    grads = run_bwd_rect(q, k, v, o, lse, do, causal, scale)
    refs = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], causal, scale)
    check(grads, refs, f"{Nq}x{Nk} causal={causal}")


def test_bwd256_several_heads_scale():
    """B=2, H=3 (head groups of two with a remainder), a non-default scale."""
    x = workloads.draw(2, 3, 400, D, "bf16", seed=31, with_dout=True)
    scale = 0.05
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = run_fwd(q, k, v, True, scale)
    dq, dk, dv = (f64(g) for g in run_bwd(q, k, v, o, lse, do, True, scale))
    for b in range(2):
        for h in range(3):
            refs = oracle.attn_bwd(x["q"][b, h], x["k"][b, h], x["v"][b, h], x["dout"][b, h], True, scale)
            check((dq[b, h], dk[b, h], dv[b, h]), refs, f"head ({b},{h})")


@pytest.mark.parametrize("causal", [False, True])
def test_bwd256_long_sampled(causal):
    """B=1, H=4, N=4096: sampled query rows (dQ) and key rows (dK, dV) of two heads."""
    B, H, N = 1, 4, 4096
    x = workloads.draw(B, H, N, D, "bf16", seed=41, with_dout=True)
    scale = 1.0 / math.sqrt(D)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = run_fwd(q, k, v, causal, scale)
    dq, dk, dv = (f64(g) for g in run_bwd(q, k, v, o, lse, do, causal, scale))
    rows = sample_rows(N, extra=12, seed=3)
    for h in (0, 3):
        refs = oracle.attn_bwd(x["q"][0, h], x["k"][0, h], x["v"][0, h], x["dout"][0, h], causal, scale,
                               qrows=rows, kcols=rows)
        check((dq[0, h, rows], dk[0, h, rows], dv[0, h, rows]), refs, f"head {h}")


def test_bwd256_deterministic_and_stages():
    """Two calls give the same bytes; prepare + dkdv + dq and attn_bwd_noalloc give
    attn_bwd's bytes."""
    B, H, N = 1, 2, 333
    x = workloads.draw(B, H, N, D, "bf16", seed=17, with_dout=True)
    scale = 1.0 / math.sqrt(D)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = run_fwd(q, k, v, True, scale)
    g1 = run_bwd(q, k, v, o, lse, do, True, scale)
    g2 = run_bwd(q, k, v, o, lse, do, True, scale)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)

    nbytes = attn.attn_bwd_workspace_bytes(B, H, N, D)
    ws = Guarded((nbytes // 4,), torch.float32)
    dq, dk, dv = (Guarded((B, H, N, D), q.dtype) for _ in range(3))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert attn.attn_bwd_prepare(o, do, lse, ws.t, nbytes, B, H, N, D, q.dtype) == attn.ATTN_OK
    assert attn.attn_bwd_dkdv(q, k, v, do, ws.t, nbytes, dk.t, dv.t, B, H, N, D, q.dtype, 1, scale,
                              status) == attn.ATTN_OK
    assert attn.attn_bwd_dq(q, k, v, do, ws.t, nbytes, dq.t, B, H, N, D, q.dtype, 1, scale, status) == attn.ATTN_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and dq.intact() and dk.intact() and dv.intact() and ws.intact()
    for a, b in zip((dq.t, dk.t, dv.t), g1):
        assert torch.equal(a, b)

    na = [torch.empty_like(q) for _ in range(3)]
    assert attn.attn_bwd_noalloc(q, k, v, o, do, lse, na[0], na[1], na[2], B, H, N, D, q.dtype, 1, scale,
                                 status) == attn.ATTN_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for a, b in zip(na, g1):
        assert torch.equal(a, b)


def test_bwd256_autograd():
    """The torch.autograd wrapper at d = 256 gives the oracle's gradients."""
    x = workloads.draw(1, 2, 300, D, "bf16", seed=61, with_dout=True)
    q, k, v = (x[n].cuda().requires_grad_() for n in ("q", "k", "v"))
    o = attn.attention(q, k, v, causal=True)
    (o.float() * x["dout"].cuda().float()).sum().backward()
    refs = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], True, 1 / math.sqrt(D))
    check((q.grad, k.grad, v.grad), refs, "autograd")


def test_bwd256_dropout_zero_is_plain():
    """attn_bwd_dropout with p_drop = 0 gives attn_bwd's bytes at d = 256."""
    x = workloads.draw(1, 2, 300, D, "bf16", seed=1, with_dout=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = run_fwd(q, k, v, True)
    nbytes = attn.attn_bwd_workspace_bytes(1, 2, 300, D)
    ws = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
    g = [torch.empty_like(q) for _ in range(3)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = attn.attn_bwd_dropout(q, k, v, o, do, lse, g[0], g[1], g[2], ws, nbytes, 1, 2, 300, D, q.dtype, 1,
                               1 / 16, 0.0, 5, status)
    assert rc == attn.ATTN_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for a, b in zip(g, run_bwd(q, k, v, o, lse, do, True, 1 / 16)):
        assert torch.equal(a, b)
