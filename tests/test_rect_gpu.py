"""Parity of the rectangular entry points (Nq queries against Nk keys; causal aligned to
the last key) with the FP64 oracle, through the C ABI, forward and backward."""
import math

import numpy as np
import pytest
import torch

import oracle
import tiled_online_softmax_attention_gb300 as attn
from gpu_util import GRAD_REL_L2, LSE_REL, O_MAX_ABS, Guarded, f64, grad_err, lse_err, o_err, sample_rows

pytestmark = pytest.mark.gpu


def draw_rect(B, H, Nq, Nk, d, dtype, seed):
    """FP32 randn q, dout [B,H,Nq,d] and k, v [B,H,Nk,d] (drawn q, k, v, dout), cast to dtype."""
    g = torch.Generator().manual_seed(seed)
    t = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    q = torch.randn((B, H, Nq, d), generator=g)
    k = torch.randn((B, H, Nk, d), generator=g)
    v = torch.randn((B, H, Nk, d), generator=g)
    do = torch.randn((B, H, Nq, d), generator=g)
    return {"q": q.to(t), "k": k.to(t), "v": v.to(t), "dout": do.to(t)}


def run_fwd_rect(q, k, v, causal, scale):
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    o = Guarded((B, H, Nq, d), q.dtype)
    lse = Guarded((B, H, Nq), torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = attn.attn_fwd_rect(q, k, v, o.t, lse.t, B, H, Nq, Nk, d, q.dtype, causal, scale, status)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and o.intact() and lse.intact()
    return o.t, lse.t


def run_bwd_rect(q, k, v, o, lse, do, causal, scale):
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    dq = Guarded((B, H, Nq, d), q.dtype)
    dk, dv = Guarded((B, H, Nk, d), q.dtype), Guarded((B, H, Nk, d), q.dtype)
    nbytes = attn.attn_bwd_workspace_bytes(B, H, Nq, d)
    ws = Guarded((nbytes // 4,), torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = attn.attn_bwd_rect(q, k, v, o, do, lse, dq.t, dk.t, dv.t, ws.t, nbytes, B, H, Nq, Nk, d, q.dtype, causal,
                            scale, status)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and dq.intact() and dk.intact() and dv.intact() and ws.intact()
    return dq.t, dk.t, dv.t


SHAPES = [(1, 1), (1, 300), (100, 300), (128, 129), (129, 128), (200, 513), (300, 300), (513, 700), (64, 1100)]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", SHAPES)
def test_rect_fwd(Nq, Nk, causal, d):
    if causal and Nk < Nq:
        pytest.skip("causal needs Nk >= Nq")
    x = draw_rect(1, 2, Nq, Nk, d, "bf16", seed=Nq * 7 + Nk + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_fwd_rect(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal, scale)
    ro, rl = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, scale)
    assert o_err(o, ro) <= O_MAX_ABS, f"O error {o_err(o, ro):.3e}"
    assert lse_err(lse, rl) <= LSE_REL


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", SHAPES)
def test_rect_bwd(Nq, Nk, causal, d, dtype):
    if causal and Nk < Nq:
        pytest.skip("causal needs Nk >= Nq")
    x = draw_rect(1, 2, Nq, Nk, d, dtype, seed=Nq * 11 + Nk + d)
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = run_fwd_rect(q, k, v, causal, scale)
    dq, dk, dv = run_bwd_rect(q, k, v, o, lse, do, causal, scale)
    rq, rk, rv = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], causal, scale)
    for name, g, r in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        e = grad_err(g, r)
        assert e <= GRAD_REL_L2, f"{name} relative L2 {e:.3e} ({Nq}x{Nk} d={d} causal={causal} {dtype})"


@pytest.mark.parametrize("causal", [False, True])
def test_rect_long_prefix_sampled(causal):
    """2048 new queries after 6144 earlier positions (Nk = 8192), B=1, H=8, d=128: sampled
    query rows (O, LSE, dQ) and key rows (dK, dV) of three heads."""
    B, H, Nq, Nk, d = 1, 8, 2048, 8192, 128
    x = draw_rect(B, H, Nq, Nk, d, "bf16", seed=77)
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = run_fwd_rect(q, k, v, causal, scale)
    dq, dk, dv = run_bwd_rect(q, k, v, o, lse, do, causal, scale)
    qrows, krows = sample_rows(Nq, extra=8, seed=5), sample_rows(Nk, extra=8, seed=6)
    for h in (0, 3, 7):
        ro, rl = oracle.attn_fwd(x["q"][0, h], x["k"][0, h], x["v"][0, h], causal, scale, rows=qrows)
        assert o_err(o[0, h], ro, qrows) <= O_MAX_ABS
        assert float(np.max(np.abs(f64(lse[0, h])[qrows] - rl) / np.maximum(np.abs(rl), 1))) <= LSE_REL
        rq, rk, rv = oracle.attn_bwd(x["q"][0, h], x["k"][0, h], x["v"][0, h], x["dout"][0, h], causal, scale,
                                     qrows=qrows, kcols=krows)
        for name, g, r in (("dQ", f64(dq[0, h])[qrows], rq), ("dK", f64(dk[0, h])[krows], rk),
                           ("dV", f64(dv[0, h])[krows], rv)):
            e = grad_err(g, r)
            assert e <= GRAD_REL_L2, f"head {h} {name} relative L2 {e:.3e}"


def test_rect_square_matches_attn_fwd():
    """Nq = Nk through the rectangular entry points gives attn_fwd / attn_bwd's bytes."""
    x = draw_rect(1, 3, 700, 700, 128, "bf16", seed=3)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    o1, l1 = run_fwd_rect(q, k, v, True, 0.1)
    o2, l2 = attn.forward(q, k, v, True, 0.1)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    g1 = run_bwd_rect(q, k, v, o1, l1, do, True, 0.1)
    g2 = attn.backward(q, k, v, o2, l2, do, True, 0.1)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
