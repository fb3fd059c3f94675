"""The extreme cases the kwkr page's section 10 lists for an online-softmax
implementation: an all-zero input, a 32K-token sequence (values > 100 and lengths that
are not tile multiples are covered by the stress workload and the sweeps)."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import GRAD_REL_L2, LSE_REL, O_MAX_ABS, f64, grad_err, o_err, run_bwd, run_fwd, sample_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
def test_all_zero_input(causal):
    """Q = K = V = 0: every score is 0, so O = 0 and LSE_i = ln(visible keys); dO arbitrary
    gives dV_j = sum over the queries that see j of dO_i / n_i and dQ = dK = 0."""
    B, H, N, d = 1, 2, 300, 128
    z = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    do = workloads.draw(B, H, N, d, "bf16", seed=60, with_dout=True)["dout"].cuda()
    o, lse = run_fwd(z, z, z, causal)
    assert torch.count_nonzero(o) == 0
    n = np.arange(1, N + 1) if causal else np.full(N, N)
    assert np.max(np.abs(f64(lse) - np.log(n)) / np.log(np.maximum(n, 2))) <= LSE_REL
    dq, dk, dv = run_bwd(z, z, z, o, lse, do, causal)
    assert torch.count_nonzero(dq) == 0 and torch.count_nonzero(dk) == 0
    dof = do.double().cpu().numpy()
    w = dof / n[None, None, :, None]
    ref = np.cumsum(w[:, :, ::-1], axis=2)[:, :, ::-1] if causal else np.broadcast_to(w.sum(axis=2, keepdims=True), w.shape)
    assert grad_err(dv, ref) <= GRAD_REL_L2


@pytest.mark.parametrize("causal", [False, True])
def test_32k_sequence_sampled(causal):
    """One 32768-token sequence (B=1, H=2, d=128): sampled rows of O, LSE, dQ, dK, dV."""
    B, H, N, d = 1, 2, 32768, 128
    x = workloads.draw(B, H, N, d, "bf16", seed=61, with_dout=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    scale = 1.0 / math.sqrt(d)
    o, lse = run_fwd(q, k, v, causal, scale)
    dq, dk, dv = run_bwd(q, k, v, o, lse, do, causal, scale)
    o, lse, dq, dk, dv = (f64(t) for t in (o, lse, dq, dk, dv))
    rows = sample_rows(N, extra=8, seed=62)
    for h in range(H):
        ro, rl = oracle.attn_fwd(x["q"][0, h], x["k"][0, h], x["v"][0, h], causal, scale, rows=rows)
        assert float(np.max(np.abs(o[0, h, rows] - ro))) <= O_MAX_ABS
        assert float(np.max(np.abs(lse[0, h, rows] - rl) / np.maximum(np.abs(rl), 1))) <= LSE_REL
        rq, rk, rv = oracle.attn_bwd(x["q"][0, h], x["k"][0, h], x["v"][0, h], x["dout"][0, h], causal, scale,
                                     qrows=rows, kcols=rows)
        for name, g, r in (("dQ", dq[0, h, rows], rq), ("dK", dk[0, h, rows], rk), ("dV", dv[0, h, rows], rv)):
            e = grad_err(g, r)
            assert e <= GRAD_REL_L2, f"head {h} {name} relative L2 {e:.3e}"


@pytest.mark.parametrize("d", [64, 128, 256])
def test_largest_element_count(d):
    """The most elements a call takes, B*H*N*d just under 2^31 (65535 to 262143 heads of
    one 128-row tile): every element index of the tensors is exercised.  Forward and
    backward, causal; all outputs finite, and three heads (first, middle, last) against
    the oracle.  Inputs are drawn on the device from a seeded generator."""
    B, N = 1, 128
    H = (1 << 31) // (N * d) - 1
    g = torch.Generator(device="cuda").manual_seed(70 + d)

    def draw():
        return torch.randn((B, H, N, d), device="cuda", generator=g).to(torch.bfloat16)

    q, k, v, do = draw(), draw(), draw(), draw()
    scale = 1.0 / math.sqrt(d)
    o, lse = run_fwd(q, k, v, True, scale)
    dq, dk, dv = run_bwd(q, k, v, o, lse, do, True, scale)
    for t in (o, lse, dq, dk, dv):
        assert bool(torch.isfinite(t).all())
    for h in (0, H // 2, H - 1):
        qh, kh, vh, dh = (t[0, h].cpu() for t in (q, k, v, do))
        ro, rl = oracle.attn_fwd(qh, kh, vh, True, scale)
        assert o_err(o[0, h], ro) <= O_MAX_ABS
        assert float(np.max(np.abs(f64(lse[0, h]) - rl) / np.maximum(np.abs(rl), 1))) <= LSE_REL
        refs = oracle.attn_bwd(qh, kh, vh, dh, True, scale)
        for name, gr, r in zip(("dQ", "dK", "dV"), (dq[0, h], dk[0, h], dv[0, h]), refs):
            e = grad_err(gr, r)
            assert e <= GRAD_REL_L2, f"head {h} {name} relative L2 {e:.3e}"
