"""Whole-tensor parity on the two large workloads: every head and every row of the
long-sequence forward (B=1, H=32, N=16384, d=128, both masks) and of the training step
(B=2, H=16, N=8192, d=128, causal: the forward, and dQ, dK, dV of attn_bwd and of the
fused pass, with the relative L2 taken over each whole gradient tensor).  The launches
are exactly the full-size calls the benchmark times; the FP64 oracle evaluates every
output (tens of seconds to a few minutes of host time).  The errors are printed (run
with -s to see them)."""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import GRAD_REL_L2, LSE_REL, O_MAX_ABS, f64, lse_err, o_err, rel_l2, run_bwd, run_bwd_fused, run_fwd

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
def test_long_forward_every_head(causal):
    w = workloads.WORKLOADS["c3"]
    x = workloads.inputs("c3")
    o, lse = run_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal, w.scale)
    assert np.all(np.isfinite(f64(o))) and np.all(np.isfinite(f64(lse)))
    o_ref, lse_ref = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, w.scale)
    eo, el = o_err(o, o_ref), lse_err(lse, lse_ref)
    print(f"\nc3 causal={causal} all {w.B * w.H} heads x {w.N} rows: O max-abs {eo:.3e}, LSE rel {el:.3e}")
    assert eo <= O_MAX_ABS, f"O max-abs error {eo:.3e}"
    assert el <= LSE_REL, f"LSE relative error {el:.3e}"


def test_training_step_every_head():
    w = workloads.WORKLOADS["c5"]
    x = workloads.inputs("c5")
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = run_fwd(q, k, v, True, w.scale)
    grads = {"attn_bwd": run_bwd(q, k, v, o, lse, do, True, w.scale),
             "fused": run_bwd_fused(q, k, v, o, lse, do, True, w.scale)}
    o_ref, lse_ref = oracle.attn_fwd(x["q"], x["k"], x["v"], True, w.scale)
    eo, el = o_err(o, o_ref), lse_err(lse, lse_ref)
    rq, rk, rv = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], True, w.scale)
    print(f"\nc5 all {w.B * w.H} heads x {w.N} rows: O max-abs {eo:.3e}, LSE rel {el:.3e}")
    assert eo <= O_MAX_ABS, f"O max-abs error {eo:.3e}"
    assert el <= LSE_REL, f"LSE relative error {el:.3e}"
    for path, (dq, dk, dv) in grads.items():
        errs = {name: rel_l2(g, r) for name, g, r in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv))}
        print(f"c5 backward ({path}): " + ", ".join(f"{n} rel-L2 {e:.3e}" for n, e in errs.items()))
        for g in (dq, dk, dv):
            assert np.all(np.isfinite(f64(g)))
        for n, e in errs.items():
            assert e <= GRAD_REL_L2, f"{path} {n} relative L2 over the whole tensor {e:.3e}"
