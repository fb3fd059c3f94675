"""attn_bwd_noalloc, the backward entry point that allocates nothing.

Some callers cannot allocate device memory (a plugin whose host framework owns
all device memory, an engine with a budget fixed at start-up, an FFI caller with
no CUDA runtime of its own); this entry point takes its workspace from a fixed
array inside the library and runs the kernels of attn_bwd_deterministic.  Its
gradients must be the bytes attn_bwd_deterministic (the entry point that takes a
caller-provided workspace) gives, on two calls in a row (the second call reuses
the array the first one left behind), and must match the FP64 oracle.  The file
is named so that pytest collects it last.
"""
import math

import pytest
import torch

import oracle
import tiled_online_softmax_attention_gb300 as attn
import workloads
from gpu_util import GRAD_REL_L2, Guarded, grad_err, run_bwd, run_fwd

pytestmark = pytest.mark.gpu


def noalloc_grads(q, k, v, o, lse, do, causal, scale):
    B, H, N, d = q.shape
    outs = [Guarded((B, H, N, d), q.dtype) for _ in range(3)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = attn.attn_bwd_noalloc(q, k, v, o, do, lse, outs[0].t, outs[1].t, outs[2].t, B, H, N, d, q.dtype, causal,
                               scale, status)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert all(g.intact() for g in outs), "attn_bwd_noalloc wrote outside its outputs"
    return [g.t for g in outs]


@pytest.mark.parametrize("B,H,N,d,dtype,causal,seed",
                         [(1, 3, 700, 128, "bf16", True, 41), (2, 2, 300, 64, "fp16", False, 42)])
def test_noalloc_matches_deterministic_on_two_calls_in_a_row(B, H, N, d, dtype, causal, seed):
    x = workloads.draw(B, H, N, d, dtype, seed=seed, with_dout=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    scale = 1.0 / math.sqrt(d)
    o, lse = run_fwd(q, k, v, causal, scale)
    ref = run_bwd(q, k, v, o, lse, do, causal, scale, deterministic=True)
    for call in range(2):
        got = noalloc_grads(q, k, v, o, lse, do, causal, scale)
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert torch.equal(g, r), f"call {call + 1}: attn_bwd_noalloc {name} differs from attn_bwd_deterministic"
    rq, rk, rv = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], causal, scale)
    for name, g, r in zip(("dQ", "dK", "dV"), got, (rq, rk, rv)):
        e = grad_err(g, r)
        assert e <= GRAD_REL_L2, f"attn_bwd_noalloc {name} vs the oracle: relative L2 {e:.3e}"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # 129 heads of N = 8192 need 8 * 129 * 8192 bytes, just over the 8 MiB array
    B, H, N, d = 1, 129, 8192, 64
    assert attn.attn_bwd_deterministic_workspace_bytes(B, H, N, d) > 8 * 1024 * 1024
    t = torch.empty(16, device="cuda", dtype=torch.bfloat16)
    p = [t] * 9
    rc = attn.attn_bwd_noalloc(*p, B, H, N, d, torch.bfloat16, True, 0.125)
    assert rc == attn.ATTN_ERR_INVALID_ARG
