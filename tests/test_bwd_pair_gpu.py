"""The d = 128 dK/dV stage on CTA pairs (bwd_pair.cu) against the FP64 oracle, and against
the one-CTA kernel, which does the same arithmetic per key row and must give the same bytes.

ATTN_BWD_CTA_PAIR=1 / =0 forces the kernel the dK/dV stage runs.  Shapes cover one tile,
ragged query and key ends, an odd number of key tiles (the second CTA of the last pair has
no keys), fewer query tiles than the two-stage ring, and enough to cycle it; under the
causal mask the later key tile of a pair also visits its earlier tile's first query tile,
which is wholly masked for it."""
import math
import os

import pytest
import torch

import oracle
import tiled_online_softmax_attention_gb300 as attn
import workloads
from gpu_util import GRAD_REL_L2, Guarded, grad_err, run_fwd

pytestmark = pytest.mark.gpu


def dkdv(q, k, v, o, lse, do, causal, pair):
    old = os.environ.get("ATTN_BWD_CTA_PAIR")
    os.environ["ATTN_BWD_CTA_PAIR"] = "1" if pair else "0"
    try:
        B, H, N, d = q.shape
        scale = 1 / math.sqrt(d)
        nbytes = attn.attn_bwd_deterministic_workspace_bytes(B, H, N, d)
        ws = Guarded((nbytes // 4,), torch.float32)
        dk, dv = (Guarded((B, H, N, d), q.dtype) for _ in range(2))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert attn.attn_bwd_prepare(o, do, lse, ws.t, nbytes, B, H, N, d, q.dtype) == attn.ATTN_OK
        rc = attn.attn_bwd_dkdv(q, k, v, do, ws.t, nbytes, dk.t, dv.t, B, H, N, d, q.dtype, causal, scale, status)
        assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"device status {int(status.item())}"
        assert dk.intact() and dv.intact() and ws.intact(), "the dK/dV stage wrote outside its buffers"
        return dk.t, dv.t
    finally:
        if old is None:
            del os.environ["ATTN_BWD_CTA_PAIR"]
        else:
            os.environ["ATTN_BWD_CTA_PAIR"] = old


CASES = [  # B, H, N
    (1, 1, 128), (1, 2, 256), (2, 3, 512), (1, 2, 300), (1, 2, 640), (1, 1, 1100), (2, 2, 2048), (1, 1, 1),
    (1, 3, 383), (1, 2, 129),
]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N", CASES)
def test_pair_dkdv_matches_oracle_and_one_cta(B, H, N, causal, dtype):
    x = workloads.draw(B, H, N, 128, dtype, seed=6000 + N + causal, with_dout=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    scale = 1 / math.sqrt(128)
    o, lse = run_fwd(q, k, v, causal, scale)
    dk2, dv2 = dkdv(q, k, v, o, lse, do, causal, True)
    dk1, dv1 = dkdv(q, k, v, o, lse, do, causal, False)
    _, rk, rv = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], causal, scale)
    for name, g, r in (("dK", dk2, rk), ("dV", dv2, rv)):
        e = grad_err(g, r)
        assert e <= GRAD_REL_L2, f"{name} relative L2 {e:.3e}"
    assert torch.equal(dk2, dk1) and torch.equal(dv2, dv1), "the pair kernel differs from the one-CTA kernel"


@pytest.mark.parametrize("causal", [False, True])
def test_pair_dkdv_long_rows_and_stress(causal):
    """The stress recipe (a head of zero queries, a dominant key, 20x scaled scores) over
    4096 queries: 32 query tiles cycle the ring many times; compared with the one-CTA kernel."""
    x = workloads.draw(1, 3, 4096, 128, "bf16", seed=17, stress=True, with_dout=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = run_fwd(q, k, v, causal, 1 / math.sqrt(128))
    dk2, dv2 = dkdv(q, k, v, o, lse, do, causal, True)
    dk1, dv1 = dkdv(q, k, v, o, lse, do, causal, False)
    assert torch.equal(dk2, dk1) and torch.equal(dv2, dv1)
