"""The d = 128 forward on CTA pairs (fwd_pair.cu) against the FP64 oracle, and against the
one-CTA kernel, which does the same arithmetic per row and must give the same bytes.

ATTN_FWD_CTA_PAIR=1 / =0 forces the kernel attn_fwd and attn_fwd_rect run (by default
the pair kernel takes only long rows without the causal mask).  Shapes cover one tile, ragged ends of the query
and the key range, an odd number of query tiles (the second CTA of the last pair has no
rows), fewer key tiles than the pair kernel's three score buffers, rectangular causal
masks, and enough key tiles to cycle the buffers, the K/V ring and the rescale path."""
import math
import os

import pytest
import torch

import oracle
import tiled_online_softmax_attention_gb300 as attn
import workloads
from gpu_util import LSE_REL, O_MAX_ABS, Guarded, lse_err, o_err

pytestmark = pytest.mark.gpu


def draw(B, H, Nq, Nk, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    t = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    q = torch.randn((B, H, Nq, 128), generator=g)
    k = torch.randn((B, H, Nk, 128), generator=g)
    v = torch.randn((B, H, Nk, 128), generator=g)
    return q.to(t), k.to(t), v.to(t)


def fwd(q, k, v, causal, pair):
    old = os.environ.get("ATTN_FWD_CTA_PAIR")
    os.environ["ATTN_FWD_CTA_PAIR"] = "1" if pair else "0"
    try:
        B, H, Nq, d = q.shape
        Nk = k.shape[2]
        o = Guarded((B, H, Nq, d), q.dtype)
        lse = Guarded((B, H, Nq), torch.float32)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = attn.attn_fwd_rect(q, k, v, o.t, lse.t, B, H, Nq, Nk, d, q.dtype, causal, 1 / math.sqrt(d), status)
        assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"device status {int(status.item())}"
        assert o.intact() and lse.intact(), "the forward wrote outside its outputs"
        return o.t, lse.t
    finally:
        if old is None:
            del os.environ["ATTN_FWD_CTA_PAIR"]
        else:
            os.environ["ATTN_FWD_CTA_PAIR"] = old


CASES = [  # B, H, Nq, Nk
    (1, 1, 128, 128), (1, 2, 256, 256), (2, 3, 512, 512), (1, 2, 300, 300), (1, 2, 640, 640),
    (1, 1, 1100, 1100), (2, 2, 2048, 2048), (1, 2, 256, 512), (1, 2, 300, 1000), (1, 1, 130, 1),
    (1, 3, 1024, 1088), (1, 1, 1, 7), (1, 2, 383, 129),
]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Nq,Nk", CASES)
def test_pair_forward_matches_oracle_and_one_cta(B, H, Nq, Nk, causal, dtype):
    if causal and Nk < Nq:
        pytest.skip("causal needs Nk >= Nq")
    q, k, v = draw(B, H, Nq, Nk, dtype, seed=Nq * 7 + Nk + causal)
    o2, l2 = fwd(q.cuda(), k.cuda(), v.cuda(), causal, True)
    o1, l1 = fwd(q.cuda(), k.cuda(), v.cuda(), causal, False)
    ro, rl = oracle.attn_fwd(q, k, v, causal, 1 / math.sqrt(128))
    eo, el = o_err(o2, ro), lse_err(l2, rl)
    assert eo <= O_MAX_ABS, f"O max-abs error {eo:.3e}"
    assert el <= LSE_REL, f"LSE relative error {el:.3e}"
    assert torch.equal(o2, o1) and torch.equal(l2, l1), "the pair kernel differs from the one-CTA kernel"


@pytest.mark.parametrize("causal", [False, True])
def test_pair_forward_stress_inputs(causal):
    """The stress recipe (a head of zero queries, a head whose last key dominates every
    row, heads of 20x scaled scores): the lazily moved reference maximum moves on late and
    on early key tiles, so the O rescale runs between the pair's products."""
    x = workloads.draw(1, 3, 2048, 128, "bf16", seed=5, stress=True)
    q, k, v = x["q"], x["k"], x["v"]
    o2, l2 = fwd(q.cuda(), k.cuda(), v.cuda(), causal, True)
    o1, l1 = fwd(q.cuda(), k.cuda(), v.cuda(), causal, False)
    ro, rl = oracle.attn_fwd(q, k, v, causal, 1 / math.sqrt(128))
    assert o_err(o2, ro) <= O_MAX_ABS and lse_err(l2, rl) <= LSE_REL
    assert torch.equal(o2, o1) and torch.equal(l2, l1)


def test_pair_forward_is_the_default_on_long_rows():
    """Without the override, Nk = 16384 non-causal (128 key tiles) takes the pair kernel and
    Nk = 1024 the one-CTA kernel; both give the same bytes, so the check is the dispatch
    rule through ATTN_FWD_CTA_PAIR's absence leaving results unchanged."""
    old = os.environ.pop("ATTN_FWD_CTA_PAIR", None)
    try:
        q, k, v = draw(1, 1, 256, 16384, "bf16", seed=9)
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        o = torch.empty_like(qd)
        lse = torch.empty((1, 1, 256), device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert attn.attn_fwd_rect(qd, kd, vd, o, lse, 1, 1, 256, 16384, 128, qd.dtype, False, 1 / math.sqrt(128),
                                  status) == attn.ATTN_OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        o1, l1 = fwd(qd, kd, vd, False, False)
        assert torch.equal(o, o1) and torch.equal(lse, l1)
    finally:
        if old is not None:
            os.environ["ATTN_FWD_CTA_PAIR"] = old
