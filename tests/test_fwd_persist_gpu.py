"""The d = 64 forward on a persistent grid (fwd_persist.cu: CTAs take further work units
with cluster launch control) against the FP64 oracle, and against the one-unit-per-CTA
kernel, which does the same arithmetic per row and must give the same bytes.

ATTN_FWD_PERSIST=1 / =0 forces the kernel attn_fwd and attn_fwd_rect run at d = 64 (the
persistent one needs an even number of query tiles; other shapes keep the one-unit
kernel).  Shapes cover one unit, fewer units than SMs (every request cancels nothing),
several units per SM (the GPT-2-shaped 96 heads x 1024 and more), ragged key ends,
rectangular causal masks, and causal units of different lengths."""
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
    q = torch.randn((B, H, Nq, 64), generator=g)
    k = torch.randn((B, H, Nk, 64), generator=g)
    v = torch.randn((B, H, Nk, 64), generator=g)
    return q.to(t), k.to(t), v.to(t)


def fwd(q, k, v, causal, persist):
    old = os.environ.get("ATTN_FWD_PERSIST")
    os.environ["ATTN_FWD_PERSIST"] = "1" if persist else "0"
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
            del os.environ["ATTN_FWD_PERSIST"]
        else:
            os.environ["ATTN_FWD_PERSIST"] = old


SMALL = [  # B, H, Nq, Nk: checked against the oracle
    (1, 1, 256, 256), (2, 3, 512, 512), (1, 2, 256, 300), (1, 2, 1000, 1000), (1, 1, 256, 1100),
    (2, 2, 2048, 2048), (1, 3, 384, 512),
]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Nq,Nk", SMALL)
def test_persist_forward_matches_oracle_and_one_unit(B, H, Nq, Nk, causal, dtype):
    if causal and Nk < Nq:
        pytest.skip("causal needs Nk >= Nq")
    q, k, v = draw(B, H, Nq, Nk, dtype, seed=Nq * 5 + Nk + causal)
    o2, l2 = fwd(q.cuda(), k.cuda(), v.cuda(), causal, True)
    o1, l1 = fwd(q.cuda(), k.cuda(), v.cuda(), causal, False)
    ro, rl = oracle.attn_fwd(q, k, v, causal, 1 / math.sqrt(64))
    eo, el = o_err(o2, ro), lse_err(l2, rl)
    assert eo <= O_MAX_ABS, f"O max-abs error {eo:.3e}"
    assert el <= LSE_REL, f"LSE relative error {el:.3e}"
    assert torch.equal(o2, o1) and torch.equal(l2, l1), "the persistent kernel differs from the one-unit kernel"


MANY = [  # B, H, N: several units per SM; compared with the one-unit kernel byte for byte
    (8, 12, 1024), (4, 16, 2048), (16, 12, 512), (1, 40, 4096), (3, 100, 256),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N", MANY)
def test_persist_forward_many_units(B, H, N, causal):
    q, k, v = draw(B, H, N, N, "bf16", seed=N + B * H + causal)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o2, l2 = fwd(qd, kd, vd, causal, True)
    o1, l1 = fwd(qd, kd, vd, causal, False)
    assert torch.equal(o2, o1) and torch.equal(l2, l1)
    # and a few heads against the oracle
    for bh in (0, B * H // 2, B * H - 1):
        b, h = divmod(bh, H)
        ro, rl = oracle.attn_fwd(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], causal, 1 / 8)
        assert o_err(o2[b:b + 1, h:h + 1], ro) <= O_MAX_ABS and lse_err(l2[b:b + 1, h:h + 1], rl) <= LSE_REL


def test_persist_forward_stress_inputs():
    """The stress recipe at d = 64 (zero queries, a dominant last key, 20x scaled scores):
    the reference maximum moves on early and late key tiles of units that follow each
    other on one CTA."""
    x = workloads.draw(2, 96, 1024, 64, "bf16", seed=3, stress=True)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    for causal in (False, True):
        o2, l2 = fwd(q, k, v, causal, True)
        o1, l1 = fwd(q, k, v, causal, False)
        assert torch.equal(o2, o1) and torch.equal(l2, l1)


@pytest.mark.parametrize("persist", [False, True], ids=["one_unit", "persistent"])
@pytest.mark.parametrize("B,H,N", [(32, 12, 1024), (8, 12, 2048)])
def test_d64_repeated_calls_complete(B, H, N, persist):
    """Causal d = 64 forwards of many heads, back to back: every call must finish without a
    wait running out (the softmax of one query tile can run a key tile ahead of the
    product issuer, so a hand-off that could complete two phases of one barrier before the
    issuer looks would stall the CTA until the wait limit) and give the same bytes."""
    q, k, v = draw(B, H, N, N, "bf16", seed=N + H)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ref_o, ref_l = fwd(qd, kd, vd, True, persist)
    old = os.environ.get("ATTN_FWD_PERSIST")
    os.environ["ATTN_FWD_PERSIST"] = "1" if persist else "0"
    try:
        o = torch.empty_like(qd)
        lse = torch.empty((B, H, N), device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        for _ in range(40):
            assert attn.attn_fwd(qd, kd, vd, o, lse, B, H, N, 64, qd.dtype, True, 1 / 8, status) == attn.ATTN_OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"device status {int(status.item())}"
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)
    finally:
        if old is None:
            del os.environ["ATTN_FWD_PERSIST"]
        else:
            os.environ["ATTN_FWD_PERSIST"] = old
