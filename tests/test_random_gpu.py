"""Randomised parity: seeded random shapes across the entry points (square, rectangular,
split-KV, d in {64, 128, 256}, both masks, bf16/fp16), forward and backward, against the
FP64 oracle.  The fixed seed makes every run the same set of cases; the sizes keep the
oracle to a fraction of a second per case."""
import math
import random

import numpy as np
import pytest
import torch

import oracle
import tiled_online_softmax_attention_gb300 as attn
from gpu_util import GRAD_REL_L2, LSE_REL, O_MAX_ABS, Guarded, grad_err, lse_err, o_err

pytestmark = pytest.mark.gpu


def cases(n, seed=2024):
    rnd = random.Random(seed)
    out = []
    for i in range(n):
        d = rnd.choice([64, 128, 256])
        causal = rnd.random() < 0.5
        nq = rnd.choice([1, 2, 63, 127, 128, 129, 200, 255, 256, 257, 384, 511, 640])
        nk = nq if rnd.random() < 0.5 else rnd.choice([nq, nq + 1, nq + 127, nq + 300, 2 * nq + 5])
        if not causal and rnd.random() < 0.25:
            nk = max(1, nq // 3)  # fewer keys than queries (non-causal only)
        split = rnd.choice([0, 0, 2, 3]) if d != 256 else 0
        dt = rnd.choice(["bf16", "fp16"])
        B, H = rnd.choice([(1, 1), (1, 3), (2, 2)])
        out.append((i, B, H, nq, nk, d, causal, split, dt))
    return out


@pytest.mark.parametrize("i,B,H,Nq,Nk,d,causal,split,dt", cases(200))
def test_random_case(i, B, H, Nq, Nk, d, causal, split, dt):
    g = torch.Generator().manual_seed(9000 + i)
    t = {"bf16": torch.bfloat16, "fp16": torch.float16}[dt]
    q = torch.randn((B, H, Nq, d), generator=g).to(t)
    k = torch.randn((B, H, Nk, d), generator=g).to(t)
    v = torch.randn((B, H, Nk, d), generator=g).to(t)
    do = torch.randn((B, H, Nq, d), generator=g).to(t)
    scale = 1.0 / math.sqrt(d)
    qc, kc, vc, dc = (x.cuda() for x in (q, k, v, do))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = Guarded((B, H, Nq, d), t)
    lse = Guarded((B, H, Nq), torch.float32)
    if split:
        nb = attn.attn_fwd_splitkv_workspace_bytes(B, H, Nq, d, split)
        ws = Guarded((nb // 4,), torch.float32)
        rc = attn.attn_fwd_splitkv_rect(qc, kc, vc, o.t, lse.t, ws.t, nb, B, H, Nq, Nk, d, t, causal, scale, split,
                                        status)
    else:
        ws = None
        rc = attn.attn_fwd_rect(qc, kc, vc, o.t, lse.t, B, H, Nq, Nk, d, t, causal, scale, status)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and o.intact() and lse.intact() and (ws is None or ws.intact())
    ro, rl = oracle.attn_fwd(q, k, v, causal, scale)
    assert o_err(o.t, ro) <= O_MAX_ABS, f"O error {o_err(o.t, ro):.3e}"
    assert lse_err(lse.t, rl) <= LSE_REL

    dq = Guarded((B, H, Nq, d), t)
    dk, dv = Guarded((B, H, Nk, d), t), Guarded((B, H, Nk, d), t)
    nb = attn.attn_bwd_workspace_bytes(B, H, Nq, d)
    wsb = Guarded((nb // 4,), torch.float32)
    rc = attn.attn_bwd_rect(qc, kc, vc, o.t, dc, lse.t, dq.t, dk.t, dv.t, wsb.t, nb, B, H, Nq, Nk, d, t, causal,
                            scale, status)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and dq.intact() and dk.intact() and dv.intact() and wsb.intact()
    refs = oracle.attn_bwd(q, k, v, do, causal, scale)
    for name, gr, r in zip(("dQ", "dK", "dV"), (dq.t, dk.t, dv.t), refs):
        e = grad_err(gr, r)
        assert e <= GRAD_REL_L2, f"{name} relative L2 {e:.3e}"
