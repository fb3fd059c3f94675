"""The torch.autograd wrapper (`attention`) against the FP64 oracle: a loss through the
library's forward and backward gives the oracle's output and gradients."""
import math

import numpy as np
import pytest
import torch

import oracle
import tiled_online_softmax_attention_gb300 as attn
import workloads
from gpu_util import GRAD_REL_L2, O_MAX_ABS, f64, grad_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nk", [300, 700])
def test_autograd_matches_oracle(causal, Nk):
    N, d = 300, 64
    x = workloads.draw(1, 2, N, d, "bf16", seed=50, with_dout=True)
    g = torch.Generator().manual_seed(51)
    k = torch.randn((1, 2, Nk, d), generator=g).to(torch.bfloat16)
    v = torch.randn((1, 2, Nk, d), generator=g).to(torch.bfloat16)
    q = x["q"].cuda().requires_grad_()
    kc, vc = k.cuda().requires_grad_(), v.cuda().requires_grad_()
    o = attn.attention(q, kc, vc, causal=causal)
    (o.float() * x["dout"].cuda().float()).sum().backward()
    ro, _ = oracle.attn_fwd(x["q"], k, v, causal, 1 / math.sqrt(d))
    assert float(np.max(np.abs(f64(o) - ro))) <= O_MAX_ABS
    rq, rk, rv = oracle.attn_bwd(x["q"], k, v, x["dout"], causal, 1 / math.sqrt(d))
    for g_, r in ((q.grad, rq), (kc.grad, rk), (vc.grad, rv)):
        assert grad_err(g_, r) <= GRAD_REL_L2


@pytest.mark.parametrize("d", [128, 256])
def test_autograd_dropout_matches_oracle(d):
    N = 400
    x = workloads.draw(1, 2, N, d, "bf16", seed=52, with_dout=True)
    q, k, v = (x[n].cuda().requires_grad_() for n in ("q", "k", "v"))
    o = attn.attention(q, k, v, causal=True, dropout_p=0.2, seed=99)
    (o.float() * x["dout"].cuda().float()).sum().backward()
    t = round(256 * 0.2)
    ro, _ = oracle.attn_fwd_dropout(x["q"], x["k"], x["v"], True, 1 / math.sqrt(d), t, 99)
    assert float(np.max(np.abs(f64(o) - ro))) <= O_MAX_ABS * 256 / (256 - t)
    r = oracle.attn_bwd_dropout(x["q"], x["k"], x["v"], x["dout"], True, 1 / math.sqrt(d), t, 99)
    for g_, rr in zip((q.grad, k.grad, v.grad), r):
        assert grad_err(g_, rr) <= GRAD_REL_L2
