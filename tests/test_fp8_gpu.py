"""Parity of the FP8 forward (attn_fwd_fp8: E4M3 inputs with one scale per 128-row
block) with the FP64 oracle, through the C ABI.

The oracle computes the exact attention of the dequantised inputs.  Beyond float32
arithmetic, the kernel makes one approximation: P (with V's block scale folded in) is
rounded to E4M3 for the second product.  The tolerance follows from that rounding:

  * an E4M3 number >= 2^-6 (normal) is within 2^-4 of its value relatively, so those
    terms move O_ic by at most 2^-4 * sum_j P_ij |V_jc| = 2^-4 * A_ic, where A is the
    attention of the same inputs with |V| in place of V (one more oracle call);
  * a term below 2^-6 is off by at most 2^-10 in the kernel's scaling, where the row's
    reference term is 2^6.  Only keys j whose log2-domain weight w_j = log2(e) * S_ij
    + log2 v_scale_j lies more than 12 below the row's largest can be that small; with
    the row's base-2 logsumexp lse2 and largest weight w_max the error they add is at
    most F_ic = 2^-16 * 2^(w_max - lse2) * sum_{those j} |V8_jc|;
  * rounding the output to 16 bits adds at most 2^-8 |O_ic|; float32 scores,
    exponentials and sums add far less (1e-3 * A_ic covers them).

So |O_gpu - O| <= 2^-4 A (1 + 1e-3) + 2^-8 |O| + F + 1e-6 element by element, and,
since the rounding errors of independent terms do not add up coherently, the relative
L2 error over a whole output stays below the rms of a uniform relative error of
half-width 2^-4, 2^-4 / sqrt(3).  The logsumexp comes from unrounded float32 sums and
keeps the 16-bit forward's tolerance.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import LSE_REL, f64, lse_err, run_fwd_fp8, sample_rows

pytestmark = pytest.mark.gpu

LOG2E = 1.0 / math.log(2.0)
REL_L2_MAX = 2.0 ** -4 / math.sqrt(3.0)
P_EXP = 6  # the kernel's P~ scaling: the reference term is 2^6, normals start at 2^-6


def to_dev(x):
    return {k: v.cuda() for k, v in x.items()}


def fp8_reference(x, causal, scale, rows=None):
    """Oracle output and logsumexp, and the element-wise error bound described above."""
    q = oracle.dequant_e4m3(x["q8"], x["q_scale"])
    k = oracle.dequant_e4m3(x["k8"], x["k_scale"])
    v = oracle.dequant_e4m3(x["v8"], x["v_scale"])
    o, lse = oracle.attn_fwd(q, k, v, causal, scale, rows)
    a, _ = oracle.attn_fwd(q, k, np.abs(v), causal, scale, rows)
    B, H, N, d = q.shape
    rr = np.arange(N) if rows is None else np.asarray(rows)
    v8abs = np.abs(oracle.dequant_e4m3(x["v8"], torch.ones_like(x["v_scale"])))
    g = np.log2(x["v_scale"].double().numpy())  # [B, H, nblk]
    blk = np.arange(N) // 128
    F = np.zeros_like(o)
    for b in range(B):
        for h in range(H):
            w = LOG2E * scale * (q[b, h, rr] @ k[b, h].T) + g[b, h, blk][None, :]
            if causal:
                w = np.where(np.arange(N)[None, :] <= rr[:, None], w, -np.inf)
            wmax = w.max(axis=1, keepdims=True)
            small = (w < wmax - (P_EXP + 6)).astype(np.float64)
            lse2 = (lse[b, h] * LOG2E)[:, None]
            F[b, h] = 2.0 ** (-10 - P_EXP) * 2.0 ** (wmax - lse2) * (small @ v8abs[b, h])
    bound = 2.0 ** -4 * a * (1 + 1e-3) + 2.0 ** -8 * np.abs(o) + F + 1e-6
    return o, lse, bound


def check(o_gpu, lse_gpu, ref, rows=None, what=""):
    o_ref, lse_ref, bound = ref
    og = f64(o_gpu)
    lg = f64(lse_gpu)
    if rows is not None:
        og, lg = og[:, :, rows], lg[:, :, rows]
    err = np.abs(og - o_ref)
    worst = float((err / bound).max()) if err.size else 0.0
    assert worst <= 1.0, f"{what}: element error {worst:.3f} x its bound (max abs {err.max():.3e})"
    rel = float(np.linalg.norm(og - o_ref) / max(np.linalg.norm(o_ref), 1e-30))
    assert rel <= REL_L2_MAX, f"{what}: relative L2 {rel:.4f} > {REL_L2_MAX:.4f}"
    le = lse_err(torch.from_numpy(lg), lse_ref)
    assert le <= LSE_REL, f"{what}: lse error {le:.2e}"


@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 255, 256, 300, 513, 1024])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("spread", [0.0, 3.0])
def test_fp8_sweep(N, causal, spread):
    x = workloads.draw_fp8(1, 3, N, 128, seed=100 + N, block_spread=spread)
    scale = 1.0 / math.sqrt(128)
    o, lse = run_fwd_fp8(to_dev(x), causal, scale)
    check(o, lse, fp8_reference(x, causal, scale), what=f"N={N} causal={causal} spread={spread}")


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_fp16_output_and_pow2_scales(causal):
    x = workloads.draw_fp8(2, 2, 700, 128, seed=7, block_spread=2.0, pow2=True)
    o, lse = run_fwd_fp8(to_dev(x), causal, 0.05, out_dtype=torch.float16)
    assert o.dtype == torch.float16
    check(o, lse, fp8_reference(x, causal, 0.05), what="fp16 output, power-of-two scales")


def test_fp8_large_scores():
    """Scores with std ~ 400 (Q and K scales x 20): the reference max moves often, and
    rows are nearly one-hot."""
    x = workloads.draw_fp8(1, 4, 1000, 128, seed=8, block_spread=1.0)
    x["q_scale"] = x["q_scale"] * 20
    x["k_scale"] = x["k_scale"] * 20
    for causal in (False, True):
        o, lse = run_fwd_fp8(to_dev(x), causal, 1 / math.sqrt(128))
        check(o, lse, fp8_reference(x, causal, 1 / math.sqrt(128)), what=f"large scores causal={causal}")


def test_fp8_one_hot_key():
    """One key scores ~1000 above the others in every row (its K block has a huge
    scale): every output row is that key's V row."""
    N = 777
    x = workloads.draw_fp8(1, 2, N, 128, seed=9)
    q8 = x["q8"].clone()
    k8 = x["k8"].clone()
    q8[..., 127] = 0x38                       # 1.0
    q8[..., :127] = 0
    k8[..., 127] = 0
    k8[:, :, N - 1, 127] = 0x7E               # 448 in the last (ragged) block
    x["q8"], x["k8"] = q8, k8
    x["q_scale"] = torch.ones_like(x["q_scale"])
    x["k_scale"] = torch.ones_like(x["k_scale"])
    x["k_scale"][..., -1] = 1000.0 * math.sqrt(128) / 448.0
    o, lse = run_fwd_fp8(to_dev(x), False, 1 / math.sqrt(128))
    ref = fp8_reference(x, False, 1 / math.sqrt(128))
    check(o, lse, ref, what="one-hot key")
    v_last = oracle.dequant_e4m3(x["v8"], x["v_scale"])[:, :, N - 1]
    assert np.abs(f64(o) - v_last[:, :, None, :]).max() <= 2.0 ** -8 * np.abs(v_last).max() + 1e-6


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_long_sequence_sampled(causal):
    """The long-sequence shape (B=1, H=32, N=16384, d=128) in the launch configuration
    the benchmark times, checked on sampled rows."""
    x = workloads.draw_fp8(1, 32, 16384, 128, seed=2)
    scale = 1.0 / math.sqrt(128)
    o, lse = run_fwd_fp8(to_dev(x), causal, scale)
    rows = sample_rows(16384, extra=16, seed=3 + causal)
    check(o, lse, fp8_reference(x, causal, scale, rows), rows=rows, what=f"N=16384 causal={causal}")


def test_fp8_deterministic():
    x = to_dev(workloads.draw_fp8(2, 4, 1500, 128, seed=11, block_spread=1.0))
    o1, l1 = run_fwd_fp8(x, True)
    o2, l2 = run_fwd_fp8(x, True)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
