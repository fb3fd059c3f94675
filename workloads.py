"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws random tensors and
applies the stress-case edits, so the oracle and the CUDA library can be fed
identical bytes without sharing any of the method's code.

Recipe (the same for every workload): a CPU ``torch.Generator`` seeded with the
workload's seed draws FP32 ``randn`` tensors of shape [B, H, N, d] in the order
Q, K, V, dO; the stress edits (``c4`` only) are applied in FP32; the tensors are
then cast to the workload's 16-bit type with round-to-nearest-even.

Workloads (sizes from the pages' shapes: GPT-2-small heads, the L=16384, d=128
memory example, a length that is not a multiple of any tile, a training step):

  c1  B=1  H=1  N=256   d=64  bf16  non-causal          forward
  c2  B=8  H=12 N=1024  d=64  bf16  non-causal + causal forward
  c3  B=1  H=32 N=16384 d=128 bf16  non-causal + causal forward
  c4  B=2  H=8  N=4097  d=128 fp16  non-causal          forward, stress edits
  c5  B=2  H=16 N=8192  d=128 bf16  causal              forward + backward

Stress edits for c4 (scores near +-1000, exercising the running-max rescale):
  head 0      Q = 0                      -> every score 0, uniform softmax
  head 1      unscaled Q, K; Q[..., d-1] = 1 and K[N-1, d-1] = 1000*sqrt(d), so
              key N-1 (the lone key of the ragged last tile) scores ~1000 above
              every other key in every row -> near one-hot rows
  heads 2..7  Q and K multiplied by 20   -> scores with std ~400, |s| up to ~1500
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str
    seed: int
    causal: tuple = (False,)
    backward: bool = False
    stress: bool = False
    note: str = ""

    @property
    def BH(self) -> int:
        return self.B * self.H

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


WORKLOADS = {
    "c1": Workload("c1", 1, 1, 256, 64, "bf16", 0, (False,), note="single head, two tiles"),
    "c2": Workload("c2", 8, 12, 1024, 64, "bf16", 1, (False, True), note="GPT-2-small-shaped heads"),
    "c3": Workload("c3", 1, 32, 16384, 128, "bf16", 2, (False, True), note="long-sequence forward"),
    "c4": Workload("c4", 2, 8, 4097, 128, "fp16", 3, (False,), stress=True, note="numerics stress"),
    "c5": Workload("c5", 2, 16, 8192, 128, "bf16", 4, (True,), backward=True, note="training step"),
}


def draw(B, H, N, d, dtype="bf16", seed=0, with_dout=False, stress=False, qk_mult=1.0):
    """Return a dict of CPU tensors q, k, v (and dout) of shape [B,H,N,d] in ``dtype``."""
    g = torch.Generator().manual_seed(int(seed))
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    dout = torch.randn(shape, generator=g, dtype=torch.float32) if with_dout else None
    if qk_mult != 1.0:
        q.mul_(qk_mult)
        k.mul_(qk_mult)
    if stress:
        _stress_edits(q, k)
    t = DTYPES[dtype]
    out = {"q": q.to(t), "k": k.to(t), "v": v.to(t)}
    if dout is not None:
        out["dout"] = dout.to(t)
    return out


def _stress_edits(q, k):
    B, H, N, d = q.shape
    if H < 3:
        raise ValueError("the stress edits need at least 3 heads")
    q[:, 2:].mul_(20.0)
    k[:, 2:].mul_(20.0)
    q[:, 0].zero_()
    q[:, 1, :, d - 1] = 1.0
    k[:, 1, N - 1, d - 1] = 1000.0 * math.sqrt(d)


E4M3_MAX = 448.0  # largest finite E4M3 value


def quantize_e4m3(x, block_rows: int = 128, pow2: bool = False):
    """Block-scaled E4M3 encoding of x [..., N, d] (float32).

    Each block of ``block_rows`` consecutive rows of one head gets one float32 scale,
    absmax / 448 (rounded up to a power of two when ``pow2``; 1 for an all-zero block),
    and the codes are x / scale rounded to nearest even E4M3.  Returns (codes as uint8
    [..., N, d], scales float32 [..., ceil(N / block_rows)]).
    """
    *lead, N, d = x.shape
    nblk = -(-N // block_rows)
    pad = nblk * block_rows - N
    xp = torch.nn.functional.pad(x.float(), (0, 0, 0, pad)).reshape(*lead, nblk, block_rows, d)
    amax = xp.abs().amax(dim=(-2, -1))
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    if pow2:
        scale = torch.exp2(torch.ceil(torch.log2(scale)))
    codes = (xp / scale[..., None, None]).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    codes = codes.reshape(*lead, nblk * block_rows, d)[..., :N, :].contiguous().view(torch.uint8)
    return codes, scale.to(torch.float32).contiguous()


def draw_fp8(B, H, N, d, seed=0, block_spread=0.0, pow2=False, block_rows=128):
    """Block-scaled E4M3 inputs: FP32 randn Q, K, V (drawn as in ``draw``); with
    ``block_spread`` > 0 every block of ``block_rows`` rows of every head and tensor is
    multiplied by 2^u, u uniform in [-block_spread, block_spread] (drawn after V, in the
    order Q, K, V), so that block scales differ; then each tensor is quantised with
    ``quantize_e4m3``.  Returns a dict of CPU tensors q8, k8, v8 (uint8 [B,H,N,d]) and
    q_scale, k_scale, v_scale (float32 [B,H,ceil(N/block_rows)])."""
    g = torch.Generator().manual_seed(int(seed))
    shape = (B, H, N, d)
    xs = [torch.randn(shape, generator=g, dtype=torch.float32) for _ in range(3)]
    nblk = -(-N // block_rows)
    if block_spread > 0:
        for x in xs:
            u = (torch.rand((B, H, nblk), generator=g, dtype=torch.float32) * 2 - 1) * block_spread
            f = torch.exp2(u).repeat_interleave(block_rows, dim=-1)[..., :N]
            x.mul_(f[..., None])
    out = {}
    for name, x in zip(("q", "k", "v"), xs):
        codes, sc = quantize_e4m3(x, block_rows, pow2)
        out[name + "8"] = codes
        out[name + "_scale"] = sc
    return out


def inputs(name: str):
    """Inputs of a named workload (CPU tensors, 16-bit)."""
    w = WORKLOADS[name]
    return draw(w.B, w.H, w.N, w.d, w.dtype, w.seed, with_dout=w.backward, stress=w.stress)


def fwd_flops(B, H, N, d, causal) -> float:
    """Algorithmic forward FLOPs: two N x N x d contractions, 4*B*H*N^2*d, halved when causal."""
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


def bwd_flops(B, H, N, d, causal) -> float:
    """Algorithmic backward FLOPs: five N x N x d contractions (the recompute of S included),
    10*B*H*N^2*d, halved when causal."""
    f = 10.0 * B * H * N * N * d
    return f / 2 if causal else f
