"""Helpers for the GPU parity tests: guarded output buffers, calls through the
C ABI with a device status word, and the error measures the tolerances use."""
from __future__ import annotations

import math

import numpy as np
import torch

import tiled_online_softmax_attention_gb300 as attn

PAD = 4096                  # guard elements on each side of every output buffer
SENTINEL16 = 0x7E5A         # a NaN pattern in both bf16 and fp16
SENTINEL32 = 0x7FC5A5A5     # an fp32 NaN pattern

# Tolerances (GPU result upcast to float64 against the float64 oracle).
O_MAX_ABS = 1e-2
LSE_REL = 1e-3              # |d lse| / max(|lse_ref|, 1)
GRAD_REL_L2 = 2e-2


class Guarded:
    """An output tensor with sentinel-filled guard zones before and after it."""

    def __init__(self, shape, dtype, device="cuda"):
        n = int(np.prod(shape))
        self.n = n
        self.buf = torch.empty(n + 2 * PAD, dtype=dtype, device=device)
        self.raw = self.buf.view(torch.int16 if dtype.itemsize == 2 else torch.int32)
        s = SENTINEL16 if dtype.itemsize == 2 else SENTINEL32
        if dtype.itemsize == 4:
            s = s - (1 << 32) if s >= (1 << 31) else s
        self.sentinel = s
        self.raw.fill_(s)
        self.t = self.buf[PAD:PAD + n].view(shape)

    def intact(self) -> bool:
        head = self.raw[:PAD]
        tail = self.raw[PAD + self.n:]
        return bool((head == self.sentinel).all().item() and (tail == self.sentinel).all().item())


def run_fwd(q, k, v, causal, scale=None, stream=None):
    """attn_fwd through the C ABI with guarded outputs; returns (o, lse) on the device."""
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = Guarded((B, H, N, d), q.dtype)
    lse = Guarded((B, H, N), torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = attn.attn_fwd(q, k, v, o.t, lse.t, B, H, N, d, q.dtype, causal, scale, status, stream)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    assert o.intact() and lse.intact(), "the forward wrote outside its outputs"
    return o.t, lse.t


def run_fwd_fp8(x, causal, scale=None, out_dtype=torch.bfloat16, stream=None):
    """attn_fwd_fp8 through the C ABI with guarded outputs.  ``x`` holds device tensors
    q8, k8, v8 (uint8 [B,H,N,d]) and q_scale, k_scale, v_scale; returns (o, lse)."""
    B, H, N, d = x["q8"].shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = Guarded((B, H, N, d), out_dtype)
    lse = Guarded((B, H, N), torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = attn.attn_fwd_fp8(x["q8"], x["k8"], x["v8"], x["q_scale"], x["k_scale"], x["v_scale"], o.t, lse.t,
                           B, H, N, d, out_dtype, causal, scale, status, stream)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    assert o.intact() and lse.intact(), "the FP8 forward wrote outside its outputs"
    return o.t, lse.t


def run_bwd(q, k, v, o, lse, dout, causal, scale=None, stream=None, deterministic=False):
    """attn_bwd (or attn_bwd_deterministic) through the C ABI with guarded outputs; returns
    (dq, dk, dv)."""
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    outs = [Guarded((B, H, N, d), q.dtype) for _ in range(3)]
    size = attn.attn_bwd_deterministic_workspace_bytes if deterministic else attn.attn_bwd_workspace_bytes
    call = attn.attn_bwd_deterministic if deterministic else attn.attn_bwd
    nbytes = size(B, H, N, d)
    ws = Guarded((nbytes // 4,), torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = call(q, k, v, o, dout, lse, outs[0].t, outs[1].t, outs[2].t, ws.t, nbytes, B, H, N, d,
              q.dtype, causal, scale, status, stream)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    assert all(g.intact() for g in outs) and ws.intact(), "the backward wrote outside its buffers"
    return tuple(g.t for g in outs)


def run_bwd_fused(q, k, v, o, lse, dout, causal, scale=None, stream=None):
    """The fused backward through its stage entry points (attn_bwd_prepare, attn_bwd_dkdvdq,
    attn_bwd_dq_finish) with guarded outputs; returns (dq, dk, dv)."""
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    outs = [Guarded((B, H, N, d), q.dtype) for _ in range(3)]
    nbytes = attn.attn_bwd_workspace_bytes(B, H, N, d)
    ws = Guarded((nbytes // 4,), torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = attn.attn_bwd_prepare(o, dout, lse, ws.t, nbytes, B, H, N, d, q.dtype, stream)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    rc = attn.attn_bwd_dkdvdq(q, k, v, dout, ws.t, nbytes, outs[1].t, outs[2].t, B, H, N, d, q.dtype, causal, scale,
                              status, stream)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    rc = attn.attn_bwd_dq_finish(ws.t, nbytes, outs[0].t, B, H, N, d, q.dtype, scale, stream)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    assert all(g.intact() for g in outs) and ws.intact(), "the fused backward wrote outside its buffers"
    return tuple(g.t for g in outs)


def f64(t):
    return t.detach().double().cpu().numpy()


def half_ulp(ref, dtype):
    """Half the spacing of ``dtype`` (bf16: 8 significant bits, fp16: 11) at |ref|: the
    error of rounding the exact value to the output type, which no kernel can avoid."""
    bits = 8 if dtype == torch.bfloat16 else 11
    a = np.abs(np.asarray(ref, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - bits), 0.0)


def o_err(o, ref, rows=None):
    """Max-abs error of O beyond the rounding of the exact value to O's 16-bit type.

    O_MAX_ABS = 1e-2 bounds the computation; the exact result rounded to bf16 is itself
    up to 2^-8 |O| away (0.0156 for |O| in [4, 8)), more than 1e-2, so that final
    rounding step is allowed on top."""
    g = f64(o) if hasattr(o, "detach") else np.asarray(o, np.float64)
    if rows is not None:
        g = g[..., rows, :]
    if not ref.size:
        return 0.0
    return float(np.max(np.abs(g - ref) - half_ulp(ref, o.dtype)))


def lse_err(lse, ref):
    return float(np.max(np.abs(f64(lse) - ref) / np.maximum(np.abs(ref), 1.0))) if ref.size else 0.0


def rel_l2(g, ref):
    g = f64(g) if hasattr(g, "detach") else g
    den = float(np.linalg.norm(ref))
    return float(np.linalg.norm(g - ref)) / max(den, 1e-30)


ZERO_GRAD_ABS = 1e-3


def grad_err(g, ref):
    """Relative L2 error; for a reference that is exactly zero (one visible key makes dS = 0,
    so dQ = dK = 0) the absolute residue, scaled so that ZERO_GRAD_ABS maps to GRAD_REL_L2."""
    g = f64(g) if hasattr(g, "detach") else g
    if not np.any(ref):
        return float(np.max(np.abs(g))) / ZERO_GRAD_ABS * GRAD_REL_L2 if g.size else 0.0
    return rel_l2(g, ref)


def sample_rows(N, extra=24, seed=0):
    """Rows at both ends, on tile boundaries and at random."""
    rows = {0, 1, N - 1, N - 2}
    for t in range(128, N, 128):
        rows.update({t - 1, t})
    rows = sorted(r for r in rows if 0 <= r < N)
    rng = np.random.default_rng(seed)
    if len(rows) > 40:
        rows = sorted(set(rng.choice(rows, 40, replace=False).tolist()) | {0, N - 1})
    rows = sorted(set(rows) | set(rng.integers(0, N, extra).tolist()))
    return np.array(rows, dtype=np.int64)


def dq_close(a, b) -> bool:
    """Two dQ results of the fused backward, whose float32 accumulator adds the key tiles'
    shares in an order that varies from run to run: equal up to the rounding that order
    can move (one 16-bit step of the value, plus a cancellation allowance scaled by the
    tensor's largest entry)."""
    x, y = f64(a), f64(b)
    tol = 2.0 ** -7 * np.abs(y) + 1e-4 * float(np.max(np.abs(y)) if y.size else 0.0)
    return bool(np.all(np.abs(x - y) <= tol))


def assert_same_grads(got, want, what=""):
    """dK and dV byte for byte; dQ as dq_close allows (the fused backward's accumulator)."""
    dq, dk, dv = got
    rq, rk, rv = want
    assert torch.equal(dk, rk), f"{what} dK differs"
    assert torch.equal(dv, rv), f"{what} dV differs"
    assert dq_close(dq, rq), f"{what} dQ differs beyond the accumulator's reordering"
