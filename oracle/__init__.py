"""FP64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  The product library
never imports this package and shares no code with it.

The arithmetic lives in ``attn_oracle.c`` (plain double-precision loops over
the definition, OpenMP across rows); this module compiles it with gcc and
marshals NumPy float64 arrays in and out.  Every input is first upcast to
float64, which is exact for BF16 and FP16.

Functions
---------
attn_fwd(q, k, v, causal, scale, rows=None) -> (o, lse)
    O = softmax(scale * Q K^T) V and the natural-log row logsumexp
    ("FlashAttention hardware-aware analysis" (huaweicloud), section one,
    part 2; "Understanding online softmax in Flash Attention from scratch",
    section 3.1).
attn_bwd(q, k, v, dout, causal, scale, qrows=None, kcols=None) -> (dq, dk, dv)
    chain rule of the same definition ("Understanding FlashAttention,
    Part 2", section 2.4, Figs 16-19).
dequant_e4m3(codes, scales, block_rows=128) -> float64 array
    value of each E4M3 code times the scale of its block of rows (FP8 with
    per-block scale factors: huaweicloud page, section four, part 3).
attn_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal, scale) -> (o, lse)
    attn_fwd of the dequantised inputs.
attn_fwd_varlen(q, k, v, cu_q, cu_k, causal, scale) / attn_bwd_varlen(...)
    packed [tokens, H, d] sequences with offsets cu_q, cu_k: attn_fwd /
    attn_bwd of every sequence's own slices.
attn_fwd_dropout / attn_bwd_dropout(..., t, seed)
    the same with dropout on the probabilities: keep iff a Philox4x32-10 byte
    >= t, kept probabilities scaled by 256 / (256 - t) (definition in the C
    source; "Understanding FlashAttention, Part 2", section 2.4 names dropout).

Pins (tests/test_oracle_pins.py): hand-derived closed forms under
tests/golden/, brute force with Python ``math`` on tiny inputs, the two-block
merge rule of the huaweicloud page (section two), the all-equal-scores closed
form, one-hot rows at scores near 1000, causal row 0, finite differences and
an independent autograd evaluation for the backward, the invariants
sum_j dV_j = sum_i dO_i, sum_j dK_j = 0, and K/V permutation symmetry; for
the FP8 decoding, closed-form codes of the format definition, all 256 codes
against PyTorch's float8_e4m3fn conversion, and a brute-force block
dequantisation.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_default = None


def build(force: bool = False, src: str = SOURCE, out: str = _LIB) -> str:
    """Compile the oracle source into a shared library (gcc, OpenMP, IEEE semantics)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _as_f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor: upcast exactly, then view as NumPy
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _rows(r):
    if r is None:
        return None
    return np.ascontiguousarray(np.asarray(r, dtype=np.int64).reshape(-1))


class Oracle:
    """One loaded copy of the oracle library (the default one, or a test build)."""

    def __init__(self, libpath: str):
        lib = ctypes.CDLL(libpath)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.oracle_attn_fwd.argtypes = [P, P, P, I64, I64, I64, I64, ctypes.c_int, ctypes.c_double,
                                        P, I64, P, P]
        lib.oracle_attn_fwd.restype = ctypes.c_int
        lib.oracle_attn_bwd.argtypes = [P, P, P, P, I64, I64, I64, I64, ctypes.c_int, ctypes.c_double,
                                        P, I64, P, I64, P, P, P]
        lib.oracle_attn_bwd.restype = ctypes.c_int
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_dequant_e4m3.argtypes = [P, P, I64, I64, I64, I64, P]
        lib.oracle_dequant_e4m3.restype = ctypes.c_int
        U32 = ctypes.c_uint32
        lib.oracle_philox4x32_10.argtypes = [P, P, P]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_dropout_factor.argtypes = [I64, I64, I64, ctypes.c_int, U32, U32]
        lib.oracle_dropout_factor.restype = ctypes.c_double
        lib.oracle_attn_fwd_dropout.argtypes = [P, P, P, I64, I64, I64, I64, ctypes.c_int, ctypes.c_double,
                                                ctypes.c_int, U32, U32, I64, P, I64, P, P]
        lib.oracle_attn_fwd_dropout.restype = ctypes.c_int
        lib.oracle_attn_bwd_dropout.argtypes = [P, P, P, P, I64, I64, I64, I64, ctypes.c_int, ctypes.c_double,
                                                ctypes.c_int, U32, U32, I64, P, I64, P, I64, P, P, P]
        lib.oracle_attn_bwd_dropout.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        self.lib = lib
        self.path = libpath

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def attn_fwd(self, q, k, v, causal: bool, scale: float, rows=None):
        """Exact attention forward in FP64.

        q: [..., N, d]; k, v: [..., Nk, d] with the same leading dims (causal
        needs Nk >= N and aligns the mask to the last key: query i sees keys
        j <= i + Nk - N).  Returns (o, lse) with shapes [..., R, d] and [..., R],
        R = N or len(rows).
        """
        q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
        if q.ndim < 2 or k.shape != v.shape or q.shape[:-2] != k.shape[:-2] or q.shape[-1] != k.shape[-1]:
            raise ValueError("q must be [..., N, d] and k, v [..., Nk, d] with matching dims")
        lead, (N, d), Nk = q.shape[:-2], q.shape[-2:], k.shape[-2]
        BH = int(np.prod(lead)) if lead else 1
        rr = _rows(rows)
        R = N if rr is None else rr.size
        o = np.empty((BH, R, d), np.float64)
        lse = np.empty((BH, R), np.float64)
        rc = self.lib.oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), BH, N, Nk, d, int(bool(causal)),
                                      float(scale), _ptr(rr), 0 if rr is None else rr.size,
                                      _ptr(o), _ptr(lse))
        if rc != 0:
            raise RuntimeError("oracle_attn_fwd failed (bad argument or out of memory)")
        return o.reshape(*lead, R, d), lse.reshape(*lead, R)

    def e4m3_value(self, code: int) -> float:
        """The real number one E4M3 code (0..255) stands for (NaN for the NaN codes)."""
        return float(self.lib.oracle_e4m3_value(int(code) & 0xFF))

    def dequant_e4m3(self, codes, scales, block_rows: int = 128):
        """Block dequantisation: codes [..., N, d] (uint8 E4M3 bytes, or a float8_e4m3fn
        tensor), scales [..., ceil(N / block_rows)] float32 -> float64 [..., N, d]."""
        if hasattr(codes, "detach"):  # a torch tensor
            import torch

            codes = codes.detach().to("cpu")
            if codes.dtype != torch.uint8:
                codes = codes.view(torch.uint8)
            codes = codes.numpy()
        if hasattr(scales, "detach"):
            scales = scales.detach().to("cpu").numpy()
        c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
        sc = np.ascontiguousarray(np.asarray(scales, dtype=np.float32))
        if c.ndim < 2:
            raise ValueError("codes must be [..., N, d]")
        lead, (N, d) = c.shape[:-2], c.shape[-2:]
        nblk = -(-N // int(block_rows))
        if sc.shape != tuple(lead) + (nblk,):
            raise ValueError(f"scales must be {tuple(lead) + (nblk,)}, got {sc.shape}")
        BH = int(np.prod(lead)) if lead else 1
        out = np.empty(c.shape, np.float64)
        if self.lib.oracle_dequant_e4m3(_ptr(c), _ptr(sc), BH, N, d, int(block_rows), _ptr(out)) != 0:
            raise RuntimeError("oracle_dequant_e4m3 failed (bad argument)")
        return out

    def attn_fwd_fp8(self, q8, k8, v8, q_scale, k_scale, v_scale, causal: bool, scale: float,
                     rows=None, block_rows: int = 128):
        """Exact FP64 attention of block-scaled E4M3 inputs: the inputs are dequantised
        (dequant_e4m3) and passed to attn_fwd.  Returns (o, lse) as attn_fwd does."""
        q = self.dequant_e4m3(q8, q_scale, block_rows)
        k = self.dequant_e4m3(k8, k_scale, block_rows)
        v = self.dequant_e4m3(v8, v_scale, block_rows)
        return self.attn_fwd(q, k, v, causal, scale, rows)

    def philox(self, counter, key):
        """Philox4x32-10 of a 4-word counter and a 2-word key -> 4 uint32 words."""
        c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint32).reshape(4))
        k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32).reshape(2))
        out = np.zeros(4, np.uint32)
        self.lib.oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
        return out

    def dropout_factor(self, bh, i, j, t, seed):
        """Z_ij of the dropout definition: 0 or 256 / (256 - t)."""
        seed = int(seed) & 0xFFFFFFFFFFFFFFFF
        return float(self.lib.oracle_dropout_factor(int(bh), int(i), int(j), int(t), seed & 0xFFFFFFFF, seed >> 32))

    def attn_fwd_dropout(self, q, k, v, causal: bool, scale: float, t: int, seed: int, rows=None, bh0: int = 0):
        """attn_fwd with dropout on the probabilities (threshold t in 0..255, 64-bit seed); the
        arrays' heads are heads bh0, bh0 + 1, ... of the mask."""
        q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
        if q.ndim < 2 or k.shape != v.shape or q.shape[:-2] != k.shape[:-2] or q.shape[-1] != k.shape[-1]:
            raise ValueError("q must be [..., N, d] and k, v [..., Nk, d] with matching dims")
        lead, (N, d), Nk = q.shape[:-2], q.shape[-2:], k.shape[-2]
        BH = int(np.prod(lead)) if lead else 1
        rr = _rows(rows)
        R = N if rr is None else rr.size
        o = np.empty((BH, R, d), np.float64)
        lse = np.empty((BH, R), np.float64)
        seed = int(seed) & 0xFFFFFFFFFFFFFFFF
        rc = self.lib.oracle_attn_fwd_dropout(_ptr(q), _ptr(k), _ptr(v), BH, N, Nk, d, int(bool(causal)),
                                              float(scale), int(t), seed & 0xFFFFFFFF, seed >> 32, int(bh0), _ptr(rr),
                                              0 if rr is None else rr.size, _ptr(o), _ptr(lse))
        if rc != 0:
            raise RuntimeError("oracle_attn_fwd_dropout failed (bad argument or out of memory)")
        return o.reshape(*lead, R, d), lse.reshape(*lead, R)

    def attn_bwd_dropout(self, q, k, v, dout, causal: bool, scale: float, t: int, seed: int, qrows=None,
                         kcols=None, want_dq: bool = True, want_dkv: bool = True, bh0: int = 0):
        """attn_bwd with dropout on the probabilities (same t and seed as the forward)."""
        q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
        if not (q.shape == do.shape and k.shape == v.shape) or q.ndim < 2 or \
                q.shape[:-2] != k.shape[:-2] or q.shape[-1] != k.shape[-1]:
            raise ValueError("q, dout must be [..., N, d] and k, v [..., Nk, d] with matching dims")
        lead, (N, d), Nk = q.shape[:-2], q.shape[-2:], k.shape[-2]
        BH = int(np.prod(lead)) if lead else 1
        qr, kc = _rows(qrows), _rows(kcols)
        nq = N if qr is None else qr.size
        nk = Nk if kc is None else kc.size
        dq = np.empty((BH, nq, d), np.float64) if want_dq else None
        dk = np.empty((BH, nk, d), np.float64) if want_dkv else None
        dv = np.empty((BH, nk, d), np.float64) if want_dkv else None
        seed = int(seed) & 0xFFFFFFFFFFFFFFFF
        rc = self.lib.oracle_attn_bwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(do), BH, N, Nk, d,
                                              int(bool(causal)), float(scale), int(t), seed & 0xFFFFFFFF,
                                              seed >> 32, int(bh0), _ptr(qr), 0 if qr is None else qr.size,
                                              _ptr(kc), 0 if kc is None else kc.size,
                                              _ptr(dq), _ptr(dk), _ptr(dv))
        if rc != 0:
            raise RuntimeError("oracle_attn_bwd_dropout failed (bad argument or out of memory)")
        shp = lambda a, r: None if a is None else a.reshape(*lead, r, d)
        return shp(dq, nq), shp(dk, nk), shp(dv, nk)

    def attn_bwd(self, q, k, v, dout, causal: bool, scale: float, qrows=None, kcols=None,
                 want_dq: bool = True, want_dkv: bool = True):
        """Exact attention backward in FP64: gradients of sum(dO * O).

        q, dout: [..., N, d]; k, v: [..., Nk, d] (masking as in attn_fwd).
        Returns (dq, dk, dv); dq covers ``qrows`` (all rows if None), dk and dv
        cover ``kcols`` (all keys if None).  A skipped output is None.
        """
        q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
        if not (q.shape == do.shape and k.shape == v.shape) or q.ndim < 2 or \
                q.shape[:-2] != k.shape[:-2] or q.shape[-1] != k.shape[-1]:
            raise ValueError("q, dout must be [..., N, d] and k, v [..., Nk, d] with matching dims")
        lead, (N, d), Nk = q.shape[:-2], q.shape[-2:], k.shape[-2]
        BH = int(np.prod(lead)) if lead else 1
        qr, kc = _rows(qrows), _rows(kcols)
        nq = N if qr is None else qr.size
        nk = Nk if kc is None else kc.size
        dq = np.empty((BH, nq, d), np.float64) if want_dq else None
        dk = np.empty((BH, nk, d), np.float64) if want_dkv else None
        dv = np.empty((BH, nk, d), np.float64) if want_dkv else None
        rc = self.lib.oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), BH, N, Nk, d,
                                      int(bool(causal)), float(scale),
                                      _ptr(qr), 0 if qr is None else qr.size,
                                      _ptr(kc), 0 if kc is None else kc.size,
                                      _ptr(dq), _ptr(dk), _ptr(dv))
        if rc != 0:
            raise RuntimeError("oracle_attn_bwd failed (bad argument or out of memory)")
        shp = lambda a, r: None if a is None else a.reshape(*lead, r, d)
        return shp(dq, nq), shp(dk, nk), shp(dv, nk)


    def _degenerate(self, nq: int, nk: int, causal: bool) -> bool:
        """A packed sequence whose rows have no defined softmax: no keys, or causal with
        fewer keys than queries (some query would see no key)."""
        return nk == 0 or (causal and nk < nq)

    def attn_fwd_varlen(self, q, k, v, cu_q, cu_k, causal: bool, scale: float):
        """Variable-length packed attention: q [Tq, H, d], k, v [Tk, H, d], sequence b owning query
        tokens cu_q[b] .. cu_q[b+1]-1 and key tokens cu_k[b] .. cu_k[b+1]-1.  Each sequence and head
        is attn_fwd of its own slices (causal aligned to the sequence's last key).  A sequence
        without keys, or causal with fewer keys than queries, gets O = 0 and lse = -inf on
        every row (the library's stated convention for rows with no defined softmax).
        Returns (o [Tq, H, d], lse [H, Tq])."""
        q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
        cq, ck = _cu(cu_q), _cu(cu_k)
        Tq, H, d = q.shape
        o = np.zeros_like(q)
        lse = np.zeros((H, Tq))
        for b in range(len(cq) - 1):
            qs, ks = slice(cq[b], cq[b + 1]), slice(ck[b], ck[b + 1])
            nq, nk = cq[b + 1] - cq[b], ck[b + 1] - ck[b]
            if nq == 0:
                continue
            if self._degenerate(nq, nk, causal):
                lse[:, qs] = -np.inf
                continue
            t = lambda x, s_: x[s_].transpose(1, 0, 2)
            ob, lb = self.attn_fwd(t(q, qs), t(k, ks), t(v, ks), causal, scale)
            o[qs] = ob.transpose(1, 0, 2)
            lse[:, qs] = lb
        return o, lse

    def attn_bwd_varlen(self, q, k, v, dout, cu_q, cu_k, causal: bool, scale: float):
        """Gradients of sum(dO * O) for attn_fwd_varlen: (dq [Tq, H, d], dk, dv [Tk, H, d]).  Each
        sequence is attn_bwd of its own slices; a degenerate sequence (see attn_fwd_varlen) has
        a constant output, so its gradients are zero."""
        q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
        cq, ck = _cu(cu_q), _cu(cu_k)
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        for b in range(len(cq) - 1):
            qs, ks = slice(cq[b], cq[b + 1]), slice(ck[b], ck[b + 1])
            nq, nk = cq[b + 1] - cq[b], ck[b + 1] - ck[b]
            if nq == 0 or self._degenerate(nq, nk, causal):
                continue
            t = lambda x, s_: x[s_].transpose(1, 0, 2)
            gq, gk, gv = self.attn_bwd(t(q, qs), t(k, ks), t(v, ks), t(do, qs), causal, scale)
            dq[qs], dk[ks], dv[ks] = gq.transpose(1, 0, 2), gk.transpose(1, 0, 2), gv.transpose(1, 0, 2)
        return dq, dk, dv


def default() -> Oracle:
    """The oracle built from this package's source (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def num_threads() -> int:
    """Threads the oracle's OpenMP loops run on."""
    return default().num_threads()


def attn_fwd(q, k, v, causal: bool, scale: float, rows=None):
    return default().attn_fwd(q, k, v, causal, scale, rows)


def attn_bwd(q, k, v, dout, causal: bool, scale: float, qrows=None, kcols=None,
             want_dq: bool = True, want_dkv: bool = True):
    return default().attn_bwd(q, k, v, dout, causal, scale, qrows, kcols, want_dq, want_dkv)


attn_fwd.__doc__ = Oracle.attn_fwd.__doc__
attn_bwd.__doc__ = Oracle.attn_bwd.__doc__


def dequant_e4m3(codes, scales, block_rows: int = 128):
    return default().dequant_e4m3(codes, scales, block_rows)


def attn_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal: bool, scale: float, rows=None,
                 block_rows: int = 128):
    return default().attn_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal, scale, rows, block_rows)


dequant_e4m3.__doc__ = Oracle.dequant_e4m3.__doc__
attn_fwd_fp8.__doc__ = Oracle.attn_fwd_fp8.__doc__


def attn_fwd_dropout(q, k, v, causal: bool, scale: float, t: int, seed: int, rows=None, bh0: int = 0):
    return default().attn_fwd_dropout(q, k, v, causal, scale, t, seed, rows, bh0)


def attn_bwd_dropout(q, k, v, dout, causal: bool, scale: float, t: int, seed: int, qrows=None, kcols=None,
                     want_dq: bool = True, want_dkv: bool = True, bh0: int = 0):
    return default().attn_bwd_dropout(q, k, v, dout, causal, scale, t, seed, qrows, kcols, want_dq, want_dkv, bh0)


attn_fwd_dropout.__doc__ = Oracle.attn_fwd_dropout.__doc__
attn_bwd_dropout.__doc__ = Oracle.attn_bwd_dropout.__doc__


def _cu(cu):
    return [int(x) for x in (cu.tolist() if hasattr(cu, "tolist") else cu)]


def attn_fwd_varlen(q, k, v, cu_q, cu_k, causal: bool, scale: float):
    return default().attn_fwd_varlen(q, k, v, cu_q, cu_k, causal, scale)


def attn_bwd_varlen(q, k, v, dout, cu_q, cu_k, causal: bool, scale: float):
    return default().attn_bwd_varlen(q, k, v, dout, cu_q, cu_k, causal, scale)


attn_fwd_varlen.__doc__ = Oracle.attn_fwd_varlen.__doc__
attn_bwd_varlen.__doc__ = Oracle.attn_bwd_varlen.__doc__
