"""Exact tiled online-softmax attention for one GB300 (sm_103a).

A thin ctypes binding over ``libattn.so`` (the C ABI in ``include/attn.h``):
argument marshalling only, every step of the computation runs in the
library's CUDA kernels.  There is no CPU fallback: if the library is missing
or cannot load, every call raises.

Low level (same names and argument order as the C ABI; tensors may be passed
where the C ABI takes device pointers, and ``stream=None`` means torch's
current stream):

    attn_fwd(q, k, v, o, lse, B, H, N, d, dt, causal, scale, dev_status=None, stream=None)
    attn_fwd_rect(q, k, v, o, lse, B, H, Nq, Nk, d, dt, causal, scale, dev_status=None, stream=None)
    attn_fwd_varlen(q, k, v, o, lse, cu_q, cu_k, B, H, max_q, max_k, Tq, Tk, d, dt, causal, scale, ...)
    attn_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, cu_q, cu_k,
                    B, H, max_q, max_k, Tq, Tk, d, dt, causal, scale, ...)
    attn_fwd_varlen_dropout / attn_bwd_varlen_dropout: the two above plus p_drop, seed
    attn_fwd_rect_dropout / attn_bwd_rect_dropout: attn_fwd_rect / attn_bwd_rect plus p_drop, seed
    attn_dropout_bits_bytes(B, H, Nq, Nk)
    attn_fwd_dropout_bits(q, k, v, o, lse, keep_bits, keep_bits_bytes, B, H, N, d, dt, causal, scale, p_drop, seed, ...)
    attn_bwd_dropout_bits(q, k, v, o, dout, lse, keep_bits, keep_bits_bytes, dq, dk, dv, workspace, workspace_bytes,
                          B, H, N, d, dt, causal, scale, p_drop, ...)   (the keep decisions drawn once)
    attn_fwd_varlen_splitkv_workspace_bytes(H, Tq, d, n_splits)
    attn_fwd_varlen_splitkv(q, k, v, o, lse, workspace, workspace_bytes, cu_q, cu_k, B, H, max_q, max_k,
                            Tq, Tk, d, dt, causal, scale, n_splits, dev_status=None, stream=None)
    attn_fwd_dropout(q, k, v, o, lse, B, H, N, d, dt, causal, scale, p_drop, seed, dev_status=None, stream=None)
    attn_bwd_dropout(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes,
                     B, H, N, d, dt, causal, scale, p_drop, seed, dev_status=None, stream=None)
    attn_bwd_rect(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes,
                  B, H, Nq, Nk, d, dt, causal, scale, dev_status=None, stream=None)
    attn_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, B, H, N, d, out_dt, causal, scale,
                 dev_status=None, stream=None)
    attn_fwd_splitkv_workspace_bytes(B, H, N, d, n_splits)
    attn_fwd_splitkv_rect(q, k, v, o, lse, workspace, workspace_bytes, B, H, Nq, Nk, d, dt, causal,
                          scale, n_splits, dev_status=None, stream=None)
    attn_fwd_splitkv(q, k, v, o, lse, workspace, workspace_bytes, B, H, N, d, dt, causal, scale,
                     n_splits, dev_status=None, stream=None)
    attn_bwd_workspace_bytes(B, H, N, d)
    attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes,
             B, H, N, d, dt, causal, scale, dev_status=None, stream=None)
    attn_bwd_prepare / attn_bwd_dkdvdq / attn_bwd_dq_finish  (the stages of attn_bwd, d <= 128)
    attn_bwd_deterministic_workspace_bytes(B, H, N, d)
    attn_bwd_deterministic(...)                     (attn_bwd's arguments; identical bytes every call)
    attn_bwd_prepare / attn_bwd_dkdv / attn_bwd_dq   (the three stages of attn_bwd_deterministic)
    attn_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, dt, causal, scale, ...)
                                                     (attn_bwd with library-owned scratch)
    attn_status_string(status)
    attn_selftest_bounded_wait(dev_status, limit_ns, stream=None)

Convenience wrappers over torch tensors of shape [B, H, N, d]:

    attention(q, k, v, causal=False, scale=None, dropout_p=0.0, seed=0)  -> o
        (differentiable: a torch.autograd.Function over the forward / backward calls)

    forward(q, k, v, causal=False, scale=None)            -> (o, lse)
    forward_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal=False, scale=None,
                out_dtype=torch.bfloat16)                 -> (o, lse)
    backward(q, k, v, o, lse, dout, causal=False, scale=None) -> (dq, dk, dv)
"""
from __future__ import annotations

import ctypes
import math
import os

from . import _build

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4
ATTN_BF16 = 0
ATTN_FP16 = 1

LIB_PATH = _build.LIB
EXPORTS = ("attn_fwd", "attn_fwd_rect", "attn_bwd_rect", "attn_fwd_varlen", "attn_bwd_varlen", "attn_fwd_varlen_dropout", "attn_bwd_varlen_dropout", "attn_fwd_rect_dropout", "attn_bwd_rect_dropout", "attn_fwd_dropout", "attn_bwd_dropout", "attn_fwd_fp8", "attn_fwd_splitkv_workspace_bytes", "attn_fwd_splitkv", "attn_fwd_splitkv_rect", "attn_fwd_varlen_splitkv_workspace_bytes", "attn_fwd_varlen_splitkv", "attn_bwd_workspace_bytes", "attn_bwd", "attn_bwd_prepare", "attn_bwd_dkdv",
           "attn_bwd_dq", "attn_bwd_deterministic_workspace_bytes", "attn_bwd_deterministic", "attn_bwd_dkdvdq",
           "attn_bwd_dq_finish", "attn_dropout_bits_bytes", "attn_fwd_dropout_bits", "attn_bwd_dropout_bits", "attn_bwd_noalloc", "attn_status_string", "attn_selftest_bounded_wait")

_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {attn_status_string(status)}")


def load(build_if_missing: bool = True):
    """Load libattn.so (building it in-tree first if it is absent or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libattn.so not found at {LIB_PATH}; run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, P, P]
    U64 = ctypes.c_uint64
    lib.attn_fwd_varlen.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, P, P]
    lib.attn_fwd_varlen.restype = I
    lib.attn_bwd_varlen.argtypes = [P, P, P, P, P, P, P, P, P, P, SZ, P, P, I, I, I, I, I, I, I, I, I, F, P, P]
    lib.attn_bwd_varlen.restype = I
    lib.attn_fwd_rect_dropout.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, F, U64, P, P]
    lib.attn_fwd_rect_dropout.restype = I
    lib.attn_bwd_rect_dropout.argtypes = [P, P, P, P, P, P, P, P, P, P, SZ, I, I, I, I, I, I, I, F, F, U64, P, P]
    lib.attn_bwd_rect_dropout.restype = I
    lib.attn_fwd_varlen_dropout.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, F, U64, P, P]
    lib.attn_fwd_varlen_dropout.restype = I
    lib.attn_bwd_varlen_dropout.argtypes = [P, P, P, P, P, P, P, P, P, P, SZ, P, P, I, I, I, I, I, I, I, I, I, F, F,
                                            U64, P, P]
    lib.attn_bwd_varlen_dropout.restype = I
    lib.attn_fwd_dropout.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, F, U64, P, P]
    lib.attn_fwd_dropout.restype = I
    lib.attn_bwd_dropout.argtypes = [P, P, P, P, P, P, P, P, P, P, SZ, I, I, I, I, I, I, F, F, U64, P, P]
    lib.attn_bwd_dropout.restype = I
    lib.attn_fwd_rect.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, P, P]
    lib.attn_fwd_rect.restype = I
    lib.attn_bwd_rect.argtypes = [P, P, P, P, P, P, P, P, P, P, SZ, I, I, I, I, I, I, I, F, P, P]
    lib.attn_bwd_rect.restype = I
    lib.attn_fwd_fp8.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P, P]
    lib.attn_fwd_fp8.restype = I
    lib.attn_fwd.restype = I
    lib.attn_fwd_splitkv_workspace_bytes.argtypes = [I, I, I, I, I]
    lib.attn_fwd_splitkv_workspace_bytes.restype = SZ
    lib.attn_fwd_splitkv.argtypes = [P, P, P, P, P, P, SZ, I, I, I, I, I, I, F, I, P, P]
    lib.attn_fwd_splitkv.restype = I
    lib.attn_fwd_splitkv_rect.argtypes = [P, P, P, P, P, P, SZ, I, I, I, I, I, I, I, F, I, P, P]
    lib.attn_fwd_splitkv_rect.restype = I
    lib.attn_fwd_varlen_splitkv_workspace_bytes.argtypes = [I, I, I, I]
    lib.attn_fwd_varlen_splitkv_workspace_bytes.restype = SZ
    lib.attn_fwd_varlen_splitkv.argtypes = [P, P, P, P, P, P, SZ, P, P, I, I, I, I, I, I, I, I, I, F, I, P, P]
    lib.attn_fwd_varlen_splitkv.restype = I
    lib.attn_bwd_workspace_bytes.argtypes = [I, I, I, I]
    lib.attn_bwd_workspace_bytes.restype = SZ
    lib.attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, SZ, I, I, I, I, I, I, F, P, P]
    lib.attn_bwd.restype = I
    lib.attn_bwd_prepare.argtypes = [P, P, P, P, SZ, I, I, I, I, I, P]
    lib.attn_bwd_prepare.restype = I
    lib.attn_bwd_dkdv.argtypes = [P, P, P, P, P, SZ, P, P, I, I, I, I, I, I, F, P, P]
    lib.attn_bwd_dkdv.restype = I
    lib.attn_bwd_dq.argtypes = [P, P, P, P, P, SZ, P, I, I, I, I, I, I, F, P, P]
    lib.attn_bwd_dq.restype = I
    lib.attn_bwd_deterministic_workspace_bytes.argtypes = [I, I, I, I]
    lib.attn_bwd_deterministic_workspace_bytes.restype = SZ
    lib.attn_bwd_deterministic.argtypes = [P, P, P, P, P, P, P, P, P, P, SZ, I, I, I, I, I, I, F, P, P]
    lib.attn_bwd_deterministic.restype = I
    lib.attn_bwd_dkdvdq.argtypes = [P, P, P, P, P, SZ, P, P, I, I, I, I, I, I, F, P, P]
    lib.attn_bwd_dkdvdq.restype = I
    lib.attn_bwd_dq_finish.argtypes = [P, SZ, P, I, I, I, I, I, F, P]
    lib.attn_bwd_dq_finish.restype = I
    lib.attn_dropout_bits_bytes.argtypes = [I, I, I, I]
    lib.attn_dropout_bits_bytes.restype = SZ
    lib.attn_fwd_dropout_bits.argtypes = [P, P, P, P, P, P, SZ, I, I, I, I, I, I, F, F, U64, P, P]
    lib.attn_fwd_dropout_bits.restype = I
    lib.attn_bwd_dropout_bits.argtypes = [P, P, P, P, P, P, P, SZ, P, P, P, P, SZ, I, I, I, I, I, I, F, F, P, P]
    lib.attn_bwd_dropout_bits.restype = I
    lib.attn_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P, P]
    lib.attn_bwd_noalloc.restype = I
    lib.attn_status_string.argtypes = [I]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_selftest_bounded_wait.argtypes = [P, ctypes.c_uint64, P]
    lib.attn_selftest_bounded_wait.restype = I
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr() or None
    return int(x) or None


def _stream(s):
    if s is None:
        import torch

        return torch.cuda.current_stream().cuda_stream or None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream or None
    return int(s) or None


def _dt(x):
    if isinstance(x, int):
        return x
    import torch

    if x == torch.bfloat16:
        return ATTN_BF16
    if x == torch.float16:
        return ATTN_FP16
    raise ValueError(f"unsupported dtype {x}")


def attn_status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()


def attn_fwd(q, k, v, o, lse, B, H, N, d, dt, causal, scale, dev_status=None, stream=None) -> int:
    return int(load().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(N), int(d),
                               _dt(dt), int(bool(causal)), float(scale), _ptr(dev_status), _stream(stream)))


def attn_fwd_varlen(q, k, v, o, lse, cu_q, cu_k, B, H, max_q, max_k, Tq, Tk, d, dt, causal, scale, dev_status=None,
                    stream=None) -> int:
    return int(load().attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_q), _ptr(cu_k), int(B),
                                      int(H), int(max_q), int(max_k), int(Tq), int(Tk), int(d), _dt(dt),
                                      int(bool(causal)), float(scale), _ptr(dev_status), _stream(stream)))


def attn_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, cu_q, cu_k, B, H, max_q, max_k, Tq,
                    Tk, d, dt, causal, scale, dev_status=None, stream=None) -> int:
    return int(load().attn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                                      _ptr(dv), _ptr(workspace), int(workspace_bytes), _ptr(cu_q), _ptr(cu_k), int(B),
                                      int(H), int(max_q), int(max_k), int(Tq), int(Tk), int(d), _dt(dt),
                                      int(bool(causal)), float(scale), _ptr(dev_status), _stream(stream)))


def attn_fwd_varlen_splitkv_workspace_bytes(H, Tq, d, n_splits) -> int:
    return int(load().attn_fwd_varlen_splitkv_workspace_bytes(int(H), int(Tq), int(d), int(n_splits)))


def attn_fwd_varlen_splitkv(q, k, v, o, lse, workspace, workspace_bytes, cu_q, cu_k, B, H, max_q, max_k, Tq, Tk, d, dt,
                            causal, scale, n_splits, dev_status=None, stream=None) -> int:
    return int(load().attn_fwd_varlen_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(workspace),
                                              int(workspace_bytes), _ptr(cu_q), _ptr(cu_k), int(B), int(H),
                                              int(max_q), int(max_k), int(Tq), int(Tk), int(d), _dt(dt),
                                              int(bool(causal)), float(scale), int(n_splits), _ptr(dev_status),
                                              _stream(stream)))


def attn_fwd_rect_dropout(q, k, v, o, lse, B, H, Nq, Nk, d, dt, causal, scale, p_drop, seed, dev_status=None,
                          stream=None) -> int:
    return int(load().attn_fwd_rect_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(Nq),
                                            int(Nk), int(d), _dt(dt), int(bool(causal)), float(scale), float(p_drop),
                                            int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(dev_status), _stream(stream)))


def attn_bwd_rect_dropout(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, Nq, Nk, d, dt, causal,
                          scale, p_drop, seed, dev_status=None, stream=None) -> int:
    return int(load().attn_bwd_rect_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                                            _ptr(dk), _ptr(dv), _ptr(workspace), int(workspace_bytes), int(B), int(H),
                                            int(Nq), int(Nk), int(d), _dt(dt), int(bool(causal)), float(scale),
                                            float(p_drop), int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(dev_status),
                                            _stream(stream)))


def attn_fwd_varlen_dropout(q, k, v, o, lse, cu_q, cu_k, B, H, max_q, max_k, Tq, Tk, d, dt, causal, scale, p_drop,
                            seed, dev_status=None, stream=None) -> int:
    return int(load().attn_fwd_varlen_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_q), _ptr(cu_k),
                                              int(B), int(H), int(max_q), int(max_k), int(Tq), int(Tk), int(d),
                                              _dt(dt), int(bool(causal)), float(scale), float(p_drop),
                                              int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(dev_status), _stream(stream)))


def attn_bwd_varlen_dropout(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, cu_q, cu_k, B, H, max_q,
                            max_k, Tq, Tk, d, dt, causal, scale, p_drop, seed, dev_status=None, stream=None) -> int:
    return int(load().attn_bwd_varlen_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                                              _ptr(dk), _ptr(dv), _ptr(workspace), int(workspace_bytes), _ptr(cu_q),
                                              _ptr(cu_k), int(B), int(H), int(max_q), int(max_k), int(Tq), int(Tk),
                                              int(d), _dt(dt), int(bool(causal)), float(scale), float(p_drop),
                                              int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(dev_status), _stream(stream)))


def attn_fwd_dropout(q, k, v, o, lse, B, H, N, d, dt, causal, scale, p_drop, seed, dev_status=None,
                     stream=None) -> int:
    return int(load().attn_fwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(N), int(d),
                                       _dt(dt), int(bool(causal)), float(scale), float(p_drop),
                                       int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(dev_status), _stream(stream)))


def attn_bwd_dropout(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, d, dt, causal, scale,
                     p_drop, seed, dev_status=None, stream=None) -> int:
    return int(load().attn_bwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                                       _ptr(dk), _ptr(dv), _ptr(workspace), int(workspace_bytes), int(B), int(H),
                                       int(N), int(d), _dt(dt), int(bool(causal)), float(scale), float(p_drop),
                                       int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(dev_status), _stream(stream)))


def attn_fwd_rect(q, k, v, o, lse, B, H, Nq, Nk, d, dt, causal, scale, dev_status=None, stream=None) -> int:
    return int(load().attn_fwd_rect(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(Nq), int(Nk),
                                    int(d), _dt(dt), int(bool(causal)), float(scale), _ptr(dev_status),
                                    _stream(stream)))


def attn_bwd_rect(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, Nq, Nk, d, dt, causal, scale,
                  dev_status=None, stream=None) -> int:
    return int(load().attn_bwd_rect(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                                    _ptr(dv), _ptr(workspace), int(workspace_bytes), int(B), int(H), int(Nq),
                                    int(Nk), int(d), _dt(dt), int(bool(causal)), float(scale), _ptr(dev_status),
                                    _stream(stream)))


def attn_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, B, H, N, d, out_dt, causal, scale,
                 dev_status=None, stream=None) -> int:
    return int(load().attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
                                   _ptr(o), _ptr(lse), int(B), int(H), int(N), int(d), _dt(out_dt),
                                   int(bool(causal)), float(scale), _ptr(dev_status), _stream(stream)))


def attn_fwd_splitkv_workspace_bytes(B, H, N, d, n_splits) -> int:
    return int(load().attn_fwd_splitkv_workspace_bytes(int(B), int(H), int(N), int(d), int(n_splits)))


def attn_fwd_splitkv(q, k, v, o, lse, workspace, workspace_bytes, B, H, N, d, dt, causal, scale, n_splits,
                     dev_status=None, stream=None) -> int:
    return int(load().attn_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(workspace),
                                       int(workspace_bytes), int(B), int(H), int(N), int(d), _dt(dt),
                                       int(bool(causal)), float(scale), int(n_splits), _ptr(dev_status),
                                       _stream(stream)))


def attn_fwd_splitkv_rect(q, k, v, o, lse, workspace, workspace_bytes, B, H, Nq, Nk, d, dt, causal, scale,
                          n_splits, dev_status=None, stream=None) -> int:
    return int(load().attn_fwd_splitkv_rect(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(workspace),
                                            int(workspace_bytes), int(B), int(H), int(Nq), int(Nk), int(d),
                                            _dt(dt), int(bool(causal)), float(scale), int(n_splits),
                                            _ptr(dev_status), _stream(stream)))


def attn_bwd_workspace_bytes(B, H, N, d) -> int:
    return int(load().attn_bwd_workspace_bytes(int(B), int(H), int(N), int(d)))


def attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, d, dt, causal, scale,
             dev_status=None, stream=None) -> int:
    return int(load().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                               _ptr(dv), _ptr(workspace), int(workspace_bytes), int(B), int(H), int(N), int(d),
                               _dt(dt), int(bool(causal)), float(scale), _ptr(dev_status), _stream(stream)))


def attn_bwd_prepare(o, dout, lse, workspace, workspace_bytes, B, H, N, d, dt, stream=None) -> int:
    return int(load().attn_bwd_prepare(_ptr(o), _ptr(dout), _ptr(lse), _ptr(workspace), int(workspace_bytes),
                                       int(B), int(H), int(N), int(d), _dt(dt), _stream(stream)))


def attn_bwd_dkdv(q, k, v, dout, workspace, workspace_bytes, dk, dv, B, H, N, d, dt, causal, scale,
                  dev_status=None, stream=None) -> int:
    return int(load().attn_bwd_dkdv(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(workspace), int(workspace_bytes),
                                    _ptr(dk), _ptr(dv), int(B), int(H), int(N), int(d), _dt(dt),
                                    int(bool(causal)), float(scale), _ptr(dev_status), _stream(stream)))


def attn_bwd_dq(q, k, v, dout, workspace, workspace_bytes, dq, B, H, N, d, dt, causal, scale,
                dev_status=None, stream=None) -> int:
    return int(load().attn_bwd_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(workspace), int(workspace_bytes),
                                  _ptr(dq), int(B), int(H), int(N), int(d), _dt(dt), int(bool(causal)),
                                  float(scale), _ptr(dev_status), _stream(stream)))


def attn_bwd_deterministic_workspace_bytes(B, H, N, d) -> int:
    return int(load().attn_bwd_deterministic_workspace_bytes(int(B), int(H), int(N), int(d)))


def attn_bwd_deterministic(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, d, dt, causal,
                           scale, dev_status=None, stream=None) -> int:
    return int(load().attn_bwd_deterministic(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                                             _ptr(dk), _ptr(dv), _ptr(workspace), int(workspace_bytes), int(B),
                                             int(H), int(N), int(d), _dt(dt), int(bool(causal)), float(scale),
                                             _ptr(dev_status), _stream(stream)))


def attn_bwd_dkdvdq(q, k, v, dout, workspace, workspace_bytes, dk, dv, B, H, N, d, dt, causal, scale,
                    dev_status=None, stream=None) -> int:
    return int(load().attn_bwd_dkdvdq(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(workspace), int(workspace_bytes),
                                      _ptr(dk), _ptr(dv), int(B), int(H), int(N), int(d), _dt(dt),
                                      int(bool(causal)), float(scale), _ptr(dev_status), _stream(stream)))


def attn_bwd_dq_finish(workspace, workspace_bytes, dq, B, H, N, d, dt, scale, stream=None) -> int:
    return int(load().attn_bwd_dq_finish(_ptr(workspace), int(workspace_bytes), _ptr(dq), int(B), int(H), int(N),
                                         int(d), _dt(dt), float(scale), _stream(stream)))


def attn_dropout_bits_bytes(B, H, Nq, Nk) -> int:
    return int(load().attn_dropout_bits_bytes(int(B), int(H), int(Nq), int(Nk)))


def attn_fwd_dropout_bits(q, k, v, o, lse, keep_bits, keep_bits_bytes, B, H, N, d, dt, causal, scale, p_drop, seed,
                          dev_status=None, stream=None) -> int:
    return int(load().attn_fwd_dropout_bits(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(keep_bits),
                                            int(keep_bits_bytes), int(B), int(H), int(N), int(d), _dt(dt),
                                            int(bool(causal)), float(scale), float(p_drop),
                                            int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(dev_status), _stream(stream)))


def attn_bwd_dropout_bits(q, k, v, o, dout, lse, keep_bits, keep_bits_bytes, dq, dk, dv, workspace, workspace_bytes,
                          B, H, N, d, dt, causal, scale, p_drop, dev_status=None, stream=None) -> int:
    return int(load().attn_bwd_dropout_bits(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                                            _ptr(keep_bits), int(keep_bits_bytes), _ptr(dq), _ptr(dk), _ptr(dv),
                                            _ptr(workspace), int(workspace_bytes), int(B), int(H), int(N), int(d),
                                            _dt(dt), int(bool(causal)), float(scale), float(p_drop),
                                            _ptr(dev_status), _stream(stream)))


def attn_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, dt, causal, scale, dev_status=None,
                     stream=None) -> int:
    return int(load().attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                                       _ptr(dk), _ptr(dv), int(B), int(H), int(N), int(d), _dt(dt),
                                       int(bool(causal)), float(scale), _ptr(dev_status), _stream(stream)))


def attn_selftest_bounded_wait(dev_status, limit_ns, stream=None) -> int:
    return int(load().attn_selftest_bounded_wait(_ptr(dev_status), int(limit_ns), _stream(stream)))


# ---------------------------------------------------------------- torch convenience


def _check(t, name):
    import torch

    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dim() == 4):
        raise ValueError(f"{name} must be a CUDA tensor of shape [B, H, N, d]")
    return t.contiguous()


def forward(q, k, v, causal: bool = False, scale=None, dev_status=None, out=None):
    """O = softmax(scale Q K^T) V and the row logsumexp; q: [B, H, Nq, d], k, v: [B, H, Nk, d]
    bf16/fp16 CUDA tensors (Nk != Nq goes through attn_fwd_rect; causal then needs Nk >= Nq)."""
    import torch

    q, k, v = _check(q, "q"), _check(k, "k"), _check(v, "v")
    B, H, N, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != k.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q must be [B, H, Nq, d] and k, v [B, H, Nk, d], all of one dtype")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o, lse = out if out is not None else (torch.empty_like(q), torch.empty((B, H, N), device=q.device,
                                                                            dtype=torch.float32))
    if Nk == N:
        st, name = attn_fwd(q, k, v, o, lse, B, H, N, d, q.dtype, causal, scale, dev_status), "attn_fwd"
    else:
        st, name = attn_fwd_rect(q, k, v, o, lse, B, H, N, Nk, d, q.dtype, causal, scale, dev_status), "attn_fwd_rect"
    if st != ATTN_OK:
        raise AttnError(st, name)
    return o, lse


def forward_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal: bool = False, scale=None, out_dtype=None,
                dev_status=None, out=None):
    """Attention of block-scaled E4M3 inputs: q8, k8, v8 [B, H, N, d] uint8 (or float8_e4m3fn)
    CUDA tensors, scales [B, H, ceil(N/128)] float32 CUDA tensors.  Returns (o, lse), o in
    ``out_dtype`` (bf16 by default)."""
    import torch

    q8, k8, v8 = _check(q8, "q8"), _check(k8, "k8"), _check(v8, "v8")
    B, H, N, d = q8.shape
    if k8.shape != q8.shape or v8.shape != q8.shape or any(t.element_size() != 1 for t in (q8, k8, v8)):
        raise ValueError("q8, k8, v8 must share one shape and hold one byte per element")
    nblk = -(-N // 128)
    scales = []
    for t, n in ((q_scale, "q_scale"), (k_scale, "k_scale"), (v_scale, "v_scale")):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.float32 and t.numel() == B * H * nblk):
            raise ValueError(f"{n} must be a float32 CUDA tensor of {B * H * nblk} scales [B, H, ceil(N/128)]")
        scales.append(t.contiguous())
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out_dtype = torch.bfloat16 if out_dtype is None else out_dtype
    o, lse = out if out is not None else (torch.empty((B, H, N, d), device=q8.device, dtype=out_dtype),
                                          torch.empty((B, H, N), device=q8.device, dtype=torch.float32))
    st = attn_fwd_fp8(q8, k8, v8, *scales, o, lse, B, H, N, d, o.dtype, causal, scale, dev_status)
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_fp8")
    return o, lse


def backward(q, k, v, o, lse, dout, causal: bool = False, scale=None, dev_status=None, workspace=None,
             out=None, deterministic: bool = False):
    """dQ, dK, dV of sum(dout * O) for O = forward(q, k, v); q, o, dout [B, H, Nq, d], k, v
    [B, H, Nk, d] CUDA tensors (Nk != Nq goes through attn_bwd_rect).  ``deterministic``
    selects attn_bwd_deterministic (same bytes on every call; Nk == Nq only)."""
    import torch

    q, k, v, o, dout = (_check(t, n) for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")))
    B, H, N, d = q.shape
    Nk = k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    nbytes = (attn_bwd_deterministic_workspace_bytes if deterministic else attn_bwd_workspace_bytes)(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), device=q.device, dtype=torch.uint8)
    dq, dk, dv = out if out is not None else (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    if deterministic:
        if Nk != N:
            raise ValueError("deterministic backward needs Nk == Nq")
        st = attn_bwd_deterministic(q, k, v, o, dout, lse.contiguous(), dq, dk, dv, workspace, workspace.numel(),
                                    B, H, N, d, q.dtype, causal, scale, dev_status)
        if st != ATTN_OK:
            raise AttnError(st, "attn_bwd_deterministic")
        return dq, dk, dv
    if Nk != N:
        st = attn_bwd_rect(q, k, v, o, dout, lse.contiguous(), dq, dk, dv, workspace, workspace.numel(), B, H, N, Nk,
                           d, q.dtype, causal, scale, dev_status)
        if st != ATTN_OK:
            raise AttnError(st, "attn_bwd_rect")
        return dq, dk, dv
    st = attn_bwd(q, k, v, o, dout, lse.contiguous(), dq, dk, dv, workspace, workspace.numel(), B, H, N, d,
                  q.dtype, causal, scale, dev_status)
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd")
    return dq, dk, dv


# ---------------------------------------------------------------- autograd


def _autograd_function():
    import torch

    class _Attention(torch.autograd.Function):
        """O = softmax(scale Q K^T) V through attn_fwd / attn_fwd_rect / attn_fwd_dropout,
        with the matching backward entry point; argument marshalling only."""

        @staticmethod
        def forward(ctx, q, k, v, causal, scale, dropout_p, seed):
            q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
            B, H, N, d = q.shape
            Nk = k.shape[2]
            o = torch.empty_like(q)
            lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
            if dropout_p > 0:
                if Nk != N:
                    raise ValueError("dropout needs Nq == Nk")
                st, name = attn_fwd_dropout(q, k, v, o, lse, B, H, N, d, q.dtype, causal, scale, dropout_p, seed), \
                    "attn_fwd_dropout"
            elif Nk != N:
                st, name = attn_fwd_rect(q, k, v, o, lse, B, H, N, Nk, d, q.dtype, causal, scale), "attn_fwd_rect"
            else:
                st, name = attn_fwd(q, k, v, o, lse, B, H, N, d, q.dtype, causal, scale), "attn_fwd"
            if st != ATTN_OK:
                raise AttnError(st, name)
            ctx.save_for_backward(q, k, v, o, lse)
            ctx.args = (causal, scale, dropout_p, seed)
            return o

        @staticmethod
        def backward(ctx, do):
            q, k, v, o, lse = ctx.saved_tensors
            causal, scale, dropout_p, seed = ctx.args
            do = do.contiguous()
            B, H, N, d = q.shape
            Nk = k.shape[2]
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            nb = attn_bwd_workspace_bytes(B, H, N, d)
            ws = torch.empty(max(nb, 16), device=q.device, dtype=torch.uint8)
            if dropout_p > 0:
                st, name = attn_bwd_dropout(q, k, v, o, do, lse, dq, dk, dv, ws, ws.numel(), B, H, N, d, q.dtype,
                                            causal, scale, dropout_p, seed), "attn_bwd_dropout"
            elif Nk != N:
                st, name = attn_bwd_rect(q, k, v, o, do, lse, dq, dk, dv, ws, ws.numel(), B, H, N, Nk, d, q.dtype,
                                         causal, scale), "attn_bwd_rect"
            else:
                st, name = attn_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, ws.numel(), B, H, N, d, q.dtype, causal,
                                    scale), "attn_bwd"
            if st != ATTN_OK:
                raise AttnError(st, name)
            return dq, dk, dv, None, None, None, None

    return _Attention


_ATTN_FN = None


def attention(q, k, v, causal: bool = False, scale=None, dropout_p: float = 0.0, seed: int = 0):
    """Differentiable attention on [B, H, N, d] bf16/fp16 CUDA tensors (k, v may have their
    own length Nk; dropout needs Nk == Nq): the forward and backward of this library behind a
    torch.autograd.Function.  Pass a fresh ``seed`` per call when dropout_p > 0."""
    global _ATTN_FN
    if _ATTN_FN is None:
        _ATTN_FN = _autograd_function()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else float(scale)
    return _ATTN_FN.apply(q, k, v, bool(causal), scale, float(dropout_p), int(seed))
