"""The C ABI without a GPU: the library builds for sm_103a, loads, exports every
entry point include/attn.h declares, and rejects bad arguments before it touches
CUDA."""
import ctypes
import os
import re

import pytest

import tiled_online_softmax_attention_gb300 as attn

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "attn.h")


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    assert declared_functions() == sorted(attn.EXPORTS)


def test_library_loads_and_exports_every_symbol():
    lib = attn.load()
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_library_exports_nothing_else():
    out = os.popen(f"nm -D --defined-only {attn.LIB_PATH}").read()
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert {s for s in exported if s.startswith("attn_")} == set(attn.EXPORTS)


def test_status_strings():
    assert attn.attn_status_string(0) == "ATTN_OK"
    assert attn.attn_status_string(4) == "ATTN_ERR_TIMEOUT"
    assert attn.attn_status_string(99) == "ATTN_ERR_UNKNOWN"


def test_workspace_size():
    # two float32 values per padded row, plus d float32 dQ-accumulator values for d <= 128
    assert attn.attn_bwd_workspace_bytes(2, 16, 8192, 128) == (2 + 128) * 32 * 8192 * 4
    assert attn.attn_bwd_workspace_bytes(2, 8, 4097, 128) == (2 + 128) * 16 * 4224 * 4
    assert attn.attn_bwd_workspace_bytes(1, 1, 1, 64) == (2 + 64) * 128 * 4
    assert attn.attn_bwd_workspace_bytes(1, 1, 0, 64) == 0
    assert attn.attn_bwd_workspace_bytes(1, 1, 16, 96) == 0
    assert attn.attn_bwd_workspace_bytes(1, 2, 300, 256) == 2 * 2 * 384 * 4
    assert attn.attn_bwd_deterministic_workspace_bytes(2, 16, 8192, 128) == 2 * 32 * 8192 * 4
    assert attn.attn_bwd_deterministic_workspace_bytes(2, 8, 4097, 64) == 2 * 16 * 4224 * 4
    assert attn.attn_bwd_deterministic_workspace_bytes(1, 2, 300, 256) == 2 * 2 * 384 * 4
    assert attn.attn_bwd_deterministic_workspace_bytes(1, 1, 16, 96) == 0


# fake, aligned, non-overlapping "device" addresses: validation fails before any CUDA call
A = [0x10000000 * (i + 1) for i in range(12)]


def fwd(**kw):
    args = dict(q=A[0], k=A[1], v=A[2], o=A[3], lse=A[4], B=1, H=2, N=256, d=128, dt=0, causal=0, scale=0.088, stream=0)
    args.update(kw)
    return attn.attn_fwd(**args)


def bwd(**kw):
    args = dict(q=A[0], k=A[1], v=A[2], o=A[3], dout=A[4], lse=A[5], dq=A[6], dk=A[7], dv=A[8],
                workspace=A[9], workspace_bytes=1 << 20, B=1, H=2, N=256, d=128, dt=0, causal=1, scale=0.088, stream=0)
    args.update(kw)
    return attn.attn_bwd(**args)


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(o=A[3] + 8), attn.ATTN_ERR_INVALID_ARG),          # misaligned
    (dict(lse=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(N=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(B=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(d=192), attn.ATTN_ERR_UNSUPPORTED),
    (dict(d=512), attn.ATTN_ERR_UNSUPPORTED),
    (dict(dt=7), attn.ATTN_ERR_UNSUPPORTED),
    (dict(scale=0.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), attn.ATTN_ERR_INVALID_ARG),
    (dict(o=A[0]), attn.ATTN_ERR_INVALID_ARG),               # output aliases an input
    (dict(B=1 << 12, H=1 << 12, N=1 << 8), attn.ATTN_ERR_INVALID_ARG),  # > 2^31 elements
])
def test_fwd_rejects(kw, status):
    assert fwd(**kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(dq=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(workspace=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(workspace_bytes=2 * 2 * 256 * 4 - 4), attn.ATTN_ERR_INVALID_ARG),
    (dict(workspace_bytes=(2 + 128) * 2 * 256 * 4 - 4), attn.ATTN_ERR_INVALID_ARG),  # no room for the dQ accumulator
    (dict(dq=A[9] + 2 * 2 * 256 * 4), attn.ATTN_ERR_INVALID_ARG),  # dq inside the dQ accumulator
    (dict(dk=A[6]), attn.ATTN_ERR_INVALID_ARG),              # two outputs alias
    (dict(dv=A[2]), attn.ATTN_ERR_INVALID_ARG),              # output aliases an input
    (dict(workspace=A[0]), attn.ATTN_ERR_INVALID_ARG),       # workspace aliases an input
    (dict(d=32), attn.ATTN_ERR_UNSUPPORTED),
    (dict(d=192), attn.ATTN_ERR_UNSUPPORTED),
    (dict(d=256, workspace_bytes=16), attn.ATTN_ERR_INVALID_ARG),  # 256 passes the d check
    (dict(scale=-1.0), attn.ATTN_ERR_INVALID_ARG),
])
def test_bwd_rejects(kw, status):
    assert bwd(**kw) == status


def test_deterministic_and_fused_stages_validate():
    det = dict(q=A[0], k=A[1], v=A[2], o=A[3], dout=A[4], lse=A[5], dq=A[6], dk=A[7], dv=A[8], workspace=A[9],
               workspace_bytes=2 * 2 * 256 * 4 - 4, B=1, H=2, N=256, d=128, dt=0, causal=1, scale=0.088, stream=0)
    assert attn.attn_bwd_deterministic(**det) == attn.ATTN_ERR_INVALID_ARG           # workspace one value short
    assert attn.attn_bwd_deterministic(**dict(det, workspace_bytes=1 << 20, dk=A[6])) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_bwd_deterministic(**dict(det, workspace_bytes=1 << 20, d=80)) == attn.ATTN_ERR_UNSUPPORTED
    full = attn.attn_bwd_workspace_bytes(1, 2, 256, 128)
    assert attn.attn_bwd_dkdvdq(A[0], A[1], A[2], A[4], A[9], full - 4, A[7], A[8], 1, 2, 256, 128, 0, 1, 0.1,
                                stream=0) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_bwd_dkdvdq(A[0], A[1], A[2], A[4], A[9], full, A[7], A[7], 1, 2, 256, 128, 0, 1, 0.1,
                                stream=0) == attn.ATTN_ERR_INVALID_ARG                # dk == dv
    assert attn.attn_bwd_dkdvdq(A[0], A[1], A[2], A[4], A[9], 1 << 24, A[7], A[8], 1, 2, 256, 256, 0, 1, 0.1,
                                stream=0) == attn.ATTN_ERR_UNSUPPORTED                # no fused path at d = 256
    assert attn.attn_bwd_dq_finish(A[9], full - 4, A[6], 1, 2, 256, 128, 0, 0.1, stream=0) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_bwd_dq_finish(A[9], full, A[9] + 64, 1, 2, 256, 128, 0, 0.1,
                                   stream=0) == attn.ATTN_ERR_INVALID_ARG             # dq inside the workspace
    assert attn.attn_bwd_dq_finish(A[9], full, A[6], 1, 2, 256, 128, 0, 0.0, stream=0) == attn.ATTN_ERR_INVALID_ARG


def test_selftest_needs_status_pointer():
    assert attn.attn_selftest_bounded_wait(None, 1000, stream=0) == attn.ATTN_ERR_INVALID_ARG


def test_stage_entry_points_validate():
    assert attn.attn_bwd_prepare(A[3], A[4], A[5], A[9], 16, 1, 2, 256, 128, 0, stream=0) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_bwd_prepare(A[3], A[4], None, A[9], 1 << 20, 1, 2, 256, 128, 0, stream=0) == \
        attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_bwd_dkdv(A[0], A[1], A[2], A[4], A[9], 1 << 20, A[7], A[7], 1, 2, 256, 128, 0, 1, 0.1,
                              stream=0) == attn.ATTN_ERR_INVALID_ARG      # dk == dv
    assert attn.attn_bwd_dq(A[0], A[1], A[2], A[4], A[9], 1 << 20, A[6], 1, 2, 256, 80, 0, 1, 0.1,
                            stream=0) == attn.ATTN_ERR_UNSUPPORTED


def test_splitkv_validates():
    assert attn.attn_fwd_splitkv_workspace_bytes(1, 2, 256, 128, 4) == 4 * 2 * 256 * 129 * 4
    assert attn.attn_fwd_splitkv_workspace_bytes(1, 2, 256, 256, 4) == 4 * 2 * 256 * 257 * 4
    assert attn.attn_fwd_splitkv_workspace_bytes(1, 2, 256, 192, 4) == 0
    assert attn.attn_fwd_splitkv_workspace_bytes(1, 2, 256, 128, 0) == 0
    assert attn.attn_fwd_splitkv_workspace_bytes(1, 2, 256, 128, 65) == 0
    args = dict(q=A[0], k=A[1], v=A[2], o=A[3], lse=A[4], workspace=A[9], workspace_bytes=1 << 24, B=1, H=2,
                N=256, d=128, dt=0, causal=1, scale=0.088, n_splits=4, stream=0)
    for kw, st in [(dict(n_splits=0), attn.ATTN_ERR_INVALID_ARG), (dict(n_splits=65), attn.ATTN_ERR_INVALID_ARG),
                   (dict(workspace_bytes=100), attn.ATTN_ERR_INVALID_ARG), (dict(workspace=A[0]), attn.ATTN_ERR_INVALID_ARG),
                   (dict(workspace=0), attn.ATTN_ERR_INVALID_ARG), (dict(d=80), attn.ATTN_ERR_UNSUPPORTED),
                   (dict(d=256, workspace_bytes=100), attn.ATTN_ERR_INVALID_ARG)]:  # 256 passes the d check
        a2 = dict(args)
        a2.update(kw)
        assert attn.attn_fwd_splitkv(**a2) == st, kw


def test_splitkv_rect_validates():
    args = dict(q=A[0], k=A[1], v=A[2], o=A[3], lse=A[4], workspace=A[9], workspace_bytes=1 << 24, B=1, H=2,
                Nq=128, Nk=4096, d=128, dt=0, causal=1, scale=0.088, n_splits=4, stream=0)
    for kw, st in [(dict(Nq=600, Nk=500), attn.ATTN_ERR_INVALID_ARG),       # causal needs Nk >= Nq
                   (dict(n_splits=0), attn.ATTN_ERR_INVALID_ARG), (dict(d=192), attn.ATTN_ERR_UNSUPPORTED),
                   (dict(o=A[1] + 128 * 128 * 2 * 2), attn.ATTN_ERR_INVALID_ARG),  # o inside k (Nk rows)
                   (dict(workspace_bytes=4 * 2 * 128 * 129 * 4 - 4), attn.ATTN_ERR_INVALID_ARG),  # sized by Nq
                   (dict(Nk=0), attn.ATTN_ERR_INVALID_ARG)]:
        a2 = dict(args)
        a2.update(kw)
        assert attn.attn_fwd_splitkv_rect(**a2) == st, kw


def fwd_fp8(**kw):
    args = dict(q8=A[0], k8=A[1], v8=A[2], q_scale=A[5], k_scale=A[6], v_scale=A[7], o=A[3], lse=A[4], B=1, H=2,
                N=256, d=128, out_dt=0, causal=0, scale=0.088, stream=0)
    args.update(kw)
    return attn.attn_fwd_fp8(**args)


@pytest.mark.parametrize("kw,status", [
    (dict(q8=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(v8=A[2] + 4), attn.ATTN_ERR_INVALID_ARG),          # misaligned codes
    (dict(k_scale=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(v_scale=A[7] + 2), attn.ATTN_ERR_INVALID_ARG),     # misaligned scales
    (dict(d=64), attn.ATTN_ERR_UNSUPPORTED),                 # E4M3 inputs: d = 128 only
    (dict(out_dt=5), attn.ATTN_ERR_UNSUPPORTED),
    (dict(N=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), attn.ATTN_ERR_INVALID_ARG),
    (dict(o=A[1]), attn.ATTN_ERR_INVALID_ARG),               # output aliases an input
    (dict(q_scale=A[4] + 16), attn.ATTN_ERR_INVALID_ARG),    # scales inside lse
])
def test_fwd_fp8_rejects(kw, status):
    assert fwd_fp8(**kw) == status


def test_rect_validates():
    fa = dict(q=A[0], k=A[1], v=A[2], o=A[3], lse=A[4], B=1, H=2, Nq=256, Nk=512, d=128, dt=0, causal=1,
              scale=0.088, stream=0)
    for kw, st in [(dict(Nq=600), attn.ATTN_ERR_INVALID_ARG),        # causal needs Nk >= Nq
                   (dict(Nk=0), attn.ATTN_ERR_INVALID_ARG), (dict(d=96), attn.ATTN_ERR_UNSUPPORTED),
                   (dict(o=A[1] + 256 * 128 * 2 * 2), attn.ATTN_ERR_INVALID_ARG)]:  # o inside k (Nk rows)
        a2 = dict(fa)
        a2.update(kw)
        assert attn.attn_fwd_rect(**a2) == st, kw
    ba = dict(q=A[0], k=A[1], v=A[2], o=A[3], dout=A[4], lse=A[5], dq=A[6], dk=A[7], dv=A[8], workspace=A[9],
              workspace_bytes=1 << 20, B=1, H=2, Nq=256, Nk=512, d=128, dt=0, causal=1, scale=0.088, stream=0)
    for kw, st in [(dict(Nq=600), attn.ATTN_ERR_INVALID_ARG), (dict(d=192), attn.ATTN_ERR_UNSUPPORTED),
                   (dict(d=256, workspace_bytes=16), attn.ATTN_ERR_INVALID_ARG),
                   (dict(dk=A[7], dv=A[7] + 512 * 128 * 2), attn.ATTN_ERR_INVALID_ARG),  # dv inside dk's Nk rows
                   (dict(workspace_bytes=16), attn.ATTN_ERR_INVALID_ARG)]:
        a2 = dict(ba)
        a2.update(kw)
        assert attn.attn_bwd_rect(**a2) == st, kw


def test_dropout_validates():
    fa = dict(q=A[0], k=A[1], v=A[2], o=A[3], lse=A[4], B=1, H=2, N=256, d=128, dt=0, causal=1, scale=0.088,
              p_drop=0.1, seed=7, stream=0)
    for kw, st in [(dict(p_drop=1.0), attn.ATTN_ERR_INVALID_ARG), (dict(p_drop=-0.1), attn.ATTN_ERR_INVALID_ARG),
                   (dict(p_drop=float("nan")), attn.ATTN_ERR_INVALID_ARG),
                   (dict(p_drop=0.999), attn.ATTN_ERR_INVALID_ARG),      # round(256 p) = 256
                   (dict(d=192), attn.ATTN_ERR_UNSUPPORTED), (dict(d=96), attn.ATTN_ERR_UNSUPPORTED),
                   (dict(o=A[0]), attn.ATTN_ERR_INVALID_ARG)]:
        a2 = dict(fa)
        a2.update(kw)
        assert attn.attn_fwd_dropout(**a2) == st, kw
    ba = dict(q=A[0], k=A[1], v=A[2], o=A[3], dout=A[4], lse=A[5], dq=A[6], dk=A[7], dv=A[8], workspace=A[9],
              workspace_bytes=1 << 20, B=1, H=2, N=256, d=128, dt=0, causal=1, scale=0.088, p_drop=0.1, seed=7,
              stream=0)
    for kw, st in [(dict(p_drop=1.5), attn.ATTN_ERR_INVALID_ARG), (dict(d=192), attn.ATTN_ERR_UNSUPPORTED),
                   (dict(dq=A[7]), attn.ATTN_ERR_INVALID_ARG)]:
        a2 = dict(ba)
        a2.update(kw)
        assert attn.attn_bwd_dropout(**a2) == st, kw


def test_varlen_validates():
    fa = dict(q=A[0], k=A[1], v=A[2], o=A[3], lse=A[4], cu_q=A[5], cu_k=A[6], B=3, H=2, max_q=300, max_k=300,
              Tq=600, Tk=600, d=128, dt=0, causal=1, scale=0.088, stream=0)
    for kw, st in [(dict(B=0), attn.ATTN_ERR_INVALID_ARG), (dict(Tk=0), attn.ATTN_ERR_INVALID_ARG),
                   (dict(cu_q=A[5] + 2), attn.ATTN_ERR_INVALID_ARG), (dict(cu_k=0), attn.ATTN_ERR_INVALID_ARG),
                   (dict(d=192), attn.ATTN_ERR_UNSUPPORTED), (dict(o=A[0]), attn.ATTN_ERR_INVALID_ARG),
                   (dict(lse=A[3] + 16), attn.ATTN_ERR_INVALID_ARG)]:
        a2 = dict(fa)
        a2.update(kw)
        assert attn.attn_fwd_varlen(**a2) == st, kw
    ba = dict(q=A[0], k=A[1], v=A[2], o=A[3], dout=A[4], lse=A[5], dq=A[6], dk=A[7], dv=A[8], workspace=A[9],
              workspace_bytes=1 << 20, cu_q=A[10], cu_k=A[11], B=3, H=2, max_q=300, max_k=300, Tq=600, Tk=600, d=128,
              dt=0, causal=1, scale=0.088, stream=0)
    for kw, st in [(dict(workspace_bytes=100), attn.ATTN_ERR_INVALID_ARG), (dict(dq=A[7]), attn.ATTN_ERR_INVALID_ARG),
                   (dict(workspace=A[0]), attn.ATTN_ERR_INVALID_ARG), (dict(d=96), attn.ATTN_ERR_UNSUPPORTED)]:
        a2 = dict(ba)
        a2.update(kw)
        assert attn.attn_bwd_varlen(**a2) == st, kw


def test_varlen_splitkv_validates():
    assert attn.attn_fwd_varlen_splitkv_workspace_bytes(2, 600, 128, 4) == 4 * 600 * 2 * 129 * 4
    assert attn.attn_fwd_varlen_splitkv_workspace_bytes(2, 600, 256, 1) == 600 * 2 * 257 * 4
    assert attn.attn_fwd_varlen_splitkv_workspace_bytes(2, 600, 96, 4) == 0
    assert attn.attn_fwd_varlen_splitkv_workspace_bytes(2, 600, 128, 65) == 0
    fa = dict(q=A[0], k=A[1], v=A[2], o=A[3], lse=A[4], workspace=A[9], workspace_bytes=1 << 24, cu_q=A[5], cu_k=A[6],
              B=3, H=2, max_q=300, max_k=300, Tq=600, Tk=600, d=128, dt=0, causal=1, scale=0.088, n_splits=4,
              stream=0)
    for kw, st in [(dict(n_splits=0), attn.ATTN_ERR_INVALID_ARG), (dict(n_splits=65), attn.ATTN_ERR_INVALID_ARG),
                   (dict(workspace_bytes=100), attn.ATTN_ERR_INVALID_ARG), (dict(workspace=A[0]), attn.ATTN_ERR_INVALID_ARG),
                   (dict(workspace=0), attn.ATTN_ERR_INVALID_ARG), (dict(d=192), attn.ATTN_ERR_UNSUPPORTED),
                   (dict(B=0), attn.ATTN_ERR_INVALID_ARG)]:
        a2 = dict(fa)
        a2.update(kw)
        assert attn.attn_fwd_varlen_splitkv(**a2) == st, kw


def test_rect_dropout_validates():
    fa = dict(q=A[0], k=A[1], v=A[2], o=A[3], lse=A[4], B=1, H=2, Nq=256, Nk=512, d=128, dt=0, causal=1,
              scale=0.088, p_drop=0.1, seed=3, stream=0)
    for kw, st in [(dict(Nq=600), attn.ATTN_ERR_INVALID_ARG), (dict(p_drop=2.0), attn.ATTN_ERR_INVALID_ARG),
                   (dict(d=96), attn.ATTN_ERR_UNSUPPORTED), (dict(o=A[1] + 256 * 128 * 2 * 2), attn.ATTN_ERR_INVALID_ARG)]:
        a2 = dict(fa)
        a2.update(kw)
        assert attn.attn_fwd_rect_dropout(**a2) == st, kw
    ba = dict(q=A[0], k=A[1], v=A[2], o=A[3], dout=A[4], lse=A[5], dq=A[6], dk=A[7], dv=A[8], workspace=A[9],
              workspace_bytes=1 << 20, B=1, H=2, Nq=256, Nk=512, d=128, dt=0, causal=1, scale=0.088, p_drop=0.1,
              seed=3, stream=0)
    for kw, st in [(dict(Nq=600), attn.ATTN_ERR_INVALID_ARG), (dict(p_drop=-1.0), attn.ATTN_ERR_INVALID_ARG),
                   (dict(d=192), attn.ATTN_ERR_UNSUPPORTED), (dict(workspace_bytes=16), attn.ATTN_ERR_INVALID_ARG)]:
        a2 = dict(ba)
        a2.update(kw)
        assert attn.attn_bwd_rect_dropout(**a2) == st, kw


def test_varlen_dropout_validates():
    fa = dict(q=A[0], k=A[1], v=A[2], o=A[3], lse=A[4], cu_q=A[5], cu_k=A[6], B=3, H=2, max_q=300, max_k=300,
              Tq=600, Tk=600, d=128, dt=0, causal=1, scale=0.088, p_drop=0.1, seed=7, stream=0)
    for kw, st in [(dict(p_drop=1.0), attn.ATTN_ERR_INVALID_ARG), (dict(p_drop=float("nan")), attn.ATTN_ERR_INVALID_ARG),
                   (dict(B=0), attn.ATTN_ERR_INVALID_ARG), (dict(d=192), attn.ATTN_ERR_UNSUPPORTED),
                   (dict(o=A[0]), attn.ATTN_ERR_INVALID_ARG)]:
        a2 = dict(fa)
        a2.update(kw)
        assert attn.attn_fwd_varlen_dropout(**a2) == st, kw
    ba = dict(q=A[0], k=A[1], v=A[2], o=A[3], dout=A[4], lse=A[5], dq=A[6], dk=A[7], dv=A[8], workspace=A[9],
              workspace_bytes=1 << 20, cu_q=A[10], cu_k=A[11], B=3, H=2, max_q=300, max_k=300, Tq=600, Tk=600, d=128,
              dt=0, causal=1, scale=0.088, p_drop=0.1, seed=7, stream=0)
    for kw, st in [(dict(p_drop=-0.5), attn.ATTN_ERR_INVALID_ARG), (dict(workspace_bytes=100), attn.ATTN_ERR_INVALID_ARG),
                   (dict(dq=A[7]), attn.ATTN_ERR_INVALID_ARG), (dict(d=96), attn.ATTN_ERR_UNSUPPORTED)]:
        a2 = dict(ba)
        a2.update(kw)
        assert attn.attn_bwd_varlen_dropout(**a2) == st, kw


def test_dropout_bits_validate():
    assert attn.attn_dropout_bits_bytes(2, 16, 8192, 8192) == 2 * 16 * 64 * 4 * 8192 * 4
    assert attn.attn_dropout_bits_bytes(1, 1, 300, 129) == 2 * 4 * 384 * 4
    assert attn.attn_dropout_bits_bytes(1, 1, 0, 128) == 0
    nbits = attn.attn_dropout_bits_bytes(1, 2, 256, 256)
    f = dict(q=A[0], k=A[1], v=A[2], o=A[3], lse=A[4], keep_bits=A[10], keep_bits_bytes=nbits, B=1, H=2, N=256, d=128,
             dt=0, causal=1, scale=0.088, p_drop=0.1, seed=7, stream=0)
    for kw, st in [(dict(p_drop=0.0), attn.ATTN_ERR_INVALID_ARG),        # nothing dropped: no bits to store
                   (dict(p_drop=1.0), attn.ATTN_ERR_INVALID_ARG),
                   (dict(keep_bits_bytes=nbits - 4), attn.ATTN_ERR_INVALID_ARG),
                   (dict(keep_bits=A[10] + 4), attn.ATTN_ERR_INVALID_ARG),
                   (dict(keep_bits=A[3]), attn.ATTN_ERR_INVALID_ARG),     # the bits over o
                   (dict(d=256), attn.ATTN_ERR_UNSUPPORTED)]:
        assert attn.attn_fwd_dropout_bits(**dict(f, **kw)) == st, kw
    b = dict(q=A[0], k=A[1], v=A[2], o=A[3], dout=A[4], lse=A[5], keep_bits=A[10], keep_bits_bytes=nbits, dq=A[6],
             dk=A[7], dv=A[8], workspace=A[9], workspace_bytes=1 << 22, B=1, H=2, N=256, d=128, dt=0, causal=1,
             scale=0.088, p_drop=0.1, stream=0)
    for kw, st in [(dict(p_drop=0.001), attn.ATTN_ERR_INVALID_ARG),
                   (dict(keep_bits_bytes=16), attn.ATTN_ERR_INVALID_ARG),
                   (dict(keep_bits=A[6]), attn.ATTN_ERR_INVALID_ARG),     # the bits over dq
                   (dict(d=256), attn.ATTN_ERR_UNSUPPORTED),
                   (dict(dk=A[6]), attn.ATTN_ERR_INVALID_ARG)]:
        assert attn.attn_bwd_dropout_bits(**dict(b, **kw)) == st, kw
