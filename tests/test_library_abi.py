"""The C-ABI library on the host: it builds, loads, exports every function include/sa2.h
declares, and rejects bad arguments before touching the GPU (no compute calls here)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sa2.h")

OK, INVALID, UNSUPPORTED, ALIGN, WORKSPACE = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def lib():
    from block_sparse_attention_sa2_gb300 import build_lib, sa2
    if not build_lib.up_to_date():
        build_lib.build()
    return sa2.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sa2_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert {"sa2_build_mask", "sa2_attn_fwd", "sa2_attn_bwd", "sa2_attn_bwd_with_fwd_ws", "sa2_build_mask_noalloc",
            "sa2_vd_loss"} <= set(names)
    from block_sparse_attention_sa2_gb300.sa2 import LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (sa2_\w+)", out))
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n), n


def _shape(sa2, **kw):
    base = dict(B=1, H=2, N=1000, d=128, bq=128, bk=64, dtype=0, reserved=0, stride_b=2 * 1000 * 128,
                stride_h=1000 * 128, stride_n=128)
    base.update(kw)
    return sa2.Shape(*[base[f] for f, _ in sa2.Shape._fields_])


def test_version_and_status_strings(lib):
    assert lib.sa2_version() >= 100
    for code in range(9):
        assert lib.sa2_status_string(code)
    assert b"unknown" in lib.sa2_status_string(99)


def test_workspace_sizes_cover_their_buffers(lib):
    from block_sparse_attention_sa2_gb300 import sa2
    s = _shape(sa2)
    Tq, Tk, B, H, N, d = 8, 16, 1, 2, 1000, 128
    mws = lib.sa2_mask_workspace_size(ctypes.byref(s))
    assert mws >= 4 * B * H * d * (Tq + Tk) + B * H * Tq * Tk
    fws = lib.sa2_fwd_workspace_size(ctypes.byref(s))
    assert fws >= 2 * B * H * N * d  # fp16 copy of V
    bws = lib.sa2_bwd_workspace_size(ctypes.byref(s))
    Tp = (Tk + 1) // 2
    stats = 4 * B * H * Tq * 128 * 2  # two floats per row of the 64-row sub-tiles (bq = 128)
    assert bws >= stats + 4 * B * H * Tp * (1 + Tq) + 4 * 2 * B * H * N * d  # + pair lists, fp16 copies
    f32 = _shape(sa2, dtype=1, stride_b=2 * 1000 * 128, stride_h=1000 * 128)
    assert lib.sa2_fwd_workspace_size(ctypes.byref(f32)) >= 3 * 2 * B * H * N * d
    bad = _shape(sa2, d=96)
    assert lib.sa2_mask_workspace_size(ctypes.byref(bad)) == 0


def test_arguments_are_rejected_before_any_launch(lib):
    from block_sparse_attention_sa2_gb300 import sa2
    M = sa2.BlockMaskStruct
    m = M(16, 16, 16, 16, 16, None)
    good = _shape(sa2)
    P = 256  # a fake, aligned device pointer: never dereferenced on these paths
    mask = lambda sh, q=P, k=P, tk=0.1, tp=0.5, mm=m: lib.sa2_build_mask(  # noqa: E731
        ctypes.byref(sh), q, k, tk, tp, ctypes.byref(mm), P, 1 << 30, None)
    assert mask(_shape(sa2, d=96)) == UNSUPPORTED
    assert mask(_shape(sa2, bk=128)) == UNSUPPORTED
    assert mask(_shape(sa2, dtype=7)) == UNSUPPORTED
    assert mask(_shape(sa2, N=0)) == INVALID
    assert mask(_shape(sa2, reserved=1)) == INVALID
    assert mask(_shape(sa2, stride_n=100)) == INVALID
    assert mask(_shape(sa2, stride_n=132)) == ALIGN  # 264-byte rows
    assert mask(good, q=None) == INVALID
    assert mask(good, tk=1.5) == INVALID
    assert mask(good, tp=float("nan")) == INVALID
    assert mask(good, q=P + 8) == ALIGN
    assert mask(good, mm=M(16, None, 16, 16, 16, None)) == INVALID
    assert lib.sa2_build_mask(ctypes.byref(good), P, P, 0.1, 0.5, ctypes.byref(m), P, 16, None) == WORKSPACE
    assert lib.sa2_build_mask(ctypes.byref(_shape(sa2, N=64 * 8000)), P, P, 0.1, 0.5, ctypes.byref(m), P, 1 << 40,
                              None) == UNSUPPORTED  # Tk > 7680
    # forward / backward
    fwd = lambda sh, o=P, ws=P, wsb=1 << 40: lib.sa2_attn_fwd(  # noqa: E731
        ctypes.byref(sh), P, P, P, ctypes.byref(m), 0.0, o, None, P, ws, wsb, None)
    assert fwd(_shape(sa2, d=80)) == UNSUPPORTED
    assert fwd(good, o=None) == INVALID
    assert fwd(good, o=P + 4) == ALIGN
    assert fwd(good, wsb=8) == WORKSPACE
    assert lib.sa2_attn_fwd(ctypes.byref(good), P, P, P, ctypes.byref(m), float("inf"), P, None, P, P, 1 << 40,
                            None) == INVALID
    bwd = lambda sh, dq=P, wsb=1 << 40: lib.sa2_attn_bwd(  # noqa: E731
        ctypes.byref(sh), P, P, P, P, None, P, P, ctypes.byref(m), 0.0, dq, P, P, P, wsb, None)
    assert bwd(_shape(sa2, bq=32)) == UNSUPPORTED
    assert bwd(good, dq=None) == INVALID
    assert bwd(good, wsb=1024) == WORKSPACE
    assert lib.sa2_attn_bwd(ctypes.byref(good), P, P, P, P, None, P, P, ctypes.byref(M(16, 16, None, 16, 16, None)),
                            0.0, P, P, P, P, 1 << 40, None) == INVALID
    # backward taking the forward's workspace
    bwdf = lambda sh, fws=P, fwsb=1 << 40, wsb=1 << 40: lib.sa2_attn_bwd_with_fwd_ws(  # noqa: E731
        ctypes.byref(sh), P, P, P, P, None, P, P, ctypes.byref(m), 0.0, P, P, P, P, wsb, fws, fwsb, None)
    assert bwdf(_shape(sa2, bq=32)) == UNSUPPORTED
    assert bwdf(good, fws=None) == INVALID
    assert bwdf(good, fws=P + 8) == ALIGN
    assert bwdf(good, fwsb=lib.sa2_fwd_workspace_size(ctypes.byref(good)) - 1) == WORKSPACE
    assert bwdf(good, wsb=1024) == WORKSPACE


def test_noalloc_rejects_oversized_shapes_on_the_host(lib):
    from block_sparse_attention_sa2_gb300 import sa2
    lib.sa2_build_mask_noalloc.restype = ctypes.c_int
    m = sa2.BlockMaskStruct(16, 16, 16, 16, 16, None)
    big = _shape(sa2, H=40, N=75600, stride_b=40 * 75600 * 128, stride_h=75600 * 128)
    assert lib.sa2_build_mask_noalloc(ctypes.byref(big), 256, 256, ctypes.c_float(0.1), ctypes.c_float(0.5),
                                      ctypes.byref(m), None) == WORKSPACE
    # the lists are required (the u8 mask and P-bar are optional outputs)
    no_cols = sa2.BlockMaskStruct(16, 16, None, 16, None, None)
    assert lib.sa2_build_mask_noalloc(ctypes.byref(_shape(sa2)), 256, 256, ctypes.c_float(0.1), ctypes.c_float(0.5),
                                      ctypes.byref(no_cols), None) == INVALID


def test_profiler_size_query_needs_no_gpu(lib):
    lib.sa2_profiler_enable(0)
    assert lib.sa2_profiler_collect(None, 0) == 12


def test_vd_loss_rejects_bad_arguments_before_any_launch(lib):
    from block_sparse_attention_sa2_gb300 import sa2
    good = _shape(sa2)
    P = 256
    lib.sa2_vd_loss.restype = ctypes.c_int
    call = lambda sh, os=P, os_lo=None, ot_lo=None, do=P, loss=P, wsb=1 << 20: lib.sa2_vd_loss(  # noqa: E731
        ctypes.byref(sh), ctypes.c_void_p(os), ctypes.c_void_p(os_lo), ctypes.c_void_p(P), ctypes.c_void_p(ot_lo),
        ctypes.c_void_p(do), ctypes.c_void_p(loss), ctypes.c_void_p(P), ctypes.c_size_t(wsb), None)
    assert lib.sa2_vd_loss_workspace_size(ctypes.byref(good)) >= 8 * 152
    assert call(_shape(sa2, d=80)) == UNSUPPORTED
    assert call(good, os=None) == INVALID
    assert call(good, loss=None) == INVALID
    assert call(good, os_lo=P) == INVALID  # one residual without the other
    assert call(good, do=P + 8) == ALIGN
    assert call(good, loss=P + 4) == ALIGN
    assert call(good, wsb=8) == WORKSPACE
