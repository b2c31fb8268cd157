"""Thin Python binding of libsa2 (include/sa2.h): argument marshalling only.

Every step of the hot path runs in the library's CUDA kernels; this module allocates the
output tensors and workspaces with PyTorch, passes raw device pointers and the current CUDA
stream through ctypes, and turns status codes into exceptions.  It fails loudly when the
library is missing.  Names follow the C ABI: ``build_mask``, ``attn_fwd``, ``attn_bwd``.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsa2.so")

SA2_BF16, SA2_FP32 = 0, 1
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "alignment", 4: "workspace", 5: "cuda",
          6: "device timeout", 7: "device bounds", 8: "input beyond fp16 range"}


class Sa2Error(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: status {code} ({STATUS.get(code, 'unknown')})")
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("N", ctypes.c_int32), ("d", ctypes.c_int32),
                ("bq", ctypes.c_int32), ("bk", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("stride_b", ctypes.c_int64), ("stride_h", ctypes.c_int64),
                ("stride_n", ctypes.c_int64)]


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_int), ("total_ms", ctypes.c_double)]


class BlockMaskStruct(ctypes.Structure):
    _fields_ = [("row_cnt", ctypes.c_void_p), ("row_idx", ctypes.c_void_p), ("col_cnt", ctypes.c_void_p),
                ("col_idx", ctypes.c_void_p), ("mask", ctypes.c_void_p), ("pooled_p", ctypes.c_void_p)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libsa2.so (built by ``build_lib.build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libsa2.so not found at {path}: run block_sparse_attention_sa2_gb300.build_lib.build()")
    lib = ctypes.CDLL(path)
    P, S, F, Z = ctypes.c_void_p, ctypes.POINTER(Shape), ctypes.c_float, ctypes.c_size_t
    M = ctypes.POINTER(BlockMaskStruct)
    lib.sa2_version.restype = ctypes.c_int
    lib.sa2_status_string.restype = ctypes.c_char_p
    lib.sa2_status_string.argtypes = [ctypes.c_int]
    for fn in ("sa2_mask_workspace_size", "sa2_fwd_workspace_size", "sa2_bwd_workspace_size"):
        getattr(lib, fn).restype = Z
        getattr(lib, fn).argtypes = [S]
    lib.sa2_build_mask.restype = ctypes.c_int
    lib.sa2_build_mask.argtypes = [S, P, P, F, F, M, P, Z, P]
    lib.sa2_attn_fwd.restype = ctypes.c_int
    lib.sa2_attn_fwd.argtypes = [S, P, P, P, M, F, P, P, P, P, Z, P]
    lib.sa2_attn_bwd.restype = ctypes.c_int
    lib.sa2_attn_bwd.argtypes = [S, P, P, P, P, P, P, P, M, F, P, P, P, P, Z, P]
    lib.sa2_attn_bwd_with_fwd_ws.restype = ctypes.c_int
    lib.sa2_attn_bwd_with_fwd_ws.argtypes = [S, P, P, P, P, P, P, P, M, F, P, P, P, P, Z, P, Z, P]
    lib.sa2_vd_loss_workspace_size.restype = Z
    lib.sa2_vd_loss_workspace_size.argtypes = [S]
    lib.sa2_vd_loss.restype = ctypes.c_int
    lib.sa2_vd_loss.argtypes = [S, P, P, P, P, P, P, P, Z, P]
    lib.sa2_get_device_status.restype = ctypes.c_int
    lib.sa2_get_device_status.argtypes = [P]
    lib.sa2_debug_set_wait_limit.restype = None
    lib.sa2_debug_set_wait_limit.argtypes = [ctypes.c_ulonglong, ctypes.c_ulonglong]
    lib.sa2_profiler_enable.restype = None
    lib.sa2_profiler_enable.argtypes = [ctypes.c_int]
    lib.sa2_profiler_collect.restype = ctypes.c_int
    lib.sa2_profiler_collect.argtypes = [ctypes.POINTER(KernelTime), ctypes.c_int]
    _lib = lib
    return lib


def make_shape(x: torch.Tensor, bq: int, bk: int) -> Shape:
    """sa2_shape of a [B, H, N, d] token tensor (last dimension contiguous)."""
    if x.dim() != 4:
        raise ValueError("token tensors are [B, H, N, d]")
    if x.stride(3) != 1:
        raise ValueError("the last dimension must be contiguous")
    if x.dtype == torch.bfloat16:
        dt = SA2_BF16
    elif x.dtype == torch.float32:
        dt = SA2_FP32
    else:
        raise ValueError(f"unsupported dtype {x.dtype}")
    B, H, N, d = x.shape
    return Shape(B, H, N, d, bq, bk, dt, 0, x.stride(0), x.stride(1), x.stride(2))


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(fn: str, code: int):
    if code != 0:
        raise Sa2Error(fn, code)


@dataclass
class BlockMask:
    """The block mask in compact form (device tensors).  Only the first row_cnt / col_cnt
    entries of row_idx / col_idx are defined."""
    row_cnt: torch.Tensor  # [B, H, Tq] int32
    row_idx: torch.Tensor  # [B, H, Tq, Tk] int32
    col_cnt: torch.Tensor  # [B, H, Tk] int32
    col_idx: torch.Tensor  # [B, H, Tk, Tq] int32
    mask: Optional[torch.Tensor] = None  # [B, H, Tq, Tk] uint8
    pooled_p: Optional[torch.Tensor] = None  # [B, H, Tq, Tk] float32

    def struct(self) -> BlockMaskStruct:
        return BlockMaskStruct(_ptr(self.row_cnt), _ptr(self.row_idx), _ptr(self.col_cnt), _ptr(self.col_idx),
                               _ptr(self.mask), _ptr(self.pooled_p))

    @staticmethod
    def empty(B: int, H: int, Tq: int, Tk: int, device, mask: bool = True, pooled: bool = False) -> "BlockMask":
        i32 = dict(dtype=torch.int32, device=device)
        return BlockMask(torch.empty((B, H, Tq), **i32), torch.empty((B, H, Tq, Tk), **i32),
                         torch.empty((B, H, Tk), **i32), torch.empty((B, H, Tk, Tq), **i32),
                         torch.empty((B, H, Tq, Tk), dtype=torch.uint8, device=device) if mask else None,
                         torch.empty((B, H, Tq, Tk), dtype=torch.float32, device=device) if pooled else None)


def blocks(N: int, b: int) -> int:
    return -(-N // b)


def workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def build_mask(q: torch.Tensor, k: torch.Tensor, topk: float, topp: float, bq: int = 128, bk: int = 64,
               want_mask: bool = True, want_pooled: bool = False, out: Optional[BlockMask] = None,
               ws: Optional[torch.Tensor] = None, stream=None) -> BlockMask:
    """sa2_build_mask: the hybrid Top-k + Top-p block mask of q, k ([B, H, N, d])."""
    lib = load_library()
    shp = make_shape(q, bq, bk)
    if make_shape(k, bq, bk).stride_n != shp.stride_n or k.shape != q.shape:
        raise ValueError("q and k must have the same shape and strides")
    B, H, N, _ = q.shape
    Tq, Tk = blocks(N, bq), blocks(N, bk)
    if out is None:
        out = BlockMask.empty(B, H, Tq, Tk, q.device, mask=want_mask, pooled=want_pooled)
    if ws is None:
        ws = workspace(lib.sa2_mask_workspace_size(ctypes.byref(shp)), q.device)
    m = out.struct()
    _check("sa2_build_mask", lib.sa2_build_mask(ctypes.byref(shp), q.data_ptr(), k.data_ptr(), float(topk),
                                                float(topp), ctypes.byref(m), ws.data_ptr(), ws.numel(),
                                                _stream(stream)))
    return out


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: BlockMask, bq: int = 128, bk: int = 64,
             scale: Optional[float] = None, o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
             o_lo: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None, stream=None):
    """sa2_attn_fwd: block-sparse attention forward; returns (O, LSE).  Pass ``o_lo`` (a
    tensor like q) to also receive the low-order bf16 part of O for the backward."""
    lib = load_library()
    shp = make_shape(q, bq, bk)
    B, H, N, d = q.shape
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(lib.sa2_fwd_workspace_size(ctypes.byref(shp)), q.device)
    m = mask.struct()
    _check("sa2_attn_fwd", lib.sa2_attn_fwd(ctypes.byref(shp), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                            ctypes.byref(m), float(scale or 0.0), o.data_ptr(), _ptr(o_lo),
                                            lse.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)))
    return o, lse


def attn_bwd(q, k, v, o, lse, do, mask: BlockMask, bq: int = 128, bk: int = 64, scale: Optional[float] = None,
             o_lo: Optional[torch.Tensor] = None, dq=None, dk=None, dv=None, ws: Optional[torch.Tensor] = None,
             fwd_ws: Optional[torch.Tensor] = None, stream=None):
    """sa2_attn_bwd: gradients (dQ, dK, dV) of the block-sparse attention, mask fixed.

    ``fwd_ws``: the ``ws`` tensor given to the attn_fwd call on these q, k, v (untouched
    since); its fp16 copies are used instead of converting again
    (sa2_attn_bwd_with_fwd_ws)."""
    lib = load_library()
    shp = make_shape(q, bq, bk)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if ws is None:
        ws = workspace(lib.sa2_bwd_workspace_size(ctypes.byref(shp)), q.device)
    m = mask.struct()
    args = (ctypes.byref(shp), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), _ptr(o_lo), lse.data_ptr(),
            do.data_ptr(), ctypes.byref(m), float(scale or 0.0), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
            ws.data_ptr(), ws.numel())
    if fwd_ws is None:
        _check("sa2_attn_bwd", lib.sa2_attn_bwd(*args, _stream(stream)))
    else:
        _check("sa2_attn_bwd_with_fwd_ws",
               lib.sa2_attn_bwd_with_fwd_ws(*args, fwd_ws.data_ptr(), fwd_ws.numel(), _stream(stream)))
    return dq, dk, dv


def vd_loss(o_s: torch.Tensor, o_t: torch.Tensor, o_s_lo: Optional[torch.Tensor] = None,
            o_t_lo: Optional[torch.Tensor] = None, d_o: Optional[torch.Tensor] = None,
            ws: Optional[torch.Tensor] = None, stream=None):
    """sa2_vd_loss: the toy distillation loss sum (O_s - O_t)^2 (a float64 scalar tensor on
    the device) and d_o = 2 (O_s - O_t), ready for attn_bwd of the student."""
    lib = load_library()
    shp = make_shape(o_s, 128, 64)
    if o_t.shape != o_s.shape or o_t.stride() != o_s.stride():
        raise ValueError("o_s and o_t must have the same shape and strides")
    d_o = torch.empty_like(o_s) if d_o is None else d_o
    loss = torch.empty((), dtype=torch.float64, device=o_s.device)
    if ws is None:
        ws = workspace(lib.sa2_vd_loss_workspace_size(ctypes.byref(shp)), o_s.device)
    _check("sa2_vd_loss", lib.sa2_vd_loss(ctypes.byref(shp), o_s.data_ptr(), _ptr(o_s_lo), o_t.data_ptr(),
                                          _ptr(o_t_lo), d_o.data_ptr(), loss.data_ptr(), ws.data_ptr(),
                                          ws.numel(), _stream(stream)))
    return loss, d_o


def device_status(stream=None) -> int:
    """sa2_get_device_status: synchronizes the stream and returns (and clears) the status."""
    return load_library().sa2_get_device_status(_stream(stream))


def profiler_enable(on: bool = True):
    """sa2_profiler_enable: bracket every later kernel launch with CUDA events."""
    load_library().sa2_profiler_enable(1 if on else 0)


def profiler_collect() -> dict:
    """sa2_profiler_collect: {kernel name: (launches, total device ms)} since the last call."""
    lib = load_library()
    n = lib.sa2_profiler_collect(None, 0)
    arr = (KernelTime * n)()
    got = lib.sa2_profiler_collect(arr, n)
    if got < 0:
        raise Sa2Error("sa2_profiler_collect", 5)
    return {arr[i].name.decode(): (arr[i].launches, arr[i].total_ms) for i in range(got)}


def debug_set_wait_limit(limit_ns: int = 0, stall_ns: int = 0):
    """sa2_debug_set_wait_limit: test hook of the failure path (limit of the attention
    kernels' bounded waits, 0 = default; stall of their first CTA's row warps)."""
    load_library().sa2_debug_set_wait_limit(int(limit_ns), int(stall_ns))


def check_device(stream=None):
    code = device_status(stream)
    _check("device", code)


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)
