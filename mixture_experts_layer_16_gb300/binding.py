"""Thin ctypes binding of libmm_moe.so (include/mm_moe.h).

Argument marshalling only: every step of the layer runs in the CUDA library.
PyTorch is used for device memory and streams.  There is no fallback: if the
library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmm_moe.so")

MM_MOE_BF16, MM_MOE_MXFP8, MM_MOE_FP8_BWD, MM_MOE_FP8_BLOCK = 0, 1, 2, 3
PRECISION = {"bf16": MM_MOE_BF16, "mxfp8": MM_MOE_MXFP8, "fp8_bwd": MM_MOE_FP8_BWD,
             "fp8_block": MM_MOE_FP8_BLOCK}
STATUS = {0: "MM_MOE_OK", 1: "MM_MOE_EINVAL", 2: "MM_MOE_ENOTSUP", 3: "MM_MOE_EBADIDX",
          4: "MM_MOE_ETIMEOUT", 5: "MM_MOE_ECUDA"}
MM_MOE_OK, MM_MOE_EINVAL, MM_MOE_ENOTSUP, MM_MOE_EBADIDX, MM_MOE_ETIMEOUT, MM_MOE_ECUDA = range(6)

# every symbol include/mm_moe.h declares
EXPORTS = ("mm_moe_workspace_size", "mm_moe_forward", "mm_moe_backward", "mm_moe_get_routing",
           "mm_moe_read_status", "mm_moe_last_launch_count", "mm_moe_profile_start",
           "mm_moe_profile_stop", "mm_moe_kernel_name", "mm_moe_kernel_count",
           "mm_moe_route_noalloc", "mm_moe_mx_qdq", "mm_moe_router_forward",
           "mm_moe_router_backward", "mm_moe_fp8_block_qdq", "mm_moe_mx_quantize",
           "mm_moe_fp8_block_quantize")


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")
        self.status = status


class Shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int64), ("I", ctypes.c_int64),
                ("E", ctypes.c_int64), ("k", ctypes.c_int64), ("prec", ctypes.c_int32),
                ("flags", ctypes.c_int32)]


MM_MOE_RECOMPUTE = 1  # activation checkpointing (include/mm_moe.h)
MM_MOE_MULTICAST = 2  # A-multicast clusters of two SM pairs (include/mm_moe.h)


def make_shape(T, H, I, E, k, prec="bf16", recompute: bool = False,
               multicast: bool = False) -> Shape:
    return Shape(int(T), int(H), int(I), int(E), int(k), PRECISION.get(prec, prec),
                 (MM_MOE_RECOMPUTE if recompute else 0) | (MM_MOE_MULTICAST if multicast else 0))


_lib: Optional[ctypes.CDLL] = None
_vp = ctypes.c_void_p


def lib() -> ctypes.CDLL:
    """Load the library once; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "mixture_experts_layer_16_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        sp = ctypes.POINTER(Shape)
        L.mm_moe_workspace_size.argtypes = [sp, ctypes.POINTER(ctypes.c_size_t),
                                            ctypes.POINTER(ctypes.c_size_t)]
        L.mm_moe_forward.argtypes = [sp] + [_vp] * 10
        L.mm_moe_backward.argtypes = [sp] + [_vp] * 13
        L.mm_moe_get_routing.argtypes = [sp, _vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                         ctypes.POINTER(_vp)]
        L.mm_moe_read_status.argtypes = [_vp, _vp]
        L.mm_moe_last_launch_count.argtypes = []
        L.mm_moe_profile_start.argtypes = []
        L.mm_moe_profile_stop.argtypes = [ctypes.POINTER(ctypes.c_float),
                                          ctypes.POINTER(ctypes.c_int), ctypes.c_int]
        L.mm_moe_kernel_name.argtypes = [ctypes.c_int]
        L.mm_moe_kernel_count.argtypes = []
        L.mm_moe_route_noalloc.argtypes = [sp] + [_vp] * 6
        L.mm_moe_mx_qdq.argtypes = [_vp, _vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, _vp]
        L.mm_moe_fp8_block_qdq.argtypes = [_vp, _vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                           _vp]
        L.mm_moe_mx_quantize.argtypes = [_vp, _vp, _vp, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_int, _vp]
        L.mm_moe_fp8_block_quantize.argtypes = [_vp, _vp, _vp, ctypes.c_int64, ctypes.c_int64,
                                                ctypes.c_int, _vp]
        L.mm_moe_router_forward.argtypes = [sp] + [_vp] * 6
        L.mm_moe_router_backward.argtypes = [sp] + [_vp] * 9
        for fn in EXPORTS:
            getattr(L, fn).restype = ctypes.c_int
        L.mm_moe_kernel_name.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    return int(getattr(stream, "cuda_stream", stream))


def _check(fn: str, st: int) -> None:
    if st != MM_MOE_OK:
        raise MoEError(fn, st)


def mm_moe_workspace_size(shape: Shape) -> Tuple[int, int]:
    sc, sv = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check("mm_moe_workspace_size",
           lib().mm_moe_workspace_size(ctypes.byref(shape), ctypes.byref(sc), ctypes.byref(sv)))
    return sc.value, sv.value


def mm_moe_forward(shape: Shape, x, topk_idx, topk_w, W_gate, W_up, W_down, y, scratch, saved,
                   stream=None, check: bool = True) -> int:
    st = lib().mm_moe_forward(ctypes.byref(shape), _ptr(x), _ptr(topk_idx), _ptr(topk_w),
                              _ptr(W_gate), _ptr(W_up), _ptr(W_down), _ptr(y), _ptr(scratch),
                              _ptr(saved), _stream(stream))
    if check:
        _check("mm_moe_forward", st)
    return st


def mm_moe_backward(shape: Shape, dy, saved, W_gate, W_up, W_down, x, dx, dW_gate, dW_up,
                    dW_down, dtopk_w, scratch, stream=None, check: bool = True) -> int:
    st = lib().mm_moe_backward(ctypes.byref(shape), _ptr(dy), _ptr(saved), _ptr(W_gate),
                               _ptr(W_up), _ptr(W_down), _ptr(x), _ptr(dx), _ptr(dW_gate),
                               _ptr(dW_up), _ptr(dW_down), _ptr(dtopk_w), _ptr(scratch),
                               _stream(stream))
    if check:
        _check("mm_moe_backward", st)
    return st


def mm_moe_get_routing(shape: Shape, saved):
    """Views of `saved` (a uint8 device tensor): offsets [E+1], perm [T*k], inv [T*k], int32."""
    import torch
    o, p, i = _vp(), _vp(), _vp()
    _check("mm_moe_get_routing",
           lib().mm_moe_get_routing(ctypes.byref(shape), _ptr(saved), ctypes.byref(o),
                                    ctypes.byref(p), ctypes.byref(i)))
    base = saved.data_ptr()
    R = shape.T * shape.k

    def view(ptr, n):
        off = ptr.value - base
        return saved[off:off + 4 * n].view(torch.int32)
    return view(o, shape.E + 1), view(p, R), view(i, R)


def mm_moe_route_noalloc(shape: Shape, topk_idx, topk_w, offsets, perm, inv, stream=None,
                         check: bool = True) -> int:
    """Routing into caller-provided offsets/perm/inv with no scratch buffer (the
    library's own fixed device array is used; calls on different streams race)."""
    st = lib().mm_moe_route_noalloc(ctypes.byref(shape), _ptr(topk_idx), _ptr(topk_w),
                                    _ptr(offsets), _ptr(perm), _ptr(inv), _stream(stream))
    if check:
        _check("mm_moe_route_noalloc", st)
    return st


def mm_moe_mx_qdq(inp, out, axis: int, stream=None) -> None:
    """MXFP8 quantise-dequantise of a 2-D bf16 CUDA tensor into `out` (may be `inp`):
    32-element blocks along rows (axis=1) or down columns (axis=0)."""
    import torch
    if inp.dim() != 2 or inp.dtype != torch.bfloat16 or not inp.is_contiguous():
        raise ValueError("inp must be a contiguous 2-D bf16 tensor")
    if out.shape != inp.shape or out.dtype != inp.dtype or not out.is_contiguous():
        raise ValueError("out must match inp")
    _check("mm_moe_mx_qdq", lib().mm_moe_mx_qdq(_ptr(inp), _ptr(out), inp.shape[0],
                                                inp.shape[1], int(axis), _stream(stream)))


def mm_moe_mx_quantize(inp, codes, scales, axis: int, stream=None) -> None:
    """MXFP8 quantisation of a 2-D bf16 CUDA tensor [rows, cols] (multiples of 128)
    into e4m3 codes (uint8, same shape) and E8M0 scales (uint8, rows * cols / 32 bytes
    in the block-scaled tensor cores' atom arrangement): 32-element blocks along rows
    (axis=1) or down columns (axis=0)."""
    import torch
    if inp.dim() != 2 or inp.dtype != torch.bfloat16 or not inp.is_contiguous():
        raise ValueError("inp must be a contiguous 2-D bf16 tensor")
    if codes.shape != inp.shape or codes.dtype != torch.uint8 or not codes.is_contiguous():
        raise ValueError("codes must be a contiguous uint8 tensor of inp's shape")
    if scales.dtype != torch.uint8 or scales.numel() != inp.numel() // 32:
        raise ValueError("scales must hold rows * cols / 32 uint8")
    _check("mm_moe_mx_quantize", lib().mm_moe_mx_quantize(
        _ptr(inp), _ptr(codes), _ptr(scales), inp.shape[0], inp.shape[1], int(axis),
        _stream(stream)))


def mm_moe_fp8_block_quantize(inp, codes, scales, layout: int, stream=None) -> None:
    """Blockwise FP8 quantisation of a 2-D bf16 CUDA tensor [rows, cols] (multiples of
    128) into e4m3 codes (uint8, same shape) and E8M0 scales (uint8, in the block-scaled
    tensor cores' atom arrangement; rows * cols / 32 bytes, twice that for tiles):
    128-element blocks along rows (layout 0), down columns (1), or 128 x 128 tiles (2)."""
    import torch
    if inp.dim() != 2 or inp.dtype != torch.bfloat16 or not inp.is_contiguous():
        raise ValueError("inp must be a contiguous 2-D bf16 tensor")
    if codes.shape != inp.shape or codes.dtype != torch.uint8 or not codes.is_contiguous():
        raise ValueError("codes must be a contiguous uint8 tensor of inp's shape")
    n = inp.numel() // 32 * (2 if int(layout) == 2 else 1)
    if scales.dtype != torch.uint8 or scales.numel() != n:
        raise ValueError("scales must hold rows * cols / 32 uint8 (twice that for tiles)")
    _check("mm_moe_fp8_block_quantize", lib().mm_moe_fp8_block_quantize(
        _ptr(inp), _ptr(codes), _ptr(scales), inp.shape[0], inp.shape[1], int(layout),
        _stream(stream)))


def mm_moe_fp8_block_qdq(inp, out, layout: int, stream=None) -> None:
    """Blockwise FP8 quantise-dequantise of a 2-D bf16 CUDA tensor into `out` (may be
    `inp`): 128-element blocks along rows (layout 0), down columns (1), or 128 x 128
    tiles (2)."""
    import torch
    if inp.dim() != 2 or inp.dtype != torch.bfloat16 or not inp.is_contiguous():
        raise ValueError("inp must be a contiguous 2-D bf16 tensor")
    if out.shape != inp.shape or out.dtype != inp.dtype or not out.is_contiguous():
        raise ValueError("out must match inp")
    _check("mm_moe_fp8_block_qdq", lib().mm_moe_fp8_block_qdq(
        _ptr(inp), _ptr(out), inp.shape[0], inp.shape[1], int(layout), _stream(stream)))


def mm_moe_router_forward(shape: Shape, x, W_router, logits, topk_idx, topk_w, stream=None,
                          check: bool = True) -> int:
    st = lib().mm_moe_router_forward(ctypes.byref(shape), _ptr(x), _ptr(W_router), _ptr(logits),
                                     _ptr(topk_idx), _ptr(topk_w), _stream(stream))
    if check:
        _check("mm_moe_router_forward", st)
    return st


def mm_moe_router_backward(shape: Shape, x, W_router, topk_idx, topk_w, dtopk_w, dlogits, dx,
                           dW_router, stream=None, check: bool = True) -> int:
    st = lib().mm_moe_router_backward(ctypes.byref(shape), _ptr(x), _ptr(W_router),
                                      _ptr(topk_idx), _ptr(topk_w), _ptr(dtopk_w),
                                      _ptr(dlogits), _ptr(dx), _ptr(dW_router), _stream(stream))
    if check:
        _check("mm_moe_router_backward", st)
    return st


def mm_moe_read_status(scratch, stream=None) -> int:
    return int(lib().mm_moe_read_status(_ptr(scratch), _stream(stream)))


def mm_moe_last_launch_count() -> int:
    return int(lib().mm_moe_last_launch_count())


def mm_moe_kernel_count() -> int:
    return int(lib().mm_moe_kernel_count())


def mm_moe_kernel_name(i: int) -> str:
    n = lib().mm_moe_kernel_name(int(i))
    return n.decode() if n else ""


def mm_moe_profile_start() -> None:
    _check("mm_moe_profile_start", lib().mm_moe_profile_start())


def mm_moe_profile_stop():
    """{kernel name: (total ms, launches)} of the calls since mm_moe_profile_start."""
    n = mm_moe_kernel_count()
    ms = (ctypes.c_float * n)()
    cnt = (ctypes.c_int * n)()
    _check("mm_moe_profile_stop", lib().mm_moe_profile_stop(ms, cnt, n))
    return {mm_moe_kernel_name(i): (float(ms[i]), int(cnt[i])) for i in range(n)}


class Workspace:
    """The two caller-owned device buffers of one layer shape, allocated with torch."""

    def __init__(self, shape: Shape, device="cuda"):
        import torch
        self.shape = shape
        sc, sv = mm_moe_workspace_size(shape)
        self.scratch = torch.empty(max(sc, 256), dtype=torch.uint8, device=device)
        self.saved = torch.empty(max(sv, 256), dtype=torch.uint8, device=device)
