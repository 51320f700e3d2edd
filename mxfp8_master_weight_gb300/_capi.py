"""ctypes view of the C ABI in include/mxfp8_partial.h.

Loads the in-tree ``libmxfp8_gb300.so``.  There is no fallback: when the library
is missing or cannot be loaded, every call raises ``RuntimeError``.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmxfp8_gb300.so")

DTYPE_F32, DTYPE_BF16, DTYPE_U8 = 0, 1, 2

STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "shape mismatch", 3: "dtype mismatch",
                4: "missing required tensor", 5: "non-contiguous", 6: "CUDA error"}

EXPORTED = ("mxfp8_partial_amax", "mxfp8_amax_max_reduce", "mxfp8_update_scales",
            "mxfp8_partial_cast", "mxfp8_partial_amax_batched", "mxfp8_update_scales_batched",
            "mxfp8_partial_cast_batched", "mxfp8_quantize_whole_blocks",
            "mxfp8_quantize_whole_blocks_batched", "mxfp8_swizzle_scales",
            "mxfp8_swizzled_scales_size", "mxfp8_device_can_access",
            "mxfp8_amax_max_reduce_update_scales", "mxfp8_amax_max_reduce_update_scales_ranged",
            "mxfp8_sharded_update_noalloc", "nvfp4_partial_amax", "nvfp4_update_scales",
            "nvfp4_partial_cast", "mxfp8_last_error", "mxfp8_version")


class Tensor(ctypes.Structure):
    """mxfp8_tensor: {void* data; int32 dtype; int32 ndim; int64 shape[2]}."""

    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 2)]


class AmaxJob(ctypes.Structure):
    _fields_ = [("input", Tensor), ("amax_rowwise", Tensor), ("amax_colwise", Tensor),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("start_offset", ctypes.c_int64)]


class CastJob(ctypes.Structure):
    _fields_ = [("input", Tensor), ("scale_inv_rowwise", Tensor), ("scale_inv_colwise", Tensor),
                ("output_rowwise", Tensor), ("output_colwise", Tensor),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("start_offset", ctypes.c_int64), ("out_offset", ctypes.c_int64),
                ("model_dtype", ctypes.c_int32)]


class ScaleJob(ctypes.Structure):
    _fields_ = [("amax_rowwise", Tensor), ("amax_colwise", Tensor), ("scale_inv_rowwise", Tensor),
                ("scale_inv_colwise", Tensor), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


class QuantizeJob(ctypes.Structure):
    _fields_ = [("input", Tensor), ("amax_rowwise", Tensor), ("amax_colwise", Tensor),
                ("scale_inv_rowwise", Tensor), ("scale_inv_colwise", Tensor),
                ("output_rowwise", Tensor), ("output_colwise", Tensor),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("start_offset", ctypes.c_int64), ("out_offset", ctypes.c_int64),
                ("model_dtype", ctypes.c_int32)]


MODEL_BF16, MODEL_F16 = 0, 1
MODELS = {"bf16": MODEL_BF16, "f16": MODEL_F16, MODEL_BF16: MODEL_BF16, MODEL_F16: MODEL_F16}


def empty_tensor() -> Tensor:
    return Tensor(None, DTYPE_U8, 1, (ctypes.c_int64 * 2)(0, 0))


class MXFP8Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)} ({status}): {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load (once) and return the CUDA library; raise RuntimeError if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: build the sm_103a library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(p)
        T = ctypes.POINTER(Tensor)
        i64, vp = ctypes.c_int64, ctypes.c_void_p
        lib.mxfp8_partial_amax.argtypes = [T, T, T, i64, i64, i64, vp]
        lib.mxfp8_amax_max_reduce.argtypes = [T, T, vp]
        lib.mxfp8_update_scales.argtypes = [T, T, T, T, i64, i64, vp]
        lib.mxfp8_partial_cast.argtypes = [T, T, T, T, T, i64, i64, i64, i64, vp]
        i32 = ctypes.c_int32
        lib.mxfp8_partial_amax_batched.argtypes = [ctypes.POINTER(AmaxJob), i32, vp]
        lib.mxfp8_update_scales_batched.argtypes = [ctypes.POINTER(ScaleJob), i32, vp]
        lib.mxfp8_partial_cast_batched.argtypes = [ctypes.POINTER(CastJob), i32, vp]
        lib.mxfp8_quantize_whole_blocks.argtypes = [T, T, T, T, T, T, T, i64, i64, i64, i64, vp]
        lib.mxfp8_quantize_whole_blocks_batched.argtypes = [ctypes.POINTER(QuantizeJob), i32, vp]
        lib.mxfp8_swizzle_scales.argtypes = [T, T, i64, i64, i32, vp]
        lib.mxfp8_swizzled_scales_size.argtypes = [i64, i64, i32]
        lib.mxfp8_swizzled_scales_size.restype = i64
        lib.mxfp8_amax_max_reduce_update_scales.argtypes = [T, T, ctypes.POINTER(ScaleJob), i32, vp]
        lib.mxfp8_amax_max_reduce_update_scales.restype = ctypes.c_int
        lib.mxfp8_amax_max_reduce_update_scales_ranged.argtypes = [
            T, T, ctypes.POINTER(ScaleJob), i32, ctypes.POINTER(i64), i32, vp]
        lib.mxfp8_amax_max_reduce_update_scales_ranged.restype = ctypes.c_int
        lib.nvfp4_partial_amax.argtypes = [T, T, T, T, i64, i64, i64, vp]
        lib.nvfp4_update_scales.argtypes = [T, T, T, T, T, i64, i64, vp]
        lib.nvfp4_partial_cast.argtypes = [T, T, T, T, T, T, i64, i64, i64, i64, vp]
        for name in ("nvfp4_partial_amax", "nvfp4_update_scales", "nvfp4_partial_cast"):
            getattr(lib, name).restype = ctypes.c_int
        lib.mxfp8_device_can_access.argtypes = [vp, i64]
        lib.mxfp8_device_can_access.restype = ctypes.c_int
        for name in ("mxfp8_partial_amax", "mxfp8_amax_max_reduce", "mxfp8_update_scales",
                     "mxfp8_partial_cast", "mxfp8_partial_amax_batched",
                     "mxfp8_update_scales_batched", "mxfp8_partial_cast_batched",
                     "mxfp8_quantize_whole_blocks", "mxfp8_quantize_whole_blocks_batched",
                     "mxfp8_swizzle_scales", "mxfp8_version"):
            getattr(lib, name).restype = ctypes.c_int
        lib.mxfp8_last_error.argtypes = []
        lib.mxfp8_last_error.restype = ctypes.c_char_p
        _lib = lib
        return lib


def check(status: int) -> None:
    if status != 0:
        msg = load().mxfp8_last_error().decode(errors="replace")
        raise MXFP8Error(status, msg)
