"""CPU oracle for the partial MXFP8 cast of master weights (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The product (the ``mxfp8_master_weight_gb300``
package and its CUDA library) never does.

The arithmetic lives in ``mxfp8_oracle.c`` (plain scalar C, double precision);
this module compiles it with the host C compiler on first use and wraps it with
numpy-level functions.  It shares no code with the CUDA path.

Parity pins: every function here is checked in ``tests/test_oracle_pins.py``
against brute force, closed forms, library conversions and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxfp8_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cc = os.environ.get("CC", "gcc")
        subprocess.check_call([cc, "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, vp, dbl = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
            lib.oracle_partial_amax.argtypes = [vp, ctypes.c_int, i64, i64, i64, i64, vp, i64, vp, i64]
            lib.oracle_partial_amax.restype = ctypes.c_int
            lib.oracle_max_reduce.argtypes = [vp, ctypes.c_int, i64, ctypes.c_int, vp]
            lib.oracle_update_scales.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp, i64]
            lib.oracle_partial_cast.argtypes = [vp, ctypes.c_int, i64, i64, i64, i64, vp, i64, vp, i64,
                                                vp, vp, i64]
            lib.oracle_partial_cast_model.argtypes = [vp, ctypes.c_int, ctypes.c_int, i64, i64, i64, i64,
                                                      vp, i64, vp, i64, vp, vp, i64]
            lib.oracle_f16_bits_array.argtypes = [vp, vp, i64]
            lib.oracle_swizzle_scales.argtypes = [vp, i64, i64, i64, ctypes.c_int, vp]
            lib.oracle_bf16_rne_bits_array.argtypes = [vp, vp, i64]
            lib.oracle_e4m3_encode_array.argtypes = [vp, vp, i64]
            lib.oracle_e8m0_array.argtypes = [vp, vp, i64]
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_decode.restype = dbl
            lib.oracle_quantize.argtypes = [dbl, ctypes.c_uint8]
            lib.oracle_quantize.restype = ctypes.c_uint8
            flt = ctypes.c_float
            lib.oracle_e2m1_encode_array.argtypes = [vp, vp, i64]
            lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e2m1_decode.restype = dbl
            lib.oracle_nvfp4_tensor_scale.argtypes = [flt]
            lib.oracle_nvfp4_tensor_scale.restype = flt
            lib.oracle_nvfp4_block_scale.argtypes = [flt, flt]
            lib.oracle_nvfp4_block_scale.restype = ctypes.c_uint8
            lib.oracle_nvfp4_block_scale_array.argtypes = [vp, flt, vp, i64]
            lib.oracle_nvfp4_multiplier.argtypes = [ctypes.c_uint8, flt]
            lib.oracle_nvfp4_multiplier.restype = flt
            lib.oracle_nvfp4_quantize.argtypes = [flt, flt]
            lib.oracle_nvfp4_quantize.restype = ctypes.c_uint8
            lib.oracle_nvfp4_partial_amax.argtypes = [vp, ctypes.c_int, i64, i64, i64, i64, vp, i64,
                                                      vp, i64, vp]
            lib.oracle_nvfp4_partial_amax.restype = ctypes.c_int
            lib.oracle_nvfp4_update_scales.argtypes = [vp, i64, i64, i64, flt, vp, i64]
            lib.oracle_nvfp4_partial_cast.argtypes = [vp, ctypes.c_int, i64, i64, i64, i64, vp, i64,
                                                      vp, i64, flt, vp, vp, i64]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle input must be float32 or uint16 (bf16 bits), got {a.dtype}")


def _c(a):
    if a is not None and not a.flags.c_contiguous:
        raise ValueError("oracle buffers must be C-contiguous")
    return a


# ---------------------------------------------------------------- element-wise

def bf16_rne_bits(x: np.ndarray) -> np.ndarray:
    """BF16 bit patterns of FP32 values, round to nearest, ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().oracle_bf16_rne_bits_array(_ptr(x), _ptr(out), x.size)
    return out


def f16_bits(v: np.ndarray) -> np.ndarray:
    """IEEE FP16 bit patterns of float64 values, round to nearest, ties to even."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().oracle_f16_bits_array(_ptr(v), _ptr(out), v.size)
    return out


MODELS = {"bf16": 0, "f16": 1}


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """E4M3 bytes of float64 values: nearest, ties to even, saturate to 448, NaN -> 0x7F."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(v), _ptr(out), v.size)
    return out


def e4m3_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_e4m3_decode(int(b)) for b in c.reshape(-1)]).reshape(c.shape)


def e8m0_from_amax(amax: np.ndarray) -> np.ndarray:
    """E8M0 scale bytes of block amax values (convention: floor(log2 amax) - 8)."""
    a = np.ascontiguousarray(amax, dtype=np.float64)
    out = np.empty(a.shape, np.uint8)
    _load().oracle_e8m0_array(_ptr(a), _ptr(out), a.size)
    return out


def quantize(y: float, scale_byte: int) -> int:
    return int(_load().oracle_quantize(float(y), int(scale_byte)))


# ---------------------------------------------------------------- path steps

def partial_amax(frag: np.ndarray, rows: int, cols: int, start: int,
                 amax_r: np.ndarray, amax_c: np.ndarray | None) -> None:
    """In place: block maxima of the fragment into amax_r [rows][ld] / amax_c [ceil(rows/32)][ld]."""
    frag = _c(np.ascontiguousarray(frag))
    dt = _dtype_code(frag)
    _c(amax_r)
    _c(amax_c)
    for a in (amax_r, amax_c):
        if a is not None and a.dtype != frag.dtype:
            raise TypeError("amax dtype must equal the input dtype")
    rc = _load().oracle_partial_amax(_ptr(frag), dt, rows, cols, start, frag.size,
                                     _ptr(amax_r), amax_r.shape[1],
                                     _ptr(amax_c), 0 if amax_c is None else amax_c.shape[1])
    if rc:
        raise MemoryError("oracle_partial_amax could not allocate its accumulators")


def max_reduce(slots: np.ndarray) -> np.ndarray:
    """Element-wise max of |.| over the leading (shard) axis of a [S][E] packed buffer."""
    slots = _c(np.ascontiguousarray(slots))
    out = np.empty(slots.shape[1:], slots.dtype)
    _load().oracle_max_reduce(_ptr(slots), _dtype_code(slots), int(np.prod(slots.shape[1:])),
                              slots.shape[0], _ptr(out))
    return out


def update_scales(amax: np.ndarray, nrows: int, ncols: int, scale: np.ndarray) -> None:
    """In place: scale[r][c] = E8M0(amax[r][c]) for r < nrows, c < ncols."""
    _c(amax)
    _c(scale)
    _load().oracle_update_scales(_ptr(amax), _dtype_code(amax), nrows, ncols, amax.shape[1],
                                 _ptr(scale), scale.shape[1])


def partial_cast(frag: np.ndarray, rows: int, cols: int, start: int,
                 scale_r: np.ndarray, scale_c: np.ndarray | None,
                 out_r: np.ndarray, out_c: np.ndarray | None, out_offset: int,
                 model: str = "bf16") -> None:
    """In place: E4M3 bytes of the fragment into out_r / out_c at out_offset + (k - start);
    values are first rounded to the model dtype (``"bf16"`` or ``"f16"``)."""
    frag = _c(np.ascontiguousarray(frag))
    for o in (out_r, out_c):
        if o is not None:
            _c(o)
            if o.size < out_offset + frag.size:
                raise ValueError("output too small")
    if out_c is not None and scale_c is None:
        raise ValueError("columnwise scales are required for a columnwise output")
    _load().oracle_partial_cast_model(_ptr(frag), _dtype_code(frag), MODELS[model], rows, cols,
                                      start, frag.size, _ptr(scale_r), scale_r.shape[1],
                                _ptr(scale_c) if out_c is not None else None,
                                scale_c.shape[1] if out_c is not None else 0,
                                _ptr(out_r), _ptr(out_c), out_offset)


def swizzled_size(nr: int, nc: int, transpose: bool) -> int:
    lr, lc = (nc, nr) if transpose else (nr, nc)
    return ((lr + 127) // 128 * 128) * ((lc + 3) // 4 * 4)


def swizzle_scales(S: np.ndarray, nr: int, nc: int, transpose: bool = False) -> np.ndarray:
    """The E8M0 grid S[:nr, :nc] in the 128x4-tile layout of block-scaled GEMMs."""
    _c(S)
    out = np.empty(swizzled_size(nr, nc, transpose), np.uint8)
    _load().oracle_swizzle_scales(_ptr(S), nr, nc, S.shape[1], int(transpose), _ptr(out))
    return out


# ---------------------------------------------------------------- whole flows

def block_dims(rows: int, cols: int):
    return (rows, (cols + 31) // 32), ((rows + 31) // 32, cols)


def full_cast(x: np.ndarray, rows: int, cols: int, colwise: bool = True, model: str = "bf16"):
    """Whole-weight flow: amax over every element, scales, cast.

    Returns (amax_r, amax_c, scale_r, scale_c, q_r, q_c); the columnwise items are
    None for a row-only weight.
    """
    x = np.ascontiguousarray(x).reshape(-1)
    rdim, cdim = block_dims(rows, cols)
    amax_r = np.zeros(rdim, x.dtype)
    amax_c = np.zeros(cdim, x.dtype) if colwise else None
    partial_amax(x, rows, cols, 0, amax_r, amax_c)
    scale_r = np.zeros(rdim, np.uint8)
    update_scales(amax_r, *rdim, scale_r)
    scale_c = None
    if colwise:
        scale_c = np.zeros(cdim, np.uint8)
        update_scales(amax_c, *cdim, scale_c)
    q_r = np.zeros(rows * cols, np.uint8)
    q_c = np.zeros(rows * cols, np.uint8) if colwise else None
    partial_cast(x, rows, cols, 0, scale_r, scale_c, q_r, q_c, 0, model=model)
    return amax_r, amax_c, scale_r, scale_c, q_r, q_c


# ---------------------------------------------------------------- NVFP4 (stated convention)
# E2M1 data in 1x16 / 16x1 blocks with E4M3 block scales and one FP32 tensor scale
# S = 2688 / G (G = tensor amax); see the NVFP4 section of mxfp8_oracle.c.

def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """E2M1 codes (0..15) of float64 values: nearest, ties to the even code, saturate to 6."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint8)
    _load().oracle_e2m1_encode_array(_ptr(v), _ptr(out), v.size)
    return out


def e2m1_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_e2m1_decode(int(b)) for b in c.reshape(-1)]).reshape(c.shape)


def nvfp4_tensor_scale(g: float) -> float:
    return float(_load().oracle_nvfp4_tensor_scale(float(g)))


def nvfp4_block_scales(amax: np.ndarray, s_enc: float) -> np.ndarray:
    a = np.ascontiguousarray(amax, dtype=np.float32)
    out = np.empty(a.shape, np.uint8)
    _load().oracle_nvfp4_block_scale_array(_ptr(a), float(s_enc), _ptr(out), a.size)
    return out


def nvfp4_multiplier(s: int, s_enc: float) -> float:
    return float(_load().oracle_nvfp4_multiplier(int(s), float(s_enc)))


def nvfp4_quantize(y: float, m: float) -> int:
    return int(_load().oracle_nvfp4_quantize(float(y), float(m)))


def nvfp4_block_dims(rows: int, cols: int):
    return (rows, (cols + 15) // 16), ((rows + 15) // 16, cols)


def nvfp4_partial_amax(frag: np.ndarray, rows: int, cols: int, start: int, amax_r: np.ndarray,
                       amax_c: np.ndarray | None, amax_t: np.ndarray) -> None:
    """In place: FP32 1x16 / 16x1 block maxima of the fragment into amax_r / amax_c, and
    amax_t[0] max-accumulated with the fragment's largest |x|."""
    frag = _c(np.ascontiguousarray(frag))
    for a in (amax_r, amax_c, amax_t):
        if a is not None and (a.dtype != np.float32 or not a.flags.c_contiguous):
            raise TypeError("NVFP4 amax buffers are contiguous float32")
    rc = _load().oracle_nvfp4_partial_amax(_ptr(frag), _dtype_code(frag), rows, cols, start,
                                           frag.size, _ptr(amax_r), amax_r.shape[1], _ptr(amax_c),
                                           0 if amax_c is None else amax_c.shape[1], _ptr(amax_t))
    if rc:
        raise MemoryError("oracle_nvfp4_partial_amax could not allocate its accumulators")


def nvfp4_update_scales(amax: np.ndarray, nrows: int, ncols: int, g: float, scale: np.ndarray) -> None:
    _c(amax)
    _c(scale)
    if amax.dtype != np.float32:
        raise TypeError("NVFP4 amax grids are float32")
    _load().oracle_nvfp4_update_scales(_ptr(amax), nrows, ncols, amax.shape[1], float(g),
                                       _ptr(scale), scale.shape[1])


def nvfp4_partial_cast(frag: np.ndarray, rows: int, cols: int, start: int, scale_r: np.ndarray,
                       scale_c: np.ndarray | None, g: float, out_r: np.ndarray,
                       out_c: np.ndarray | None, out_offset: int) -> None:
    """In place: E2M1 codes of the fragment into nibble out_offset + (k - start) of the
    packed outputs (low nibble = even position)."""
    frag = _c(np.ascontiguousarray(frag))
    for o in (out_r, out_c):
        if o is not None:
            _c(o)
            if 2 * o.size < out_offset + frag.size:
                raise ValueError("output too small")
    if out_c is not None and scale_c is None:
        raise ValueError("columnwise scales are required for a columnwise output")
    _load().oracle_nvfp4_partial_cast(_ptr(frag), _dtype_code(frag), rows, cols, start, frag.size,
                                      _ptr(scale_r), scale_r.shape[1],
                                      _ptr(scale_c) if out_c is not None else None,
                                      scale_c.shape[1] if out_c is not None else 0, float(g),
                                      _ptr(out_r), _ptr(out_c), out_offset)


def nvfp4_full_cast(x: np.ndarray, rows: int, cols: int, colwise: bool = True):
    """Whole-weight NVFP4 flow.  Returns (amax_r, amax_c, amax_t, scale_r, scale_c, q_r,
    q_c); columnwise items None for a row-only weight; q_* packed, ceil(n/2) bytes."""
    x = np.ascontiguousarray(x).reshape(-1)
    rdim, cdim = nvfp4_block_dims(rows, cols)
    amax_r = np.zeros(rdim, np.float32)
    amax_c = np.zeros(cdim, np.float32) if colwise else None
    amax_t = np.zeros(1, np.float32)
    nvfp4_partial_amax(x, rows, cols, 0, amax_r, amax_c, amax_t)
    scale_r = np.zeros(rdim, np.uint8)
    nvfp4_update_scales(amax_r, *rdim, amax_t[0], scale_r)
    scale_c = None
    if colwise:
        scale_c = np.zeros(cdim, np.uint8)
        nvfp4_update_scales(amax_c, *cdim, amax_t[0], scale_c)
    nbytes = (rows * cols + 1) // 2
    q_r = np.zeros(nbytes, np.uint8)
    q_c = np.zeros(nbytes, np.uint8) if colwise else None
    nvfp4_partial_cast(x, rows, cols, 0, scale_r, scale_c, amax_t[0], q_r, q_c, 0)
    return amax_r, amax_c, amax_t, scale_r, scale_c, q_r, q_c
