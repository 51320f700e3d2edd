"""Python binding of the C ABI, with the same entry-point names.

Argument marshalling only: torch tensors are turned into ``mxfp8_tensor``
handles and the call goes to the CUDA library on the tensor's current stream.
Every step of the computation runs in the library's kernels.

Omission contract ("Support row-only MXFP8 distributed master-weight casts",
section "Changes"): ``None`` and every zero-element tensor -- including a view
that still has backing storage -- become an EMPTY handle, which the library reads
as "this direction is absent".
"""
from __future__ import annotations

import ctypes

import torch

from . import _capi
from ._capi import (DTYPE_BF16, DTYPE_F32, DTYPE_U8, AmaxJob, CastJob, MXFP8Error, QuantizeJob,
                    ScaleJob, Tensor)

_DTYPES = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16, torch.uint8: DTYPE_U8,
           torch.float8_e4m3fn: DTYPE_U8}
if hasattr(torch, "float8_e8m0fnu"):
    _DTYPES[torch.float8_e8m0fnu] = DTYPE_U8


def device_can_access(t: torch.Tensor) -> bool:
    """True when the current CUDA device can dereference the tensor's storage directly
    (device memory, or page-locked host memory mapped into the device's address space)."""
    nbytes = t.numel() * t.element_size()
    return bool(_capi.load().mxfp8_device_can_access(ctypes.c_void_p(t.data_ptr()), nbytes))


def mxfp8_device_can_access(t: torch.Tensor) -> bool:
    """The C entry of the same name for a tensor's storage (see device_can_access)."""
    return device_can_access(t)


def mxfp8_last_error() -> str:
    """Message of the calling thread's most recent non-zero status ("" if none)."""
    return _capi.load().mxfp8_last_error().decode(errors="replace")


def mxfp8_version() -> int:
    """Library version as major*10000 + minor*100 + patch."""
    return int(_capi.load().mxfp8_version())


def handle(t: torch.Tensor | None, name: str, allow_host: bool = False) -> Tensor:
    """mxfp8_tensor for a CUDA tensor; None / zero-element tensors give an empty handle.
    With ``allow_host``, a page-locked CPU tensor is accepted when the device can access
    it directly (checked by the library)."""
    if t is None or t.numel() == 0:
        return _capi.empty_tensor()
    if not t.is_cuda:
        if not allow_host:
            raise ValueError(f"{name}: expected a CUDA tensor, got device {t.device}")
        if not t.is_pinned() or not device_can_access(t):
            raise ValueError(f"{name}: host tensor is not page-locked memory the device can access")
    if not t.is_contiguous():
        raise MXFP8Error(5, f"{name}: tensor must be contiguous")
    if t.dtype not in _DTYPES:
        raise MXFP8Error(3, f"{name}: unsupported dtype {t.dtype}")
    if t.dim() > 2:
        raise ValueError(f"{name}: expected at most 2 dimensions, got {t.dim()}")
    shape = tuple(t.shape) if t.dim() == 2 else (t.numel(), 0)
    return Tensor(ctypes.c_void_p(t.data_ptr()), _DTYPES[t.dtype], 2 if t.dim() == 2 else 1,
                  (ctypes.c_int64 * 2)(*shape))


def _stream(stream, like: torch.Tensor | None):
    if stream is None:
        dev = like.device if like is not None and like.is_cuda else None
        stream = torch.cuda.current_stream(dev)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _device_of(*ts):
    for t in ts:
        if t is not None and t.numel() > 0 and t.is_cuda:
            return t.device
    return None


def _call(fn, dev, *args):
    lib = _capi.load()
    if dev is not None:
        with torch.cuda.device(dev):
            _capi.check(getattr(lib, fn)(*args))
    else:
        _capi.check(getattr(lib, fn)(*args))


def mxfp8_partial_amax(input, amax_rowwise, amax_colwise, rows: int, cols: int,
                       start_offset: int, stream=None) -> None:
    """Block maxima of |x| over the fragment, written in place (see include/mxfp8_partial.h)."""
    dev = _device_of(input, amax_rowwise, amax_colwise)
    args = [handle(input, "input"), handle(amax_rowwise, "amax_rowwise"),
            handle(amax_colwise, "amax_colwise")]
    _call("mxfp8_partial_amax", dev, *[ctypes.byref(a) for a in args], int(rows), int(cols),
          int(start_offset), _stream(stream, input))


def mxfp8_amax_max_reduce(slots, out, stream=None) -> None:
    """out[k] = max_s |slots[s][k]| over the leading (shard) axis of a [S][E] buffer."""
    dev = _device_of(slots, out)
    args = [handle(slots, "slots"), handle(out, "out")]
    _call("mxfp8_amax_max_reduce", dev, *[ctypes.byref(a) for a in args], _stream(stream, out))


def mxfp8_update_scales(amax_rowwise, amax_colwise, scale_inv_rowwise, scale_inv_colwise,
                        rows: int, cols: int, stream=None) -> None:
    """E8M0 scale bytes of the (reduced) block amaxes for the present directions."""
    dev = _device_of(amax_rowwise, amax_colwise, scale_inv_rowwise)
    args = [handle(amax_rowwise, "amax_rowwise"), handle(amax_colwise, "amax_colwise"),
            handle(scale_inv_rowwise, "scale_inv_rowwise"),
            handle(scale_inv_colwise, "scale_inv_colwise")]
    _call("mxfp8_update_scales", dev, *[ctypes.byref(a) for a in args], int(rows), int(cols),
          _stream(stream, amax_rowwise))


def mxfp8_partial_cast(input, scale_inv_rowwise, scale_inv_colwise, output_rowwise,
                       output_colwise, rows: int, cols: int, start_offset: int,
                       out_offset: int | None = None, stream=None, model_dtype="bf16") -> None:
    """E4M3 bytes of the fragment into the outputs (out_offset defaults to start_offset:
    a full-size output written in place; pass 0 for a fragment-sized output).
    ``model_dtype``: "bf16" (default) or "f16", the dtype values are rounded through."""
    if out_offset is None:
        out_offset = start_offset
    if _capi.MODELS[model_dtype] != _capi.MODEL_BF16:
        mxfp8_partial_cast_batched([(input, scale_inv_rowwise, scale_inv_colwise, output_rowwise,
                                     output_colwise, rows, cols, start_offset, out_offset,
                                     model_dtype)], stream=stream)
        return
    dev = _device_of(input, output_rowwise, output_colwise)
    args = [handle(input, "input"), handle(scale_inv_rowwise, "scale_inv_rowwise"),
            handle(scale_inv_colwise, "scale_inv_colwise"),
            handle(output_rowwise, "output_rowwise"), handle(output_colwise, "output_colwise")]
    _call("mxfp8_partial_cast", dev, *[ctypes.byref(a) for a in args], int(rows), int(cols),
          int(start_offset), int(out_offset), _stream(stream, input))


def _amax_jobs(jobs):
    arr = (AmaxJob * max(1, len(jobs)))()
    keep = []
    for k, (inp, ar, ac, rows, cols, start) in enumerate(jobs):
        arr[k] = AmaxJob(handle(inp, "input"), handle(ar, "amax_rowwise"), handle(ac, "amax_colwise"),
                         int(rows), int(cols), int(start))
        keep += [t for t in (inp, ar, ac) if t is not None]
    return arr, keep


def _cast_jobs(jobs):
    arr = (CastJob * max(1, len(jobs)))()
    keep = []
    for k, job in enumerate(jobs):
        inp, sr, sc, qr, qc, rows, cols, start = job[:8]
        out_offset = job[8] if len(job) > 8 and job[8] is not None else start
        model = _capi.MODELS[job[9]] if len(job) > 9 else _capi.MODEL_BF16
        arr[k] = CastJob(handle(inp, "input"), handle(sr, "scale_inv_rowwise"),
                         handle(sc, "scale_inv_colwise"), handle(qr, "output_rowwise"),
                         handle(qc, "output_colwise"), int(rows), int(cols), int(start),
                         int(out_offset), model)
        keep += [t for t in (inp, sr, sc, qr, qc) if t is not None]
    return arr, keep


def _scale_jobs(jobs):
    arr = (ScaleJob * max(1, len(jobs)))()
    keep = []
    for k, (ar, ac, sr, sc, rows, cols) in enumerate(jobs):
        arr[k] = ScaleJob(handle(ar, "amax_rowwise"), handle(ac, "amax_colwise"),
                          handle(sr, "scale_inv_rowwise"), handle(sc, "scale_inv_colwise"),
                          int(rows), int(cols))
        keep += [t for t in (ar, ac, sr, sc) if t is not None]
    return arr, keep


def mxfp8_partial_amax_batched(jobs, stream=None) -> None:
    """Many fragments in as few launches as possible.  ``jobs``: sequence of
    (input, amax_rowwise, amax_colwise, rows, cols, start_offset)."""
    arr, keep = _amax_jobs(jobs)
    _call("mxfp8_partial_amax_batched", _device_of(*keep), arr, len(jobs),
          _stream(stream, keep[0] if keep else None))


def mxfp8_update_scales_batched(jobs, stream=None) -> None:
    """``jobs``: sequence of (amax_rowwise, amax_colwise, scale_inv_rowwise, scale_inv_colwise,
    rows, cols)."""
    arr, keep = _scale_jobs(jobs)
    _call("mxfp8_update_scales_batched", _device_of(*keep), arr, len(jobs),
          _stream(stream, keep[0] if keep else None))


def mxfp8_amax_max_reduce_update_scales(slots, reduced, jobs, stream=None) -> None:
    """One pass: reduced = max over the slots of the packed amax, and the E8M0 scales of
    every job, whose amax grids are views into ``reduced``.  ``jobs`` as for
    mxfp8_update_scales_batched."""
    arr, keep = _scale_jobs(jobs)
    hs = [handle(slots, "slots"), handle(reduced, "reduced")]
    _call("mxfp8_amax_max_reduce_update_scales", _device_of(slots, reduced),
          ctypes.byref(hs[0]), ctypes.byref(hs[1]), arr, len(jobs), _stream(stream, reduced))


def _ranges_array(slot_ranges):
    flat = [int(v) for r in slot_ranges for v in r]
    return (ctypes.c_int64 * max(1, len(flat)))(*flat), len(flat) // 3


def mxfp8_amax_max_reduce_update_scales_ranged(slots, reduced, jobs, slot_ranges,
                                               stream=None) -> None:
    """As mxfp8_amax_max_reduce_update_scales, reading slot s only on the packed entries
    its ranges name: ``slot_ranges`` is a sequence of (slot, begin, end) triples."""
    arr, keep = _scale_jobs(jobs)
    rng, nr = _ranges_array(slot_ranges)
    hs = [handle(slots, "slots"), handle(reduced, "reduced")]
    _call("mxfp8_amax_max_reduce_update_scales_ranged", _device_of(slots, reduced),
          ctypes.byref(hs[0]), ctypes.byref(hs[1]), arr, len(jobs), rng, nr,
          _stream(stream, reduced))


def mxfp8_partial_cast_batched(jobs, stream=None) -> None:
    """``jobs``: sequence of (input, scale_inv_rowwise, scale_inv_colwise, output_rowwise,
    output_colwise, rows, cols, start_offset[, out_offset])."""
    arr, keep = _cast_jobs(jobs)
    _call("mxfp8_partial_cast_batched", _device_of(*keep), arr, len(jobs),
          _stream(stream, keep[0] if keep else None))


def mxfp8_quantize_whole_blocks(input, amax_rowwise, amax_colwise, scale_inv_rowwise,
                                scale_inv_colwise, output_rowwise, output_colwise, rows: int,
                                cols: int, start_offset: int, out_offset: int | None = None,
                                stream=None, model_dtype="bf16", allow_host=False) -> None:
    """One-pass amax -> scales -> cast of a fragment made of whole blocks (amax outputs
    optional); bit-identical to the split calls on the same fragment.  With
    ``allow_host``, any tensor may be page-locked host memory the device can access
    (zero-copy: the kernel reads and writes host memory over the CPU-GPU link)."""
    if out_offset is None:
        out_offset = start_offset
    if _capi.MODELS[model_dtype] != _capi.MODEL_BF16:
        if allow_host:
            raise ValueError("host buffers are supported with the BF16 model dtype only")
        mxfp8_quantize_whole_blocks_batched(
            [(input, amax_rowwise, amax_colwise, scale_inv_rowwise, scale_inv_colwise,
              output_rowwise, output_colwise, rows, cols, start_offset, out_offset, model_dtype)],
            stream=stream)
        return
    names = ("input", "amax_rowwise", "amax_colwise", "scale_inv_rowwise", "scale_inv_colwise",
             "output_rowwise", "output_colwise")
    ts = (input, amax_rowwise, amax_colwise, scale_inv_rowwise, scale_inv_colwise,
          output_rowwise, output_colwise)
    dev = _device_of(*ts)
    if dev is None and allow_host:
        dev = torch.device("cuda", torch.cuda.current_device())
    args = [handle(t, n, allow_host) for t, n in zip(ts, names)]
    _call("mxfp8_quantize_whole_blocks", dev, *[ctypes.byref(a) for a in args], int(rows),
          int(cols), int(start_offset), int(out_offset),
          _stream(stream, input if input.is_cuda else None))


def _quantize_jobs(jobs):
    arr = (QuantizeJob * max(1, len(jobs)))()
    keep = []
    names = ("input", "amax_rowwise", "amax_colwise", "scale_inv_rowwise", "scale_inv_colwise",
             "output_rowwise", "output_colwise")
    for k, job in enumerate(jobs):
        ts = job[:7]
        rows, cols, start = job[7:10]
        out_offset = job[10] if len(job) > 10 and job[10] is not None else start
        model = _capi.MODELS[job[11]] if len(job) > 11 else _capi.MODEL_BF16
        arr[k] = QuantizeJob(*[handle(t, n) for t, n in zip(ts, names)], int(rows), int(cols),
                             int(start), int(out_offset), model)
        keep += [t for t in ts if t is not None]
    return arr, keep


def mxfp8_quantize_whole_blocks_batched(jobs, stream=None) -> None:
    """``jobs``: sequence of (input, amax_rowwise, amax_colwise, scale_inv_rowwise,
    scale_inv_colwise, output_rowwise, output_colwise, rows, cols, start_offset[, out_offset])."""
    arr, keep = _quantize_jobs(jobs)
    _call("mxfp8_quantize_whole_blocks_batched", _device_of(*keep), arr, len(jobs),
          _stream(stream, keep[0] if keep else None))


def mxfp8_swizzled_scales_size(nrows: int, ncols: int, transpose: bool = False) -> int:
    """Bytes of the GEMM scale layout of an nrows x ncols E8M0 grid."""
    return int(_capi.load().mxfp8_swizzled_scales_size(int(nrows), int(ncols), int(bool(transpose))))


def mxfp8_swizzle_scales(scale_inv, out, nrows: int, ncols: int, transpose: bool = False,
                         stream=None) -> None:
    """E8M0 grid -> the 128x4-tile layout block-scaled GEMMs read (see the C header)."""
    dev = _device_of(scale_inv, out)
    args = [handle(scale_inv, "scale_inv"), handle(out, "out")]
    _call("mxfp8_swizzle_scales", dev, *[ctypes.byref(a) for a in args], int(nrows), int(ncols),
          int(bool(transpose)), _stream(stream, scale_inv))


def mxfp8_sharded_update_noalloc(fragments, start_offsets, scale_inv_rowwise, scale_inv_colwise,
                                 output_rowwise, output_colwise, rows: int, cols: int,
                                 stream=None) -> None:
    """Sharded update of one weight (amax of every fragment, MAX reduction, scales, casts)
    for callers that cannot allocate device memory: the library keeps the amax working
    memory in a fixed 64 MiB device array of its own (limits and sharing rules in the C
    header).  ``fragments``: one tensor per shard; ``start_offsets``: their flat starts."""
    lib = _capi.load()
    fn = lib.mxfp8_sharded_update_noalloc
    T = ctypes.POINTER(Tensor)
    fn.argtypes = [T, ctypes.POINTER(ctypes.c_int64), ctypes.c_int32, T, T, T, T,
                   ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    n = len(fragments)
    frs = (Tensor * max(1, n))(*[handle(f, "fragment") for f in fragments])
    starts = (ctypes.c_int64 * max(1, n))(*[int(s) for s in start_offsets])
    outs = [handle(scale_inv_rowwise, "scale_inv_rowwise"), handle(scale_inv_colwise, "scale_inv_colwise"),
            handle(output_rowwise, "output_rowwise"), handle(output_colwise, "output_colwise")]
    dev = _device_of(*fragments, scale_inv_rowwise, output_rowwise)
    _call("mxfp8_sharded_update_noalloc", dev, frs, starts, n, *[ctypes.byref(o) for o in outs],
          int(rows), int(cols), _stream(stream, output_rowwise))


# ---------------------------------------------------------------- NVFP4
def nvfp4_block_shapes(rows: int, cols: int):
    """((rows, ceil(cols/16)), (ceil(rows/16), cols)): the NVFP4 rowwise and columnwise
    block grids of a rows x cols weight."""
    return (rows, (cols + 15) // 16), ((rows + 15) // 16, cols)


def nvfp4_partial_amax(input, amax_rowwise, amax_colwise, amax_tensor, rows: int, cols: int,
                       start_offset: int, stream=None) -> None:
    """1x16 / 16x1 block maxima (F32) of a fragment, and its largest |x| max-accumulated
    into ``amax_tensor[0]`` (see the C header for the NVFP4 convention)."""
    hs = [handle(input, "input"), handle(amax_rowwise, "amax_rowwise"),
          handle(amax_colwise, "amax_colwise"), handle(amax_tensor, "amax_tensor")]
    _call("nvfp4_partial_amax", _device_of(input, amax_rowwise), *[ctypes.byref(h) for h in hs],
          int(rows), int(cols), int(start_offset), _stream(stream, amax_rowwise))


def nvfp4_update_scales(amax_rowwise, amax_colwise, amax_tensor, scale_rowwise, scale_colwise,
                        rows: int, cols: int, stream=None) -> None:
    """E4M3 block scales of the present directions under the tensor amax."""
    hs = [handle(amax_rowwise, "amax_rowwise"), handle(amax_colwise, "amax_colwise"),
          handle(amax_tensor, "amax_tensor"), handle(scale_rowwise, "scale_rowwise"),
          handle(scale_colwise, "scale_colwise")]
    _call("nvfp4_update_scales", _device_of(amax_rowwise, scale_rowwise),
          *[ctypes.byref(h) for h in hs], int(rows), int(cols), _stream(stream, scale_rowwise))


def nvfp4_partial_cast(input, scale_rowwise, scale_colwise, amax_tensor, output_rowwise,
                       output_colwise, rows: int, cols: int, start_offset: int,
                       out_offset: int | None = None, stream=None) -> None:
    """Packed E2M1 codes of a fragment into the rowwise and (optional) columnwise outputs,
    element k at nibble out_offset + k (default: start_offset, full-size outputs)."""
    if out_offset is None:
        out_offset = start_offset
    hs = [handle(input, "input"), handle(scale_rowwise, "scale_rowwise"),
          handle(scale_colwise, "scale_colwise"), handle(amax_tensor, "amax_tensor"),
          handle(output_rowwise, "output_rowwise"), handle(output_colwise, "output_colwise")]
    _call("nvfp4_partial_cast", _device_of(input, output_rowwise), *[ctypes.byref(h) for h in hs],
          int(rows), int(cols), int(start_offset), int(out_offset), _stream(stream, output_rowwise))


def prepare_nvfp4_partial_amax(input, amax_rowwise, amax_colwise, amax_tensor, rows, cols,
                               start_offset):
    ts = (input, amax_rowwise, amax_colwise, amax_tensor)
    hs = [handle(t, n) for t, n in zip(ts, ("input", "amax_rowwise", "amax_colwise", "amax_tensor"))]
    return Prepared("nvfp4_partial_amax", hs, (rows, cols, start_offset), [t for t in ts if t is not None])


def prepare_nvfp4_update_scales(amax_rowwise, amax_colwise, amax_tensor, scale_rowwise,
                                scale_colwise, rows, cols):
    ts = (amax_rowwise, amax_colwise, amax_tensor, scale_rowwise, scale_colwise)
    hs = [handle(t, n) for t, n in zip(ts, ("amax_rowwise", "amax_colwise", "amax_tensor",
                                            "scale_rowwise", "scale_colwise"))]
    return Prepared("nvfp4_update_scales", hs, (rows, cols), [t for t in ts if t is not None])


def prepare_nvfp4_partial_cast(input, scale_rowwise, scale_colwise, amax_tensor, output_rowwise,
                               output_colwise, rows, cols, start_offset, out_offset=None):
    if out_offset is None:
        out_offset = start_offset
    ts = (input, scale_rowwise, scale_colwise, amax_tensor, output_rowwise, output_colwise)
    hs = [handle(t, n) for t, n in zip(ts, ("input", "scale_rowwise", "scale_colwise", "amax_tensor",
                                            "output_rowwise", "output_colwise"))]
    return Prepared("nvfp4_partial_cast", hs, (rows, cols, start_offset, out_offset),
                    [t for t in ts if t is not None])


class Prepared:
    """One library call with its tensor handles marshalled once.

    ``call(stream)`` launches it on the given stream (a torch stream or a raw
    cudaStream_t value) with the current CUDA device, which must be the device the
    tensors live on.  The tensors are kept alive by this object; their storage must
    not move between calls (re-prepare after reallocating).
    """

    __slots__ = ("fn", "args", "handles", "tensors", "device")

    def __init__(self, fn_name, handles, scalars, tensors, job_array=None):
        self.fn = getattr(_capi.load(), fn_name)
        self.handles = handles
        if job_array is not None:  # batched entry: (job array, count)
            self.args = (job_array, int(scalars[0]))
        else:
            self.args = tuple(ctypes.byref(h) for h in handles) + tuple(int(v) for v in scalars)
        self.tensors = tensors
        self.device = _device_of(*tensors)

    def call(self, stream=None) -> None:
        if stream is None or hasattr(stream, "cuda_stream"):
            stream = _stream(stream, self.tensors[0] if self.tensors else None)
        rc = self.fn(*self.args, stream)
        if rc != 0:
            _capi.check(rc)


def prepare_partial_amax(input, amax_rowwise, amax_colwise, rows, cols, start_offset) -> Prepared:
    hs = [handle(input, "input"), handle(amax_rowwise, "amax_rowwise"),
          handle(amax_colwise, "amax_colwise")]
    return Prepared("mxfp8_partial_amax", hs, (rows, cols, start_offset),
                    [t for t in (input, amax_rowwise, amax_colwise) if t is not None])


def prepare_amax_max_reduce(slots, out) -> Prepared:
    return Prepared("mxfp8_amax_max_reduce", [handle(slots, "slots"), handle(out, "out")], (),
                    [slots, out])


def prepare_update_scales(amax_rowwise, amax_colwise, scale_inv_rowwise, scale_inv_colwise,
                          rows, cols) -> Prepared:
    ts = (amax_rowwise, amax_colwise, scale_inv_rowwise, scale_inv_colwise)
    hs = [handle(t, n) for t, n in zip(ts, ("amax_rowwise", "amax_colwise", "scale_inv_rowwise",
                                            "scale_inv_colwise"))]
    return Prepared("mxfp8_update_scales", hs, (rows, cols), [t for t in ts if t is not None])


def prepare_partial_cast(input, scale_inv_rowwise, scale_inv_colwise, output_rowwise,
                         output_colwise, rows, cols, start_offset, out_offset=None,
                         allow_host=False) -> Prepared:
    """``allow_host``: the outputs may be page-locked host memory the device can access
    (the kernel's stores then cross the CPU-GPU link)."""
    if out_offset is None:
        out_offset = start_offset
    ts = (input, scale_inv_rowwise, scale_inv_colwise, output_rowwise, output_colwise)
    names = ("input", "scale_inv_rowwise", "scale_inv_colwise", "output_rowwise", "output_colwise")
    hs = [handle(t, n, allow_host and n.startswith("output")) for t, n in zip(ts, names)]
    return Prepared("mxfp8_partial_cast", hs, (rows, cols, start_offset, out_offset),
                    [t for t in ts if t is not None])


def prepare_partial_amax_batched(jobs) -> Prepared:
    arr, keep = _amax_jobs(jobs)
    return Prepared("mxfp8_partial_amax_batched", [arr], (len(jobs),), keep, job_array=arr)


def prepare_update_scales_batched(jobs) -> Prepared:
    arr, keep = _scale_jobs(jobs)
    return Prepared("mxfp8_update_scales_batched", [arr], (len(jobs),), keep, job_array=arr)


def prepare_amax_max_reduce_update_scales(slots, reduced, jobs) -> Prepared:
    arr, keep = _scale_jobs(jobs)
    hs = [handle(slots, "slots"), handle(reduced, "reduced")]
    pr = Prepared("mxfp8_amax_max_reduce_update_scales", hs, (), keep + [slots, reduced])
    pr.args = (ctypes.byref(hs[0]), ctypes.byref(hs[1]), arr, len(jobs))
    pr.handles = hs + [arr]
    return pr


def prepare_amax_max_reduce_update_scales_ranged(slots, reduced, jobs, slot_ranges) -> Prepared:
    arr, keep = _scale_jobs(jobs)
    rng, nr = _ranges_array(slot_ranges)
    hs = [handle(slots, "slots"), handle(reduced, "reduced")]
    pr = Prepared("mxfp8_amax_max_reduce_update_scales_ranged", hs, (), keep + [slots, reduced])
    pr.args = (ctypes.byref(hs[0]), ctypes.byref(hs[1]), arr, len(jobs), rng, nr)
    pr.handles = hs + [arr, rng]
    return pr


def prepare_partial_cast_batched(jobs) -> Prepared:
    arr, keep = _cast_jobs(jobs)
    return Prepared("mxfp8_partial_cast_batched", [arr], (len(jobs),), keep, job_array=arr)


def prepare_quantize_whole_blocks_batched(jobs) -> Prepared:
    arr, keep = _quantize_jobs(jobs)
    return Prepared("mxfp8_quantize_whole_blocks_batched", [arr], (len(jobs),), keep, job_array=arr)


def block_shapes(rows: int, cols: int):
    """Compact (rowwise, columnwise) block-grid shapes: [rows, ceil(cols/32)], [ceil(rows/32), cols]."""
    return (rows, (cols + 31) // 32), ((rows + 31) // 32, cols)
