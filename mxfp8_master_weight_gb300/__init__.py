"""GB300 (sm_103a) partial MXFP8 cast of high-precision master weights.

The data-parallel hot path of a distributed master-weight writeback: partial
amax over a contiguous fragment -> packed MAX reduction -> E8M0 scale update ->
partial cast to E4M3 (rowwise and optionally columnwise), as hand-written CUDA
kernels behind a C ABI (``include/mxfp8_partial.h``).  This package holds the
ctypes binding (``api``), the multi-fragment driver (``driver``), the build
script (``build``) and the seeded synthetic workloads (``workloads``).

Importing the package does not load the CUDA library; the first call does, and
raises if the library was not built.
"""
from .api import (block_shapes, mxfp8_amax_max_reduce, mxfp8_amax_max_reduce_update_scales,
                  mxfp8_amax_max_reduce_update_scales_ranged, mxfp8_partial_amax,
                  mxfp8_partial_amax_batched, mxfp8_partial_cast, mxfp8_partial_cast_batched,
                  mxfp8_quantize_whole_blocks, mxfp8_quantize_whole_blocks_batched,
                  mxfp8_swizzle_scales, mxfp8_swizzled_scales_size, mxfp8_update_scales,
                  mxfp8_update_scales_batched)

__all__ = ["mxfp8_partial_amax", "mxfp8_amax_max_reduce", "mxfp8_amax_max_reduce_update_scales",
           "mxfp8_amax_max_reduce_update_scales_ranged",
           "mxfp8_update_scales",
           "mxfp8_partial_cast", "mxfp8_partial_amax_batched", "mxfp8_update_scales_batched",
           "mxfp8_partial_cast_batched", "mxfp8_quantize_whole_blocks",
           "mxfp8_quantize_whole_blocks_batched", "mxfp8_swizzle_scales",
           "mxfp8_swizzled_scales_size", "block_shapes"]
