// Partial cast kernel templates: master values of a contiguous fragment -> model
// dtype (BF16, or FP16; nearest-even) -> E4M3 (nearest-even, saturating at 448),
// scaled by the E8M0 block scales, written in place into the rowwise and
// (optionally) columnwise outputs.  cast_f32.cu / cast_bf16.cu instantiate them for
// FP32 and BF16 master values with word-aligned outputs, cast_*_unaligned.cu for
// outputs that are not.
//
// Follows "Support row-only MXFP8 distributed master-weight casts" (sections
// "Changes" and the flow diagram): rounding goes through the model dtype, the
// rowwise output is always written, and the columnwise output -- with every read
// of its scales -- is removed at compile time when the weight has none (a batch
// mixing row-only and bidirectional weights picks the specialisation per tile).
//
// Work unit and tile classes as in the amax kernel: one warp per 32 x (32*V)
// tile, one 16-byte input chunk per lane per row; a row's V output bytes per
// direction leave as one 4- (FP32) or 8-byte (BF16) store when the output is
// word-aligned (naturally aligned pieces otherwise), so a warp writes 128 or 256
// contiguous bytes per row and direction.  The columnwise multipliers of a
// lane's V columns are loaded once per tile; the rowwise multiplier once per row.
#pragma once

#include "common.cuh"

namespace mxfp8 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowBatch = 8;     // rows per batch of 16-byte loads, aligned fast path
constexpr int kShiftBatch = 4;   // rows per batch on the realigning path (extra words per row)
constexpr int kMaskBatch = 4;    // rows per batch of predicated per-element loads
// Resident blocks per SM the register allocation must allow (an unconstrained allocation
// leaves room for 1-2): 3, where some variants then spill a few dozen bytes to L1 and
// still run faster (FP32 config-5 cast phase -4 %, BF16 16384x6144 cast -4 %); 2 for the
// BF16 kernels with unaligned outputs, whose piece stores spill more.
#ifndef MXFP8_CAST_SHIFT_MIN_BLOCKS
#define MXFP8_CAST_SHIFT_MIN_BLOCKS 3
#endif
template <class T, int N, bool kVec, bool kShift>
constexpr int min_blocks() {
  return (T::kBytes == 2 && !kVec) ? 2 : (kShift ? MXFP8_CAST_SHIFT_MIN_BLOCKS : 3);
}

// Columnwise multipliers 2^(127 - s) of this lane's V columns in column band row0/32.
template <class T>
__device__ __forceinline__ void colwise_multipliers(const CastParams& p, int64_t row0, int64_t j,
                                                    float (&mc)[T::V]) {
  const uint8_t* sc = p.s_c + (row0 >> 5) * p.ld_sc + j;
  if (p.vec_sc) {
    if constexpr (T::V == 4) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(sc);
#pragma unroll
      for (int k = 0; k < 4; ++k) mc[k] = scale_multiplier((w >> (8 * k)) & 0xffu);
    } else {
      const uint2 w = *reinterpret_cast<const uint2*>(sc);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        mc[k] = scale_multiplier((w.x >> (8 * k)) & 0xffu);
        mc[k + 4] = scale_multiplier((w.y >> (8 * k)) & 0xffu);
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < T::V; ++k) mc[k] = scale_multiplier(sc[k]);
  }
}

// Whole tile inside the fragment: 16-byte loads (realigned for a shifted virtual
// base), one scale byte per row, word stores when the outputs are aligned.
// kM: byte offset of the outputs' virtual bases past a V-byte boundary (0: word
// stores; > 0: aligned pieces; < 0: bytes, the two outputs differ).
// kEdge: a tile cut by the matrix's right edge (kTileEdge, word-aligned outputs): the lanes
// past it read no input, scale or multiplier and store nothing.
template <class T, bool kCol, int kS, int kM, int kModel, bool kEdge = false>
__device__ __forceinline__ void cast_tile_fast(const CastParams& p, int64_t row0, int64_t col0,
                                               int lane, int r_lo, int r_hi) {
  static_assert(!kEdge || (kS == 0 && kM == 0), "edge tiles are aligned, with word stores");
  const int64_t cols = p.g.cols;
  const int64_t j = col0 + lane * T::V;
  const bool active = !kEdge || j < cols;
  const char* src = static_cast<const char*>(p.in) + (row0 * cols + j - p.g.start) * T::kBytes;
  const int64_t row_bytes = cols * T::kBytes;
  const uint8_t* srow = p.s_r + row0 * p.ld_sr + (j >> 5);
  const int64_t o0 = row0 * cols + j + p.out_shift;
  // FP32 realigning tiles batch 8 rows (the extra words loaded by row lanes keep the
  // registers in bounds); BF16 ones 4 rows with lane 31 loading them
  constexpr bool kRowLanes = kS != 0 && T::kBytes == 4;
  constexpr int NB = kS ? (kRowLanes ? kRowBatch : kShiftBatch) : kRowBatch;
  float mc[T::V];
  if constexpr (kCol) {
    if (active) {
      colwise_multipliers<T>(p, row0, j, mc);
    } else {
#pragma unroll
      for (int k = 0; k < T::V; ++k) mc[k] = 0.0f;
    }
  }
#pragma unroll 1
  for (int rb = r_lo; rb < r_hi; rb += NB) {
    uint4 v[NB];
    uint32_t sb[NB];
    if constexpr (kEdge) {
#pragma unroll
      for (int r = 0; r < NB; ++r) {
        sb[r] = active ? srow[(rb + r) * p.ld_sr] : 0u;
        v[r] = active ? ld_stream16(src + (rb + r) * row_bytes) : make_uint4(0u, 0u, 0u, 0u);
      }
    } else {
#pragma unroll
      for (int r = 0; r < NB; ++r) sb[r] = srow[(rb + r) * p.ld_sr];
      load_rows<NB, kS, false, kRowLanes>(v, src + rb * row_bytes, row_bytes, lane);
    }
#pragma unroll
    for (int r = 0; r < NB; ++r) {
      float mr[T::V];
      const float m = scale_multiplier(sb[r]);
#pragma unroll
      for (int k = 0; k < T::V; ++k) mr[k] = m;
      uint2 qr, qc;
      cast_chunk<T, kModel, kCol>(v[r], mr, mc, qr, qc);
      const int64_t o = o0 + (rb + r) * cols;
      if (active) {
        store_chunk_at<T, kM>(p.out_r + o, qr);
        if constexpr (kCol) store_chunk_at<T, kM>(p.out_c + o, qc);
      }
    }
  }
}

// Fast tile with outputs that are not V-aligned (kVec false).  The offset m of each
// output past a V-byte boundary is the same for every row and lane of the tile; when
// both outputs share it, it selects a specialisation with aligned piece stores: for
// an aligned input any m, for a realigned input the m that a fragment-sized output in
// an aligned allocation has (input offset / element size) -- other combinations store
// bytes.
template <class T, bool kCol, int kS, int kModel>
__device__ __forceinline__ void cast_tile_unaligned(const CastParams& p, int64_t row0, int64_t col0,
                                                    int lane, int r_lo, int r_hi) {
  constexpr uint32_t V = T::V;
  const uint32_t mr = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(p.out_r) + uintptr_t(p.out_shift)) & (V - 1);
  const uint32_t mc =
      kCol ? static_cast<uint32_t>(reinterpret_cast<uintptr_t>(p.out_c) + uintptr_t(p.out_shift)) & (V - 1) : mr;
  if (mr != mc || mr == 0) {
    cast_tile_fast<T, kCol, kS, -1, kModel>(p, row0, col0, lane, r_lo, r_hi);
  } else if constexpr (kS != 0) {
    constexpr int M = (kS / T::kBytes) % int(V);
    if (M != 0 && mr == uint32_t(M)) {
      cast_tile_fast<T, kCol, kS, M, kModel>(p, row0, col0, lane, r_lo, r_hi);
    } else {
      cast_tile_fast<T, kCol, kS, -1, kModel>(p, row0, col0, lane, r_lo, r_hi);
    }
  } else {
    with_out_offset<T>(mr, [&](auto m) {
      cast_tile_fast<T, kCol, 0, decltype(m)::value, kModel>(p, row0, col0, lane, r_lo, r_hi);
    });
  }
}

// A fast tile of a launch whose fragments are all aligned (kShift false) or of a launch
// that holds realigning fragments (kShift true: each fragment's own offset, 0 included,
// picks the specialisation).
template <class T, bool kCol, bool kShift, bool kVec, int kModel>
__device__ __forceinline__ void cast_fast(const CastParams& p, int64_t row0, int64_t col0, int lane,
                                          int r_lo = 0, int r_hi = 32) {
  if constexpr (kShift) {
    if (p.g.shift == 0) {
      if constexpr (kVec) {
        cast_tile_fast<T, kCol, 0, 0, kModel>(p, row0, col0, lane, r_lo, r_hi);
      } else {
        cast_tile_unaligned<T, kCol, 0, kModel>(p, row0, col0, lane, r_lo, r_hi);
      }
      return;
    }
    with_shift<T>(p.g.shift, [&](auto s) {
      if constexpr (kVec) {
        cast_tile_fast<T, kCol, decltype(s)::value, 0, kModel>(p, row0, col0, lane, r_lo, r_hi);
      } else {
        cast_tile_unaligned<T, kCol, decltype(s)::value, kModel>(p, row0, col0, lane, r_lo, r_hi);
      }
    });
  } else {
    if constexpr (kVec) {
      cast_tile_fast<T, kCol, 0, 0, kModel>(p, row0, col0, lane, r_lo, r_hi);
    } else {
      cast_tile_unaligned<T, kCol, 0, kModel>(p, row0, col0, lane, r_lo, r_hi);
    }
  }
}

// Tile cut by the fragment boundary or the matrix edge: loads a batch of rows at a
// time (16-byte loads for chunks wholly inside the fragment, predicated per-element
// loads otherwise), one scale byte per row and block, and stores only the
// fragment's elements (a word per whole chunk when the output is aligned).  Inlined
// into the kernel, as in the amax kernel.
// MB: rows per batch of predicated loads.
template <class T, bool kCol, bool kVec, int kModel, int MB = kMaskBatch>
__device__ __forceinline__ void cast_tile_masked(const CastParams& p, int64_t row0, int64_t col0,
                                              int lane, int r_lo = 0, int r_hi = 32) {
  constexpr uint64_t kChunkBits = (uint64_t(1) << T::V) - 1;
  const FragGeom& g = p.g;
  const int64_t j = col0 + lane * T::V;
  if (j >= g.cols) return;  // no element of this lane is inside the matrix
  const bool word_ok = kVec && g.fast_ok;  // whole chunks sit on V-aligned output addresses
  const int64_t blk = j >> 5;              // the lane's V columns share one row block
  float mc[T::V];
  if constexpr (kCol) {
#pragma unroll
    for (int k = 0; k < T::V; ++k)
      mc[k] = j + k < g.cols ? scale_multiplier(p.s_c[(row0 >> 5) * p.ld_sc + j + k]) : 0.0f;
  }
#pragma unroll 1
  for (int rb = r_lo; rb < r_hi && row0 + rb < g.rows; rb += MB) {
    uint4 v[MB];
    const uint64_t valid = load_rows_masked<T, MB>(v, g, p.in, row0 + rb, j);
    if (valid == 0) continue;
    float mrow[MB];
#pragma unroll
    for (int r = 0; r < MB; ++r) {
      const int64_t i = row0 + rb + r;
      mrow[r] = ((valid >> (r * T::V)) & kChunkBits) ? scale_multiplier(p.s_r[i * p.ld_sr + blk]) : 0.0f;
    }
#pragma unroll
    for (int r = 0; r < MB; ++r) {
      const uint64_t bits = (valid >> (r * T::V)) & kChunkBits;
      if (bits == 0) continue;
      const int64_t i = row0 + rb + r;
      float mr[T::V];
#pragma unroll
      for (int k = 0; k < T::V; ++k) mr[k] = mrow[r];
      uint2 qr, qc = make_uint2(0u, 0u);
      cast_chunk<T, kModel, kCol>(v[r], mr, mc, qr, qc);
      const int64_t o = i * g.cols + j + p.out_shift;
      if (word_ok && bits == kChunkBits) {
        store_chunk<T, true>(p.out_r + o, qr);
        if constexpr (kCol) store_chunk<T, true>(p.out_c + o, qc);
      } else {
#pragma unroll
        for (int k = 0; k < T::V; ++k) {
          if (bits & (uint64_t(1) << k)) {
            const int sh = 8 * (k & 3);
            p.out_r[o + k] = static_cast<uint8_t>((k < 4 ? qr.x : qr.y) >> sh);
            if constexpr (kCol) p.out_c[o + k] = static_cast<uint8_t>((k < 4 ? qc.x : qc.y) >> sh);
          }
        }
      }
    }
  }
}

// kSplit: four warps per tile, a quarter of its rows each (the cast needs no exchange
// between them), for single-fragment launches with few tiles; kSplit 2 also takes tiles cut
// by the matrix's right edge on the fast path (instantiated only for weights whose width is
// not a multiple of the tile's: the extra path costs registers).
template <class T, int kDirs, bool kShift, bool kVec, int kModel, int N, int kSplit>
__global__ void __launch_bounds__(kThreads, min_blocks<T, N, kVec, kShift>()) k_partial_cast(
    const __grid_constant__ JobBatch<CastParams, N> b) {
  grid_dependency_sync();
  constexpr int TW = tile_width<T>();
  constexpr int kParts = kSplit ? 4 : 1;
  const int lane = threadIdx.x & 31;
  const int64_t total = (b.prefix_a[b.njobs] + b.prefix_b[b.njobs]) * kParts;
  const int64_t stride = int64_t(gridDim.x) * kWarps;
  for (int64_t u = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5); u < total; u += stride) {
    const int64_t t = kSplit ? u >> 2 : u;
    const int r_lo = kSplit ? 8 * int(u & 3) : 0, r_hi = kSplit ? r_lo + 8 : 32;
    int64_t row0, col0;
    const CastParams& p = b.job[batch_tile(b, t, TW, row0, col0)];
    const int kind = kSplit == 2 && kVec ? classify_tile_edge<T>(p.g, row0, col0, TW)
                                         : classify_tile<T>(p.g, row0, col0, TW);
    const bool col = kDirs == kMixed ? p.out_c != nullptr : kDirs == kBidir;
    if constexpr (kSplit == 2 && kVec) {
      if (kind == kTileEdge) {
        if (col) {
          if constexpr (kDirs != kRowOnly) cast_tile_fast<T, true, 0, 0, kModel, true>(p, row0, col0, lane, r_lo, r_hi);
        } else {
          if constexpr (kDirs != kBidir) cast_tile_fast<T, false, 0, 0, kModel, true>(p, row0, col0, lane, r_lo, r_hi);
        }
        continue;
      }
    }
    if (kind == kTileFast) {
      if (col) {
        if constexpr (kDirs != kRowOnly) cast_fast<T, true, kShift, kVec, kModel>(p, row0, col0, lane, r_lo, r_hi);
      } else {
        if constexpr (kDirs != kBidir) cast_fast<T, false, kShift, kVec, kModel>(p, row0, col0, lane, r_lo, r_hi);
      }
    } else if (kind == kTileMasked) {
      if (col) {
        if constexpr (kDirs != kRowOnly) cast_tile_masked<T, true, kVec, kModel>(p, row0, col0, lane, r_lo, r_hi);
      } else {
        if constexpr (kDirs != kBidir) cast_tile_masked<T, false, kVec, kModel>(p, row0, col0, lane, r_lo, r_hi);
      }
    }
  }
}

template <class T, int kDirs, bool kShift, bool kVec, int kModel, int N>
cudaError_t launch_n(const CastParams* jobs, int n, const DeviceInfo& dev, cudaStream_t stream) {
  JobBatch<CastParams, N> b;
  const int64_t total = fill_batch(b, jobs, n);
  if (total == 0) return cudaSuccess;
  if constexpr (N == 1 && !kShift && kDirs != kMixed) {
    if (total <= split_max_tiles(dev, MXFP8_CAST_SPLIT_TILES_PER_SM)) {  // few tiles: four warps per tile
      const unsigned grid = tile_grid(total * 4, kWarps);
      if constexpr (kVec) {  // the edge path stores whole words
        if (jobs[0].g.cols % tile_width<T>() != 0)
          return launch_kernel(k_partial_cast<T, kDirs, kShift, kVec, kModel, N, 2>, grid, kThreads, 0, stream, b);
      }
      return launch_kernel(k_partial_cast<T, kDirs, kShift, kVec, kModel, N, 1>, grid, kThreads, 0, stream, b);
    }
  }
  const unsigned grid = tile_grid(total, kWarps);
  return launch_kernel(k_partial_cast<T, kDirs, kShift, kVec, kModel, N, 0>, grid, kThreads, 0, stream, b);
}

// One launch per batch of at most kMaxBatchJobs jobs, with the kernel for the batch's
// direction set; single BF16-model jobs use the one-entry job table.
template <class T, bool kShift, bool kVec, int kModel>
cudaError_t launch(const CastParams* jobs, int n, const DeviceInfo& dev, cudaStream_t stream) {
  auto colwise = [](const CastParams& p) { return p.out_c != nullptr; };
  if constexpr (kModel == kModelBF16) {
    if (n == 1) {
      return colwise(jobs[0]) ? launch_n<T, kBidir, kShift, kVec, kModel, 1>(jobs, 1, dev, stream)
                              : launch_n<T, kRowOnly, kShift, kVec, kModel, 1>(jobs, 1, dev, stream);
    }
  }
  for (int k = 0; k < n; k += kMaxBatchJobs) {
    const int m = n - k < kMaxBatchJobs ? n - k : kMaxBatchJobs;
    cudaError_t e;
    switch (batch_dirs(jobs + k, m, colwise)) {
      case kRowOnly:
        e = launch_n<T, kRowOnly, kShift, kVec, kModel, kMaxBatchJobs>(jobs + k, m, dev, stream);
        break;
      case kBidir:
        e = launch_n<T, kBidir, kShift, kVec, kModel, kMaxBatchJobs>(jobs + k, m, dev, stream);
        break;
      default:
        e = launch_n<T, kMixed, kShift, kVec, kModel, kMaxBatchJobs>(jobs + k, m, dev, stream);
        break;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// All launches for one input dtype T, output alignment kVec and model dtype kModel.
template <class T, bool kVec, int kModel>
cudaError_t launch_for_model(const CastParams* jobs, int n, bool shifted, const DeviceInfo& dev,
                             cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  return shifted ? launch<T, true, kVec, kModel>(jobs, n, dev, stream)
                 : launch<T, false, kVec, kModel>(jobs, n, dev, stream);
}

// All launches for one input dtype T and output alignment kVec (instantiated by that
// combination's translation unit).
template <class T, bool kVec>
cudaError_t launch_for_dtype(const CastParams* jobs, int n, bool shifted, int model,
                             const DeviceInfo& dev, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  if (model == kModelF16) {
    return shifted ? launch<T, true, kVec, kModelF16>(jobs, n, dev, stream)
                   : launch<T, false, kVec, kModelF16>(jobs, n, dev, stream);
  }
  return shifted ? launch<T, true, kVec, kModelBF16>(jobs, n, dev, stream)
                 : launch<T, false, kVec, kModelBF16>(jobs, n, dev, stream);
}

}  // namespace

}  // namespace mxfp8
