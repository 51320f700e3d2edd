// One-pass MXFP8 quantisation of fragments made of whole blocks.
//
// When every 1x32 (and, for a bidirectional weight, every 32x1) block a fragment
// touches lies wholly inside it -- a rank that owns whole weights or whole 32-row
// bands, or a single rank -- the block maxima need no cross-rank reduction, and the
// four steps of "Support row-only MXFP8 distributed master-weight casts" (amax,
// MAX reduction, scale update, cast; flow diagram) collapse into one kernel with
// the same results: the MAX over one rank is the identity.
//
// Each warp owns a 32-row tile, as in the split kernels, and reads it twice: pass 1
// folds the block maxima, derives and stores the E8M0 scales (and, on request, the
// amaxes); pass 2 re-reads the tile and writes the E4M3 data.  Pass 1 loads carry an
// L2 evict_last policy and pass 2 loads evict_first, so the second read is served
// from L2 and HBM sees the input once: 4 + 2 bytes per FP32 element (bidirectional)
// instead of 4 + 4 + 2 for the split amax and cast kernels.
#pragma once

#include <atomic>

#include "common.cuh"

namespace mxfp8 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowBatch = 8;
constexpr int kShiftBatch = 4;
constexpr int kMaskBatch = 4;
constexpr int kMaxDevices = 64;
constexpr int kMaxGroups = 8;  // row blocks per warp tile (BF16: 256 columns / 32)
// Resident blocks per SM the register allocation must allow: the two passes of a tile
// run back to back in one warp, so latency is hidden only across warps.
#ifndef MXFP8_FUSED_MIN_BLOCKS
#define MXFP8_FUSED_MIN_BLOCKS 3
#endif
constexpr int kFusedMinBlocks = MXFP8_FUSED_MIN_BLOCKS;

// Multipliers 2^(127 - s) of the E8M0 scales of the 32 rows' row blocks of each warp's
// tile, handed from pass 1 (where one lane per block derives them) to pass 2 (where every
// lane of the block reads its row's multiplier).
struct RowScales {
  float m[kWarps][32][kMaxGroups];
};

template <class T, bool kCol>
__device__ __forceinline__ void store_col_stats(const FusedParams& p, int64_t row0, int64_t j,
                                                const uint4& colmax, float (&mc)[T::V]) {
  const int64_t band = row0 >> 5;
  uint32_t sb[T::V];
#pragma unroll
  for (int k = 0; k < T::V; ++k) {
    sb[k] = e8m0_from_bits<T>(chunk_get<T>(colmax, k));
    mc[k] = scale_multiplier(sb[k]);
  }
  if (p.amax_c != nullptr) {
    const int64_t base = band * p.ld_c + j;
    const uint4 out = canonical_nan_chunk<T>(colmax);
    if (p.vec_c) {
      *reinterpret_cast<uint4*>(static_cast<char*>(p.amax_c) + base * T::kBytes) = out;
    } else {
#pragma unroll
      for (int k = 0; k < T::V; ++k) store_bits<T>(p.amax_c, base + k, chunk_get<T>(out, k));
    }
  }
  uint8_t* dst = p.s_c + band * p.ld_sc + j;
  if (p.vec_sc) {
    uint2 w = make_uint2(0u, 0u);
#pragma unroll
    for (int k = 0; k < T::V; ++k) (k < 4 ? w.x : w.y) |= sb[k] << (8 * (k & 3));
    if constexpr (T::V == 4) {
      *reinterpret_cast<uint32_t*>(dst) = w.x;
    } else {
      *reinterpret_cast<uint2*>(dst) = w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < T::V; ++k) dst[k] = static_cast<uint8_t>(sb[k]);
  }
}

// Exponent-only maxima.  A block's E8M0 scale depends only on the exponent field of its
// amax, and the maximum of |x| commutes with keeping the top 16 bits of the FP32 pattern
// (a monotone map on non-negative patterns), so when no amax output is requested the
// FP32 maxima are taken on packed high halves: two columns per register, two rows per
// butterfly.
__device__ __forceinline__ uint32_t e8m0_from_half(uint32_t h) {
  const uint32_t e = (h >> 7) & 0xffu;
  return e == 0xffu ? 0xffu : (e > 8u ? e - 8u : 0u);
}

// High halves of two FP32 words, sign cleared: (|b| >> 16) << 16 | |a| >> 16.
__device__ __forceinline__ uint32_t abs_hi_halves(uint32_t a, uint32_t b) {
  return __byte_perm(a, b, 0x7632) & 0x7fff7fffu;
}

template <bool kCol>
__device__ __forceinline__ void store_col_scales_half(const FusedParams& p, int64_t row0, int64_t j,
                                                      uint32_t c01, uint32_t c23, float (&mc)[4]) {
  const uint32_t sb[4] = {e8m0_from_half(c01 & 0xffffu), e8m0_from_half(c01 >> 16),
                          e8m0_from_half(c23 & 0xffffu), e8m0_from_half(c23 >> 16)};
#pragma unroll
  for (int k = 0; k < 4; ++k) mc[k] = scale_multiplier(sb[k]);
  uint8_t* dst = p.s_c + (row0 >> 5) * p.ld_sc + j;
  if (p.vec_sc) {
    *reinterpret_cast<uint32_t*>(dst) = sb[0] | (sb[1] << 8) | (sb[2] << 16) | (sb[3] << 24);
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) dst[k] = static_cast<uint8_t>(sb[k]);
  }
}

template <class T, bool kCol, int kS, bool kVec, int kModel, bool kExp>
__device__ __forceinline__ void fused_tile_fast(const FusedParams& p, int64_t row0, int64_t col0,
                                                int lane, RowScales& rsc, int warp) {
  const int64_t cols = p.g.cols;
  const int64_t j = col0 + lane * T::V;
  const char* src = static_cast<const char*>(p.in) + (row0 * cols + j - p.g.start) * T::kBytes;
  const int64_t row_bytes = cols * T::kBytes;
  constexpr int NB = kS ? kShiftBatch : kRowBatch;
  const int grp = lane / T::G;
  const bool writer = (lane % T::G) == 0;
  const int64_t blk = j >> 5;
  const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();

  // pass 1: block maxima -> scales
  float mc[T::V];
  if constexpr (kExp) {
    static_assert(T::kBytes == 4, "exponent-only maxima are taken on FP32 high halves");
    uint32_t c01 = 0u, c23 = 0u;  // column maxima, two columns per register
#pragma unroll 1
    for (int rb = 0; rb < 32; rb += NB) {
      uint4 v[NB];
      load_rows<NB, kS, true>(v, src + rb * row_bytes, row_bytes, lane, keep);
#pragma unroll
      for (int r = 0; r < NB; r += 2) {
        const uint32_t a01 = abs_hi_halves(v[r].x, v[r].y), a23 = abs_hi_halves(v[r].z, v[r].w);
        const uint32_t b01 = abs_hi_halves(v[r + 1].x, v[r + 1].y);
        const uint32_t b23 = abs_hi_halves(v[r + 1].z, v[r + 1].w);
        if constexpr (kCol) {
          c01 = __vmaxu2(c01, __vmaxu2(a01, b01));
          c23 = __vmaxu2(c23, __vmaxu2(a23, b23));
        }
        // rows r and r+1 in the low and high halves of one word, one butterfly for both
        const uint32_t ha = __vmaxu2(a01, a23), hb = __vmaxu2(b01, b23);
        uint32_t w = __vmaxu2(__byte_perm(ha, hb, 0x5410), __byte_perm(ha, hb, 0x7632));
#pragma unroll
        for (int off = 1; off < T::G; off <<= 1) w = __vmaxu2(w, __shfl_xor_sync(kFullMask, w, off));
        if (writer) {
          const int64_t i = row0 + rb + r;
          const uint32_t ea = e8m0_from_half(w & 0xffffu), eb = e8m0_from_half(w >> 16);
          rsc.m[warp][rb + r][grp] = scale_multiplier(ea);
          rsc.m[warp][rb + r + 1][grp] = scale_multiplier(eb);
          p.s_r[i * p.ld_sr + blk] = static_cast<uint8_t>(ea);
          p.s_r[(i + 1) * p.ld_sr + blk] = static_cast<uint8_t>(eb);
        }
      }
    }
    if constexpr (kCol) store_col_scales_half<kCol>(p, row0, j, c01, c23, mc);
  } else {
    uint4 colmax = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
    for (int rb = 0; rb < 32; rb += NB) {
      uint4 v[NB];
      load_rows<NB, kS, true>(v, src + rb * row_bytes, row_bytes, lane, keep);
#pragma unroll
      for (int r = 0; r < NB; ++r) {
        const uint4 a = chunk_abs<T>(v[r]);
        if constexpr (kCol) colmax = chunk_max<T>(colmax, a);
        const uint32_t m = group_max<T>(chunk_reduce<T>(a));
        if (writer) {
          const int64_t i = row0 + rb + r;
          const uint32_t e = e8m0_from_bits<T>(m);
          rsc.m[warp][rb + r][grp] = scale_multiplier(e);
          p.s_r[i * p.ld_sr + blk] = static_cast<uint8_t>(e);
          if (p.amax_r != nullptr) store_bits<T>(p.amax_r, i * p.ld_r + blk, canonical_nan<T>(m));
        }
      }
    }
    if constexpr (kCol) store_col_stats<T, kCol>(p, row0, j, colmax, mc);
  }
  __syncwarp();

  // pass 2: cast (the tile's lines are still in L2)
  const int64_t o0 = row0 * cols + j + p.out_shift;
#pragma unroll 1
  for (int rb = 0; rb < 32; rb += NB) {
    uint4 v[NB];
    load_rows<NB, kS, true>(v, src + rb * row_bytes, row_bytes, lane, drop);
#pragma unroll
    for (int r = 0; r < NB; ++r) {
      float mr[T::V];
      const float m = rsc.m[warp][rb + r][grp];
#pragma unroll
      for (int k = 0; k < T::V; ++k) mr[k] = m;
      uint2 qr, qc;
      cast_chunk<T, kModel, kCol>(v[r], mr, mc, qr, qc);
      const int64_t o = o0 + (rb + r) * cols;
      store_chunk<T, kVec>(p.out_r + o, qr);
      if constexpr (kCol) store_chunk<T, kVec>(p.out_c + o, qc);
    }
  }
  __syncwarp();
}

// A fast tile of a launch whose fragments are all aligned or all shifted.
template <class T, bool kCol, bool kShift, bool kVec, int kModel, bool kExp>
__device__ __forceinline__ void fused_fast(const FusedParams& p, int64_t row0, int64_t col0, int lane,
                                           RowScales& rsc, int warp) {
  if constexpr (kShift) {
    with_shift<T>(p.g.shift, [&](auto s) {
      fused_tile_fast<T, kCol, decltype(s)::value, kVec, kModel, kExp>(p, row0, col0, lane, rsc, warp);
    });
  } else {
    fused_tile_fast<T, kCol, 0, kVec, kModel, kExp>(p, row0, col0, lane, rsc, warp);
  }
}

// Tile cut by the fragment boundary or the matrix edge.  Every block the fragment
// touches is whole, so the maxima over the loaded elements are the block maxima.
template <class T, bool kCol, bool kVec, int kModel>
__device__ __noinline__ void fused_tile_masked(const FusedParams& p, int64_t row0, int64_t col0,
                                               int lane, RowScales& rsc, int warp) {
  constexpr uint64_t kChunkBits = (uint64_t(1) << T::V) - 1;
  const FragGeom& g = p.g;
  const int64_t j = col0 + lane * T::V;
  const int grp = lane / T::G;
  const bool writer = (lane % T::G) == 0;
  const int64_t b0 = j & ~int64_t(31);
  const bool word_ok = kVec && g.fast_ok;
  uint4 colmax = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
  for (int rb = 0; rb < 32; rb += kMaskBatch) {  // warp-uniform
    uint4 v[kMaskBatch];
    load_rows_masked<T, kMaskBatch>(v, g, p.in, row0 + rb, j);
#pragma unroll
    for (int r = 0; r < kMaskBatch; ++r) {
      const uint4 a = chunk_abs<T>(v[r]);
      if constexpr (kCol) colmax = chunk_max<T>(colmax, a);
      const uint32_t m = group_max<T>(chunk_reduce<T>(a));
      const int64_t i = row0 + rb + r;
      const uint32_t e = e8m0_from_bits<T>(m);
      if (writer) rsc.m[warp][rb + r][grp] = scale_multiplier(e);
      if (writer && i < g.rows && b0 < g.cols &&
          row_span_meets(g, i, b0, min(b0 + 31, g.cols - 1))) {
        p.s_r[i * p.ld_sr + (b0 >> 5)] = static_cast<uint8_t>(e);
        if (p.amax_r != nullptr) store_bits<T>(p.amax_r, i * p.ld_r + (b0 >> 5), canonical_nan<T>(m));
      }
    }
  }
  float mc[T::V];
  if constexpr (kCol) {
    const int64_t r_end = min(row0 + 32, g.rows);
#pragma unroll
    for (int k = 0; k < T::V; ++k) {
      const int64_t col = j + k;
      const uint32_t m = chunk_get<T>(colmax, k);
      const uint32_t e = e8m0_from_bits<T>(m);
      mc[k] = scale_multiplier(e);
      if (col < g.cols && column_meets(g, col, row0, r_end)) {
        p.s_c[(row0 >> 5) * p.ld_sc + col] = static_cast<uint8_t>(e);
        if (p.amax_c != nullptr) store_bits<T>(p.amax_c, (row0 >> 5) * p.ld_c + col, canonical_nan<T>(m));
      }
    }
  }
  __syncwarp();
#pragma unroll 1
  for (int rb = 0; rb < 32 && row0 + rb < g.rows; rb += kMaskBatch) {
    uint4 v[kMaskBatch];
    const uint64_t valid = load_rows_masked<T, kMaskBatch>(v, g, p.in, row0 + rb, j);
    if (valid == 0) continue;
#pragma unroll
    for (int r = 0; r < kMaskBatch; ++r) {
      const uint64_t bits = (valid >> (r * T::V)) & kChunkBits;
      if (bits == 0) continue;
      float mr[T::V];
      const float m = rsc.m[warp][rb + r][grp];
#pragma unroll
      for (int k = 0; k < T::V; ++k) mr[k] = m;
      uint2 qr, qc = make_uint2(0u, 0u);
      cast_chunk<T, kModel, kCol>(v[r], mr, mc, qr, qc);
      const int64_t o = (row0 + rb + r) * g.cols + j + p.out_shift;
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
  __syncwarp();
}

template <class T, int kDirs, bool kShift, bool kVec, int kModel, int N, bool kExp>
__global__ void __launch_bounds__(kThreads, kFusedMinBlocks) k_fused_quantize(
    const __grid_constant__ JobBatch<FusedParams, N> b) {
  __shared__ RowScales rsc;
  grid_dependency_sync();
  constexpr int TW = tile_width<T>();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t total = b.prefix_a[b.njobs] + b.prefix_b[b.njobs];
  const int64_t stride = int64_t(gridDim.x) * kWarps;
  for (int64_t t = int64_t(blockIdx.x) * kWarps + warp; t < total; t += stride) {
    int64_t row0, col0;
    const FusedParams& p = b.job[batch_tile(b, t, TW, row0, col0)];
    const int kind = classify_tile<T>(p.g, row0, col0, TW);
    const bool col = kDirs == kMixed ? p.out_c != nullptr : kDirs == kBidir;
    if (kind == kTileFast) {
      if (col) {
        if constexpr (kDirs != kRowOnly) fused_fast<T, true, kShift, kVec, kModel, kExp>(p, row0, col0, lane, rsc, warp);
      } else {
        if constexpr (kDirs != kBidir) fused_fast<T, false, kShift, kVec, kModel, kExp>(p, row0, col0, lane, rsc, warp);
      }
    } else if (kind == kTileMasked) {
      if (col) {
        if constexpr (kDirs != kRowOnly) fused_tile_masked<T, true, kVec, kModel>(p, row0, col0, lane, rsc, warp);
      } else {
        if constexpr (kDirs != kBidir) fused_tile_masked<T, false, kVec, kModel>(p, row0, col0, lane, rsc, warp);
      }
    }
  }
}

template <class T, int kDirs, bool kShift, bool kVec, int kModel, int N, bool kExp>
cudaError_t launch_n(const FusedParams* jobs, int n, const DeviceInfo& dev, cudaStream_t stream) {
  static std::atomic<int> occupancy[kMaxDevices];
  int occ = dev.device < kMaxDevices ? occupancy[dev.device].load() : 0;
  if (occ == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &occ, k_fused_quantize<T, kDirs, kShift, kVec, kModel, N, kExp>, kThreads, 0);
    if (e != cudaSuccess) return e;
    if (occ < 1) occ = 1;
    if (dev.device < kMaxDevices) occupancy[dev.device].store(occ);
  }
  JobBatch<FusedParams, N> b;
  const int64_t total = fill_batch(b, jobs, n);
  if (total == 0) return cudaSuccess;
  const unsigned grid = balanced_grid(total, kWarps, int64_t(dev.sms) * occ);
  return launch_kernel(k_fused_quantize<T, kDirs, kShift, kVec, kModel, N, kExp>, grid, kThreads, 0,
                       stream, b);
}

// One launch per batch of at most kMaxBatchJobs jobs, with the kernel for the batch's
// direction set; single BF16-model jobs use the one-entry job table.
template <class T, bool kShift, bool kVec, int kModel, bool kExp>
cudaError_t launch(const FusedParams* jobs, int n, const DeviceInfo& dev, cudaStream_t stream) {
  auto colwise = [](const FusedParams& p) { return p.out_c != nullptr; };
  if constexpr (kModel == kModelBF16) {
    if (n == 1) {
      return colwise(jobs[0]) ? launch_n<T, kBidir, kShift, kVec, kModel, 1, kExp>(jobs, 1, dev, stream)
                              : launch_n<T, kRowOnly, kShift, kVec, kModel, 1, kExp>(jobs, 1, dev, stream);
    }
  }
  for (int k = 0; k < n; k += kMaxBatchJobs) {
    const int m = n - k < kMaxBatchJobs ? n - k : kMaxBatchJobs;
    cudaError_t e;
    switch (batch_dirs(jobs + k, m, colwise)) {
      case kRowOnly:
        e = launch_n<T, kRowOnly, kShift, kVec, kModel, kMaxBatchJobs, kExp>(jobs + k, m, dev, stream);
        break;
      case kBidir:
        e = launch_n<T, kBidir, kShift, kVec, kModel, kMaxBatchJobs, kExp>(jobs + k, m, dev, stream);
        break;
      default:
        e = launch_n<T, kMixed, kShift, kVec, kModel, kMaxBatchJobs, kExp>(jobs + k, m, dev, stream);
        break;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <class T, int kModel>
cudaError_t launch_variant(const FusedParams* jobs, int n, bool shifted, bool vec_out,
                           const DeviceInfo& dev, cudaStream_t stream) {
  // FP32 input with word-aligned outputs and no amax output requested: exponent-only
  // maxima (packed high halves)
  if constexpr (T::kBytes == 4 && kModel == kModelBF16) {
    bool exp_only = vec_out;
    for (int k = 0; k < n && exp_only; ++k) exp_only = jobs[k].amax_r == nullptr && jobs[k].amax_c == nullptr;
    if (exp_only) {
      return shifted ? launch<T, true, true, kModel, true>(jobs, n, dev, stream)
                     : launch<T, false, true, kModel, true>(jobs, n, dev, stream);
    }
  }
  if (shifted) {
    return vec_out ? launch<T, true, true, kModel, false>(jobs, n, dev, stream)
                   : launch<T, true, false, kModel, false>(jobs, n, dev, stream);
  }
  return vec_out ? launch<T, false, true, kModel, false>(jobs, n, dev, stream)
                 : launch<T, false, false, kModel, false>(jobs, n, dev, stream);
}

// ---------------------------------------------------------------- staged one-pass kernel
// A single fragment made of whole 32-row bands, columns a multiple of the tile width, a
// 16-byte aligned virtual base and word-aligned outputs (a rank or a host pipeline chunk
// holding whole bands, a single rank holding a whole weight): a block of 8 warps owns one
// tile at a time.  Every thread copies 4 of the tile's 16-byte chunks into shared memory
// with cp.async, kStages tiles deep, so the DRAM reads of the next tile run while the
// block works on this one; both passes then read shared memory.  Warp w owns rows 4w..4w+3
// of the tile: pass 1 folds their row-block maxima (butterflies, as in the register
// kernel) and their column maxima, which go to shared memory; after one barrier every lane
// combines the 8 warps' column maxima of its V columns, and pass 2 casts the warp's rows.
// Tiles in flight per block: 2 (36 KB of shared memory, up to 6 blocks per SM) measured
// faster than 3 or 4 (fewer resident blocks).
#ifndef MXFP8_STAGED_STAGES
#define MXFP8_STAGED_STAGES 2
#endif
constexpr int kStages = MXFP8_STAGED_STAGES;
constexpr int kTileChunks = 32 * 32;                    // 16-byte chunks per tile
// tiles, the warps' column maxima, and the 256 multipliers 2^(127 - s) of the E8M0 bytes
constexpr int kStagedSmem = (kStages * kTileChunks + kWarps * 32) * 16 + 256 * 4;  // 37 KB at 2 stages

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <class T, bool kCol, bool kExp>
__device__ __forceinline__ void staged_tile(const FusedParams& p, const uint4 (&tile)[32][32],
                                            uint4 (&colpart)[kWarps][32], const float* mult,
                                            int64_t row0, int64_t col0,
                                            int warp, int lane) {
  const int64_t cols = p.g.cols;
  const int64_t j = col0 + lane * T::V;
  const int64_t blk = j >> 5;
  const bool writer = (lane % T::G) == 0;
  float rowmul[4];
  // pass 1: rows 4w .. 4w+3
  if constexpr (kExp) {
    static_assert(T::kBytes == 4, "exponent-only maxima are taken on FP32 high halves");
    uint32_t c01 = 0u, c23 = 0u;
#pragma unroll
    for (int rr = 0; rr < 4; rr += 2) {
      const int r = warp * 4 + rr;
      const uint4 va = tile[r][lane], vb = tile[r + 1][lane];
      const uint32_t a01 = abs_hi_halves(va.x, va.y), a23 = abs_hi_halves(va.z, va.w);
      const uint32_t b01 = abs_hi_halves(vb.x, vb.y), b23 = abs_hi_halves(vb.z, vb.w);
      if constexpr (kCol) {
        c01 = __vmaxu2(c01, __vmaxu2(a01, b01));
        c23 = __vmaxu2(c23, __vmaxu2(a23, b23));
      }
      const uint32_t ha = __vmaxu2(a01, a23), hb = __vmaxu2(b01, b23);
      uint32_t w = __vmaxu2(__byte_perm(ha, hb, 0x5410), __byte_perm(ha, hb, 0x7632));
#pragma unroll
      for (int off = 1; off < T::G; off <<= 1) w = __vmaxu2(w, __shfl_xor_sync(kFullMask, w, off));
      const uint32_t ea = e8m0_from_half(w & 0xffffu), eb = e8m0_from_half(w >> 16);
      rowmul[rr] = mult[ea];
      rowmul[rr + 1] = mult[eb];
      if (writer) {
        const int64_t i = row0 + r;
        p.s_r[i * p.ld_sr + blk] = static_cast<uint8_t>(ea);
        p.s_r[(i + 1) * p.ld_sr + blk] = static_cast<uint8_t>(eb);
      }
    }
    if constexpr (kCol) colpart[warp][lane] = make_uint4(c01, c23, 0u, 0u);
  } else {
    uint4 cm = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = warp * 4 + rr;
      const uint4 a = chunk_abs<T>(tile[r][lane]);
      if constexpr (kCol) cm = chunk_max<T>(cm, a);
      const uint32_t m = group_max<T>(chunk_reduce<T>(a));
      const uint32_t e = e8m0_from_bits<T>(m);
      rowmul[rr] = mult[e];
      if (writer) {
        const int64_t i = row0 + r;
        p.s_r[i * p.ld_sr + blk] = static_cast<uint8_t>(e);
        if (p.amax_r != nullptr) store_bits<T>(p.amax_r, i * p.ld_r + blk, canonical_nan<T>(m));
      }
    }
    if constexpr (kCol) colpart[warp][lane] = cm;
  }
  // column maxima of this lane's V columns over the 32 rows, scales, multipliers
  float mc[T::V];
  if constexpr (kCol) {
    __syncthreads();
    if constexpr (kExp) {
      uint32_t c01 = 0u, c23 = 0u;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const uint4 q = colpart[w][lane];
        c01 = __vmaxu2(c01, q.x);
        c23 = __vmaxu2(c23, q.y);
      }
      const uint32_t sb[4] = {e8m0_from_half(c01 & 0xffffu), e8m0_from_half(c01 >> 16),
                              e8m0_from_half(c23 & 0xffffu), e8m0_from_half(c23 >> 16)};
#pragma unroll
      for (int k = 0; k < 4; ++k) mc[k] = mult[sb[k]];
      if (warp == 0) {
        uint8_t* dst = p.s_c + (row0 >> 5) * p.ld_sc + j;
        if (p.vec_sc) {
          *reinterpret_cast<uint32_t*>(dst) = sb[0] | (sb[1] << 8) | (sb[2] << 16) | (sb[3] << 24);
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) dst[k] = static_cast<uint8_t>(sb[k]);
        }
      }
    } else {
      uint4 cm = colpart[0][lane];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) cm = chunk_max<T>(cm, colpart[w][lane]);
      if (warp == 0) {
        store_col_stats<T, kCol>(p, row0, j, cm, mc);
      } else {
#pragma unroll
        for (int k = 0; k < T::V; ++k) mc[k] = mult[e8m0_from_bits<T>(chunk_get<T>(cm, k))];
      }
    }
  }
  // pass 2: cast the warp's rows
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int r = warp * 4 + rr;
    float mr[T::V];
#pragma unroll
    for (int k = 0; k < T::V; ++k) mr[k] = rowmul[rr];
    uint2 qr, qc;
    cast_chunk<T, kModelBF16, kCol>(tile[r][lane], mr, mc, qr, qc);
    const int64_t o = (row0 + r) * cols + j + p.out_shift;
    store_chunk<T, true>(p.out_r + o, qr);
    if constexpr (kCol) store_chunk<T, true>(p.out_c + o, qc);
  }
}

// Position of a tile: its first row and its column-tile index.  A block's tiles are
// blockIdx.x, blockIdx.x + gridDim.x, ...; the position advances by that stride with a
// carry instead of a 64-bit division per tile.
struct TilePos {
  int64_t row0;
  int32_t ct;
};

__device__ __forceinline__ void advance(TilePos& p, int32_t step_bands, int32_t step_ct, int32_t coltiles) {
  p.ct += step_ct;
  int64_t bands = step_bands;
  if (p.ct >= coltiles) {
    p.ct -= coltiles;
    bands += 1;
  }
  p.row0 += 32 * bands;
}

template <class T, bool kCol, bool kExp>
__global__ void __launch_bounds__(kThreads) k_fused_staged(const __grid_constant__ FusedParams p) {
  extern __shared__ __align__(16) unsigned char staged_smem[];
  auto tiles = reinterpret_cast<uint4 (*)[32][32]>(staged_smem);
  auto& colpart = *reinterpret_cast<uint4 (*)[kWarps][32]>(staged_smem + kStages * kTileChunks * 16);
  float* mult = reinterpret_cast<float*>(staged_smem + (kStages * kTileChunks + kWarps * 32) * 16);
  mult[threadIdx.x] = scale_multiplier(threadIdx.x);  // 256 threads, 256 E8M0 bytes; read after
                                                      // the first barrier below
  grid_dependency_sync();
  constexpr int TW = tile_width<T>();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const FragGeom& g = p.g;
  const int64_t ntiles = g.ntiles, cols = g.cols;
  const int64_t row_bytes = cols * T::kBytes;
  // this thread copies chunks c = k * 256 + tid of every tile: row 8k + warp, chunk lane
  int64_t off[kTileChunks / kThreads];
#pragma unroll
  for (int k = 0; k < kTileChunks / kThreads; ++k) off[k] = (8 * k + warp) * row_bytes + lane * 16;
  const char* base = static_cast<const char*>(p.in) - g.start * T::kBytes;  // weight element 0
  auto issue = [&](const TilePos& tp, int stage) {
    const char* src = base + (tp.row0 * cols + int64_t(tp.ct) * TW) * T::kBytes;
#pragma unroll
    for (int k = 0; k < kTileChunks / kThreads; ++k)
      cp_async16(&tiles[stage][8 * k + warp][lane], src + off[k]);
  };
  const int32_t coltiles = g.coltiles;
  const int32_t step_bands = int32_t(gridDim.x / coltiles), step_ct = int32_t(gridDim.x % coltiles);
  const TilePos first = {(g.band0 + int64_t(blockIdx.x / coltiles)) * 32, int32_t(blockIdx.x % coltiles)};
  const int64_t step = gridDim.x;
  TilePos ip = first;
  int64_t ti = blockIdx.x;
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (ti < ntiles) issue(ip, s);
    cp_async_commit();  // one group per tile slot, empty past the last tile
    ti += step;
    advance(ip, step_bands, step_ct, coltiles);
  }
  TilePos tp = first;
  int stage = 0, istage = kStages - 1;
  for (int64_t t = blockIdx.x; t < ntiles; t += step) {
    cp_async_wait<kStages - 2>();  // this thread's copies of tile t have landed
    // every thread's copies of tile t have landed, and every thread is done with tile t - 1:
    // its stage may take the next tile and the column partials may be rewritten
    __syncthreads();
    if (ti < ntiles) issue(ip, istage);
    cp_async_commit();
    ti += step;
    advance(ip, step_bands, step_ct, coltiles);
    istage = istage + 1 == kStages ? 0 : istage + 1;
    staged_tile<T, kCol, kExp>(p, tiles[stage], colpart, mult, tp.row0, int64_t(tp.ct) * TW, warp, lane);
    stage = stage + 1 == kStages ? 0 : stage + 1;
    advance(tp, step_bands, step_ct, coltiles);
  }
  cp_async_wait<0>();
}

template <class T, bool kCol, bool kExp>
cudaError_t launch_staged_kernel(const FusedParams& p, const DeviceInfo& dev, cudaStream_t stream) {
  static std::atomic<int> occupancy[kMaxDevices];
  const auto kernel = k_fused_staged<T, kCol, kExp>;
  int occ = dev.device < kMaxDevices ? occupancy[dev.device].load() : 0;
  if (occ == 0) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kStagedSmem);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, kStagedSmem);
    if (e != cudaSuccess) return e;
    if (occ < 1) occ = 1;
    if (dev.device < kMaxDevices) occupancy[dev.device].store(occ);
  }
  const unsigned grid = balanced_grid(p.g.ntiles, 1, int64_t(dev.sms) * occ);
  return launch_kernel(kernel, grid, kThreads, kStagedSmem, stream, p);
}

// Whether one job can take the staged kernel (see above).
template <class T>
bool staged_ok(const FusedParams& p, bool shifted, bool vec_out) {
  const FragGeom& g = p.g;
  const int64_t band = 32 * g.cols;
  return !shifted && vec_out && g.cols % tile_width<T>() == 0 && g.end > g.start &&
         g.start % band == 0 && g.end % band == 0;
}

template <class T>
cudaError_t launch_staged(const FusedParams& p, const DeviceInfo& dev, cudaStream_t stream) {
  const bool col = p.out_c != nullptr;
  if constexpr (T::kBytes == 4) {
    if (p.amax_r == nullptr && p.amax_c == nullptr) {
      return col ? launch_staged_kernel<T, true, true>(p, dev, stream)
                 : launch_staged_kernel<T, false, true>(p, dev, stream);
    }
  }
  return col ? launch_staged_kernel<T, true, false>(p, dev, stream)
             : launch_staged_kernel<T, false, false>(p, dev, stream);
}

// All launches for one input dtype T (instantiated by that dtype's translation unit).
template <class T>
cudaError_t launch_for_dtype(const FusedParams* jobs, int n, bool shifted, bool vec_out, int model,
                             const DeviceInfo& dev, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  if (n == 1 && model == kModelBF16 && staged_ok<T>(jobs[0], shifted, vec_out))
    return launch_staged<T>(jobs[0], dev, stream);
  if (model == kModelF16) return launch_variant<T, kModelF16>(jobs, n, shifted, vec_out, dev, stream);
  return launch_variant<T, kModelBF16>(jobs, n, shifted, vec_out, dev, stream);
}

}  // namespace

}  // namespace mxfp8
