// Partial amax kernel: 1x32 row-block and (optionally) 32x1 column-block maxima of
// |x| over a contiguous fragment of a flattened rows x cols weight.
//
// Follows "Support row-only MXFP8 distributed master-weight casts" (sections
// "Changes" and "Bidirectional kernel performance"): the columnwise direction is a
// compile-time template parameter, so a row-only weight's kernel carries no column
// loads, reductions or stores (a run-time pointer test was measured there to slow
// the amax kernel by 21-35%).
//
// Work unit: one warp owns a 32-row x (32*V)-column tile.  Each lane owns V
// consecutive columns (one 16-byte chunk per row) and walks the 32 rows of the
// tile: the column maxima stay in the lane's registers, the row-block maximum is
// a butterfly over the G lanes of the block.  Tiles fully inside the fragment take
// 16-byte loads with no per-element tests; tiles cut by the fragment boundary or
// the matrix edge take per-element predicated loads.  The grid has one tile per
// warp (the block scheduler balances uneven tiles); tiles are numbered band-major,
// boundary bands first.
#include "common.cuh"

namespace mxfp8 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowBatch = 8;     // rows per batch of 16-byte loads, aligned and realigning
constexpr int kMaskBatch = 4;    // rows per batch of predicated per-element loads
// Resident blocks per SM the register allocation must allow: the amax is a pure
// streaming read, and 3 blocks (24 warps, at most 85 registers) keep more loads in flight
// than the 2 an unconstrained allocation leaves room for.
constexpr int kMinBlocks = 3;
// The realigning (shifted) kernels: their per-row shuffles add latency that more resident
// warps hide; 4 blocks (at most 64 registers) measured 2 us faster on the config-5 shard
// in its own buffer than 3.
#ifndef MXFP8_AMAX_SHIFT_MIN_BLOCKS
#define MXFP8_AMAX_SHIFT_MIN_BLOCKS 4
#endif
constexpr int kShiftMinBlocks = MXFP8_AMAX_SHIFT_MIN_BLOCKS;

// Per-row work shared by both tile paths: fold |x| of one chunk into the column
// maxima and return the maximum of the chunk's 32-element row block (all lanes of
// the warp must call this together: the row-block maximum is a butterfly).
template <class T, bool kCol>
__device__ __forceinline__ uint32_t fold_row(const uint4& chunk, uint4& colmax) {
  const uint4 a = chunk_abs<T>(chunk);
  if constexpr (kCol) colmax = chunk_max<T>(colmax, a);
  return group_max<T>(chunk_reduce<T>(a));
}

template <class T, bool kCol>
__device__ __forceinline__ void store_colmax(const AmaxParams& p, int64_t row0, int64_t j,
                                             const uint4& colmax) {
  const int64_t base = (row0 >> 5) * p.ld_c + j;
  const uint4 out = canonical_nan_chunk<T>(colmax);
  if (p.vec_c) {
    *reinterpret_cast<uint4*>(static_cast<char*>(p.amax_c) + base * T::kBytes) = out;
  } else {
#pragma unroll
    for (int k = 0; k < T::V; ++k) store_bits<T>(p.amax_c, base + k, chunk_get<T>(out, k));
  }
}

// Whole tile inside the fragment: 16-byte loads (realigned when the fragment's
// virtual base sits kS bytes past a 16-byte boundary), no per-element tests.  Rows
// r_lo .. r_hi-1 of the tile (all 32, or a quarter of them when four warps share the
// tile); the column maxima are stored, or left in *colpart for the warps to combine.
// kEdge: a tile cut by the matrix's right edge (kTileEdge): the lanes past it load
// nothing (their chunks read as zeros) and store nothing.
template <class T, bool kCol, int kS, bool kEdge = false>
__device__ __forceinline__ void amax_tile_fast(const AmaxParams& p, int64_t row0, int64_t col0,
                                               int lane, int r_lo, int r_hi, uint4* colpart) {
  static_assert(!kEdge || kS == 0, "edge tiles are aligned");
  const int64_t cols = p.g.cols;
  const int64_t j = col0 + lane * T::V;
  const char* src = static_cast<const char*>(p.in) + (row0 * cols + j - p.g.start) * T::kBytes;
  const int64_t row_bytes = cols * T::kBytes;
  const bool active = !kEdge || j < cols;
  const bool writer = (lane % T::G) == 0 && active;
  const int64_t out_r = row0 * p.ld_r + (j >> 5);
  // the realigning path batches 8 rows too: lane r loads the words after row r of the
  // tile (one load for the batch) and lane 31 takes them by shuffle
  constexpr bool kRowLanes = kS != 0;
  constexpr int NB = kRowBatch;
  uint4 colmax = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
  for (int rb = r_lo; rb < r_hi; rb += NB) {
    uint4 v[NB];
    if constexpr (kEdge) {
#pragma unroll
      for (int r = 0; r < NB; ++r)
        v[r] = active ? ld_stream16(src + (rb + r) * row_bytes) : make_uint4(0u, 0u, 0u, 0u);
    } else {
      load_rows<NB, kS, false, kRowLanes>(v, src + rb * row_bytes, row_bytes, lane);
    }
#pragma unroll
    for (int r = 0; r < NB; ++r) {
      const uint32_t m = fold_row<T, kCol>(v[r], colmax);
      if (writer) store_bits<T>(p.amax_r, out_r + (rb + r) * p.ld_r, canonical_nan<T>(m));
    }
  }
  if constexpr (kCol) {
    if (colpart != nullptr) {
      *colpart = colmax;
    } else if (active) {
      store_colmax<T, kCol>(p, row0, j, colmax);
    }
  }
}

// A fast tile of a launch whose fragments are all aligned (kShift false) or of a launch
// that holds realigning fragments (kShift true: each fragment's own offset, 0 included,
// picks the specialisation, so aligned and realigning fragments share one launch).
template <class T, bool kCol, bool kShift>
__device__ __forceinline__ void amax_fast(const AmaxParams& p, int64_t row0, int64_t col0, int lane,
                                          int r_lo = 0, int r_hi = 32, uint4* colpart = nullptr) {
  if constexpr (kShift) {
    if (p.g.shift == 0) {
      amax_tile_fast<T, kCol, 0>(p, row0, col0, lane, r_lo, r_hi, colpart);
    } else {
      with_shift<T>(p.g.shift, [&](auto s) {
        amax_tile_fast<T, kCol, decltype(s)::value>(p, row0, col0, lane, r_lo, r_hi, colpart);
      });
    }
  } else {
    amax_tile_fast<T, kCol, 0>(p, row0, col0, lane, r_lo, r_hi, colpart);
  }
}

// Tile cut by the fragment boundary or the matrix edge: per-element predicated
// loads, issued a batch of rows at a time; only blocks that meet the fragment are
// written.  Inlined into the kernel, so the fragment geometry is read straight from
// the kernel's parameters (behind a call, every store through an output pointer made
// the compiler reload it, which doubled the time of small, all-masked fragments).
// Column maxima of a cut tile: only the columns whose 32x1 block meets the fragment.
template <class T>
__device__ __forceinline__ void store_colmax_masked(const AmaxParams& p, int64_t row0, int64_t j,
                                                    const uint4& colmax) {
  const FragGeom& g = p.g;
  const int64_t r_end = min(row0 + 32, g.rows);
#pragma unroll
  for (int k = 0; k < T::V; ++k) {
    const int64_t col = j + k;
    if (col < g.cols && column_meets(g, col, row0, r_end))
      store_bits<T>(p.amax_c, (row0 >> 5) * p.ld_c + col, canonical_nan<T>(chunk_get<T>(colmax, k)));
  }
}

// MB: rows per batch of predicated loads (a split tile's warp takes its 8 rows at once).
template <class T, bool kCol, int MB = kMaskBatch>
__device__ __forceinline__ void amax_tile_masked(const AmaxParams& p, int64_t row0, int64_t col0,
                                              int lane, int r_lo = 0, int r_hi = 32,
                                              uint4* colpart = nullptr) {
  const FragGeom& g = p.g;
  const int64_t j = col0 + lane * T::V;
  const bool writer = (lane % T::G) == 0;
  const int64_t b0 = j & ~int64_t(31);  // first column of this lane's row block
  uint4 colmax = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
  for (int rb = r_lo; rb < r_hi; rb += MB) {  // warp-uniform: the butterfly stays converged
    uint4 v[MB];
    load_rows_masked<T, MB>(v, g, p.in, row0 + rb, j);
#pragma unroll
    for (int r = 0; r < MB; ++r) {
      const uint32_t m = fold_row<T, kCol>(v[r], colmax);
      const int64_t i = row0 + rb + r;
      if (writer && i < g.rows && b0 < g.cols && row_span_meets(g, i, b0, min(b0 + 31, g.cols - 1)))
        store_bits<T>(p.amax_r, i * p.ld_r + (b0 >> 5), canonical_nan<T>(m));
    }
  }
  if constexpr (kCol) {
    if (colpart != nullptr) {
      *colpart = colmax;
    } else {
      store_colmax_masked<T>(p, row0, j, colmax);
    }
  }
}

// kSplit: four warps share each tile, a quarter of its rows each (a block's eight warps
// take two tiles), and combine the tile's column maxima in shared memory; for launches
// with few tiles, whose time is one warp's chain of row batches rather than HBM traffic.
// kSplit 2 also takes tiles cut by the matrix's right edge on the fast path (instantiated
// only for weights whose width is not a multiple of the tile's: the extra path costs
// registers).
template <class T, int kDirs, bool kShift, int N, int kSplit>
__global__ void __launch_bounds__(kThreads, kShift ? kShiftMinBlocks : kMinBlocks) k_partial_amax(
    const __grid_constant__ JobBatch<AmaxParams, N> b) {
  grid_dependency_sync();
  constexpr int TW = tile_width<T>();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t total = b.prefix_a[b.njobs] + b.prefix_b[b.njobs];
  if constexpr (kSplit == 0) {
    const int64_t stride = int64_t(gridDim.x) * kWarps;
    for (int64_t t = int64_t(blockIdx.x) * kWarps + warp; t < total; t += stride) {
      int64_t row0, col0;
      const AmaxParams& p = b.job[batch_tile(b, t, TW, row0, col0)];
      const int kind = classify_tile<T>(p.g, row0, col0, TW);
      const bool col = kDirs == kMixed ? p.amax_c != nullptr : kDirs == kBidir;
      if (kind == kTileFast) {
        if (col) {
          if constexpr (kDirs != kRowOnly) amax_fast<T, true, kShift>(p, row0, col0, lane);
        } else {
          if constexpr (kDirs != kBidir) amax_fast<T, false, kShift>(p, row0, col0, lane);
        }
      } else if (kind == kTileMasked) {
        if (col) {
          if constexpr (kDirs != kRowOnly) amax_tile_masked<T, true>(p, row0, col0, lane);
        } else {
          if constexpr (kDirs != kBidir) amax_tile_masked<T, false>(p, row0, col0, lane);
        }
      }
    }
  } else {
    static_assert(kDirs != kMixed, "the split kernel serves single-direction-set launches");
    __shared__ uint4 part[kWarps][32];
    const int q = warp & 3;  // quarter: rows 8q .. 8q+7
    // block-uniform rounds (every warp reaches every barrier); warp w of a round takes
    // quarter w % 4 of tile (round * 8 + w) / 4
    for (int64_t base = int64_t(blockIdx.x) * kWarps; base < total * 4; base += int64_t(gridDim.x) * kWarps) {
      const int64_t t = (base + warp) >> 2;
      int kind = kTileSkip;
      int64_t row0 = 0, col0 = 0;
      const AmaxParams* pp = nullptr;
      if (t < total) {
        pp = &b.job[batch_tile(b, t, TW, row0, col0)];
        kind = kSplit == 2 ? classify_tile_edge<T>(pp->g, row0, col0, TW)
                           : classify_tile<T>(pp->g, row0, col0, TW);
        uint4* cp = kDirs == kBidir ? &part[warp][lane] : nullptr;
        if (kind == kTileFast) {
          amax_fast<T, kDirs == kBidir, kShift>(*pp, row0, col0, lane, 8 * q, 8 * q + 8, cp);
        } else if (kind == kTileEdge) {
          if constexpr (kSplit == 2)
            amax_tile_fast<T, kDirs == kBidir, 0, true>(*pp, row0, col0, lane, 8 * q, 8 * q + 8, cp);
        } else if (kind == kTileMasked) {
          amax_tile_masked<T, kDirs == kBidir, 8>(*pp, row0, col0, lane, 8 * q, 8 * q + 8, cp);
        }
      }
      if constexpr (kDirs == kBidir) {
        __syncthreads();
        if (q == 0 && kind != kTileSkip) {
          uint4 cm = part[warp][lane];
#pragma unroll
          for (int w = 1; w < 4; ++w) cm = chunk_max<T>(cm, part[warp + w][lane]);
          const int64_t j = col0 + lane * T::V;
          if (kind == kTileFast || (kind == kTileEdge && j < pp->g.cols)) {
            store_colmax<T, true>(*pp, row0, j, cm);
          } else if (kind == kTileMasked) {
            store_colmax_masked<T>(*pp, row0, j, cm);
          }
        }
        __syncthreads();
      }
    }
  }
}

template <class T, int kDirs, bool kShift, int N>
cudaError_t launch_n(const AmaxParams* jobs, int n, const DeviceInfo& dev, cudaStream_t stream) {
  JobBatch<AmaxParams, N> b;
  const int64_t total = fill_batch(b, jobs, n);
  if (total == 0) return cudaSuccess;
  if constexpr (N == 1 && !kShift && kDirs != kMixed) {
    if (total <= split_max_tiles(dev, MXFP8_AMAX_SPLIT_TILES_PER_SM)) {  // few tiles: four warps per tile
      const unsigned grid = tile_grid(total * 4, kWarps);
      if (jobs[0].g.cols % tile_width<T>() != 0)
        return launch_kernel(k_partial_amax<T, kDirs, kShift, N, 2>, grid, kThreads, 0, stream, b);
      return launch_kernel(k_partial_amax<T, kDirs, kShift, N, 1>, grid, kThreads, 0, stream, b);
    }
  }
  const unsigned grid = tile_grid(total, kWarps);
  return launch_kernel(k_partial_amax<T, kDirs, kShift, N, 0>, grid, kThreads, 0, stream, b);
}

// One launch per batch of at most kMaxBatchJobs jobs, with the kernel for the batch's
// direction set; single jobs use the one-entry job table.
template <class T, bool kShift>
cudaError_t launch(const AmaxParams* jobs, int n, const DeviceInfo& dev, cudaStream_t stream) {
  auto colwise = [](const AmaxParams& p) { return p.amax_c != nullptr; };
  if (n == 1) {
    return colwise(jobs[0]) ? launch_n<T, kBidir, kShift, 1>(jobs, 1, dev, stream)
                            : launch_n<T, kRowOnly, kShift, 1>(jobs, 1, dev, stream);
  }
  for (int k = 0; k < n; k += kMaxBatchJobs) {
    const int m = n - k < kMaxBatchJobs ? n - k : kMaxBatchJobs;
    cudaError_t e;
    switch (batch_dirs(jobs + k, m, colwise)) {
      case kRowOnly: e = launch_n<T, kRowOnly, kShift, kMaxBatchJobs>(jobs + k, m, dev, stream); break;
      case kBidir: e = launch_n<T, kBidir, kShift, kMaxBatchJobs>(jobs + k, m, dev, stream); break;
      default: e = launch_n<T, kMixed, kShift, kMaxBatchJobs>(jobs + k, m, dev, stream); break;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_partial_amax(const AmaxParams* jobs, int n, int dtype, bool shifted,
                                const DeviceInfo& dev, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  if (dtype == 0) {
    return shifted ? launch<F32T, true>(jobs, n, dev, stream) : launch<F32T, false>(jobs, n, dev, stream);
  }
  return shifted ? launch<BF16T, true>(jobs, n, dev, stream) : launch<BF16T, false>(jobs, n, dev, stream);
}

}  // namespace mxfp8
