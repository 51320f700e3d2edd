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
// the matrix edge take per-element predicated loads.  The grid is persistent
// (a multiple of the SM count) and walks tiles in band-major order.
#include <atomic>

#include "common.cuh"

namespace mxfp8 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowBatch = 8;  // 16-byte loads in flight per lane
constexpr int kMaxDevices = 64;

template <class T, bool kCol>
__device__ __forceinline__ void amax_tile_fast(const AmaxParams& p, int64_t row0, int64_t col0,
                                               int lane) {
  const int64_t cols = p.g.cols;
  const int64_t j = col0 + lane * T::V;
  const char* src = static_cast<const char*>(p.in) + (row0 * cols + j - p.g.start) * T::kBytes;
  const int64_t row_bytes = cols * T::kBytes;
  const bool writer = (lane % T::G) == 0;
  const int64_t out_r = row0 * p.ld_r + (j >> 5);
  uint4 colmax = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
  for (int rb = 0; rb < 32; rb += kRowBatch) {
    uint4 v[kRowBatch];
#pragma unroll
    for (int r = 0; r < kRowBatch; ++r) v[r] = ld_stream16(src + (rb + r) * row_bytes);
#pragma unroll
    for (int r = 0; r < kRowBatch; ++r) {
      const uint4 a = chunk_abs<T>(v[r]);
      if constexpr (kCol) colmax = chunk_max<T>(colmax, a);
      const uint32_t m = group_max<T>(chunk_reduce<T>(a));
      if (writer) store_bits<T>(p.amax_r, out_r + (rb + r) * p.ld_r, m);
    }
  }
  if constexpr (kCol) {
    const int64_t base = (row0 >> 5) * p.ld_c + j;
    if (p.vec_c) {
      *reinterpret_cast<uint4*>(static_cast<char*>(p.amax_c) + base * T::kBytes) = colmax;
    } else {
#pragma unroll
      for (int k = 0; k < T::V; ++k) store_bits<T>(p.amax_c, base + k, chunk_get<T>(colmax, k));
    }
  }
}

template <class T, bool kCol>
__device__ __noinline__ void amax_tile_masked(const AmaxParams& p, int64_t row0, int64_t col0,
                                              int lane) {
  const FragGeom& g = p.g;
  const int64_t j = col0 + lane * T::V;
  const bool writer = (lane % T::G) == 0;
  const int64_t b0 = j & ~int64_t(31);  // first column of this lane's row block
  uint4 colmax = make_uint4(0u, 0u, 0u, 0u);
  for (int r = 0; r < 32; ++r) {  // warp-uniform trip count: the butterfly stays converged
    const int64_t i = row0 + r;
    uint4 c = make_uint4(0u, 0u, 0u, 0u);
    if (i < g.rows) {
#pragma unroll
      for (int k = 0; k < T::V; ++k) {
        const int64_t col = j + k;
        const int64_t f = i * g.cols + col;
        if (col < g.cols && f >= g.start && f < g.end)
          chunk_set<T>(c, k, load_bits<T>(p.in, f - g.start));
      }
    }
    const uint4 a = chunk_abs<T>(c);
    if constexpr (kCol) colmax = chunk_max<T>(colmax, a);
    const uint32_t m = group_max<T>(chunk_reduce<T>(a));
    if (writer && i < g.rows && b0 < g.cols) {
      const int64_t lo = i * g.cols + b0;
      const int64_t hi = i * g.cols + min(b0 + 32, g.cols);
      if (meets(lo, hi, g.start, g.end)) store_bits<T>(p.amax_r, i * p.ld_r + (b0 >> 5), m);
    }
  }
  if constexpr (kCol) {
    const int64_t r_end = min(row0 + 32, g.rows);
#pragma unroll
    for (int k = 0; k < T::V; ++k) {
      const int64_t col = j + k;
      if (col < g.cols && column_meets(g, col, row0, r_end))
        store_bits<T>(p.amax_c, (row0 >> 5) * p.ld_c + col, chunk_get<T>(colmax, k));
    }
  }
}

template <class T, bool kCol>
__global__ void __launch_bounds__(kThreads) k_partial_amax(const __grid_constant__ AmaxParams p) {
  constexpr int TW = tile_width<T>();
  const int lane = threadIdx.x & 31;
  const int64_t stride = int64_t(gridDim.x) * kWarps;
  for (int64_t t = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5); t < p.g.ntiles; t += stride) {
    const int64_t row0 = (p.g.band0 + t / p.g.coltiles) * 32;
    const int64_t col0 = (t % p.g.coltiles) * TW;
    const int kind = classify_tile(p.g, row0, col0, TW);
    if (kind == kTileFast) {
      amax_tile_fast<T, kCol>(p, row0, col0, lane);
    } else if (kind == kTileMasked) {
      amax_tile_masked<T, kCol>(p, row0, col0, lane);
    }
  }
}

template <class T, bool kCol>
cudaError_t launch(const AmaxParams& p, const DeviceInfo& dev, cudaStream_t stream) {
  static std::atomic<int> occupancy[kMaxDevices];
  int occ = dev.device < kMaxDevices ? occupancy[dev.device].load() : 0;
  if (occ == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_partial_amax<T, kCol>,
                                                                  kThreads, 0);
    if (e != cudaSuccess) return e;
    if (occ < 1) occ = 1;
    if (dev.device < kMaxDevices) occupancy[dev.device].store(occ);
  }
  const int64_t want = (p.g.ntiles + kWarps - 1) / kWarps;
  const int64_t cap = int64_t(dev.sms) * occ;
  const unsigned grid = unsigned(want < cap ? want : cap);
  k_partial_amax<T, kCol><<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_partial_amax(const AmaxParams& p, int dtype, bool colwise,
                                const DeviceInfo& dev, cudaStream_t stream) {
  if (p.g.ntiles <= 0) return cudaSuccess;
  if (dtype == 0) {
    return colwise ? launch<F32T, true>(p, dev, stream) : launch<F32T, false>(p, dev, stream);
  }
  return colwise ? launch<BF16T, true>(p, dev, stream) : launch<BF16T, false>(p, dev, stream);
}

}  // namespace mxfp8
