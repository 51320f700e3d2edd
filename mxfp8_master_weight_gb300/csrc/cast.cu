// Partial cast kernel: master values of a contiguous fragment -> BF16 (model
// dtype, nearest-even) -> E4M3 (nearest-even, saturating at 448), scaled by the
// E8M0 block scales, written in place into the rowwise and (optionally)
// columnwise outputs.
//
// Follows "Support row-only MXFP8 distributed master-weight casts" (sections
// "Changes" and the flow diagram): rounding goes through the model dtype, the
// rowwise output is always written, and the columnwise output -- with every read
// of its scales -- is removed at compile time when the weight has none.
//
// Work unit and tile classes as in the amax kernel: one warp per 32 x (32*V)
// tile, one 16-byte input chunk per lane per row; a row's V output bytes per
// direction leave as one 4- (FP32) or 8-byte (BF16) store, so a warp writes 128
// or 256 contiguous bytes per row and direction.  The columnwise multipliers of a
// lane's V columns are loaded once per tile; the rowwise multiplier once per row.
#include <atomic>

#include "common.cuh"

namespace mxfp8 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowBatch = 8;
constexpr int kMaxDevices = 64;

// Model-dtype values of one input chunk.
template <class T>
__device__ __forceinline__ void model_values(const uint4& c, float (&y)[T::V]) {
  if constexpr (T::kBytes == 4) {
    const uint32_t w0 = bf16x2_rn(__uint_as_float(c.x), __uint_as_float(c.y));
    const uint32_t w1 = bf16x2_rn(__uint_as_float(c.z), __uint_as_float(c.w));
    y[0] = bf16_lo(w0); y[1] = bf16_hi(w0); y[2] = bf16_lo(w1); y[3] = bf16_hi(w1);
  } else {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) { y[2 * k] = bf16_lo(w[k]); y[2 * k + 1] = bf16_hi(w[k]); }
  }
}

// Model-dtype value of one element given as a bit pattern.
template <class T>
__device__ __forceinline__ float model_value(uint32_t bits) {
  if constexpr (T::kBytes == 4) {
    return bf16_lo(bf16x2_rn(__uint_as_float(bits), 0.0f));
  } else {
    return __uint_as_float(bits << 16);
  }
}

__device__ __forceinline__ uint8_t quantize1(float y, float mult) {
  return static_cast<uint8_t>(e4m3x2_rn_sat(y * mult, 0.0f) & 0xffu);
}

// V E4M3 bytes of y[k] * mult[k], stored as one 4- or 8-byte word.
template <class T>
__device__ __forceinline__ void store_q(uint8_t* dst, const float (&y)[T::V], const float (&mult)[T::V]) {
  if constexpr (T::V == 4) {
    const uint32_t q = e4m3x2_rn_sat(y[0] * mult[0], y[1] * mult[1]) |
                       (e4m3x2_rn_sat(y[2] * mult[2], y[3] * mult[3]) << 16);
    *reinterpret_cast<uint32_t*>(dst) = q;
  } else {
    uint2 q;
    q.x = e4m3x2_rn_sat(y[0] * mult[0], y[1] * mult[1]) |
          (e4m3x2_rn_sat(y[2] * mult[2], y[3] * mult[3]) << 16);
    q.y = e4m3x2_rn_sat(y[4] * mult[4], y[5] * mult[5]) |
          (e4m3x2_rn_sat(y[6] * mult[6], y[7] * mult[7]) << 16);
    *reinterpret_cast<uint2*>(dst) = q;
  }
}

template <class T, bool kCol>
__device__ __forceinline__ void cast_tile_fast(const CastParams& p, int64_t row0, int64_t col0,
                                               int lane) {
  const int64_t cols = p.g.cols;
  const int64_t j = col0 + lane * T::V;
  const char* src = static_cast<const char*>(p.in) + (row0 * cols + j - p.g.start) * T::kBytes;
  const int64_t row_bytes = cols * T::kBytes;
  const uint8_t* srow = p.s_r + row0 * p.ld_sr + (j >> 5);
  const int64_t o0 = row0 * cols + j + p.out_shift;
  float mc[T::V];
  if constexpr (kCol) {
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
#pragma unroll 1
  for (int rb = 0; rb < 32; rb += kRowBatch) {
    uint4 v[kRowBatch];
    uint32_t sb[kRowBatch];
#pragma unroll
    for (int r = 0; r < kRowBatch; ++r) {
      v[r] = ld_stream16(src + (rb + r) * row_bytes);
      sb[r] = srow[(rb + r) * p.ld_sr];
    }
#pragma unroll
    for (int r = 0; r < kRowBatch; ++r) {
      float y[T::V];
      model_values<T>(v[r], y);
      float mr[T::V];
      const float m = scale_multiplier(sb[r]);
#pragma unroll
      for (int k = 0; k < T::V; ++k) mr[k] = m;
      const int64_t o = o0 + (rb + r) * cols;
      store_q<T>(p.out_r + o, y, mr);
      if constexpr (kCol) store_q<T>(p.out_c + o, y, mc);
    }
  }
}

template <class T, bool kCol>
__device__ __noinline__ void cast_tile_masked(const CastParams& p, int64_t row0, int64_t col0,
                                              int lane) {
  const FragGeom& g = p.g;
  const int64_t j = col0 + lane * T::V;
  const int64_t r_end = min(row0 + 32, g.rows);
  for (int64_t i = row0; i < r_end; ++i) {
#pragma unroll
    for (int k = 0; k < T::V; ++k) {
      const int64_t col = j + k;
      const int64_t f = i * g.cols + col;
      if (col < g.cols && f >= g.start && f < g.end) {
        const float y = model_value<T>(load_bits<T>(p.in, f - g.start));
        p.out_r[f + p.out_shift] = quantize1(y, scale_multiplier(p.s_r[i * p.ld_sr + (col >> 5)]));
        if constexpr (kCol)
          p.out_c[f + p.out_shift] =
              quantize1(y, scale_multiplier(p.s_c[(i >> 5) * p.ld_sc + col]));
      }
    }
  }
}

template <class T, bool kCol>
__global__ void __launch_bounds__(kThreads) k_partial_cast(const __grid_constant__ CastParams p) {
  constexpr int TW = tile_width<T>();
  const int lane = threadIdx.x & 31;
  const int64_t stride = int64_t(gridDim.x) * kWarps;
  for (int64_t t = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5); t < p.g.ntiles; t += stride) {
    const int64_t row0 = (p.g.band0 + t / p.g.coltiles) * 32;
    const int64_t col0 = (t % p.g.coltiles) * TW;
    const int kind = classify_tile(p.g, row0, col0, TW);
    if (kind == kTileFast) {
      cast_tile_fast<T, kCol>(p, row0, col0, lane);
    } else if (kind == kTileMasked) {
      cast_tile_masked<T, kCol>(p, row0, col0, lane);
    }
  }
}

template <class T, bool kCol>
cudaError_t launch(const CastParams& p, const DeviceInfo& dev, cudaStream_t stream) {
  static std::atomic<int> occupancy[kMaxDevices];
  int occ = dev.device < kMaxDevices ? occupancy[dev.device].load() : 0;
  if (occ == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_partial_cast<T, kCol>,
                                                                  kThreads, 0);
    if (e != cudaSuccess) return e;
    if (occ < 1) occ = 1;
    if (dev.device < kMaxDevices) occupancy[dev.device].store(occ);
  }
  const int64_t want = (p.g.ntiles + kWarps - 1) / kWarps;
  const int64_t cap = int64_t(dev.sms) * occ;
  const unsigned grid = unsigned(want < cap ? want : cap);
  k_partial_cast<T, kCol><<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_partial_cast(const CastParams& p, int dtype, bool colwise,
                                const DeviceInfo& dev, cudaStream_t stream) {
  if (p.g.ntiles <= 0) return cudaSuccess;
  if (dtype == 0) {
    return colwise ? launch<F32T, true>(p, dev, stream) : launch<F32T, false>(p, dev, stream);
  }
  return colwise ? launch<BF16T, true>(p, dev, stream) : launch<BF16T, false>(p, dev, stream);
}

}  // namespace mxfp8
