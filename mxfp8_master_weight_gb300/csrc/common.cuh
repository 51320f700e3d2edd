// Device helpers shared by the partial-amax, scale and cast kernels (sm_103a).
//
// Everything here is bit-level: |x| and block maxima are taken on the raw bit
// patterns with the sign cleared (for non-negative IEEE values unsigned integer
// order equals numeric order, and NaN patterns sort above +Inf, so a NaN member
// propagates); the E8M0 exponent is read from the exponent field; the two
// roundings of the cast are the documented PTX conversions cvt.rn.bf16x2.f32
// and cvt.rn.satfinite.e4m3x2.f32.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"

namespace mxfp8 {

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------- dtype traits
// V  = elements per 16-byte chunk (one chunk per lane per row),
// G  = lanes that share one 32-element row block (32 / V),
// TW = columns covered by one warp tile (32 lanes x V).
struct F32T {
  static constexpr int V = 4;
  static constexpr int G = 8;
  static constexpr int kBytes = 4;
  static constexpr uint32_t kAbsMask = 0x7fffffffu;  // per 32-bit word
};
struct BF16T {
  static constexpr int V = 8;
  static constexpr int G = 4;
  static constexpr int kBytes = 2;
  static constexpr uint32_t kAbsMask = 0x7fff7fffu;  // two elements per word
};
template <class T>
__host__ __device__ constexpr int tile_width() { return 32 * T::V; }

// ---------------------------------------------------------------- memory ops
// 16-byte global load that does not allocate in L1 (each byte is read once).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ---------------------------------------------------------------- per-element access
template <class T>
__device__ __forceinline__ uint32_t load_bits(const void* base, int64_t idx) {
  if constexpr (T::kBytes == 4) {
    return static_cast<const uint32_t*>(base)[idx];
  } else {
    return static_cast<const uint16_t*>(base)[idx];
  }
}

template <class T>
__device__ __forceinline__ void store_bits(void* base, int64_t idx, uint32_t bits) {
  if constexpr (T::kBytes == 4) {
    static_cast<uint32_t*>(base)[idx] = bits;
  } else {
    static_cast<uint16_t*>(base)[idx] = static_cast<uint16_t>(bits);
  }
}

// Element k (0 <= k < V) of a chunk held as four 32-bit words.
template <class T>
__device__ __forceinline__ uint32_t chunk_get(const uint4& c, int k) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  if constexpr (T::kBytes == 4) {
    return w[k];
  } else {
    return (w[k >> 1] >> ((k & 1) * 16)) & 0xffffu;
  }
}

template <class T>
__device__ __forceinline__ void chunk_set(uint4& c, int k, uint32_t bits) {
  if constexpr (T::kBytes == 4) {
    if (k == 0) c.x = bits; else if (k == 1) c.y = bits; else if (k == 2) c.z = bits; else c.w = bits;
  } else {
    const int sh = (k & 1) * 16;
    const uint32_t keep = ~(0xffffu << sh);
    const uint32_t put = (bits & 0xffffu) << sh;
    switch (k >> 1) {
      case 0: c.x = (c.x & keep) | put; break;
      case 1: c.y = (c.y & keep) | put; break;
      case 2: c.z = (c.z & keep) | put; break;
      default: c.w = (c.w & keep) | put; break;
    }
  }
}

// ---------------------------------------------------------------- |x| and maxima
template <class T>
__device__ __forceinline__ uint4 chunk_abs(uint4 c) {
  c.x &= T::kAbsMask; c.y &= T::kAbsMask; c.z &= T::kAbsMask; c.w &= T::kAbsMask;
  return c;
}

// Lane-wise max of two chunks of |x| bit patterns.
template <class T>
__device__ __forceinline__ uint4 chunk_max(uint4 a, const uint4& b) {
  if constexpr (T::kBytes == 4) {
    a.x = max(a.x, b.x); a.y = max(a.y, b.y); a.z = max(a.z, b.z); a.w = max(a.w, b.w);
  } else {
    a.x = __vmaxu2(a.x, b.x); a.y = __vmaxu2(a.y, b.y);
    a.z = __vmaxu2(a.z, b.z); a.w = __vmaxu2(a.w, b.w);
  }
  return a;
}

// Max over the V elements of one chunk of |x| bit patterns.
template <class T>
__device__ __forceinline__ uint32_t chunk_reduce(const uint4& c) {
  if constexpr (T::kBytes == 4) {
    return max(max(c.x, c.y), max(c.z, c.w));
  } else {
    const uint32_t m = __vmaxu2(__vmaxu2(c.x, c.y), __vmaxu2(c.z, c.w));
    return max(m & 0xffffu, m >> 16);
  }
}

// Max over the G lanes that hold one 32-element row block (aligned lane groups).
template <class T>
__device__ __forceinline__ uint32_t group_max(uint32_t m) {
#pragma unroll
  for (int off = 1; off < T::G; off <<= 1) m = max(m, __shfl_xor_sync(kFullMask, m, off));
  return m;
}

// ---------------------------------------------------------------- scale and cast
// E8M0 byte of an amax bit pattern: max(E - 8, 0) for a finite amax with biased
// exponent field E (so that amax * 2^(127 - byte) lies in [256, 512) when the
// byte is not clamped), 0xFF for NaN / Inf.
template <class T>
__device__ __forceinline__ uint32_t e8m0_from_bits(uint32_t bits) {
  const uint32_t e = (T::kBytes == 4) ? ((bits >> 23) & 0xffu) : ((bits >> 7) & 0xffu);
  return e == 0xffu ? 0xffu : (e > 8u ? e - 8u : 0u);
}

// 2^(127 - s) as a float (the multiplier that maps a value onto the E4M3 grid of
// its block); s == 254 gives the subnormal 2^-127, s == 255 (NaN scale) gives NaN.
__device__ __forceinline__ float scale_multiplier(uint32_t s) {
  const uint32_t bits = s == 255u ? 0x7fc00000u : (s == 254u ? 0x00400000u : (254u - s) << 23);
  return __uint_as_float(bits);
}

// Two FP32 values rounded to BF16 (nearest-even); lo lands in the low half.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two FP32 values to E4M3 (nearest-even, saturating to +-448); lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2_rn_sat(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ---------------------------------------------------------------- fragment geometry
// True when the flat range [a, b) meets the fragment [start, end).
__device__ __forceinline__ bool meets(int64_t a, int64_t b, int64_t start, int64_t end) {
  return (a < b) && (a < end) && (start < b);
}

// True when column `col` has a fragment element in rows [r_a, r_b).
__device__ __forceinline__ bool column_meets(const FragGeom& g, int64_t col, int64_t r_a,
                                             int64_t r_b) {
  // rows r with start <= r*cols + col < end form one interval [lo, hi]
  const int64_t lo = g.start > col ? (g.start - col + g.cols - 1) / g.cols : 0;
  const int64_t hi = g.end - 1 >= col ? (g.end - 1 - col) / g.cols : -1;
  return max(lo, r_a) <= min(hi, r_b - 1);
}

enum TileKind { kTileSkip = 0, kTileFast = 1, kTileMasked = 2 };

// Classify the warp tile whose top-left element is (row0, col0), tw columns wide.
__device__ __forceinline__ int classify_tile(const FragGeom& g, int64_t row0, int64_t col0,
                                             int tw) {
  const int64_t row_last = min(row0 + 31, g.rows - 1);
  const int64_t col_last = min(col0 + tw, g.cols) - 1;
  const int64_t first = row0 * g.cols + col0;
  const int64_t last = row_last * g.cols + col_last;
  if (last < g.start || first >= g.end) return kTileSkip;
  const bool whole = (row0 + 32 <= g.rows) && (col0 + tw <= g.cols);
  if (g.fast_ok && whole && first >= g.start && last < g.end) return kTileFast;
  return kTileMasked;
}

}  // namespace mxfp8
