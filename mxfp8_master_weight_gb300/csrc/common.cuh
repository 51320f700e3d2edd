// Device helpers shared by the partial-amax, scale, cast and one-pass kernels
// (sm_103a).
//
// Everything here is bit-level: |x| and block maxima are taken on the raw bit
// patterns with the sign cleared (for non-negative IEEE values unsigned integer
// order equals numeric order, and NaN patterns sort above +Inf, so a NaN member
// propagates); the E8M0 exponent is read from the exponent field; the roundings of
// the cast are the documented PTX conversions cvt.rn.bf16x2.f32 (or cvt.rn.f16x2.f32
// for an FP16 model dtype) and cvt.rn.satfinite.e4m3x2.f32.
#pragma once

#include <cstdint>
#include <utility>
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

// ---------------------------------------------------------------- launches
// Programmatic dependent launch.  Every kernel starts with grid_dependency_sync():
// it returns once the kernel before it in the stream has completed and its writes
// are visible (at once when this grid was launched without a programmatic
// dependency), and then lets the next kernel's blocks be scheduled on SMs that this
// grid frees, so a launch overlaps the tail of the grid before it instead of
// following its completion.  No global memory is touched before the wait, so the
// kernel before may be any producer of this kernel's inputs.
__device__ __forceinline__ void grid_dependency_sync() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with the programmatic stream serialisation attribute (the kernel must start
// with grid_dependency_sync()).
template <class... KArgs, class... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- memory ops
// 16-byte global load that does not allocate in L1 (each byte is read once).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// L2 cache policies (createpolicy) and a 16-byte load that carries one: a tile read
// twice in a row keeps its lines in L2 between the reads (evict_last on the first
// read, evict_first on the second).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint4 ld_hint16(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
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

// A NaN amax is stored as the canonical quiet NaN (FP32 0x7FC00000, BF16 0x7FC0),
// whatever NaN pattern the block's members carried: the bit-pattern maxima above keep
// the largest member pattern, so each stored amax passes through these first.
// One element (a BF16 value in the low 16 bits):
template <class T>
__device__ __forceinline__ uint32_t canonical_nan(uint32_t m) {
  if constexpr (T::kBytes == 4) {
    return m > 0x7f800000u ? 0x7fc00000u : m;
  } else {
    return m > 0x7f80u ? 0x7fc0u : m;
  }
}

// Every element of a chunk of |x| bit patterns.
template <class T>
__device__ __forceinline__ uint4 canonical_nan_chunk(uint4 c) {
  if constexpr (T::kBytes == 4) {
    c.x = canonical_nan<T>(c.x); c.y = canonical_nan<T>(c.y);
    c.z = canonical_nan<T>(c.z); c.w = canonical_nan<T>(c.w);
  } else {
    // per 16-bit half: 0xffff where the half is a NaN, then select the canonical pattern
    uint32_t* w[4] = {&c.x, &c.y, &c.z, &c.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t nan = __vcmpgtu2(*w[k], 0x7f807f80u);
      *w[k] = (*w[k] & ~nan) | (0x7fc07fc0u & nan);
    }
  }
  return c;
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

// Two FP32 products in one packed multiply (mul.rn.f32x2), each rounded to nearest as a
// scalar multiply is; with a power-of-two multiplier the products are exact.
__device__ __forceinline__ void mul2_rn(float a0, float a1, float b0, float b1, float& p0, float& p1) {
  uint64_t x, y, z;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b0), "f"(b1));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(z) : "l"(x), "l"(y));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(p0), "=f"(p1) : "l"(z));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ---------------------------------------------------------------- cast of one chunk
// Model dtypes the master values are rounded through before quantisation.
constexpr int kModelBF16 = 0;
constexpr int kModelF16 = 1;

// Two FP32 values rounded to IEEE FP16 (nearest-even, overflow to infinity); lo in
// the low half.
__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float f16_lo(uint32_t w) {
  float f;
  asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.f32.f16 %0, l; }" : "=f"(f) : "r"(w));
  return f;
}
__device__ __forceinline__ float f16_hi(uint32_t w) {
  float f;
  asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.f32.f16 %0, h; }" : "=f"(f) : "r"(w));
  return f;
}

// Model-dtype values of one input chunk: BF16 (identity for BF16 input) or FP16.
template <class T, int kModel = kModelBF16>
__device__ __forceinline__ void model_values(const uint4& c, float (&y)[T::V]) {
  if constexpr (T::kBytes == 4) {
    const uint32_t w0 = kModel == kModelF16 ? f16x2_rn(__uint_as_float(c.x), __uint_as_float(c.y))
                                            : bf16x2_rn(__uint_as_float(c.x), __uint_as_float(c.y));
    const uint32_t w1 = kModel == kModelF16 ? f16x2_rn(__uint_as_float(c.z), __uint_as_float(c.w))
                                            : bf16x2_rn(__uint_as_float(c.z), __uint_as_float(c.w));
    if constexpr (kModel == kModelF16) {
      y[0] = f16_lo(w0); y[1] = f16_hi(w0); y[2] = f16_lo(w1); y[3] = f16_hi(w1);
    } else {
      y[0] = bf16_lo(w0); y[1] = bf16_hi(w0); y[2] = bf16_lo(w1); y[3] = bf16_hi(w1);
    }
  } else {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if constexpr (kModel == kModelF16) {
        const uint32_t h = f16x2_rn(bf16_lo(w[k]), bf16_hi(w[k]));
        y[2 * k] = f16_lo(h);
        y[2 * k + 1] = f16_hi(h);
      } else {
        y[2 * k] = bf16_lo(w[k]);
        y[2 * k + 1] = bf16_hi(w[k]);
      }
    }
  }
}

// V E4M3 bytes of y[k] * mult[k] (element k in byte k).
template <class T>
__device__ __forceinline__ uint2 quantize_chunk(const float (&y)[T::V], const float (&mult)[T::V]) {
  uint2 q;
  float p[T::V];
#pragma unroll
  for (int k = 0; k < T::V; k += 2) mul2_rn(y[k], y[k + 1], mult[k], mult[k + 1], p[k], p[k + 1]);
  q.x = e4m3x2_rn_sat(p[0], p[1]) | (e4m3x2_rn_sat(p[2], p[3]) << 16);
  if constexpr (T::V == 8) {
    q.y = e4m3x2_rn_sat(p[4], p[5]) | (e4m3x2_rn_sat(p[6], p[7]) << 16);
  } else {
    q.y = 0;
  }
  return q;
}

// Rowwise and (kCol) columnwise E4M3 bytes of one input chunk through the model dtype.
template <class T, int kModel, bool kCol>
__device__ __forceinline__ void cast_chunk(const uint4& c, const float (&mr)[T::V], const float (&mc)[T::V],
                                           uint2& qr, uint2& qc) {
  float y[T::V];
  model_values<T, kModel>(c, y);
  qr = quantize_chunk<T>(y, mr);
  if constexpr (kCol) qc = quantize_chunk<T>(y, mc);
}

// Store V bytes: one 4- or 8-byte word when the destination is aligned, else bytes.
template <class T, bool kVec>
__device__ __forceinline__ void store_chunk(uint8_t* dst, const uint2& q) {
  if constexpr (kVec) {
    if constexpr (T::V == 4) {
      *reinterpret_cast<uint32_t*>(dst) = q.x;
    } else {
      *reinterpret_cast<uint2*>(dst) = q;
    }
  } else {
#pragma unroll
    for (int k = 0; k < T::V; ++k) dst[k] = static_cast<uint8_t>((k < 4 ? q.x : q.y) >> (8 * (k & 3)));
  }
}

// A compile-time integer handed to the generic lambdas of the dispatch helpers.
template <int S>
struct ShiftC {
  static constexpr int value = S;
};

// Bytes [off, off + 4) of a lane's V output bytes (q.x, then q.y), as the low bytes.
template <class T, int kOff>
__device__ __forceinline__ uint32_t chunk_bytes(const uint2& q) {
  if constexpr (kOff == 0) {
    return q.x;
  } else if constexpr (kOff < 4) {
    return T::V == 4 ? q.x >> (8 * kOff) : __funnelshift_r(q.x, q.y, 8 * kOff);
  } else {
    return q.y >> (8 * (kOff - 4));
  }
}

// Stores the V bytes at dst, which sits kM bytes past a V-byte boundary (the same
// offset for every lane and row of a tile, known at compile time), as naturally
// aligned 1-, 2- and 4-byte pieces from byte kOff on: at most 3 stores for V = 4 and
// 4 for V = 8 instead of V byte stores.
template <class T, int kM, int kOff = 0>
__device__ __forceinline__ void store_chunk_pieces(uint8_t* dst, const uint2& q) {
  if constexpr (kOff < T::V) {
    constexpr int kA = (kM + kOff) % 4;  // address mod 4 of this piece
    constexpr int kS = (kA == 0 && kOff + 4 <= T::V) ? 4 : ((kA % 2 == 0 && kOff + 2 <= T::V) ? 2 : 1);
    const uint32_t bits = chunk_bytes<T, kOff>(q);
    if constexpr (kS == 4) {
      *reinterpret_cast<uint32_t*>(dst + kOff) = bits;
    } else if constexpr (kS == 2) {
      *reinterpret_cast<uint16_t*>(dst + kOff) = static_cast<uint16_t>(bits);
    } else {
      dst[kOff] = static_cast<uint8_t>(bits);
    }
    store_chunk_pieces<T, kM, kOff + kS>(dst, q);
  }
}

// Store of a lane's V output bytes for an output whose virtual base sits kM bytes past
// a V-byte boundary: kM == 0 one word, 0 < kM < V naturally aligned pieces, kM < 0
// (offset not known at compile time) single bytes.
template <class T, int kM>
__device__ __forceinline__ void store_chunk_at(uint8_t* dst, const uint2& q) {
  if constexpr (kM == 0) {
    store_chunk<T, true>(dst, q);
  } else if constexpr (kM > 0) {
    store_chunk_pieces<T, kM>(dst, q);
  } else {
    store_chunk<T, false>(dst, q);
  }
}

// Calls f(ShiftC<M>{}) with M the compile-time copy of a non-zero output offset m < V.
template <class T, class F>
__device__ __forceinline__ void with_out_offset(uint32_t m, F&& f) {
  if constexpr (T::V == 4) {
    switch (m) {
      case 1: f(ShiftC<1>{}); break;
      case 2: f(ShiftC<2>{}); break;
      default: f(ShiftC<3>{}); break;
    }
  } else {
    switch (m) {
      case 1: f(ShiftC<1>{}); break;
      case 2: f(ShiftC<2>{}); break;
      case 3: f(ShiftC<3>{}); break;
      case 4: f(ShiftC<4>{}); break;
      case 5: f(ShiftC<5>{}); break;
      case 6: f(ShiftC<6>{}); break;
      default: f(ShiftC<7>{}); break;
    }
  }
}

// ---------------------------------------------------------------- fragment geometry
// The fragment is every element from (rs, cs) to (re, ce) in row-major order, so row
// i holds fragment columns [row_lo(i), row_hi(i)] (none when i is outside [rs, re])
// and column c holds the fragment rows from rs (rs + 1 when c < cs) to re (re - 1
// when c > ce).
__device__ __forceinline__ int64_t row_lo(const FragGeom& g, int64_t i) {
  return i == g.rs ? g.cs : 0;
}
__device__ __forceinline__ int64_t row_hi(const FragGeom& g, int64_t i) {
  return i == g.re ? g.ce : g.cols - 1;
}
__device__ __forceinline__ bool row_in(const FragGeom& g, int64_t i) {
  return i >= g.rs && i <= g.re;
}

// True when columns [c0, c1] of row i hold a fragment element.
__device__ __forceinline__ bool row_span_meets(const FragGeom& g, int64_t i, int64_t c0,
                                               int64_t c1) {
  return row_in(g, i) && max(c0, row_lo(g, i)) <= min(c1, row_hi(g, i));
}

// True when column c has a fragment element in rows [r_a, r_b).
__device__ __forceinline__ bool column_meets(const FragGeom& g, int64_t c, int64_t r_a,
                                             int64_t r_b) {
  const int64_t lo = c >= g.cs ? g.rs : g.rs + 1;
  const int64_t hi = c <= g.ce ? g.re : g.re - 1;
  return max(lo, r_a) <= min(hi, r_b - 1);
}

enum TileKind { kTileSkip = 0, kTileFast = 1, kTileMasked = 2 };

// Classify the warp tile whose top-left element is (row0, col0), tw columns wide.
// A tile is "fast" when it lies inside the matrix and every 16-byte chunk its rows
// load -- including the chunks a non-zero shift adds before the first and after the
// last element of each row segment -- lies inside the fragment.
template <class T>
__device__ __forceinline__ int classify_tile(const FragGeom& g, int64_t row0, int64_t col0,
                                             int tw) {
  const int64_t row_last = min(row0 + 31, g.rows - 1);
  const int64_t col_last = min(col0 + tw, g.cols) - 1;
  const int64_t first = row0 * g.cols + col0;
  const int64_t last = row_last * g.cols + col_last;
  if (last < g.start || first >= g.end) return kTileSkip;
  const bool whole = (row0 + 32 <= g.rows) && (col0 + tw <= g.cols);
  const int64_t lo = g.shift / T::kBytes;                 // elements loaded before the segment
  const int64_t hi = g.shift ? T::V - lo : 0;             // elements loaded after it
  if (g.fast_ok && whole && first - lo >= g.start && last + hi < g.end) return kTileFast;
  return kTileMasked;
}

// The split kernels' extra class: a tile cut only by the matrix's right edge, whose 32 rows
// lie inside the matrix and whose every element inside the matrix belongs to the fragment
// (aligned virtual base, cols a multiple of V).  It takes the fast path with the lanes past
// the edge idle, instead of the masked path's per-row membership tests.
constexpr int kTileEdge = 3;
template <class T>
__device__ __forceinline__ int classify_tile_edge(const FragGeom& g, int64_t row0, int64_t col0,
                                                  int tw) {
  const int kind = classify_tile<T>(g, row0, col0, tw);
  if (kind != kTileMasked || !g.fast_ok || g.shift != 0 || row0 + 32 > g.rows || col0 + tw <= g.cols)
    return kind;
  const int64_t first = row0 * g.cols + col0;            // the tile's first element
  const int64_t last = (row0 + 31) * g.cols + g.cols - 1;  // its last element inside the matrix
  return (first >= g.start && last < g.end) ? kTileEdge : kind;
}

// ---------------------------------------------------------------- row loads
template <bool kHint>
__device__ __forceinline__ uint4 ld_chunk(const void* p, uint64_t pol) {
  if constexpr (kHint) {
    return ld_hint16(p, pol);
  } else {
    return ld_stream16(p);
  }
}

// The first NW words of the 16-byte aligned chunk at p (the rest read as 0), with one
// load of 4, 8 or 16 bytes.
template <int NW, bool kHint>
__device__ __forceinline__ uint4 ld_head(const void* p, uint64_t pol) {
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if constexpr (NW >= 3) {
    v = ld_chunk<kHint>(p, pol);
  } else if constexpr (NW == 2) {
    if constexpr (kHint) {
      asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;"
                   : "=r"(v.x), "=r"(v.y) : "l"(p), "l"(pol));
    } else {
      asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    }
  } else {
    if constexpr (kHint) {
      asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;"
                   : "=r"(v.x) : "l"(p), "l"(pol));
    } else {
      asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v.x) : "l"(p));
    }
  }
  return v;
}

__device__ __forceinline__ uint32_t word_of(const uint4& c, int k) {
  return k == 0 ? c.x : (k == 1 ? c.y : (k == 2 ? c.z : c.w));
}

// Chunks of NB consecutive rows of a fast tile for this lane: chunk r holds the V
// elements (row0 + r, col0 + V*lane ...).  `src` is the lane's element address in
// the first row.  kS is the byte offset of the fragment's virtual base from a
// 16-byte boundary (a multiple of the element size).  kS == 0: one aligned 16-byte
// load per row.  kS != 0: each lane loads the aligned chunk that holds its first
// element and takes the words past it from the next lane's chunk -- only the
// ceil(kS/4) words it needs, one shuffle each -- and a half-word funnel shift
// finishes a 2-byte offset.  Lane 31 takes those words from the chunk after the tile
// row: it loads them itself for every row, or (kRowLanes) lane r loads them for row
// r with a single load for the batch and lane 31 gets them by one more shuffle per
// word, which holds 4 registers instead of 4 per row for larger batches.
// All lanes of the warp must be active.
template <int NB, int kS, bool kHint = false, bool kRowLanes = false>
__device__ __forceinline__ void load_rows(uint4 (&v)[NB], const char* src, int64_t row_bytes,
                                          int lane, uint64_t pol = 0) {
  if constexpr (kS == 0) {
#pragma unroll
    for (int r = 0; r < NB; ++r) v[r] = ld_chunk<kHint>(src + r * row_bytes, pol);
  } else {
    static_assert(kS > 0 && kS < 16, "shift is a byte offset inside a 16-byte chunk");
    constexpr int Q = kS / 4;            // whole words of the own chunk to skip
    constexpr int R = (kS % 4) * 8;      // bits to skip inside the next word (0 or 16)
    constexpr int NW = Q + (R != 0);     // words taken from the next lane's chunk
    const char* a = src - kS;
    static_assert(NB <= 32, "one lane per row of the batch");
    uint4 extra[kRowLanes ? 1 : NB];
    if constexpr (kRowLanes) {  // lane r: the chunk after row r of the tile
      extra[0] = lane < NB ? ld_head<NW, kHint>(a - lane * 16 + 32 * 16 + lane * row_bytes, pol)
                           : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int r = 0; r < NB; ++r) {
      v[r] = ld_chunk<kHint>(a + r * row_bytes, pol);
      if constexpr (!kRowLanes)
        extra[r] = lane == 31 ? ld_head<NW, kHint>(a + r * row_bytes + 16, pol) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int r = 0; r < NB; ++r) {
      uint32_t w[8] = {v[r].x, v[r].y, v[r].z, v[r].w, 0u, 0u, 0u, 0u};
#pragma unroll
      for (int k = 0; k < NW; ++k) {
        const uint32_t nx = __shfl_down_sync(kFullMask, w[k], 1);
        uint32_t ex;
        if constexpr (kRowLanes) {
          ex = __shfl_sync(kFullMask, word_of(extra[0], k), r);
        } else {
          ex = word_of(extra[r], k);
        }
        w[4 + k] = lane == 31 ? ex : nx;
      }
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) o[k] = R ? __funnelshift_r(w[Q + k], w[Q + k + 1], R) : w[Q + k];
      v[r] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// Calls f(ShiftC<S>{}) with S the compile-time copy of `shift`, a non-zero byte
// offset from a 16-byte boundary that is a multiple of T's element size: each offset
// gets its own specialisation of the realigning loads.
template <class T, class F>
__device__ __forceinline__ void with_shift(int32_t shift, F&& f) {
  if constexpr (T::kBytes == 4) {
    switch (shift) {
      case 4: f(ShiftC<4>{}); break;
      case 8: f(ShiftC<8>{}); break;
      default: f(ShiftC<12>{}); break;
    }
  } else {
    switch (shift) {
      case 2: f(ShiftC<2>{}); break;
      case 4: f(ShiftC<4>{}); break;
      case 6: f(ShiftC<6>{}); break;
      case 8: f(ShiftC<8>{}); break;
      case 10: f(ShiftC<10>{}); break;
      case 12: f(ShiftC<12>{}); break;
      default: f(ShiftC<14>{}); break;
    }
  }
}

// Chunks of NB consecutive rows of a masked tile: element k of chunk r is loaded only
// when (row0 + r, j + k) is inside the matrix and the fragment; others read as 0.
// Chunks that lie wholly inside the fragment take one 16-byte load when the
// fragment's virtual base is 16-byte aligned.  Bit (r * V + k) of the returned mask
// marks the loaded elements.
template <class T, int NB>
__device__ __forceinline__ uint64_t load_rows_masked(uint4 (&v)[NB], const FragGeom& g,
                                                     const void* in, int64_t row0, int64_t j) {
  constexpr uint64_t kChunkBits = (uint64_t(1) << T::V) - 1;
  const bool vec = g.fast_ok && g.shift == 0;
  // byte offset of element (row0, j) from the fragment's first element
  int64_t off = (row0 * g.cols + j - g.start) * T::kBytes;
  const int64_t row_bytes = g.cols * T::kBytes;
  const char* base = static_cast<const char*>(in);
  uint64_t valid = 0;
#pragma unroll
  for (int r = 0; r < NB; ++r, off += row_bytes) {
    v[r] = make_uint4(0u, 0u, 0u, 0u);
    const int64_t i = row0 + r;
    if (!row_in(g, i) || i >= g.rows) continue;
    const int64_t lo = row_lo(g, i), hi = row_hi(g, i);
    if (vec && j >= lo && j + T::V - 1 <= hi) {
      v[r] = *reinterpret_cast<const uint4*>(base + off);
      valid |= kChunkBits << (r * T::V);
      continue;
    }
#pragma unroll
    for (int k = 0; k < T::V; ++k) {
      if (j + k >= lo && j + k <= hi) {
        chunk_set<T>(v[r], k, load_bits<T>(base + off, k));
        valid |= uint64_t(1) << (r * T::V + k);
      }
    }
  }
  return valid;
}

// Tile t of a job batch, in processing order: all boundary-band tiles of all jobs
// first (their masked, slower tiles then overlap the streaming of the interior
// bands instead of trailing it), then all interior tiles.  Returns the job index and
// the tile's top-left element.
template <class P, int N>
__device__ __forceinline__ int batch_tile(const JobBatch<P, N>& b, int64_t t, int tw,
                                          int64_t& row0, int64_t& col0) {
  const int n = b.njobs;
  const bool boundary = t < b.prefix_a[n];
  const int64_t* prefix = boundary ? b.prefix_a : b.prefix_b;
  if (!boundary) t -= b.prefix_a[n];
  int lo = 0, hi = N == 1 ? 1 : n;  // prefix[lo] <= t < prefix[hi]
  while (N > 1 && hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= t) lo = mid; else hi = mid;
  }
  const FragGeom& g = b.job[lo].g;
  const int64_t k = t - prefix[lo];
  int64_t band;
  if (boundary) {
    band = k < g.coltiles ? g.band0 : g.band0 + g.ntiles / g.coltiles - 1;
  } else {
    band = g.band0 + 1 + k / g.coltiles;
  }
  row0 = band * 32;
  col0 = (k % g.coltiles) * tw;
  return lo;
}

// Blocks for a persistent grid over `ntiles` warp tiles: as many rounds as the
// resident capacity (`max_blocks` blocks of `warps` warps) needs, then just enough
// blocks that every warp gets the same number of tiles (within one), instead of a
// full last round being followed by a mostly idle one.
inline unsigned balanced_grid(int64_t ntiles, int warps, int64_t max_blocks) {
  const int64_t cap = max_blocks * warps;
  const int64_t rounds = (ntiles + cap - 1) / cap;
  const int64_t warps_needed = (ntiles + rounds - 1) / rounds;
  int64_t blocks = (warps_needed + warps - 1) / warps;
  if (blocks < 1) blocks = 1;
  return unsigned(blocks < max_blocks ? blocks : max_blocks);
}

// Single-fragment launches of at most this many warp tiles per SM split every tile over
// four warps, a quarter of its rows each: with so few tiles a whole-tile grid leaves the
// SMs short of warps, and a launch lasts one warp's chain of row batches (8 dependent
// round trips on a cut tile) rather than its HBM traffic.  The cast, whose warps share
// nothing, gains up to more tiles than the amax, whose quarters meet at a barrier.
#ifndef MXFP8_AMAX_SPLIT_TILES_PER_SM
#define MXFP8_AMAX_SPLIT_TILES_PER_SM 16
#endif
#ifndef MXFP8_CAST_SPLIT_TILES_PER_SM
#define MXFP8_CAST_SPLIT_TILES_PER_SM 32
#endif
inline int64_t split_max_tiles(const DeviceInfo& dev, int tiles_per_sm) {
  return int64_t(dev.sms) * tiles_per_sm;
}

// Blocks for one tile per warp: the hardware block scheduler then hands out tiles
// dynamically, which absorbs uneven per-tile cost (tiles cut by a fragment boundary,
// row-only next to bidirectional jobs in one batch) better than a static persistent
// assignment.  The kernels' grid-stride loop covers anything beyond the 2^31-1 cap.
inline unsigned tile_grid(int64_t ntiles, int warps) {
  const int64_t blocks = (ntiles + warps - 1) / warps;
  return unsigned(blocks < 1 ? 1 : (blocks < 2147483647 ? blocks : 2147483647));
}

}  // namespace mxfp8
