// NVFP4 partial amax, scale update and partial cast (sm_103a).
//
// The page "Support row-only MXFP8 distributed master-weight casts" leaves NVFP4 out
// of its scope (section "Scope") and prints no rule for it.  These kernels take the
// same distributed steps as the MXFP8 path for the NVFP4 format as NVIDIA defines it,
// under one stated convention:
//   blocks  1x16 along rows (rowwise) and 16x1 along columns (columnwise);
//   G       tensor amax, max |x| over the whole weight (FP32);
//   S       tensor encode scale 2688 / G in FP32 (448 * 6: the largest E4M3 scale times
//           the largest E2M1 value); 1 when G == 0, the largest float on overflow;
//   s       block scale E4M3(fp32(fp32(A / 6) * S)) for block amax A (nearest-even,
//           saturating at 448);
//   M       block multiplier fp32(S / decode(s)), 0 when s decodes to 0;
//   q       data E2M1(fp32(y * M)), y the master value rounded to BF16 (nearest-even,
//           saturating at 6), two codes per byte, the even position in the low nibble.
// Every FP32 step is one correctly rounded operation (division, mul.rn), so the codes
// are decided exactly as a scalar restatement of these steps decides them.
//
// Work unit as in the MXFP8 kernels: one warp per 32-row x (32*V)-column tile, one
// 16-byte input chunk per lane per row (realigned across lanes when the fragment's
// virtual base is not 16-byte aligned), tiles cut by the fragment or the matrix edge
// on predicated loads.  A 1x16 row block is 16/V lanes (a 2- or 1-step butterfly); a
// lane keeps the maxima of its V columns over rows 0-15 and 16-31 of the tile (the two
// 16x1 column blocks of the tile).  The partial amax also folds the fragment's largest
// |x| into one shared word per block, and one atomic max per block into the tensor
// amax.  The cast kernel first builds, per block, the 256-entry table of multipliers
// M = S / decode(s) in shared memory, so that a row's multiplier is one table read.
#include <cfloat>

#include "common.cuh"

namespace mxfp8 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowBatch = 8;
constexpr int kMaskBatch = 4;
// Resident blocks per SM the amax and cast kernels are compiled for (3: at most 85
// registers, 8 rows of 16-byte loads in flight per lane).
#ifndef MXFP8_NVFP4_AMAX_MIN_BLOCKS
#define MXFP8_NVFP4_AMAX_MIN_BLOCKS 3
#endif
#ifndef MXFP8_NVFP4_CAST_MIN_BLOCKS
#define MXFP8_NVFP4_CAST_MIN_BLOCKS 3
#endif
constexpr int kAmaxMinBlocks = MXFP8_NVFP4_AMAX_MIN_BLOCKS;
constexpr int kCastMinBlocks = MXFP8_NVFP4_CAST_MIN_BLOCKS;

// Lanes that hold one 1x16 row block.
template <class T>
__device__ __host__ constexpr int lanes16() { return 16 / T::V; }

template <class T>
__device__ __forceinline__ uint32_t block16_max(uint32_t m) {
#pragma unroll
  for (int off = 1; off < lanes16<T>(); off <<= 1) m = max(m, __shfl_xor_sync(kFullMask, m, off));
  return m;
}

__device__ __forceinline__ uint32_t warp_max(uint32_t m) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(kFullMask, m, off));
  return m;
}

// FP32 bit pattern of an |x| bit pattern of the input dtype (exact), NaN canonical.
template <class T>
__device__ __forceinline__ uint32_t f32_bits(uint32_t m) {
  if constexpr (T::kBytes == 4) {
    return canonical_nan<F32T>(m);
  } else {
    return canonical_nan<F32T>(m << 16);
  }
}

// ---------------------------------------------------------------- scale arithmetic
__device__ __forceinline__ float tensor_scale(float g) {
  if (g == 0.0f) return 1.0f;
  const float s = __fdiv_rn(2688.0f, g);
  return isinf(s) ? FLT_MAX : s;
}

// fp32(a / 6), correctly rounded, by Markstein's division with a correctly rounded
// reciprocal and an exact FMA remainder (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990):
// q0 = a * RN(1/6), r = a - 6 q0 (exact), q = RN(q0 + r * RN(1/6)).  For every float a
// from 2^-124 up to the largest float this equals the IEEE quotient (checked input by
// input); below 2^-124 the remainder can be subnormal and inexact, so there, and for
// negative, infinite and NaN inputs, the IEEE division is taken.  Three operations
// instead of a full division per block amax.
__device__ __forceinline__ float div6_rn(float a) {
  constexpr float kInv6 = 0x1.555556p-3f;  // RN(1/6)
  if (a >= 0x1p-124f && a <= FLT_MAX) {
    const float q0 = __fmul_rn(a, kInv6);
    const float r = __fmaf_rn(-6.0f, q0, a);
    return __fmaf_rn(r, kInv6, q0);
  }
  return __fdiv_rn(a, 6.0f);
}

// fp32(fp32(A / 6) * S): the value the block scale is the E4M3 rounding of.
__device__ __forceinline__ float block_scale_value(float a, float s_enc) {
  return __fmul_rn(div6_rn(a), s_enc);
}

__device__ __forceinline__ uint32_t block_scale(float a, float s_enc) {
  return e4m3x2_rn_sat(block_scale_value(a, s_enc), 0.0f) & 0xffu;
}

// Value of an E4M3 byte (sign, 4 exponent bits with bias 7, 3 mantissa bits; 0x7F and
// 0xFF are NaN), exactly, from the format definition.
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  const uint32_t sign = (b & 0x80u) << 24, e = (b >> 3) & 15u, m = b & 7u;
  if (e == 15u && m == 7u) return __uint_as_float(0x7fc00000u);
  if (e == 0u) return __uint_as_float(sign | __float_as_uint(float(m) * 0x1p-9f));
  return __uint_as_float(sign | ((e + 120u) << 23) | (m << 20));
}

// Two FP32 values to E2M1 (nearest-even, saturating to +-6): lo in the low nibble.
__device__ __forceinline__ uint32_t e2m1x2_rn_sat(float lo, float hi) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The V codes of y[k] * mult[k], packed: FP32 input 2 bytes, BF16 input 4 bytes.
template <class T>
__device__ __forceinline__ uint32_t e2m1_chunk(const float (&y)[T::V], const float (&mult)[T::V]) {
  float p[T::V];
#pragma unroll
  for (int k = 0; k < T::V; k += 2) mul2_rn(y[k], y[k + 1], mult[k], mult[k + 1], p[k], p[k + 1]);
  uint32_t q = 0;
#pragma unroll
  for (int k = 0; k < T::V; k += 2) q |= e2m1x2_rn_sat(p[k], p[k + 1]) << (4 * k);
  return q;
}

// Store a lane's V/2 output bytes: one 2- or 4-byte word when aligned, else bytes.
template <class T>
__device__ __forceinline__ void store_codes(uint8_t* dst, uint32_t q, bool vec) {
  if (vec) {
    if constexpr (T::V == 4) {
      *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(q);
    } else {
      *reinterpret_cast<uint32_t*>(dst) = q;
    }
  } else {
#pragma unroll
    for (int k = 0; k < T::V / 2; ++k) dst[k] = static_cast<uint8_t>(q >> (8 * k));
  }
}

// ---------------------------------------------------------------- partial amax
template <class T>
__device__ __forceinline__ void store_col16(const Nvfp4AmaxParams& p, int64_t band16, int64_t j,
                                            const uint4& cm) {
  uint32_t* dst = reinterpret_cast<uint32_t*>(p.amax_c) + band16 * p.ld_c + j;
  uint32_t w[T::V];
#pragma unroll
  for (int k = 0; k < T::V; ++k) w[k] = f32_bits<T>(chunk_get<T>(cm, k));
  if (p.vec_c) {
#pragma unroll
    for (int k = 0; k < T::V; k += 4)
      *reinterpret_cast<uint4*>(dst + k) = make_uint4(w[k], w[k + 1], w[k + 2], w[k + 3]);
  } else {
#pragma unroll
    for (int k = 0; k < T::V; ++k) dst[k] = w[k];
  }
}

// Whole tile inside the fragment; returns the lane's largest |x| (input-dtype bits).  Rows
// r_lo .. r_hi-1 of the tile (all 32, or a quarter when four warps share it); the column
// maxima are stored, or -- colpart != nullptr, a quarter lies inside one 16-row half --
// that half's maxima are left in *colpart for the warps to combine.
template <class T, bool kCol, int kS>
__device__ __forceinline__ uint32_t amax_tile_fast(const Nvfp4AmaxParams& p, int64_t row0,
                                                   int64_t col0, int lane, int r_lo = 0,
                                                   int r_hi = 32, uint4* colpart = nullptr) {
  const int64_t cols = p.g.cols;
  const int64_t j = col0 + lane * T::V;
  const char* src = static_cast<const char*>(p.in) + (row0 * cols + j - p.g.start) * T::kBytes;
  const int64_t row_bytes = cols * T::kBytes;
  const bool writer = (lane % lanes16<T>()) == 0;
  uint32_t* out_r = reinterpret_cast<uint32_t*>(p.amax_r) + row0 * p.ld_r + (j >> 4);
  uint4 c0 = make_uint4(0u, 0u, 0u, 0u), c1 = c0;
  uint32_t tmax = 0;
#pragma unroll 1
  for (int rb = r_lo; rb < r_hi; rb += kRowBatch) {
    uint4 v[kRowBatch];
    load_rows<kRowBatch, kS, false, kS != 0>(v, src + rb * row_bytes, row_bytes, lane);
#pragma unroll
    for (int r = 0; r < kRowBatch; ++r) {
      const uint4 a = chunk_abs<T>(v[r]);
      if constexpr (kCol) {
        if (rb < 16) c0 = chunk_max<T>(c0, a); else c1 = chunk_max<T>(c1, a);
      }
      const uint32_t m = block16_max<T>(chunk_reduce<T>(a));
      tmax = max(tmax, m);
      if (writer) out_r[(rb + r) * p.ld_r] = f32_bits<T>(m);
    }
  }
  if constexpr (kCol) {
    if (colpart != nullptr) {
      *colpart = r_lo < 16 ? c0 : c1;
    } else {
      store_col16<T>(p, row0 >> 4, j, c0);
      store_col16<T>(p, (row0 >> 4) + 1, j, c1);
    }
  }
  return tmax;
}

// Tile cut by the fragment boundary or the matrix edge: predicated loads; only blocks
// that meet the fragment are written.
// Column maxima of 16-row half h of a cut tile: only the columns whose block meets the
// fragment.
template <class T>
__device__ __forceinline__ void store_col16_masked(const Nvfp4AmaxParams& p, int64_t row0, int64_t j,
                                                   int h, const uint4& cm) {
  const FragGeom& g = p.g;
  const int64_t ra = row0 + 16 * h;
  if (ra >= g.rows) return;
  const int64_t re = min(ra + 16, g.rows);
#pragma unroll
  for (int k = 0; k < T::V; ++k) {
    const int64_t col = j + k;
    if (col < g.cols && column_meets(g, col, ra, re))
      p.amax_c[(ra >> 4) * p.ld_c + col] = __uint_as_float(f32_bits<T>(chunk_get<T>(cm, k)));
  }
}

// MB: rows per batch of predicated loads (a split tile's warp takes its 8 rows at once).
template <class T, bool kCol, int MB = kMaskBatch>
__device__ __forceinline__ uint32_t amax_tile_masked(const Nvfp4AmaxParams& p, int64_t row0,
                                                     int64_t col0, int lane, int r_lo = 0,
                                                     int r_hi = 32, uint4* colpart = nullptr) {
  const FragGeom& g = p.g;
  const int64_t j = col0 + lane * T::V;
  const bool writer = (lane % lanes16<T>()) == 0;
  const int64_t b0 = j & ~int64_t(15);  // first column of this lane's row block
  uint4 c0 = make_uint4(0u, 0u, 0u, 0u), c1 = c0;
  uint32_t tmax = 0;
#pragma unroll 1
  for (int rb = r_lo; rb < r_hi; rb += MB) {  // warp-uniform: the butterflies stay converged
    uint4 v[MB];
    load_rows_masked<T, MB>(v, g, p.in, row0 + rb, j);
#pragma unroll
    for (int r = 0; r < MB; ++r) {
      const uint4 a = chunk_abs<T>(v[r]);
      if constexpr (kCol) {
        if (rb < 16) c0 = chunk_max<T>(c0, a); else c1 = chunk_max<T>(c1, a);
      }
      const uint32_t m = block16_max<T>(chunk_reduce<T>(a));
      tmax = max(tmax, m);
      const int64_t i = row0 + rb + r;
      if (writer && i < g.rows && b0 < g.cols && row_span_meets(g, i, b0, min(b0 + 15, g.cols - 1)))
        p.amax_r[i * p.ld_r + (b0 >> 4)] = __uint_as_float(f32_bits<T>(m));
    }
  }
  if constexpr (kCol) {
    if (colpart != nullptr) {
      *colpart = r_lo < 16 ? c0 : c1;
    } else {
      store_col16_masked<T>(p, row0, j, 0, c0);
      store_col16_masked<T>(p, row0, j, 1, c1);
    }
  }
  return tmax;
}

// kSplit: four warps share each tile, 8 rows each (a block's eight warps take two tiles);
// the two warps of each 16-row half combine their column maxima in shared memory.  For
// launches of few tiles, whose time is one warp's chain of row batches.
template <class T, bool kCol, bool kShift, bool kSplit>
__global__ void __launch_bounds__(kThreads, kAmaxMinBlocks) k_nvfp4_amax(
    const __grid_constant__ JobBatch<Nvfp4AmaxParams, 1> b) {
  __shared__ uint32_t block_max;
  grid_dependency_sync();
  if (threadIdx.x == 0) block_max = 0;
  __syncthreads();
  constexpr int TW = tile_width<T>();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const Nvfp4AmaxParams& p = b.job[0];
  const int64_t total = b.prefix_a[1] + b.prefix_b[1];
  uint32_t wmax = 0;
  if constexpr (!kSplit) {
    const int64_t stride = int64_t(gridDim.x) * kWarps;
    for (int64_t t = int64_t(blockIdx.x) * kWarps + warp; t < total; t += stride) {
      int64_t row0, col0;
      batch_tile(b, t, TW, row0, col0);
      const int kind = classify_tile<T>(p.g, row0, col0, TW);
      if (kind == kTileFast) {
        if constexpr (kShift) {
          with_shift<T>(p.g.shift, [&](auto s) {
            wmax = max(wmax, amax_tile_fast<T, kCol, decltype(s)::value>(p, row0, col0, lane));
          });
        } else {
          wmax = max(wmax, amax_tile_fast<T, kCol, 0>(p, row0, col0, lane));
        }
      } else if (kind == kTileMasked) {
        wmax = max(wmax, amax_tile_masked<T, kCol>(p, row0, col0, lane));
      }
    }
  } else {
    static_assert(!kShift, "the split kernel serves aligned fragments");
    __shared__ uint4 part[kWarps][32];
    const int q = warp & 3;  // quarter: rows 8q .. 8q+7, in 16-row half q / 2
    // block-uniform rounds (every warp reaches every barrier); warp w of a round takes
    // quarter w % 4 of tile (round * 8 + w) / 4
    for (int64_t base = int64_t(blockIdx.x) * kWarps; base < total * 4; base += int64_t(gridDim.x) * kWarps) {
      const int64_t t = (base + warp) >> 2;
      int kind = kTileSkip;
      int64_t row0 = 0, col0 = 0;
      if (t < total) {
        batch_tile(b, t, TW, row0, col0);
        kind = classify_tile<T>(p.g, row0, col0, TW);
        uint4* cp = kCol ? &part[warp][lane] : nullptr;
        if (kind == kTileFast) {
          wmax = max(wmax, amax_tile_fast<T, kCol, 0>(p, row0, col0, lane, 8 * q, 8 * q + 8, cp));
        } else if (kind == kTileMasked) {
          wmax = max(wmax, amax_tile_masked<T, kCol, 8>(p, row0, col0, lane, 8 * q, 8 * q + 8, cp));
        }
      }
      if constexpr (kCol) {
        __syncthreads();
        if ((q & 1) == 0 && kind != kTileSkip) {  // quarters 0 and 2 combine their half
          const uint4 cm = chunk_max<T>(part[warp][lane], part[warp + 1][lane]);
          const int64_t j = col0 + lane * T::V;
          if (kind == kTileFast) {
            store_col16<T>(p, (row0 >> 4) + (q >> 1), j, cm);
          } else {
            store_col16_masked<T>(p, row0, j, q >> 1, cm);
          }
        }
        __syncthreads();
      }
    }
  }
  wmax = warp_max(f32_bits<T>(wmax));
  if (lane == 0 && wmax != 0) atomicMax(&block_max, wmax);
  __syncthreads();
  if (threadIdx.x == 0 && block_max != 0) atomicMax(p.amax_t, block_max);
}

// ---------------------------------------------------------------- scale update
// Each thread loads kScaleItems 16-byte groups of amaxes (grid-strided) before it converts
// any of them, so that several loads per thread are in flight.
constexpr int kScaleItems = 4;
constexpr int kScaleBlocksPerSM = 6;

__global__ void __launch_bounds__(kThreads, kScaleBlocksPerSM) k_nvfp4_scales(
    const __grid_constant__ Nvfp4ScaleParams p) {
  grid_dependency_sync();
  const float s_enc = tensor_scale(*p.amax_t);
  const Nvfp4ScaleSegment& s = p.seg[blockIdx.y];
  const int64_t n = s.nrows * s.ncols;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (s.vec) {
    const int64_t nq = n / 4;
    for (int64_t q0 = tid; q0 < nq; q0 += stride * kScaleItems) {
      uint4 a[kScaleItems];
#pragma unroll
      for (int u = 0; u < kScaleItems; ++u)
        if (q0 + u * stride < nq) a[u] = ld_stream16(s.amax + 4 * (q0 + u * stride));
#pragma unroll
      for (int u = 0; u < kScaleItems; ++u) {
        const int64_t q = q0 + u * stride;
        if (q >= nq) break;
        const uint32_t out =
            e4m3x2_rn_sat(block_scale_value(__uint_as_float(a[u].x), s_enc),
                          block_scale_value(__uint_as_float(a[u].y), s_enc)) |
            (e4m3x2_rn_sat(block_scale_value(__uint_as_float(a[u].z), s_enc),
                           block_scale_value(__uint_as_float(a[u].w), s_enc)) << 16);
        reinterpret_cast<uint32_t*>(s.scale)[q] = out;
      }
    }
  } else {
    for (int64_t e = tid; e < n; e += stride) {
      const int64_t r = e / s.ncols, c = e % s.ncols;
      s.scale[r * s.ld_s + c] = static_cast<uint8_t>(block_scale(s.amax[r * s.ld_a + c], s_enc));
    }
  }
}

// ---------------------------------------------------------------- partial cast
// Whole tile inside the fragment: 16-byte loads, the row's multiplier from the table.
template <class T, bool kCol, int kS>
__device__ __forceinline__ void cast_tile_fast(const Nvfp4CastParams& p, const float* mult,
                                               int64_t row0, int64_t col0, int lane,
                                               int r_lo = 0, int r_hi = 32) {
  const int64_t cols = p.g.cols;
  const int64_t j = col0 + lane * T::V;
  const char* src = static_cast<const char*>(p.in) + (row0 * cols + j - p.g.start) * T::kBytes;
  const int64_t row_bytes = cols * T::kBytes;
  const uint8_t* srow = p.s_r + row0 * p.ld_sr + (j >> 4);
  const int64_t n0 = row0 * cols + j + p.out_shift;  // nibble of the lane's first element (even)
  constexpr bool kRowLanes = kS != 0 && T::kBytes == 4;
  constexpr int NB = kS ? (kRowLanes ? kRowBatch : 4) : kRowBatch;
  float mc0[T::V], mc1[T::V];
  if constexpr (kCol) {
    const uint8_t* sc = p.s_c + (row0 >> 4) * p.ld_sc + j;
#pragma unroll
    for (int k = 0; k < T::V; ++k) {
      mc0[k] = mult[sc[k]];
      mc1[k] = mult[sc[p.ld_sc + k]];
    }
  }
  const bool vec = p.vec_out != 0;
#pragma unroll 1
  for (int rb = r_lo; rb < r_hi; rb += NB) {
    uint4 v[NB];
    uint32_t sb[NB];
#pragma unroll
    for (int r = 0; r < NB; ++r) sb[r] = srow[(rb + r) * p.ld_sr];
    load_rows<NB, kS, false, kRowLanes>(v, src + rb * row_bytes, row_bytes, lane);
#pragma unroll
    for (int r = 0; r < NB; ++r) {
      float y[T::V];
      model_values<T, kModelBF16>(v[r], y);
      float mr[T::V];
      const float m = mult[sb[r]];
#pragma unroll
      for (int k = 0; k < T::V; ++k) mr[k] = m;
      const int64_t o = (n0 + (rb + r) * cols) >> 1;
      store_codes<T>(p.out_r + o, e2m1_chunk<T>(y, mr), vec);
      if constexpr (kCol) store_codes<T>(p.out_c + o, e2m1_chunk<T>(y, rb < 16 ? mc0 : mc1), vec);
    }
  }
}

// Tile cut by the fragment boundary or the matrix edge.  Fragments start and end on
// even flat indices and rows hold an even number of elements, so the two elements of
// an output byte are both inside the fragment or both outside: a lane writes whole
// bytes only.
template <class T, bool kCol>
__device__ __forceinline__ void cast_tile_masked(const Nvfp4CastParams& p, const float* mult,
                                                 int64_t row0, int64_t col0, int lane,
                                                 int r_lo = 0, int r_hi = 32) {
  constexpr uint64_t kChunkBits = (uint64_t(1) << T::V) - 1;
  const FragGeom& g = p.g;
  const int64_t j = col0 + lane * T::V;
  if (j >= g.cols) return;
  const int64_t blk = j >> 4;
  float mc0[T::V], mc1[T::V];
  if constexpr (kCol) {
#pragma unroll
    for (int k = 0; k < T::V; ++k) {
      const bool in = j + k < g.cols;
      mc0[k] = in ? mult[p.s_c[(row0 >> 4) * p.ld_sc + j + k]] : 0.0f;
      mc1[k] = (in && row0 + 16 < g.rows) ? mult[p.s_c[((row0 >> 4) + 1) * p.ld_sc + j + k]] : 0.0f;
    }
  }
#pragma unroll 1
  for (int rb = r_lo; rb < r_hi && row0 + rb < g.rows; rb += kMaskBatch) {
    uint4 v[kMaskBatch];
    const uint64_t valid = load_rows_masked<T, kMaskBatch>(v, g, p.in, row0 + rb, j);
    if (valid == 0) continue;
#pragma unroll
    for (int r = 0; r < kMaskBatch; ++r) {
      const uint64_t bits = (valid >> (r * T::V)) & kChunkBits;
      if (bits == 0) continue;
      const int64_t i = row0 + rb + r;
      float y[T::V];
      model_values<T, kModelBF16>(v[r], y);
      float mr[T::V];
      const float m = mult[p.s_r[i * p.ld_sr + blk]];
#pragma unroll
      for (int k = 0; k < T::V; ++k) mr[k] = m;
      const uint32_t qr = e2m1_chunk<T>(y, mr);
      uint32_t qc = 0;
      if constexpr (kCol) qc = e2m1_chunk<T>(y, rb < 16 ? mc0 : mc1);
      const int64_t o = (i * g.cols + j + p.out_shift) >> 1;
      if (p.vec_out && g.fast_ok && bits == kChunkBits) {
        store_codes<T>(p.out_r + o, qr, true);
        if constexpr (kCol) store_codes<T>(p.out_c + o, qc, true);
      } else {
#pragma unroll
        for (int k = 0; k < T::V / 2; ++k) {
          if (bits & (uint64_t(1) << (2 * k))) {
            p.out_r[o + k] = static_cast<uint8_t>(qr >> (8 * k));
            if constexpr (kCol) p.out_c[o + k] = static_cast<uint8_t>(qc >> (8 * k));
          }
        }
      }
    }
  }
}

// kSplit: four warps per tile, 8 rows each (no exchange between them), for launches of
// few tiles.
template <class T, bool kCol, bool kShift, bool kSplit>
__global__ void __launch_bounds__(kThreads, kCastMinBlocks) k_nvfp4_cast(
    const __grid_constant__ JobBatch<Nvfp4CastParams, 1> b) {
  __shared__ float mult[256];
  grid_dependency_sync();
  const Nvfp4CastParams& p = b.job[0];
  {
    const float s_enc = tensor_scale(*p.amax_t);
    for (int s = threadIdx.x; s < 256; s += blockDim.x) {
      const float d = e4m3_value(uint32_t(s));
      mult[s] = d == 0.0f ? 0.0f : __fdiv_rn(s_enc, d);
    }
  }
  __syncthreads();
  constexpr int TW = tile_width<T>();
  constexpr int kParts = kSplit ? 4 : 1;
  const int lane = threadIdx.x & 31;
  const int64_t total = (b.prefix_a[1] + b.prefix_b[1]) * kParts;
  const int64_t stride = int64_t(gridDim.x) * kWarps;
  for (int64_t u = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5); u < total; u += stride) {
    const int64_t t = kSplit ? u >> 2 : u;
    const int r_lo = kSplit ? 8 * int(u & 3) : 0, r_hi = kSplit ? r_lo + 8 : 32;
    int64_t row0, col0;
    batch_tile(b, t, TW, row0, col0);
    const int kind = classify_tile<T>(p.g, row0, col0, TW);
    if (kind == kTileFast) {
      if constexpr (kShift) {
        with_shift<T>(p.g.shift, [&](auto s) {
          cast_tile_fast<T, kCol, decltype(s)::value>(p, mult, row0, col0, lane, r_lo, r_hi);
        });
      } else {
        cast_tile_fast<T, kCol, 0>(p, mult, row0, col0, lane, r_lo, r_hi);
      }
    } else if (kind == kTileMasked) {
      cast_tile_masked<T, kCol>(p, mult, row0, col0, lane, r_lo, r_hi);
    }
  }
}

// Few tiles (at most the MXFP8 amax kernel's per-SM threshold): the split kernels.
template <class T, bool kCol, bool kShift>
cudaError_t launch_amax(const Nvfp4AmaxParams& p, const DeviceInfo& dev, cudaStream_t stream) {
  JobBatch<Nvfp4AmaxParams, 1> b;
  const int64_t total = fill_batch(b, &p, 1);
  if (total == 0) return cudaSuccess;
  if constexpr (!kShift) {
    if (total <= split_max_tiles(dev, MXFP8_AMAX_SPLIT_TILES_PER_SM))
      return launch_kernel(k_nvfp4_amax<T, kCol, kShift, true>, tile_grid(total * 4, kWarps), kThreads, 0,
                           stream, b);
  }
  return launch_kernel(k_nvfp4_amax<T, kCol, kShift, false>, tile_grid(total, kWarps), kThreads, 0, stream, b);
}

template <class T, bool kCol, bool kShift>
cudaError_t launch_cast(const Nvfp4CastParams& p, const DeviceInfo& dev, cudaStream_t stream) {
  JobBatch<Nvfp4CastParams, 1> b;
  const int64_t total = fill_batch(b, &p, 1);
  if (total == 0) return cudaSuccess;
  if constexpr (!kShift) {
    // the MXFP8 amax threshold: split measured slower on the 4096x4096 FP32 cast (4096
    // tiles, 14.1 -> 16.6 us), which the MXFP8 cast's threshold would split
    if (total <= split_max_tiles(dev, MXFP8_AMAX_SPLIT_TILES_PER_SM))
      return launch_kernel(k_nvfp4_cast<T, kCol, kShift, true>, tile_grid(total * 4, kWarps), kThreads, 0,
                           stream, b);
  }
  return launch_kernel(k_nvfp4_cast<T, kCol, kShift, false>, tile_grid(total, kWarps), kThreads, 0, stream, b);
}

template <class T>
cudaError_t amax_for(const Nvfp4AmaxParams& p, bool shifted, const DeviceInfo& dev, cudaStream_t stream) {
  const bool col = p.amax_c != nullptr;
  if (shifted) return col ? launch_amax<T, true, true>(p, dev, stream) : launch_amax<T, false, true>(p, dev, stream);
  return col ? launch_amax<T, true, false>(p, dev, stream) : launch_amax<T, false, false>(p, dev, stream);
}

template <class T>
cudaError_t cast_for(const Nvfp4CastParams& p, bool shifted, const DeviceInfo& dev, cudaStream_t stream) {
  const bool col = p.out_c != nullptr;
  if (shifted) return col ? launch_cast<T, true, true>(p, dev, stream) : launch_cast<T, false, true>(p, dev, stream);
  return col ? launch_cast<T, true, false>(p, dev, stream) : launch_cast<T, false, false>(p, dev, stream);
}

}  // namespace

cudaError_t launch_nvfp4_amax(const Nvfp4AmaxParams& p, int dtype, bool shifted,
                              const DeviceInfo& dev, cudaStream_t stream) {
  return dtype == 0 ? amax_for<F32T>(p, shifted, dev, stream) : amax_for<BF16T>(p, shifted, dev, stream);
}

cudaError_t launch_nvfp4_cast(const Nvfp4CastParams& p, int dtype, bool shifted,
                              const DeviceInfo& dev, cudaStream_t stream) {
  return dtype == 0 ? cast_for<F32T>(p, shifted, dev, stream) : cast_for<BF16T>(p, shifted, dev, stream);
}

cudaError_t launch_nvfp4_scales(const Nvfp4ScaleParams& p, const DeviceInfo& dev,
                                cudaStream_t stream) {
  int64_t work = 0;
  for (int k = 0; k < p.nseg; ++k) {
    const int64_t n = p.seg[k].nrows * p.seg[k].ncols;
    const int64_t items = p.seg[k].vec ? n / 4 : n;
    work = items > work ? items : work;
  }
  if (work == 0) return cudaSuccess;
  // at most one resident wave over the segments; each thread takes kScaleItems groups
  const int64_t per_seg = (int64_t(dev.sms) * kScaleBlocksPerSM + p.nseg - 1) / p.nseg;
  const int64_t want = (work + int64_t(kThreads) * kScaleItems - 1) / (int64_t(kThreads) * kScaleItems);
  const dim3 grid(unsigned(want < per_seg ? want : (per_seg < 1 ? 1 : per_seg)), unsigned(p.nseg));
  return launch_kernel(k_nvfp4_scales, grid, kThreads, 0, stream, p);
}

}  // namespace mxfp8
