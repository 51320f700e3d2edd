// Scale update and packed MAX reduction kernels.
//
// Scale update: "update scales for present directions" in the flow diagram of
// "Support row-only MXFP8 distributed master-weight casts"; the E8M0 byte is read
// off the amax exponent field (max(E - 8, 0), 0xFF for NaN/Inf), which is the
// scale convention e = floor(log2 amax) - 8 clamped to [-127, 127].
//
// Packed MAX reduction: the page's single packed-amax MAX all-reduce, with the
// ranks emulated as S slots of one device buffer: out[k] = max_s |slot_s[k]|; a NaN
// result is stored as the canonical quiet NaN.
// GEMM scale layout: the E8M0 grid (or its transpose) padded to 128 x 4 and cut into
// 128x4 tiles of 512 bytes in row-major tile order; inside a tile element (r, c) sits
// at (r % 32) * 16 + (r / 32) * 4 + c -- the layout block-scaled tensor-core GEMMs
// read their scale factors in.  One thread writes one 16-byte line of a tile (rows
// j, j+32, j+64, j+96 x 4 columns), so a tile leaves as 32 contiguous 16-byte stores.
// The kernels are streaming element-wise passes: 16-byte loads, grid-stride
// loops over a grid that is a multiple of the SM count.
#include "common.cuh"

namespace mxfp8 {
namespace {

constexpr int kThreads = 256;

// E8M0 bytes of four |amax| bit patterns at once, as e8m0_from_bits gives them one by one:
// the exponent fields gathered as bytes (byte 3 of bits << 1 for F32, byte 1 for BF16),
// then max(E - 8, 0) by a saturating byte subtract, and 0xFF where E is 0xFF (NaN / Inf).
template <class T>
__device__ __forceinline__ uint32_t e8m0x4(const uint32_t (&m)[4]) {
  constexpr uint32_t kSel = T::kBytes == 4 ? 0x0073u : 0x0051u;
  const uint32_t lo = __byte_perm(m[0] << 1, m[1] << 1, kSel);
  const uint32_t hi = __byte_perm(m[2] << 1, m[3] << 1, kSel);
  const uint32_t e = __byte_perm(lo, hi, 0x5410u);
  return __vsubus4(e, 0x08080808u) | __vcmpeq4(e, 0xffffffffu);
}

constexpr int kMaxSegments = 32;

struct ScaleBatch {
  int32_t nseg;
  ScaleSegment seg[kMaxSegments];
};

// blockIdx.y selects the segment; blocks stride over its entries.
template <class T>
__global__ void __launch_bounds__(kThreads) k_update_scales(const __grid_constant__ ScaleBatch b) {
  grid_dependency_sync();
  const ScaleSegment& s = b.seg[blockIdx.y];
  const int64_t n = s.nrows * s.ncols;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (s.vec) {
    for (int64_t q = tid; q < n / 4; q += stride) {
      uint32_t w[4];
      if constexpr (T::kBytes == 4) {
        const uint4 a = ld_stream16(static_cast<const uint32_t*>(s.amax) + 4 * q);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
      } else {
        const uint2 a = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(s.amax) + 4 * q);
        w[0] = a.x & 0xffffu; w[1] = a.x >> 16; w[2] = a.y & 0xffffu; w[3] = a.y >> 16;
      }
      reinterpret_cast<uint32_t*>(s.scale)[q] = e8m0x4<T>(w);
    }
  } else {
    for (int64_t e = tid; e < n; e += stride) {
      const int64_t r = e / s.ncols, c = e % s.ncols;
      s.scale[r * s.ld_s + c] =
          static_cast<uint8_t>(e8m0_from_bits<T>(load_bits<T>(s.amax, r * s.ld_a + c)));
    }
  }
}

// Fused packed MAX reduction + scale update over runs of grid entries.  Every run is cut
// into chunks of kChunk work items (an item is 4 entries of a dense run, else one entry);
// a block takes one chunk at a time, so the run -- its slots and pointers -- is the same
// for all of its threads, and each thread loads its kItems items of every contributing
// slot before it folds any of them, keeping two 16-byte loads in flight at full occupancy.  Chunks of
// all runs form one index space (prefix sums in the parameters), so large and small
// grids share the SMs evenly.
constexpr int kMaxReduceSegments = 64;
constexpr int kItems = 2;  // items per thread loaded together
// Rounds of kItems per thread and chunk: the chunk's set-up (finding its run, the run's
// pointers) is shared by kRounds rounds; 2 measured faster than 1 and 4 (config-5 reduction
// 14.4 / 12.9 / 14.1 us).
#ifndef MXFP8_REDUCE_ROUNDS
#define MXFP8_REDUCE_ROUNDS 2
#endif
constexpr int kRounds = MXFP8_REDUCE_ROUNDS;
constexpr int kChunk = kThreads * kItems * kRounds;
constexpr int kReduceBlocksPerSM = 8;  // 8 x 256 threads: every SM full, at most 32 registers

struct ReduceScaleBatch {
  int32_t nseg;
  int64_t chunk_prefix[kMaxReduceSegments + 1];  // chunks before run k
  ReduceScaleSegment seg[kMaxReduceSegments];
};

template <class T>
__device__ __forceinline__ void store_reduced(const ReduceScaleSegment& s, int64_t e, const uint32_t (&m)[4]) {
  if (s.vec) {
    if constexpr (T::kBytes == 4) {
      *reinterpret_cast<uint4*>(static_cast<uint32_t*>(s.reduced) + e) = make_uint4(m[0], m[1], m[2], m[3]);
    } else {
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(s.reduced) + e) =
          make_uint2(m[0] | (m[1] << 16), m[2] | (m[3] << 16));
    }
    *reinterpret_cast<uint32_t*>(s.scale + e) = e8m0x4<T>(m);  // dense: ld_s == ld_a == ncols
  } else {
    const int64_t r = e / s.ld_a, c = e % s.ld_a;
    store_bits<T>(s.reduced, e, m[0]);
    s.scale[r * s.ld_s + c] = static_cast<uint8_t>(e8m0_from_bits<T>(m[0]));
  }
}

template <class T>
__global__ void __launch_bounds__(kThreads, kReduceBlocksPerSM) k_reduce_update_scales(
    const __grid_constant__ ReduceScaleBatch b) {
  grid_dependency_sync();
  constexpr uint32_t kAbs = T::kBytes == 4 ? 0x7fffffffu : 0x7fffu;
  const int64_t chunks = b.chunk_prefix[b.nseg];
  for (int64_t c = blockIdx.x; c < chunks; c += gridDim.x) {
    int lo = 0, hi = b.nseg;  // chunk_prefix[lo] <= c < chunk_prefix[hi]; uniform in the block
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (b.chunk_prefix[mid] <= c) lo = mid; else hi = mid;
    }
    const ReduceScaleSegment& s = b.seg[lo];
    const int64_t items = s.vec ? (s.e1 - s.e0) / 4 : s.e1 - s.e0;
    const int step = s.vec ? 4 : 1;
#pragma unroll 1
    for (int round = 0; round < kRounds; ++round) {
    const int64_t first = (c - b.chunk_prefix[lo]) * kChunk + round * (kThreads * kItems) + threadIdx.x;
    int64_t e[kItems];
    bool live[kItems];
    uint32_t m[kItems][4];
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      const int64_t t = first + u * kThreads;
      e[u] = s.e0 + t * step;
      live[u] = t < items && (s.vec || e[u] % s.ld_a < s.ncols);  // skip padding columns
      m[u][0] = m[u][1] = m[u][2] = m[u][3] = 0u;
    }
    // the items of one slot (zeros for items past the run)
    auto load_slot = [&](int slot, uint32_t (&v)[kItems][4]) {
      const char* base = static_cast<const char*>(s.slot0) + slot * s.slot_stride * T::kBytes;
#pragma unroll
      for (int u = 0; u < kItems; ++u) {
        v[u][0] = v[u][1] = v[u][2] = v[u][3] = 0u;
        if (!live[u]) continue;
        const char* p = base + e[u] * T::kBytes;
        if (s.vec) {
          if constexpr (T::kBytes == 4) {
            const uint4 w = ld_stream16(p);
            v[u][0] = w.x; v[u][1] = w.y; v[u][2] = w.z; v[u][3] = w.w;
          } else {
            const uint2 w = *reinterpret_cast<const uint2*>(p);
            v[u][0] = w.x & 0xffffu; v[u][1] = w.x >> 16; v[u][2] = w.y & 0xffffu; v[u][3] = w.y >> 16;
          }
        } else {
          v[u][0] = load_bits<T>(p, 0);
        }
      }
    };
    // contributing slots, uniform in the block: the first one loads straight into m
    // (a run read by one slot -- every run of a single-rank reduction, most runs of a
    // ranged one -- then folds nothing), the others fold in
    uint64_t mask = s.slots;
    int next = 0;  // all_slots: the next slot
    auto next_slot = [&]() -> int {
      if (s.all_slots) return next < s.nslots ? next++ : -1;
      if (mask == 0) return -1;
      const int slot = __ffsll(static_cast<long long>(mask)) - 1;
      mask &= mask - 1;
      return slot;
    };
    int slot = next_slot();
    if (slot >= 0) {
      load_slot(slot, m);
#pragma unroll
      for (int u = 0; u < kItems; ++u)
#pragma unroll
        for (int q = 0; q < 4; ++q) m[u][q] &= kAbs;
      while ((slot = next_slot()) >= 0) {
        uint32_t v[kItems][4];
        load_slot(slot, v);
#pragma unroll
        for (int u = 0; u < kItems; ++u)
#pragma unroll
          for (int q = 0; q < 4; ++q) m[u][q] = max(m[u][q], v[u][q] & kAbs);
      }
    }
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      if (!live[u]) continue;
#pragma unroll
      for (int q = 0; q < 4; ++q) m[u][q] = canonical_nan<T>(m[u][q]);
      store_reduced<T>(s, e[u], m[u]);
    }
    }
  }
}

template <class T>
__global__ void __launch_bounds__(kThreads) k_max_reduce(const void* __restrict__ slots,
                                                         void* __restrict__ out, int64_t elems,
                                                         int nslots, int vec) {
  grid_dependency_sync();
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (vec) {
    const int64_t nchunk = elems / T::V;
    const char* base = static_cast<const char*>(slots);
    const int64_t slot_bytes = elems * T::kBytes;
    for (int64_t q = tid; q < nchunk; q += stride) {
      uint4 m = make_uint4(0u, 0u, 0u, 0u);
      for (int s = 0; s < nslots; ++s)
        m = chunk_max<T>(m, chunk_abs<T>(ld_stream16(base + s * slot_bytes + q * 16)));
      reinterpret_cast<uint4*>(out)[q] = canonical_nan_chunk<T>(m);
    }
  } else {
    for (int64_t e = tid; e < elems; e += stride) {
      uint32_t m = 0;
      for (int s = 0; s < nslots; ++s) {
        const uint32_t a = load_bits<T>(slots, s * elems + e) & (T::kBytes == 4 ? 0x7fffffffu : 0x7fffu);
        m = max(m, a);
      }
      store_bits<T>(out, e, canonical_nan<T>(m));
    }
  }
}

__global__ void __launch_bounds__(kThreads) k_swizzle_scales(const __grid_constant__ SwizzleParams p) {
  grid_dependency_sync();
  const int64_t tiles_c = p.pc / 4;
  const int64_t lines = (p.pr / 128) * tiles_c * 32;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t g = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; g < lines; g += stride) {
    const int64_t tile = g >> 5;
    const int j = int(g & 31);
    const int64_t r0 = (tile / tiles_c) * 128 + j, c0 = (tile % tiles_c) * 4;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t r = r0 + 32 * i;
      uint32_t word = 0;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int64_t c = c0 + cc;
        uint32_t v = 0;
        if (r < p.lr && c < p.lc) v = p.transpose ? p.s[c * p.ld + r] : p.s[r * p.ld + c];
        word |= v << (8 * cc);
      }
      w[i] = word;
    }
    uint8_t* dst = p.out + tile * 512 + j * 16;
    if (p.vec) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
#pragma unroll
      for (int b = 0; b < 16; ++b) dst[b] = static_cast<uint8_t>(w[b >> 2] >> (8 * (b & 3)));
    }
  }
}

unsigned grid_for(int64_t work_items, const DeviceInfo& dev) {
  const int64_t want = (work_items + kThreads - 1) / kThreads;
  const int64_t cap = int64_t(dev.sms) * 8;  // 8 x 256 threads resident per SM
  return unsigned(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

cudaError_t launch_update_scales(const ScaleSegment* segs, int nseg, int dtype,
                                 const DeviceInfo& dev, cudaStream_t stream) {
  for (int k0 = 0; k0 < nseg; k0 += kMaxSegments) {
    ScaleBatch b;
    b.nseg = nseg - k0 < kMaxSegments ? nseg - k0 : kMaxSegments;
    int64_t work = 0;
    for (int k = 0; k < b.nseg; ++k) {
      b.seg[k] = segs[k0 + k];
      const int64_t n = b.seg[k].nrows * b.seg[k].ncols;
      const int64_t items = b.seg[k].vec ? n / 4 : n;
      work = items > work ? items : work;
    }
    if (work == 0) continue;
    // spread the SM budget over the segments of this launch
    int64_t per_seg = (int64_t(dev.sms) * 8 + b.nseg - 1) / b.nseg;
    int64_t want = (work + kThreads - 1) / kThreads;
    const unsigned gx = unsigned(want < per_seg ? want : (per_seg < 1 ? 1 : per_seg));
    const dim3 grid(gx, unsigned(b.nseg));
    const cudaError_t e = dtype == 0 ? launch_kernel(k_update_scales<F32T>, grid, kThreads, 0, stream, b)
                                     : launch_kernel(k_update_scales<BF16T>, grid, kThreads, 0, stream, b);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_reduce_update_scales(const ReduceScaleSegment* segs, int nseg, int dtype,
                                       const DeviceInfo& dev, cudaStream_t stream) {
  for (int k0 = 0; k0 < nseg; k0 += kMaxReduceSegments) {
    ReduceScaleBatch b;
    b.nseg = nseg - k0 < kMaxReduceSegments ? nseg - k0 : kMaxReduceSegments;
    b.chunk_prefix[0] = 0;
    for (int k = 0; k < b.nseg; ++k) {
      b.seg[k] = segs[k0 + k];
      const int64_t n = b.seg[k].e1 - b.seg[k].e0;
      const int64_t items = b.seg[k].vec ? n / 4 : n;
      b.chunk_prefix[k + 1] = b.chunk_prefix[k] + (items + kChunk - 1) / kChunk;
    }
    const int64_t chunks = b.chunk_prefix[b.nseg];
    if (chunks == 0) continue;
    // one chunk per block: the block scheduler keeps every SM full and hands out the
    // small chunks dynamically (the loop covers anything past the grid limit)
    const unsigned grid = unsigned(chunks < 2147483647 ? chunks : 2147483647);
    const cudaError_t e = dtype == 0
                              ? launch_kernel(k_reduce_update_scales<F32T>, grid, kThreads, 0, stream, b)
                              : launch_kernel(k_reduce_update_scales<BF16T>, grid, kThreads, 0, stream, b);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_swizzle_scales(const SwizzleParams& p, const DeviceInfo& dev,
                                  cudaStream_t stream) {
  const int64_t lines = (p.pr / 128) * (p.pc / 4) * 32;
  if (lines == 0) return cudaSuccess;
  return launch_kernel(k_swizzle_scales, grid_for(lines, dev), kThreads, 0, stream, p);
}

cudaError_t launch_max_reduce(const void* slots, void* out, int64_t slot_elems, int num_slots,
                              int dtype, const DeviceInfo& dev, cudaStream_t stream) {
  if (slot_elems <= 0) return cudaSuccess;
  const int V = dtype == 0 ? F32T::V : BF16T::V;
  const int vec = (slot_elems % V == 0) && (reinterpret_cast<uintptr_t>(slots) % 16 == 0) &&
                  (reinterpret_cast<uintptr_t>(out) % 16 == 0);
  const unsigned grid = grid_for(vec ? slot_elems / V : slot_elems, dev);
  if (dtype == 0) return launch_kernel(k_max_reduce<F32T>, grid, kThreads, 0, stream, slots, out, slot_elems, num_slots, vec);
  return launch_kernel(k_max_reduce<BF16T>, grid, kThreads, 0, stream, slots, out, slot_elems, num_slots, vec);
}

}  // namespace mxfp8
