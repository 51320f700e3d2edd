// Scale update and packed MAX reduction kernels.
//
// Scale update: "update scales for present directions" in the flow diagram of
// "Support row-only MXFP8 distributed master-weight casts"; the E8M0 byte is read
// off the amax exponent field (max(E - 8, 0), 0xFF for NaN/Inf), which is the
// scale convention e = floor(log2 amax) - 8 clamped to [-127, 127].
//
// Packed MAX reduction: the page's single packed-amax MAX all-reduce, with the
// ranks emulated as S slots of one device buffer: out[k] = max_s |slot_s[k]|.
// Both kernels are streaming element-wise passes: 16-byte loads, grid-stride
// loops over a grid that is a multiple of the SM count.
#include "common.cuh"

namespace mxfp8 {
namespace {

constexpr int kThreads = 256;

template <class T>
__global__ void __launch_bounds__(kThreads) k_update_scales(const __grid_constant__ ScaleSegment s0,
                                                            const __grid_constant__ ScaleSegment s1) {
  const ScaleSegment& s = blockIdx.y == 0 ? s0 : s1;
  const int64_t n = s.nrows * s.ncols;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (s.vec) {
    for (int64_t q = tid; q < n / 4; q += stride) {
      uint32_t b[4];
      if constexpr (T::kBytes == 4) {
        const uint4 a = *reinterpret_cast<const uint4*>(static_cast<const uint32_t*>(s.amax) + 4 * q);
        b[0] = a.x; b[1] = a.y; b[2] = a.z; b[3] = a.w;
      } else {
        const uint2 a = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(s.amax) + 4 * q);
        b[0] = a.x & 0xffffu; b[1] = a.x >> 16; b[2] = a.y & 0xffffu; b[3] = a.y >> 16;
      }
      uint32_t out = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) out |= e8m0_from_bits<T>(b[k]) << (8 * k);
      reinterpret_cast<uint32_t*>(s.scale)[q] = out;
    }
  } else {
    for (int64_t e = tid; e < n; e += stride) {
      const int64_t r = e / s.ncols, c = e % s.ncols;
      s.scale[r * s.ld_s + c] =
          static_cast<uint8_t>(e8m0_from_bits<T>(load_bits<T>(s.amax, r * s.ld_a + c)));
    }
  }
}

template <class T>
__global__ void __launch_bounds__(kThreads) k_max_reduce(const void* __restrict__ slots,
                                                         void* __restrict__ out, int64_t elems,
                                                         int nslots, int vec) {
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
      reinterpret_cast<uint4*>(out)[q] = m;
    }
  } else {
    for (int64_t e = tid; e < elems; e += stride) {
      uint32_t m = 0;
      for (int s = 0; s < nslots; ++s) {
        const uint32_t a = load_bits<T>(slots, s * elems + e) & (T::kBytes == 4 ? 0x7fffffffu : 0x7fffu);
        m = max(m, a);
      }
      store_bits<T>(out, e, m);
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
  if (nseg <= 0) return cudaSuccess;
  int64_t work = 0;
  for (int k = 0; k < nseg; ++k) {
    const int64_t n = segs[k].nrows * segs[k].ncols;
    const int64_t items = segs[k].vec ? n / 4 : n;
    work = items > work ? items : work;
  }
  if (work == 0) return cudaSuccess;
  const dim3 grid(grid_for(work, dev), unsigned(nseg));
  const ScaleSegment& s1 = nseg > 1 ? segs[1] : segs[0];
  if (dtype == 0) {
    k_update_scales<F32T><<<grid, kThreads, 0, stream>>>(segs[0], s1);
  } else {
    k_update_scales<BF16T><<<grid, kThreads, 0, stream>>>(segs[0], s1);
  }
  return cudaGetLastError();
}

cudaError_t launch_max_reduce(const void* slots, void* out, int64_t slot_elems, int num_slots,
                              int dtype, const DeviceInfo& dev, cudaStream_t stream) {
  if (slot_elems <= 0) return cudaSuccess;
  const int V = dtype == 0 ? F32T::V : BF16T::V;
  const int vec = (slot_elems % V == 0) && (reinterpret_cast<uintptr_t>(slots) % 16 == 0) &&
                  (reinterpret_cast<uintptr_t>(out) % 16 == 0);
  const unsigned grid = grid_for(vec ? slot_elems / V : slot_elems, dev);
  if (dtype == 0) {
    k_max_reduce<F32T><<<grid, kThreads, 0, stream>>>(slots, out, slot_elems, num_slots, vec);
  } else {
    k_max_reduce<BF16T><<<grid, kThreads, 0, stream>>>(slots, out, slot_elems, num_slots, vec);
  }
  return cudaGetLastError();
}

}  // namespace mxfp8
