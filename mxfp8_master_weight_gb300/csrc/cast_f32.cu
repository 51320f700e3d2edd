// Cast kernels for FP32 master values with word-aligned outputs (the templates live in
// cast_impl.cuh; one translation unit per input dtype and output alignment keeps the
// build parallel), and the launcher that picks among the four units.
#include "cast_impl.cuh"

namespace mxfp8 {

cudaError_t launch_partial_cast_f32(const CastParams* jobs, int n, bool shifted, int model,
                                    const DeviceInfo& dev, cudaStream_t stream) {
  return launch_for_dtype<F32T, true>(jobs, n, shifted, model, dev, stream);
}

cudaError_t launch_partial_cast(const CastParams* jobs, int n, int dtype, bool shifted, bool vec_out,
                                int model, const DeviceInfo& dev, cudaStream_t stream) {
  if (dtype == 0) {
    return vec_out ? launch_partial_cast_f32(jobs, n, shifted, model, dev, stream)
                   : launch_partial_cast_f32_unaligned(jobs, n, shifted, model, dev, stream);
  }
  return vec_out ? launch_partial_cast_bf16(jobs, n, shifted, model, dev, stream)
                 : launch_partial_cast_bf16_unaligned(jobs, n, shifted, model, dev, stream);
}

}  // namespace mxfp8
