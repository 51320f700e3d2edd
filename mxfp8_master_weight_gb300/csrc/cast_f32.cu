// cast kernels instantiated for FP32 master values (the templates live in
// cast_impl.cuh; one translation unit per input dtype keeps the build parallel).
#include "cast_impl.cuh"

namespace mxfp8 {

cudaError_t launch_partial_cast_f32(const CastParams* jobs, int n, bool shifted, bool vec_out, int model,
                       const DeviceInfo& dev, cudaStream_t stream) {
  return launch_for_dtype<F32T>(jobs, n, shifted, vec_out, model, dev, stream);
}

cudaError_t launch_partial_cast(const CastParams* jobs, int n, int dtype, bool shifted, bool vec_out,
                 int model, const DeviceInfo& dev, cudaStream_t stream) {
  return dtype == 0 ? launch_partial_cast_f32(jobs, n, shifted, vec_out, model, dev, stream)
                    : launch_partial_cast_bf16(jobs, n, shifted, vec_out, model, dev, stream);
}

}  // namespace mxfp8
