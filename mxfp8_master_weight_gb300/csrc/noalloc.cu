// Allocation-free sharded update of one weight.
//
// Callers such as a memory-pool allocator's own maintenance code, a process whose
// device memory is fully pre-reserved by a framework, or code running where a
// cudaMalloc would synchronise the device at a bad moment cannot allocate the
// per-rank amax slots and the reduced amax buffer that the partial amax -> MAX
// reduction -> scale update -> partial cast sequence needs.  This entry point keeps
// that working memory in one file-scope device array of fixed size instead, and
// otherwise runs exactly the library's public entry points.
#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

#include "kernels.h"
#include "mxfp8_partial.h"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;  // 64 MiB on every device that loads the library
constexpr int kMaxFragments = 64;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch for the current device, resolved once per device.
int scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return mxfp8::report_error(MXFP8_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return mxfp8::report_error(MXFP8_ERR_INVALID, "device index too large");
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || p == nullptr)
      return mxfp8::report_error(MXFP8_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MXFP8_OK;
}

bool empty(const mxfp8_tensor* t) {
  if (t == nullptr || t->data == nullptr) return true;
  if (t->ndim == 1) return t->shape[0] == 0;
  return t->shape[0] == 0 || t->shape[1] == 0;
}

int64_t numel_of(const mxfp8_tensor* t) {
  return t->ndim == 1 ? t->shape[0] : t->shape[0] * t->shape[1];
}

mxfp8_tensor view(void* base, int32_t dtype, int64_t r, int64_t c) {
  mxfp8_tensor t;
  t.data = base;
  t.dtype = dtype;
  t.ndim = 2;
  t.shape[0] = r;
  t.shape[1] = c;
  return t;
}

mxfp8_tensor none_tensor() {
  mxfp8_tensor t;
  t.data = nullptr;
  t.dtype = MXFP8_DTYPE_U8;
  t.ndim = 1;
  t.shape[0] = 0;
  t.shape[1] = 0;
  return t;
}

}  // namespace

extern "C" int mxfp8_sharded_update_noalloc(const mxfp8_tensor* fragments,
                                            const int64_t* start_offsets, int32_t nfrags,
                                            mxfp8_tensor* scale_inv_rowwise,
                                            mxfp8_tensor* scale_inv_colwise,
                                            mxfp8_tensor* output_rowwise,
                                            mxfp8_tensor* output_colwise, int64_t rows,
                                            int64_t cols, void* stream) {
  // Everything is checked on the host before the first launch: a non-zero status
  // leaves every caller buffer as it was.
  if (nfrags < 1 || nfrags > kMaxFragments || fragments == nullptr || start_offsets == nullptr)
    return mxfp8::report_error(MXFP8_ERR_INVALID, "need 1 to 64 fragments and their start offsets");
  if (rows <= 0 || cols <= 0 || rows > (int64_t(1) << 40) / cols)
    return mxfp8::report_error(MXFP8_ERR_INVALID, "rows and cols must be positive and not too large");
  int32_t dtype = -1;
  for (int f = 0; f < nfrags; ++f) {
    if (empty(&fragments[f])) continue;
    if (fragments[f].dtype != MXFP8_DTYPE_F32 && fragments[f].dtype != MXFP8_DTYPE_BF16)
      return mxfp8::report_error(MXFP8_ERR_DTYPE, "fragments must be F32 or BF16");
    if (dtype >= 0 && fragments[f].dtype != dtype)
      return mxfp8::report_error(MXFP8_ERR_DTYPE, "all fragments must share one dtype");
    dtype = fragments[f].dtype;
  }
  if (dtype < 0) return MXFP8_OK;  // every fragment empty: nothing to do

  // every fragment's cast, validated as mxfp8_partial_cast_batched would (this covers
  // the fragments' extents, the scale grids and the outputs)
  const mxfp8_tensor none = none_tensor();
  mxfp8_cast_job cast_jobs[kMaxFragments];
  for (int f = 0; f < nfrags; ++f) {
    mxfp8_cast_job& j = cast_jobs[f];
    j.input = fragments[f];
    j.scale_inv_rowwise = scale_inv_rowwise ? *scale_inv_rowwise : none;
    j.scale_inv_colwise = scale_inv_colwise ? *scale_inv_colwise : none;
    j.output_rowwise = output_rowwise ? *output_rowwise : none;
    j.output_colwise = output_colwise ? *output_colwise : none;
    j.rows = rows;
    j.cols = cols;
    j.start_offset = start_offsets[f];
    j.out_offset = start_offsets[f];
    j.model_dtype = MXFP8_MODEL_BF16;
  }
  if (int rc = mxfp8::validate_cast_jobs(cast_jobs, nfrags)) return rc;

  // fragments may not overlap: two casts would race on the same output bytes
  int order[kMaxFragments];
  int live = 0;
  for (int f = 0; f < nfrags; ++f) {
    if (empty(&fragments[f])) continue;
    int k = live++;
    while (k > 0 && start_offsets[order[k - 1]] > start_offsets[f]) {
      order[k] = order[k - 1];
      --k;
    }
    order[k] = f;
  }
  for (int k = 0; k + 1 < live; ++k) {
    const int a = order[k], b = order[k + 1];
    if (start_offsets[a] + numel_of(&fragments[a]) > start_offsets[b]) {
      char msg[160];
      std::snprintf(msg, sizeof msg, "fragments %d and %d overlap", a, b);
      return mxfp8::report_error(MXFP8_ERR_INVALID, msg);
    }
  }

  const bool colwise = !empty(output_colwise);
  const int64_t eb = dtype == MXFP8_DTYPE_F32 ? 4 : 2;
  const int64_t nbr = (cols + 31) / 32, nbc = (rows + 31) / 32;
  const int64_t row_entries = rows * nbr, col_entries = colwise ? nbc * cols : 0;
  const int64_t slot_bytes = ((row_entries + col_entries) * eb + 255) / 256 * 256;
  const int64_t need = (int64_t(nfrags) + 1) * slot_bytes;
  if (need > int64_t(kScratchBytes)) {
    char msg[200];
    std::snprintf(msg, sizeof msg,
                  "needs %lld bytes of scratch (%d amax slots + the reduced amax), the static "
                  "scratch holds %lld",
                  (long long)need, nfrags, (long long)kScratchBytes);
    return mxfp8::report_error(MXFP8_ERR_SHAPE, msg);
  }
  void* base = nullptr;
  if (int rc = scratch_for_current_device(&base)) return rc;
  char* scratch = static_cast<char*>(base);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);

  // 1. every fragment's block maxima into its own zeroed slot
  cudaError_t e = cudaMemsetAsync(scratch, 0, size_t(nfrags) * size_t(slot_bytes), s);
  if (e != cudaSuccess) return mxfp8::report_error(MXFP8_ERR_CUDA, cudaGetErrorString(e));
  mxfp8_amax_job amax_jobs[kMaxFragments];
  for (int f = 0; f < nfrags; ++f) {
    char* slot = scratch + f * slot_bytes;
    mxfp8_amax_job& j = amax_jobs[f];
    j.input = fragments[f];
    j.amax_rowwise = view(slot, dtype, rows, nbr);
    j.amax_colwise = colwise ? view(slot + row_entries * eb, dtype, nbc, cols) : none_tensor();
    j.rows = rows;
    j.cols = cols;
    j.start_offset = start_offsets[f];
  }
  if (int rc = mxfp8_partial_amax_batched(amax_jobs, nfrags, stream)) return rc;

  // 2. the MAX reduction over the slots
  char* reduced = scratch + nfrags * slot_bytes;
  mxfp8_tensor slots = view(scratch, dtype, nfrags, slot_bytes / eb);
  mxfp8_tensor red = view(reduced, dtype, 1, slot_bytes / eb);
  if (int rc = mxfp8_amax_max_reduce(&slots, &red, stream)) return rc;

  // 3. scales of the present directions
  mxfp8_tensor red_r = view(reduced, dtype, rows, nbr);
  mxfp8_tensor red_c = colwise ? view(reduced + row_entries * eb, dtype, nbc, cols) : none_tensor();
  if (int rc = mxfp8_update_scales(&red_r, &red_c, scale_inv_rowwise, scale_inv_colwise, rows,
                                   cols, stream))
    return rc;

  // 4. every fragment's cast into the full-size outputs
  return mxfp8_partial_cast_batched(cast_jobs, nfrags, stream);
}
