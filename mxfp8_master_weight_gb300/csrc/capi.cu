// C ABI of the partial MXFP8 cast (declared in include/mxfp8_partial.h):
// argument validation, fragment geometry and kernel dispatch.  No entry point
// allocates memory or synchronises; all work is enqueued on the caller's stream.
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <vector>

#include <cuda_runtime.h>

#include "kernels.h"
#include "mxfp8_partial.h"

namespace {

using mxfp8::AmaxParams;
using mxfp8::CastParams;
using mxfp8::DeviceInfo;
using mxfp8::FragGeom;
using mxfp8::FusedParams;
using mxfp8::ReduceScaleSegment;
using mxfp8::ScaleSegment;
using mxfp8::SwizzleParams;

thread_local char g_err[512] = {0};

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_err[0] = 0;
  return MXFP8_OK;
}

int64_t elem_bytes(int32_t dtype) {
  switch (dtype) {
    case MXFP8_DTYPE_F32: return 4;
    case MXFP8_DTYPE_BF16: return 2;
    case MXFP8_DTYPE_U8: return 1;
    default: return 0;
  }
}

int64_t numel(const mxfp8_tensor* t) {
  if (t->ndim == 1) return t->shape[0];
  return t->shape[0] * t->shape[1];
}

// Empty handle: absent pointer, NULL data, or a zero extent (section "Changes":
// omission is expressed by an empty tensor handle).
bool is_empty(const mxfp8_tensor* t) {
  if (t == nullptr || t->data == nullptr) return true;
  if (t->ndim == 1) return t->shape[0] == 0;
  return t->shape[0] == 0 || t->shape[1] == 0;
}

// Structural checks of a present tensor: ndim, non-negative shape, known dtype,
// element alignment.
int check_tensor(const mxfp8_tensor* t, const char* name) {
  if (t->ndim != 1 && t->ndim != 2) return fail(MXFP8_ERR_INVALID, "%s: ndim must be 1 or 2", name);
  if (t->shape[0] < 0 || (t->ndim == 2 && t->shape[1] < 0))
    return fail(MXFP8_ERR_INVALID, "%s: negative shape", name);
  if (t->ndim == 2 && t->shape[1] > 0 && t->shape[0] > INT64_MAX / t->shape[1])
    return fail(MXFP8_ERR_INVALID, "%s: shape overflows int64", name);
  const int64_t eb = elem_bytes(t->dtype);
  if (eb == 0) return fail(MXFP8_ERR_DTYPE, "%s: unknown dtype %d", name, int(t->dtype));
  if (reinterpret_cast<uintptr_t>(t->data) % uintptr_t(eb) != 0)
    return fail(MXFP8_ERR_INVALID, "%s: data pointer not aligned to its element size", name);
  return MXFP8_OK;
}

// A 2-D block grid tensor of at least [r][c] (padding allowed, row stride = shape[1]).
int check_grid(const mxfp8_tensor* t, const char* name, int64_t r, int64_t c, int32_t dtype) {
  if (int rc = check_tensor(t, name)) return rc;
  if (t->dtype != dtype) return fail(MXFP8_ERR_DTYPE, "%s: wrong dtype %d (want %d)", name, int(t->dtype), int(dtype));
  if (t->ndim != 2) return fail(MXFP8_ERR_SHAPE, "%s: must be 2-D", name);
  if (t->shape[0] < r || t->shape[1] < c)
    return fail(MXFP8_ERR_SHAPE, "%s: shape [%lld, %lld] smaller than block grid [%lld, %lld]", name,
                (long long)t->shape[0], (long long)t->shape[1], (long long)r, (long long)c);
  return MXFP8_OK;
}

// Weight size limits: byte offsets of every element stay far inside int64 and a band's
// warp-tile count, ceil(cols / tile width), fits the 32-bit count the kernels keep.
// Both are far above what one device can hold.
constexpr int64_t kMaxElems = int64_t(1) << 40;
constexpr int64_t kMaxCols = int64_t(1) << 37;

int check_size(int64_t rows, int64_t cols) {
  if (rows <= 0 || cols <= 0) return fail(MXFP8_ERR_INVALID, "rows and cols must be positive");
  if (cols > kMaxCols) return fail(MXFP8_ERR_INVALID, "cols exceeds 2^37");
  if (rows > kMaxElems / cols) return fail(MXFP8_ERR_INVALID, "rows*cols exceeds 2^40 elements");
  return MXFP8_OK;
}

int check_dims(int64_t rows, int64_t cols, int64_t start, int64_t len) {
  if (int rc = check_size(rows, cols)) return rc;
  if (start < 0) return fail(MXFP8_ERR_INVALID, "start_offset must be non-negative");
  if (len < 0 || start > rows * cols - len)
    return fail(MXFP8_ERR_INVALID, "fragment [%lld, %lld) exceeds rows*cols = %lld", (long long)start,
                (long long)(start + len), (long long)(rows * cols));
  return MXFP8_OK;
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];

int device_info(DeviceInfo* d) {
  cudaError_t e = cudaGetDevice(&d->device);
  if (e != cudaSuccess) return fail(MXFP8_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  int sms = d->device < kMaxDevices ? g_sms[d->device].load() : 0;
  if (sms == 0) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d->device);
    if (e != cudaSuccess) return fail(MXFP8_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    if (d->device < kMaxDevices) g_sms[d->device].store(sms);
  }
  d->sms = sms;
  return MXFP8_OK;
}

int cuda_status(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(MXFP8_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return ok();
}

// Fragment geometry and the warp tiles (32 rows x tw columns) that cover it.
FragGeom make_geom(int64_t rows, int64_t cols, int64_t start, int64_t len, int tw) {
  FragGeom g{};
  g.rows = rows;
  g.cols = cols;
  g.start = start;
  g.end = start + len;
  g.coltiles = int32_t((cols + tw - 1) / tw);
  if (len > 0) {
    g.rs = start / cols;
    g.cs = start % cols;
    g.re = (start + len - 1) / cols;
    g.ce = (start + len - 1) % cols;
    g.band0 = g.rs / 32;
    g.ntiles = (g.re / 32 - g.band0 + 1) * g.coltiles;
  }
  return g;
}

// Virtual base address of element 0 of the weight for a fragment pointer (may lie
// outside the allocation; only used for alignment arithmetic).
uintptr_t virtual_base(const void* frag, int64_t start, int64_t eb) {
  return reinterpret_cast<uintptr_t>(frag) - uintptr_t(start * eb);
}

// ---------------------------------------------------------------- per-job preparation
// Each prep_* validates one job exactly as the single-fragment entry point documents
// and fills the kernel parameters.  *skip is set for an empty fragment.

int prep_amax(const mxfp8_amax_job& job, AmaxParams* p, int* dtype, bool* colwise, bool* skip) {
  const mxfp8_tensor* input = &job.input;
  *skip = false;
  const bool in_empty = is_empty(input);
  if (!in_empty) {
    if (int rc = check_tensor(input, "input")) return rc;
  }
  const int64_t len = in_empty ? 0 : numel(input);
  if (int rc = check_dims(job.rows, job.cols, job.start_offset, len)) return rc;
  if (len == 0) {
    *skip = true;
    return MXFP8_OK;
  }
  const int32_t dt = input->dtype;
  if (dt != MXFP8_DTYPE_F32 && dt != MXFP8_DTYPE_BF16)
    return fail(MXFP8_ERR_DTYPE, "input: dtype must be F32 or BF16");
  if (is_empty(&job.amax_rowwise)) return fail(MXFP8_ERR_MISSING, "amax_rowwise is required");
  const int64_t rows = job.rows, cols = job.cols;
  const int64_t nbr = (cols + 31) / 32, nbc = (rows + 31) / 32;
  if (int rc = check_grid(&job.amax_rowwise, "amax_rowwise", rows, nbr, dt)) return rc;
  *colwise = !is_empty(&job.amax_colwise);
  if (*colwise) {
    if (int rc = check_grid(&job.amax_colwise, "amax_colwise", nbc, cols, dt)) return rc;
  }
  const int64_t eb = elem_bytes(dt);
  const int V = int(16 / eb);
  *p = AmaxParams{};
  p->g = make_geom(rows, cols, job.start_offset, len, mxfp8::tile_width_for(dt));
  p->g.fast_ok = cols % V == 0;
  p->g.shift = int32_t(virtual_base(input->data, job.start_offset, eb) % 16);
  p->in = input->data;
  p->amax_r = job.amax_rowwise.data;
  p->ld_r = job.amax_rowwise.shape[1];
  if (*colwise) {
    p->amax_c = job.amax_colwise.data;
    p->ld_c = job.amax_colwise.shape[1];
    p->vec_c = (reinterpret_cast<uintptr_t>(p->amax_c) % 16 == 0) && (p->ld_c % V == 0);
  }
  *dtype = dt == MXFP8_DTYPE_F32 ? 0 : 1;
  return MXFP8_OK;
}

int prep_cast(const mxfp8_cast_job& job, CastParams* p, int* dtype, bool* colwise, bool* skip) {
  const mxfp8_tensor* input = &job.input;
  *skip = false;
  const bool in_empty = is_empty(input);
  if (!in_empty) {
    if (int rc = check_tensor(input, "input")) return rc;
  }
  const int64_t len = in_empty ? 0 : numel(input);
  if (int rc = check_dims(job.rows, job.cols, job.start_offset, len)) return rc;
  if (job.out_offset < 0) return fail(MXFP8_ERR_INVALID, "out_offset must be non-negative");
  if (len == 0) {
    *skip = true;
    return MXFP8_OK;
  }
  const int32_t dt = input->dtype;
  if (dt != MXFP8_DTYPE_F32 && dt != MXFP8_DTYPE_BF16)
    return fail(MXFP8_ERR_DTYPE, "input: dtype must be F32 or BF16");
  if (job.model_dtype != MXFP8_MODEL_BF16 && job.model_dtype != MXFP8_MODEL_F16)
    return fail(MXFP8_ERR_INVALID, "model_dtype must be MXFP8_MODEL_BF16 or MXFP8_MODEL_F16");
  if (is_empty(&job.scale_inv_rowwise)) return fail(MXFP8_ERR_MISSING, "scale_inv_rowwise is required");
  if (is_empty(&job.output_rowwise)) return fail(MXFP8_ERR_MISSING, "output_rowwise is required");
  const int64_t rows = job.rows, cols = job.cols, out_offset = job.out_offset;
  const int64_t nbr = (cols + 31) / 32, nbc = (rows + 31) / 32;
  if (int rc = check_grid(&job.scale_inv_rowwise, "scale_inv_rowwise", rows, nbr, MXFP8_DTYPE_U8)) return rc;
  const mxfp8_tensor* out_r = &job.output_rowwise;
  if (int rc = check_tensor(out_r, "output_rowwise")) return rc;
  if (out_r->dtype != MXFP8_DTYPE_U8) return fail(MXFP8_ERR_DTYPE, "output_rowwise: dtype must be U8");
  if (numel(out_r) - len < out_offset)
    return fail(MXFP8_ERR_SHAPE, "output_rowwise holds %lld bytes, needs out_offset + len = %lld",
                (long long)numel(out_r), (long long)(out_offset + len));
  *colwise = !is_empty(&job.output_colwise);
  const mxfp8_tensor* out_c = &job.output_colwise;
  if (*colwise) {
    if (int rc = check_tensor(out_c, "output_colwise")) return rc;
    if (out_c->dtype != MXFP8_DTYPE_U8) return fail(MXFP8_ERR_DTYPE, "output_colwise: dtype must be U8");
    if (numel(out_c) - len < out_offset)
      return fail(MXFP8_ERR_SHAPE, "output_colwise holds %lld bytes, needs out_offset + len = %lld",
                  (long long)numel(out_c), (long long)(out_offset + len));
    if (is_empty(&job.scale_inv_colwise))
      return fail(MXFP8_ERR_MISSING, "scale_inv_colwise is required when output_colwise is present");
    if (int rc = check_grid(&job.scale_inv_colwise, "scale_inv_colwise", nbc, cols, MXFP8_DTYPE_U8)) return rc;
  }
  const int64_t eb = elem_bytes(dt);
  const int V = int(16 / eb);
  const int64_t shift = out_offset - job.start_offset;
  *p = CastParams{};
  p->g = make_geom(rows, cols, job.start_offset, len, mxfp8::tile_width_for(dt));
  p->g.fast_ok = cols % V == 0;
  p->g.shift = int32_t(virtual_base(input->data, job.start_offset, eb) % 16);
  p->in = input->data;
  p->s_r = static_cast<const uint8_t*>(job.scale_inv_rowwise.data);
  p->ld_sr = job.scale_inv_rowwise.shape[1];
  p->out_r = static_cast<uint8_t*>(out_r->data);
  p->out_shift = shift;
  bool vec_out = (reinterpret_cast<uintptr_t>(p->out_r) + uintptr_t(shift)) % uintptr_t(V) == 0;
  if (*colwise) {
    p->s_c = static_cast<const uint8_t*>(job.scale_inv_colwise.data);
    p->ld_sc = job.scale_inv_colwise.shape[1];
    p->out_c = static_cast<uint8_t*>(out_c->data);
    vec_out = vec_out && ((reinterpret_cast<uintptr_t>(p->out_c) + uintptr_t(shift)) % uintptr_t(V) == 0);
    p->vec_sc = (reinterpret_cast<uintptr_t>(p->s_c) % uintptr_t(V) == 0) && (p->ld_sc % V == 0);
  }
  p->vec_out = vec_out;
  *dtype = dt == MXFP8_DTYPE_F32 ? 0 : 1;
  return MXFP8_OK;
}

int prep_fused(const mxfp8_quantize_job& job, FusedParams* p, int* dtype, bool* colwise,
               bool* skip) {
  // the data side is validated exactly as a partial cast
  const mxfp8_cast_job cj = {job.input, job.scale_inv_rowwise, job.scale_inv_colwise,
                             job.output_rowwise, job.output_colwise, job.rows, job.cols,
                             job.start_offset, job.out_offset, job.model_dtype};
  CastParams c;
  if (int rc = prep_cast(cj, &c, dtype, colwise, skip)) return rc;
  if (*skip) return MXFP8_OK;
  const int64_t rows = job.rows, cols = job.cols;
  const int64_t start = job.start_offset, end = start + numel(&job.input);
  if ((start % cols) % 32 != 0 || (end % cols) % 32 != 0)
    return fail(MXFP8_ERR_INVALID,
                "fragment [%lld, %lld) cuts a 1x32 block: use partial amax, MAX reduction, scale "
                "update and partial cast", (long long)start, (long long)end);
  if (*colwise && (start % (32 * cols) != 0 || (end % (32 * cols) != 0 && end != rows * cols)))
    return fail(MXFP8_ERR_INVALID,
                "fragment [%lld, %lld) cuts a 32x1 block: use partial amax, MAX reduction, scale "
                "update and partial cast", (long long)start, (long long)end);
  const int32_t dt = job.input.dtype;
  const int64_t nbr = (cols + 31) / 32, nbc = (rows + 31) / 32;
  const int V = int(16 / elem_bytes(dt));
  *p = FusedParams{};
  p->g = c.g;
  p->in = c.in;
  p->s_r = static_cast<uint8_t*>(job.scale_inv_rowwise.data);
  p->ld_sr = c.ld_sr;
  p->out_r = c.out_r;
  p->out_shift = c.out_shift;
  p->vec_out = c.vec_out;
  if (!is_empty(&job.amax_rowwise)) {
    if (int rc = check_grid(&job.amax_rowwise, "amax_rowwise", rows, nbr, dt)) return rc;
    p->amax_r = job.amax_rowwise.data;
    p->ld_r = job.amax_rowwise.shape[1];
  }
  if (*colwise) {
    p->s_c = static_cast<uint8_t*>(job.scale_inv_colwise.data);
    p->ld_sc = c.ld_sc;
    p->out_c = c.out_c;
    p->vec_sc = c.vec_sc;
    if (!is_empty(&job.amax_colwise)) {
      if (int rc = check_grid(&job.amax_colwise, "amax_colwise", nbc, cols, dt)) return rc;
      p->amax_c = job.amax_colwise.data;
      p->ld_c = job.amax_colwise.shape[1];
      p->vec_c = (reinterpret_cast<uintptr_t>(p->amax_c) % 16 == 0) && (p->ld_c % V == 0);
    }
  }
  return MXFP8_OK;
}

int prep_scales(const mxfp8_scale_job& job, ScaleSegment* segs, int* nseg, int* dtype) {
  const int64_t rows = job.rows, cols = job.cols;
  if (int rc = check_size(rows, cols)) return rc;
  if (is_empty(&job.amax_rowwise)) return fail(MXFP8_ERR_MISSING, "amax_rowwise is required");
  if (is_empty(&job.scale_inv_rowwise)) return fail(MXFP8_ERR_MISSING, "scale_inv_rowwise is required");
  const int32_t dt = job.amax_rowwise.dtype;
  if (dt != MXFP8_DTYPE_F32 && dt != MXFP8_DTYPE_BF16)
    return fail(MXFP8_ERR_DTYPE, "amax_rowwise: dtype must be F32 or BF16");
  const int64_t nbr = (cols + 31) / 32, nbc = (rows + 31) / 32;
  if (int rc = check_grid(&job.amax_rowwise, "amax_rowwise", rows, nbr, dt)) return rc;
  if (int rc = check_grid(&job.scale_inv_rowwise, "scale_inv_rowwise", rows, nbr, MXFP8_DTYPE_U8)) return rc;
  const bool colwise = !is_empty(&job.amax_colwise);
  if (colwise) {
    if (int rc = check_grid(&job.amax_colwise, "amax_colwise", nbc, cols, dt)) return rc;
    if (is_empty(&job.scale_inv_colwise))
      return fail(MXFP8_ERR_MISSING, "scale_inv_colwise is required when amax_colwise is present");
    if (int rc = check_grid(&job.scale_inv_colwise, "scale_inv_colwise", nbc, cols, MXFP8_DTYPE_U8)) return rc;
  }
  const int64_t eb = elem_bytes(dt);
  auto seg = [&](const mxfp8_tensor* a, const mxfp8_tensor* sc, int64_t nr, int64_t nc) {
    ScaleSegment g{};
    g.amax = a->data;
    g.scale = static_cast<uint8_t*>(sc->data);
    g.nrows = nr;
    g.ncols = nc;
    g.ld_a = a->shape[1];
    g.ld_s = sc->shape[1];
    g.vec = (g.ld_a == nc) && (g.ld_s == nc) && ((nr * nc) % 4 == 0) &&
            (reinterpret_cast<uintptr_t>(g.amax) % uintptr_t(4 * eb) == 0) &&
            (reinterpret_cast<uintptr_t>(g.scale) % 4 == 0);
    return g;
  };
  *nseg = 0;
  segs[(*nseg)++] = seg(&job.amax_rowwise, &job.scale_inv_rowwise, rows, nbr);
  if (colwise) segs[(*nseg)++] = seg(&job.amax_colwise, &job.scale_inv_colwise, nbc, cols);
  *dtype = dt == MXFP8_DTYPE_F32 ? 0 : 1;
  return MXFP8_OK;
}

// Prefix the last error message with the failing job's index.
int job_fail(int rc, int k) {
  char tmp[sizeof g_err];
  std::snprintf(tmp, sizeof tmp, "job %d: %.480s", k, g_err);
  std::snprintf(g_err, sizeof g_err, "%s", tmp);
  return rc;
}

constexpr int kGroupChunk = mxfp8::kMaxBatchJobs;
constexpr int kWindow = 64;  // jobs prepared at a time (host stack, no heap)

// ---------------------------------------------------------------- batched drivers
// Validate every job first (a failure launches nothing), then, window by window,
// launch one kernel per (dtype, direction set, alignment class) group, at most
// kMaxBatchJobs jobs per launch.

int run_amax(const mxfp8_amax_job* jobs, int32_t njobs, void* stream) {
  if (njobs < 0 || (njobs > 0 && jobs == nullptr)) return fail(MXFP8_ERR_INVALID, "bad job array");
  AmaxParams win[kWindow];
  int key[kWindow];
  int dt;
  bool col, skip;
  int live = 0;
  for (int k = 0; k < njobs; ++k) {
    if (int rc = prep_amax(jobs[k], &win[0], &dt, &col, &skip)) return njobs > 1 ? job_fail(rc, k) : rc;
    live += !skip;
  }
  if (live == 0) return ok();
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  AmaxParams batch[kGroupChunk];
  for (int base = 0; base < njobs; base += kWindow) {
    const int m = njobs - base < kWindow ? njobs - base : kWindow;
    // aligned and realigning fragments of one dtype share a launch (the realigning
    // kernel takes aligned tiles too): one grid tail per dtype instead of two
    bool any_shift[2] = {false, false};
    for (int i = 0; i < m; ++i) {
      prep_amax(jobs[base + i], &win[i], &dt, &col, &skip);
      key[i] = skip ? -1 : dt * 2;
      if (!skip && win[i].g.shift != 0) any_shift[dt] = true;
    }
    for (int i = 0; i < m; ++i)
      if (key[i] >= 0 && any_shift[key[i] >> 1]) key[i] += 1;
    for (int kk = 0; kk < 4; ++kk) {  // dtype x shifted (direction sets may mix)
      int n = 0;
      for (int i = 0; i <= m; ++i) {
        if (i < m && key[i] == kk) batch[n++] = win[i];
        if (n > 0 && (n == kGroupChunk || i == m)) {
          if (int rc = cuda_status(mxfp8::launch_partial_amax(batch, n, kk >> 1, kk & 1, dev,
                                                              static_cast<cudaStream_t>(stream)),
                                   "partial amax launch"))
            return rc;
          n = 0;
        }
      }
    }
  }
  return ok();
}

int run_cast(const mxfp8_cast_job* jobs, int32_t njobs, void* stream) {
  if (njobs < 0 || (njobs > 0 && jobs == nullptr)) return fail(MXFP8_ERR_INVALID, "bad job array");
  CastParams win[kWindow];
  int key[kWindow];
  int dt;
  bool col, skip;
  int live = 0;
  for (int k = 0; k < njobs; ++k) {
    if (int rc = prep_cast(jobs[k], &win[0], &dt, &col, &skip)) return njobs > 1 ? job_fail(rc, k) : rc;
    live += !skip;
  }
  if (live == 0) return ok();
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  CastParams batch[kGroupChunk];
  for (int base = 0; base < njobs; base += kWindow) {
    const int m = njobs - base < kWindow ? njobs - base : kWindow;
    // as for the amax: aligned and realigning fragments of one model, dtype and output
    // alignment share a launch
    bool any_shift[16] = {};
    for (int i = 0; i < m; ++i) {
      prep_cast(jobs[base + i], &win[i], &dt, &col, &skip);
      key[i] = skip ? -1 : jobs[base + i].model_dtype * 8 + dt * 4 + (win[i].vec_out != 0);
      if (!skip && win[i].g.shift != 0) any_shift[key[i]] = true;
    }
    for (int i = 0; i < m; ++i)
      if (key[i] >= 0 && any_shift[key[i]]) key[i] += 2;
    for (int kk = 0; kk < 16; ++kk) {  // model x dtype x shifted x aligned output
      int n = 0;
      for (int i = 0; i <= m; ++i) {
        if (i < m && key[i] == kk) batch[n++] = win[i];
        if (n > 0 && (n == kGroupChunk || i == m)) {
          if (int rc = cuda_status(mxfp8::launch_partial_cast(batch, n, (kk >> 2) & 1, (kk >> 1) & 1,
                                                              kk & 1, kk >> 3, dev,
                                                              static_cast<cudaStream_t>(stream)),
                                   "partial cast launch"))
            return rc;
          n = 0;
        }
      }
    }
  }
  return ok();
}

int run_scales(const mxfp8_scale_job* jobs, int32_t njobs, void* stream) {
  if (njobs < 0 || (njobs > 0 && jobs == nullptr)) return fail(MXFP8_ERR_INVALID, "bad job array");
  ScaleSegment segs[2];
  int nseg, dt;
  for (int k = 0; k < njobs; ++k) {
    if (int rc = prep_scales(jobs[k], segs, &nseg, &dt)) return njobs > 1 ? job_fail(rc, k) : rc;
  }
  if (njobs == 0) return ok();
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  ScaleSegment batch[2 * kGroupChunk];
  for (int kdt = 0; kdt < 2; ++kdt) {
    int n = 0;
    for (int k = 0; k <= njobs; ++k) {
      if (k < njobs) {
        prep_scales(jobs[k], segs, &nseg, &dt);
        if (dt == kdt)
          for (int q = 0; q < nseg; ++q) batch[n++] = segs[q];
      }
      if (n > 0 && (n > 2 * kGroupChunk - 2 || k == njobs)) {
        if (int rc = cuda_status(mxfp8::launch_update_scales(batch, n, kdt, dev,
                                                             static_cast<cudaStream_t>(stream)),
                                 "update scales launch"))
          return rc;
        n = 0;
      }
    }
  }
  return ok();
}

int run_fused(const mxfp8_quantize_job* jobs, int32_t njobs, void* stream) {
  if (njobs < 0 || (njobs > 0 && jobs == nullptr)) return fail(MXFP8_ERR_INVALID, "bad job array");
  FusedParams win[kWindow];
  int key[kWindow];
  int dt;
  bool col, skip;
  int live = 0;
  for (int k = 0; k < njobs; ++k) {
    if (int rc = prep_fused(jobs[k], &win[0], &dt, &col, &skip)) return njobs > 1 ? job_fail(rc, k) : rc;
    live += !skip;
  }
  if (live == 0) return ok();
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  FusedParams batch[kGroupChunk];
  for (int base = 0; base < njobs; base += kWindow) {
    const int m = njobs - base < kWindow ? njobs - base : kWindow;
    for (int i = 0; i < m; ++i) {
      prep_fused(jobs[base + i], &win[i], &dt, &col, &skip);
      key[i] = skip ? -1 : jobs[base + i].model_dtype * 8 + dt * 4 + (win[i].g.shift != 0) * 2 +
                               (win[i].vec_out != 0);
    }
    for (int kk = 0; kk < 16; ++kk) {  // model x dtype x shifted x aligned output
      int n = 0;
      for (int i = 0; i <= m; ++i) {
        if (i < m && key[i] == kk) batch[n++] = win[i];
        if (n > 0 && (n == kGroupChunk || i == m)) {
          if (int rc = cuda_status(mxfp8::launch_fused_quantize(batch, n, (kk >> 2) & 1, (kk >> 1) & 1,
                                                                kk & 1, kk >> 3, dev,
                                                                static_cast<cudaStream_t>(stream)),
                                   "fused quantize launch"))
            return rc;
          n = 0;
        }
      }
    }
  }
  return ok();
}

const mxfp8_tensor kEmpty = {nullptr, MXFP8_DTYPE_U8, 1, {0, 0}};

const mxfp8_tensor& or_empty(const mxfp8_tensor* t) { return t ? *t : kEmpty; }

}  // namespace

namespace mxfp8 {
int report_error(int code, const char* msg) { return fail(code, "%s", msg); }

int validate_cast_jobs(const mxfp8_cast_job* jobs, int njobs) {
  CastParams p;
  int dt;
  bool col, skip;
  for (int k = 0; k < njobs; ++k) {
    if (int rc = prep_cast(jobs[k], &p, &dt, &col, &skip)) return njobs > 1 ? job_fail(rc, k) : rc;
  }
  return MXFP8_OK;
}
}  // namespace mxfp8

extern "C" {

const char* mxfp8_last_error(void) { return g_err; }

int mxfp8_version(void) { return 200; }

int mxfp8_partial_amax(const mxfp8_tensor* input, mxfp8_tensor* amax_rowwise,
                       mxfp8_tensor* amax_colwise, int64_t rows, int64_t cols,
                       int64_t start_offset, void* stream) {
  const mxfp8_amax_job job = {or_empty(input), or_empty(amax_rowwise), or_empty(amax_colwise),
                              rows, cols, start_offset};
  return run_amax(&job, 1, stream);
}

int mxfp8_partial_amax_batched(const mxfp8_amax_job* jobs, int32_t njobs, void* stream) {
  return run_amax(jobs, njobs, stream);
}

int mxfp8_amax_max_reduce(const mxfp8_tensor* slots, mxfp8_tensor* out, void* stream) {
  if (is_empty(out)) return fail(MXFP8_ERR_MISSING, "out is required");
  if (int rc = check_tensor(out, "out")) return rc;
  if (is_empty(slots)) return fail(MXFP8_ERR_MISSING, "slots is required");
  if (int rc = check_tensor(slots, "slots")) return rc;
  if (slots->ndim != 2) return fail(MXFP8_ERR_SHAPE, "slots must be 2-D [S][E]");
  const int32_t dt = slots->dtype;
  if (dt != MXFP8_DTYPE_F32 && dt != MXFP8_DTYPE_BF16)
    return fail(MXFP8_ERR_DTYPE, "slots: dtype must be F32 or BF16");
  if (out->dtype != dt) return fail(MXFP8_ERR_DTYPE, "out: dtype must equal the slots dtype");
  const int64_t S = slots->shape[0], E = slots->shape[1];
  if (numel(out) != E) return fail(MXFP8_ERR_SHAPE, "out numel %lld != slot size %lld", (long long)numel(out), (long long)E);
  if (S > INT32_MAX) return fail(MXFP8_ERR_INVALID, "too many slots");
  const int64_t eb = elem_bytes(dt);
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(slots->data), o0 = reinterpret_cast<uintptr_t>(out->data);
  if (o0 < s0 + uintptr_t(S * E * eb) && s0 < o0 + uintptr_t(E * eb))
    return fail(MXFP8_ERR_INVALID, "out overlaps slots");
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  return cuda_status(mxfp8::launch_max_reduce(slots->data, out->data, E, int(S),
                                              dt == MXFP8_DTYPE_F32 ? 0 : 1, dev,
                                              static_cast<cudaStream_t>(stream)),
                     "max reduce launch");
}

int mxfp8_amax_max_reduce_update_scales_ranged(const mxfp8_tensor* slots, mxfp8_tensor* reduced,
                                               const mxfp8_scale_job* jobs, int32_t njobs,
                                               const int64_t* slot_ranges, int32_t nranges,
                                               void* stream) {
  if (is_empty(reduced)) return fail(MXFP8_ERR_MISSING, "reduced is required");
  if (int rc = check_tensor(reduced, "reduced")) return rc;
  if (is_empty(slots)) return fail(MXFP8_ERR_MISSING, "slots is required");
  if (int rc = check_tensor(slots, "slots")) return rc;
  if (slots->ndim != 2) return fail(MXFP8_ERR_SHAPE, "slots must be 2-D [S][P]");
  const int32_t dt = slots->dtype;
  if (dt != MXFP8_DTYPE_F32 && dt != MXFP8_DTYPE_BF16)
    return fail(MXFP8_ERR_DTYPE, "slots: dtype must be F32 or BF16");
  if (reduced->dtype != dt) return fail(MXFP8_ERR_DTYPE, "reduced: dtype must equal the slots dtype");
  const int64_t S = slots->shape[0], P = slots->shape[1];
  if (numel(reduced) != P)
    return fail(MXFP8_ERR_SHAPE, "reduced numel %lld != slot size %lld", (long long)numel(reduced), (long long)P);
  if (S > 1024) return fail(MXFP8_ERR_INVALID, "too many slots");
  const bool ranged = nranges > 0;
  if (nranges < 0 || (ranged && slot_ranges == nullptr))
    return fail(MXFP8_ERR_INVALID, "bad slot range array");
  if (ranged && S > 64) return fail(MXFP8_ERR_INVALID, "slot ranges need at most 64 slots");
  for (int32_t q = 0; q < nranges; ++q) {
    const int64_t sl = slot_ranges[3 * q], lo = slot_ranges[3 * q + 1], hi = slot_ranges[3 * q + 2];
    if (sl < 0 || sl >= S || lo < 0 || lo > hi || hi > P)
      return fail(MXFP8_ERR_INVALID, "slot range %d: (%lld, %lld, %lld) is not a slot and an entry range "
                  "inside [0, %lld)", int(q), (long long)sl, (long long)lo, (long long)hi, (long long)P);
  }
  const int64_t eb = elem_bytes(dt);
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(slots->data), r0 = reinterpret_cast<uintptr_t>(reduced->data);
  if (r0 < s0 + uintptr_t(S * P * eb) && s0 < r0 + uintptr_t(P * eb))
    return fail(MXFP8_ERR_INVALID, "reduced overlaps slots");
  if (njobs < 0 || (njobs > 0 && jobs == nullptr)) return fail(MXFP8_ERR_INVALID, "bad job array");
  ScaleSegment segs[2];
  int nseg, jdt;
  // validate every job and that each amax view lies inside `reduced`
  auto inside = [&](const ScaleSegment& g, int64_t* begin) {
    const intptr_t d = reinterpret_cast<intptr_t>(g.amax) - intptr_t(r0);
    if (d < 0 || d % eb != 0) return false;
    *begin = d / eb;
    return *begin + (g.nrows - 1) * g.ld_a + g.ncols <= P;
  };
  for (int k = 0; k < njobs; ++k) {
    if (int rc = prep_scales(jobs[k], segs, &nseg, &jdt)) return njobs > 1 ? job_fail(rc, k) : rc;
    if (jdt != (dt == MXFP8_DTYPE_F32 ? 0 : 1)) return job_fail(fail(MXFP8_ERR_DTYPE, "amax dtype differs from the slots"), k);
    for (int q = 0; q < nseg; ++q) {
      int64_t b = 0;
      if (!inside(segs[q], &b)) return job_fail(fail(MXFP8_ERR_INVALID, "amax view is not inside `reduced`"), k);
    }
  }
  if (njobs == 0) return ok();
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  // Every grid is cut into runs of entries with one set of contributing slots: the
  // breakpoints are the grid's ends and every slot range end inside it.
  std::vector<ReduceScaleSegment> runs;
  std::vector<int64_t> cuts;
  for (int k = 0; k < njobs; ++k) {
    prep_scales(jobs[k], segs, &nseg, &jdt);
    for (int q = 0; q < nseg; ++q) {
      int64_t b = 0;
      inside(segs[q], &b);  // validated above: the view lies inside `reduced`
      const ScaleSegment& g = segs[q];
      const int64_t span = (g.nrows - 1) * g.ld_a + g.ncols;  // linear entries of the view
      ReduceScaleSegment r{};
      r.slot0 = static_cast<const char*>(slots->data) + b * eb;
      r.slot_stride = P;
      r.nslots = int32_t(S);
      r.reduced = const_cast<void*>(g.amax);
      r.scale = g.scale;
      r.nrows = g.nrows;
      r.ncols = g.ncols;
      r.ld_a = g.ld_a;
      r.ld_s = g.ld_s;
      cuts.assign({0, span});
      for (int32_t i = 0; i < nranges; ++i) {
        for (int e = 1; e <= 2; ++e) {
          const int64_t c = slot_ranges[3 * i + e] - b;
          if (c > 0 && c < span) cuts.push_back(c);
        }
      }
      std::sort(cuts.begin(), cuts.end());
      cuts.erase(std::unique(cuts.begin(), cuts.end()), cuts.end());
      for (size_t i = 0; i + 1 < cuts.size(); ++i) {
        r.e0 = cuts[i];
        r.e1 = cuts[i + 1];
        r.all_slots = ranged ? 0 : 1;
        r.slots = 0;
        for (int32_t j = 0; j < nranges; ++j)
          if (slot_ranges[3 * j + 1] - b <= r.e0 && slot_ranges[3 * j + 2] - b >= r.e1)
            r.slots |= uint64_t(1) << slot_ranges[3 * j];
        if (!runs.empty() && runs.back().reduced == r.reduced && runs.back().e1 == r.e0 &&
            runs.back().slots == r.slots && runs.back().all_slots == r.all_slots) {
          runs.back().e1 = r.e1;  // same contributors: extend the previous run
        } else {
          runs.push_back(r);
        }
      }
    }
  }
  // A run of a dense, aligned grid takes 4 entries per work item from the first multiple
  // of 4 to the last: its ragged ends (a shard boundary falls anywhere) become runs of
  // single entries of their own.
  std::vector<ReduceScaleSegment> pieces;
  pieces.reserve(runs.size() * 3);
  for (const ReduceScaleSegment& r : runs) {
    const bool dense = r.ld_a == r.ncols && r.ld_s == r.ncols && (P % 4 == 0) &&
                       (reinterpret_cast<uintptr_t>(r.slot0) % uintptr_t(4 * eb) == 0) &&
                       (reinterpret_cast<uintptr_t>(r.reduced) % uintptr_t(4 * eb) == 0) &&
                       (reinterpret_cast<uintptr_t>(r.scale) % 4 == 0);
    const int64_t a = (r.e0 + 3) / 4 * 4, z = r.e1 / 4 * 4;
    if (!dense || a >= z) {
      pieces.push_back(r);
      pieces.back().vec = 0;
      continue;
    }
    ReduceScaleSegment q = r;
    q.vec = 0;
    if (r.e0 < a) {
      q.e0 = r.e0;
      q.e1 = a;
      pieces.push_back(q);
    }
    q.vec = 1;
    q.e0 = a;
    q.e1 = z;
    pieces.push_back(q);
    if (z < r.e1) {
      q.vec = 0;
      q.e0 = z;
      q.e1 = r.e1;
      pieces.push_back(q);
    }
  }
  return cuda_status(mxfp8::launch_reduce_update_scales(pieces.data(), int(pieces.size()),
                                                        dt == MXFP8_DTYPE_F32 ? 0 : 1, dev,
                                                        static_cast<cudaStream_t>(stream)),
                     "reduce and update scales launch");
}

int mxfp8_amax_max_reduce_update_scales(const mxfp8_tensor* slots, mxfp8_tensor* reduced,
                                        const mxfp8_scale_job* jobs, int32_t njobs,
                                        void* stream) {
  return mxfp8_amax_max_reduce_update_scales_ranged(slots, reduced, jobs, njobs, nullptr, 0, stream);
}

int mxfp8_update_scales(const mxfp8_tensor* amax_rowwise, const mxfp8_tensor* amax_colwise,
                        mxfp8_tensor* scale_inv_rowwise, mxfp8_tensor* scale_inv_colwise,
                        int64_t rows, int64_t cols, void* stream) {
  const mxfp8_scale_job job = {or_empty(amax_rowwise), or_empty(amax_colwise),
                               or_empty(scale_inv_rowwise), or_empty(scale_inv_colwise), rows, cols};
  return run_scales(&job, 1, stream);
}

int mxfp8_update_scales_batched(const mxfp8_scale_job* jobs, int32_t njobs, void* stream) {
  return run_scales(jobs, njobs, stream);
}

int mxfp8_partial_cast(const mxfp8_tensor* input, const mxfp8_tensor* scale_inv_rowwise,
                       const mxfp8_tensor* scale_inv_colwise, mxfp8_tensor* output_rowwise,
                       mxfp8_tensor* output_colwise, int64_t rows, int64_t cols,
                       int64_t start_offset, int64_t out_offset, void* stream) {
  const mxfp8_cast_job job = {or_empty(input), or_empty(scale_inv_rowwise),
                              or_empty(scale_inv_colwise), or_empty(output_rowwise),
                              or_empty(output_colwise), rows, cols, start_offset, out_offset,
                              MXFP8_MODEL_BF16};
  return run_cast(&job, 1, stream);
}

int mxfp8_partial_cast_batched(const mxfp8_cast_job* jobs, int32_t njobs, void* stream) {
  return run_cast(jobs, njobs, stream);
}

int mxfp8_quantize_whole_blocks(const mxfp8_tensor* input, mxfp8_tensor* amax_rowwise,
                                mxfp8_tensor* amax_colwise, mxfp8_tensor* scale_inv_rowwise,
                                mxfp8_tensor* scale_inv_colwise, mxfp8_tensor* output_rowwise,
                                mxfp8_tensor* output_colwise, int64_t rows, int64_t cols,
                                int64_t start_offset, int64_t out_offset, void* stream) {
  const mxfp8_quantize_job job = {or_empty(input), or_empty(amax_rowwise), or_empty(amax_colwise),
                                  or_empty(scale_inv_rowwise), or_empty(scale_inv_colwise),
                                  or_empty(output_rowwise), or_empty(output_colwise),
                                  rows, cols, start_offset, out_offset, MXFP8_MODEL_BF16};
  return run_fused(&job, 1, stream);
}

int mxfp8_quantize_whole_blocks_batched(const mxfp8_quantize_job* jobs, int32_t njobs,
                                        void* stream) {
  return run_fused(jobs, njobs, stream);
}

// ---------------------------------------------------------------- NVFP4
int nvfp4_partial_amax(const mxfp8_tensor* input, mxfp8_tensor* amax_rowwise,
                       mxfp8_tensor* amax_colwise, mxfp8_tensor* amax_tensor, int64_t rows,
                       int64_t cols, int64_t start_offset, void* stream) {
  const bool in_empty = is_empty(input);
  if (!in_empty) {
    if (int rc = check_tensor(input, "input")) return rc;
  }
  const int64_t len = in_empty ? 0 : numel(input);
  if (int rc = check_dims(rows, cols, start_offset, len)) return rc;
  if (len == 0) return ok();
  const int32_t dt = input->dtype;
  if (dt != MXFP8_DTYPE_F32 && dt != MXFP8_DTYPE_BF16)
    return fail(MXFP8_ERR_DTYPE, "input: dtype must be F32 or BF16");
  if (is_empty(amax_rowwise)) return fail(MXFP8_ERR_MISSING, "amax_rowwise is required");
  if (is_empty(amax_tensor)) return fail(MXFP8_ERR_MISSING, "amax_tensor is required");
  const int64_t nbr = (cols + 15) / 16, nbc = (rows + 15) / 16;
  if (int rc = check_grid(amax_rowwise, "amax_rowwise", rows, nbr, MXFP8_DTYPE_F32)) return rc;
  if (int rc = check_tensor(amax_tensor, "amax_tensor")) return rc;
  if (amax_tensor->dtype != MXFP8_DTYPE_F32) return fail(MXFP8_ERR_DTYPE, "amax_tensor: dtype must be F32");
  const bool colwise = !is_empty(amax_colwise);
  if (colwise) {
    if (int rc = check_grid(amax_colwise, "amax_colwise", nbc, cols, MXFP8_DTYPE_F32)) return rc;
  }
  const int64_t eb = elem_bytes(dt);
  const int V = int(16 / eb);
  mxfp8::Nvfp4AmaxParams p{};
  p.g = make_geom(rows, cols, start_offset, len, mxfp8::tile_width_for(dt));
  p.g.fast_ok = cols % V == 0;
  p.g.shift = int32_t(virtual_base(input->data, start_offset, eb) % 16);
  p.in = input->data;
  p.amax_r = static_cast<float*>(amax_rowwise->data);
  p.ld_r = amax_rowwise->shape[1];
  p.amax_t = static_cast<uint32_t*>(amax_tensor->data);
  if (colwise) {
    p.amax_c = static_cast<float*>(amax_colwise->data);
    p.ld_c = amax_colwise->shape[1];
    p.vec_c = (reinterpret_cast<uintptr_t>(p.amax_c) % 16 == 0) && (p.ld_c % 4 == 0);
  }
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  return cuda_status(mxfp8::launch_nvfp4_amax(p, dt == MXFP8_DTYPE_F32 ? 0 : 1, p.g.shift != 0, dev,
                                              static_cast<cudaStream_t>(stream)),
                     "nvfp4 partial amax launch");
}

int nvfp4_update_scales(const mxfp8_tensor* amax_rowwise, const mxfp8_tensor* amax_colwise,
                        const mxfp8_tensor* amax_tensor, mxfp8_tensor* scale_rowwise,
                        mxfp8_tensor* scale_colwise, int64_t rows, int64_t cols, void* stream) {
  if (int rc = check_size(rows, cols)) return rc;
  if (is_empty(amax_rowwise)) return fail(MXFP8_ERR_MISSING, "amax_rowwise is required");
  if (is_empty(amax_tensor)) return fail(MXFP8_ERR_MISSING, "amax_tensor is required");
  if (is_empty(scale_rowwise)) return fail(MXFP8_ERR_MISSING, "scale_rowwise is required");
  const int64_t nbr = (cols + 15) / 16, nbc = (rows + 15) / 16;
  if (int rc = check_grid(amax_rowwise, "amax_rowwise", rows, nbr, MXFP8_DTYPE_F32)) return rc;
  if (int rc = check_tensor(amax_tensor, "amax_tensor")) return rc;
  if (amax_tensor->dtype != MXFP8_DTYPE_F32) return fail(MXFP8_ERR_DTYPE, "amax_tensor: dtype must be F32");
  if (int rc = check_grid(scale_rowwise, "scale_rowwise", rows, nbr, MXFP8_DTYPE_U8)) return rc;
  const bool colwise = !is_empty(amax_colwise);
  if (colwise) {
    if (int rc = check_grid(amax_colwise, "amax_colwise", nbc, cols, MXFP8_DTYPE_F32)) return rc;
    if (is_empty(scale_colwise))
      return fail(MXFP8_ERR_MISSING, "scale_colwise is required when amax_colwise is present");
    if (int rc = check_grid(scale_colwise, "scale_colwise", nbc, cols, MXFP8_DTYPE_U8)) return rc;
  }
  mxfp8::Nvfp4ScaleParams p{};
  p.amax_t = static_cast<const float*>(amax_tensor->data);
  auto seg = [](const mxfp8_tensor* a, mxfp8_tensor* sc, int64_t nr, int64_t nc) {
    mxfp8::Nvfp4ScaleSegment g{};
    g.amax = static_cast<const float*>(a->data);
    g.scale = static_cast<uint8_t*>(sc->data);
    g.nrows = nr;
    g.ncols = nc;
    g.ld_a = a->shape[1];
    g.ld_s = sc->shape[1];
    g.vec = g.ld_a == nc && g.ld_s == nc && (nr * nc) % 4 == 0 &&
            reinterpret_cast<uintptr_t>(g.amax) % 16 == 0 && reinterpret_cast<uintptr_t>(g.scale) % 4 == 0;
    return g;
  };
  p.seg[p.nseg++] = seg(amax_rowwise, scale_rowwise, rows, nbr);
  if (colwise) p.seg[p.nseg++] = seg(amax_colwise, scale_colwise, nbc, cols);
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  return cuda_status(mxfp8::launch_nvfp4_scales(p, dev, static_cast<cudaStream_t>(stream)),
                     "nvfp4 scale update launch");
}

int nvfp4_partial_cast(const mxfp8_tensor* input, const mxfp8_tensor* scale_rowwise,
                       const mxfp8_tensor* scale_colwise, const mxfp8_tensor* amax_tensor,
                       mxfp8_tensor* output_rowwise, mxfp8_tensor* output_colwise, int64_t rows,
                       int64_t cols, int64_t start_offset, int64_t out_offset, void* stream) {
  const bool in_empty = is_empty(input);
  if (!in_empty) {
    if (int rc = check_tensor(input, "input")) return rc;
  }
  const int64_t len = in_empty ? 0 : numel(input);
  if (int rc = check_dims(rows, cols, start_offset, len)) return rc;
  if (out_offset < 0) return fail(MXFP8_ERR_INVALID, "out_offset must be non-negative");
  if (cols % 2 != 0 || start_offset % 2 != 0 || len % 2 != 0 || out_offset % 2 != 0)
    return fail(MXFP8_ERR_INVALID,
                "NVFP4 packs two codes per byte: cols, start_offset, the fragment length and "
                "out_offset must be even");
  if (len == 0) return ok();
  const int32_t dt = input->dtype;
  if (dt != MXFP8_DTYPE_F32 && dt != MXFP8_DTYPE_BF16)
    return fail(MXFP8_ERR_DTYPE, "input: dtype must be F32 or BF16");
  if (is_empty(scale_rowwise)) return fail(MXFP8_ERR_MISSING, "scale_rowwise is required");
  if (is_empty(amax_tensor)) return fail(MXFP8_ERR_MISSING, "amax_tensor is required");
  if (is_empty(output_rowwise)) return fail(MXFP8_ERR_MISSING, "output_rowwise is required");
  const int64_t nbr = (cols + 15) / 16, nbc = (rows + 15) / 16;
  if (int rc = check_grid(scale_rowwise, "scale_rowwise", rows, nbr, MXFP8_DTYPE_U8)) return rc;
  if (int rc = check_tensor(amax_tensor, "amax_tensor")) return rc;
  if (amax_tensor->dtype != MXFP8_DTYPE_F32) return fail(MXFP8_ERR_DTYPE, "amax_tensor: dtype must be F32");
  const int64_t need = (out_offset + len) / 2;
  auto check_out = [&](const mxfp8_tensor* o, const char* name) {
    if (int rc = check_tensor(o, name)) return rc;
    if (o->dtype != MXFP8_DTYPE_U8) return fail(MXFP8_ERR_DTYPE, "%s: dtype must be U8", name);
    if (numel(o) < need)
      return fail(MXFP8_ERR_SHAPE, "%s holds %lld bytes, needs (out_offset + len) / 2 = %lld", name,
                  (long long)numel(o), (long long)need);
    return int(MXFP8_OK);
  };
  if (int rc = check_out(output_rowwise, "output_rowwise")) return rc;
  const bool colwise = !is_empty(output_colwise);
  if (colwise) {
    if (int rc = check_out(output_colwise, "output_colwise")) return rc;
    if (is_empty(scale_colwise))
      return fail(MXFP8_ERR_MISSING, "scale_colwise is required when output_colwise is present");
    if (int rc = check_grid(scale_colwise, "scale_colwise", nbc, cols, MXFP8_DTYPE_U8)) return rc;
  }
  const int64_t eb = elem_bytes(dt);
  const int V = int(16 / eb);
  mxfp8::Nvfp4CastParams p{};
  p.g = make_geom(rows, cols, start_offset, len, mxfp8::tile_width_for(dt));
  p.g.fast_ok = cols % V == 0;
  p.g.shift = int32_t(virtual_base(input->data, start_offset, eb) % 16);
  p.in = input->data;
  p.s_r = static_cast<const uint8_t*>(scale_rowwise->data);
  p.ld_sr = scale_rowwise->shape[1];
  p.amax_t = static_cast<const float*>(amax_tensor->data);
  p.out_r = static_cast<uint8_t*>(output_rowwise->data);
  p.out_shift = out_offset - start_offset;
  // a lane's V codes (V/2 bytes) start at nibble address 2 * out + row * cols + j +
  // out_shift, with cols and j multiples of V when whole tiles take the vector path: one
  // V/2-byte word store when 2 * out + out_shift is a multiple of V
  auto word_ok = [&](const void* o) {
    const int64_t m = V;
    const int64_t nib = (2 * int64_t(reinterpret_cast<uintptr_t>(o) % uintptr_t(m)) + p.out_shift % m) % m;
    return (nib + m) % m == 0;
  };
  bool vec = p.g.fast_ok && word_ok(p.out_r);
  if (colwise) {
    p.s_c = static_cast<const uint8_t*>(scale_colwise->data);
    p.ld_sc = scale_colwise->shape[1];
    p.out_c = static_cast<uint8_t*>(output_colwise->data);
    vec = vec && word_ok(p.out_c);
  }
  p.vec_out = vec;
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  return cuda_status(mxfp8::launch_nvfp4_cast(p, dt == MXFP8_DTYPE_F32 ? 0 : 1, p.g.shift != 0, dev,
                                              static_cast<cudaStream_t>(stream)),
                     "nvfp4 partial cast launch");
}

int mxfp8_device_can_access(const void* ptr, int64_t bytes) {
  if (ptr == nullptr || bytes < 0) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const char* first = static_cast<const char*>(ptr);
  const char* last = first + (bytes > 0 ? bytes - 1 : 0);
  for (const char* q : {first, last}) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, q) != cudaSuccess) {
      cudaGetLastError();  // clear the sticky-free error of an unknown pointer
      return 0;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
      if (a.type == cudaMemoryTypeDevice && a.device != dev) return 0;
      continue;
    }
    if (a.type == cudaMemoryTypeHost && a.devicePointer == static_cast<const void*>(q)) continue;
    return 0;
  }
  return 1;
}

int64_t mxfp8_swizzled_scales_size(int64_t nrows, int64_t ncols, int32_t transpose) {
  if (nrows < 0 || ncols < 0) return -1;
  const int64_t lr = transpose ? ncols : nrows, lc = transpose ? nrows : ncols;
  return (lr + 127) / 128 * 128 * ((lc + 3) / 4 * 4);
}

int mxfp8_swizzle_scales(const mxfp8_tensor* scale_inv, mxfp8_tensor* out, int64_t nrows,
                         int64_t ncols, int32_t transpose, void* stream) {
  if (nrows <= 0 || ncols <= 0) return fail(MXFP8_ERR_INVALID, "nrows and ncols must be positive");
  if (transpose != 0 && transpose != 1) return fail(MXFP8_ERR_INVALID, "transpose must be 0 or 1");
  if (nrows > (int64_t(1) << 40) || ncols > (int64_t(1) << 40))
    return fail(MXFP8_ERR_INVALID, "grid too large");
  if (is_empty(scale_inv)) return fail(MXFP8_ERR_MISSING, "scale_inv is required");
  if (is_empty(out)) return fail(MXFP8_ERR_MISSING, "out is required");
  if (int rc = check_grid(scale_inv, "scale_inv", nrows, ncols, MXFP8_DTYPE_U8)) return rc;
  if (int rc = check_tensor(out, "out")) return rc;
  if (out->dtype != MXFP8_DTYPE_U8) return fail(MXFP8_ERR_DTYPE, "out: dtype must be U8");
  const int64_t need = mxfp8_swizzled_scales_size(nrows, ncols, transpose);
  if (numel(out) < need)
    return fail(MXFP8_ERR_SHAPE, "out holds %lld bytes, the layout needs %lld",
                (long long)numel(out), (long long)need);
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  SwizzleParams p{};
  p.s = static_cast<const uint8_t*>(scale_inv->data);
  p.ld = scale_inv->shape[1];
  p.out = static_cast<uint8_t*>(out->data);
  p.lr = transpose ? ncols : nrows;
  p.lc = transpose ? nrows : ncols;
  p.pr = (p.lr + 127) / 128 * 128;
  p.pc = (p.lc + 3) / 4 * 4;
  p.transpose = transpose;
  p.vec = reinterpret_cast<uintptr_t>(p.out) % 16 == 0;
  return cuda_status(mxfp8::launch_swizzle_scales(p, dev, static_cast<cudaStream_t>(stream)),
                     "swizzle scales launch");
}

}  // extern "C"
