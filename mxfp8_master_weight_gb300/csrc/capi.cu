// C ABI of the partial MXFP8 cast (declared in include/mxfp8_partial.h):
// argument validation, fragment geometry and kernel dispatch.  No entry point
// allocates memory or synchronises; all work is enqueued on the caller's stream.
#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>

#include <cuda_runtime.h>

#include "kernels.h"
#include "mxfp8_partial.h"

namespace {

using mxfp8::AmaxParams;
using mxfp8::CastParams;
using mxfp8::DeviceInfo;
using mxfp8::FragGeom;
using mxfp8::ScaleSegment;

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

int check_dims(int64_t rows, int64_t cols, int64_t start, int64_t len) {
  if (rows <= 0 || cols <= 0) return fail(MXFP8_ERR_INVALID, "rows and cols must be positive");
  if (rows > INT64_MAX / cols) return fail(MXFP8_ERR_INVALID, "rows*cols overflows int64");
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
    const int64_t r0 = start / cols, r1 = (start + len - 1) / cols;
    g.band0 = r0 / 32;
    g.ntiles = (r1 / 32 - g.band0 + 1) * g.coltiles;
  }
  return g;
}

// Virtual base address of element 0 of the weight for a fragment pointer (may lie
// outside the allocation; only used for alignment arithmetic).
uintptr_t virtual_base(const void* frag, int64_t start, int64_t eb) {
  return reinterpret_cast<uintptr_t>(frag) - uintptr_t(start * eb);
}

}  // namespace

extern "C" {

const char* mxfp8_last_error(void) { return g_err; }

int mxfp8_version(void) { return 100; }

int mxfp8_partial_amax(const mxfp8_tensor* input, mxfp8_tensor* amax_rowwise,
                       mxfp8_tensor* amax_colwise, int64_t rows, int64_t cols,
                       int64_t start_offset, void* stream) {
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
  const int64_t nbr = (cols + 31) / 32, nbc = (rows + 31) / 32;
  if (int rc = check_grid(amax_rowwise, "amax_rowwise", rows, nbr, dt)) return rc;
  const bool colwise = !is_empty(amax_colwise);
  if (colwise) {
    if (int rc = check_grid(amax_colwise, "amax_colwise", nbc, cols, dt)) return rc;
  }
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;

  const int64_t eb = elem_bytes(dt);
  const int V = int(16 / eb);
  AmaxParams p{};
  p.g = make_geom(rows, cols, start_offset, len, mxfp8::tile_width_for(dt));
  p.g.fast_ok = (virtual_base(input->data, start_offset, eb) % 16 == 0) && (cols % V == 0);
  p.in = input->data;
  p.amax_r = amax_rowwise->data;
  p.ld_r = amax_rowwise->shape[1];
  if (colwise) {
    p.amax_c = amax_colwise->data;
    p.ld_c = amax_colwise->shape[1];
    p.vec_c = (reinterpret_cast<uintptr_t>(p.amax_c) % 16 == 0) && (p.ld_c % V == 0);
  }
  return cuda_status(mxfp8::launch_partial_amax(p, dt == MXFP8_DTYPE_F32 ? 0 : 1, colwise, dev,
                                                static_cast<cudaStream_t>(stream)),
                     "partial amax launch");
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

int mxfp8_update_scales(const mxfp8_tensor* amax_rowwise, const mxfp8_tensor* amax_colwise,
                        mxfp8_tensor* scale_inv_rowwise, mxfp8_tensor* scale_inv_colwise,
                        int64_t rows, int64_t cols, void* stream) {
  if (rows <= 0 || cols <= 0) return fail(MXFP8_ERR_INVALID, "rows and cols must be positive");
  if (rows > INT64_MAX / cols) return fail(MXFP8_ERR_INVALID, "rows*cols overflows int64");
  if (is_empty(amax_rowwise)) return fail(MXFP8_ERR_MISSING, "amax_rowwise is required");
  if (is_empty(scale_inv_rowwise)) return fail(MXFP8_ERR_MISSING, "scale_inv_rowwise is required");
  const int32_t dt = amax_rowwise->dtype;
  if (dt != MXFP8_DTYPE_F32 && dt != MXFP8_DTYPE_BF16)
    return fail(MXFP8_ERR_DTYPE, "amax_rowwise: dtype must be F32 or BF16");
  const int64_t nbr = (cols + 31) / 32, nbc = (rows + 31) / 32;
  if (int rc = check_grid(amax_rowwise, "amax_rowwise", rows, nbr, dt)) return rc;
  if (int rc = check_grid(scale_inv_rowwise, "scale_inv_rowwise", rows, nbr, MXFP8_DTYPE_U8)) return rc;
  const bool colwise = !is_empty(amax_colwise);
  if (colwise) {
    if (int rc = check_grid(amax_colwise, "amax_colwise", nbc, cols, dt)) return rc;
    if (is_empty(scale_inv_colwise))
      return fail(MXFP8_ERR_MISSING, "scale_inv_colwise is required when amax_colwise is present");
    if (int rc = check_grid(scale_inv_colwise, "scale_inv_colwise", nbc, cols, MXFP8_DTYPE_U8)) return rc;
  }
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  const int64_t eb = elem_bytes(dt);
  auto seg = [&](const mxfp8_tensor* a, mxfp8_tensor* s, int64_t nr, int64_t nc) {
    ScaleSegment g{};
    g.amax = a->data;
    g.scale = static_cast<uint8_t*>(s->data);
    g.nrows = nr;
    g.ncols = nc;
    g.ld_a = a->shape[1];
    g.ld_s = s->shape[1];
    g.vec = (g.ld_a == nc) && (g.ld_s == nc) && ((nr * nc) % 4 == 0) &&
            (reinterpret_cast<uintptr_t>(g.amax) % uintptr_t(4 * eb) == 0) &&
            (reinterpret_cast<uintptr_t>(g.scale) % 4 == 0);
    return g;
  };
  ScaleSegment segs[2];
  int nseg = 0;
  segs[nseg++] = seg(amax_rowwise, scale_inv_rowwise, rows, nbr);
  if (colwise) segs[nseg++] = seg(amax_colwise, scale_inv_colwise, nbc, cols);
  return cuda_status(mxfp8::launch_update_scales(segs, nseg, dt == MXFP8_DTYPE_F32 ? 0 : 1, dev,
                                                 static_cast<cudaStream_t>(stream)),
                     "update scales launch");
}

int mxfp8_partial_cast(const mxfp8_tensor* input, const mxfp8_tensor* scale_inv_rowwise,
                       const mxfp8_tensor* scale_inv_colwise, mxfp8_tensor* output_rowwise,
                       mxfp8_tensor* output_colwise, int64_t rows, int64_t cols,
                       int64_t start_offset, int64_t out_offset, void* stream) {
  const bool in_empty = is_empty(input);
  if (!in_empty) {
    if (int rc = check_tensor(input, "input")) return rc;
  }
  const int64_t len = in_empty ? 0 : numel(input);
  if (int rc = check_dims(rows, cols, start_offset, len)) return rc;
  if (out_offset < 0) return fail(MXFP8_ERR_INVALID, "out_offset must be non-negative");
  if (len == 0) return ok();
  const int32_t dt = input->dtype;
  if (dt != MXFP8_DTYPE_F32 && dt != MXFP8_DTYPE_BF16)
    return fail(MXFP8_ERR_DTYPE, "input: dtype must be F32 or BF16");
  if (is_empty(scale_inv_rowwise)) return fail(MXFP8_ERR_MISSING, "scale_inv_rowwise is required");
  if (is_empty(output_rowwise)) return fail(MXFP8_ERR_MISSING, "output_rowwise is required");
  const int64_t nbr = (cols + 31) / 32, nbc = (rows + 31) / 32;
  if (int rc = check_grid(scale_inv_rowwise, "scale_inv_rowwise", rows, nbr, MXFP8_DTYPE_U8)) return rc;
  if (int rc = check_tensor(output_rowwise, "output_rowwise")) return rc;
  if (output_rowwise->dtype != MXFP8_DTYPE_U8) return fail(MXFP8_ERR_DTYPE, "output_rowwise: dtype must be U8");
  if (numel(output_rowwise) - len < out_offset)
    return fail(MXFP8_ERR_SHAPE, "output_rowwise holds %lld bytes, needs out_offset + len = %lld",
                (long long)numel(output_rowwise), (long long)(out_offset + len));
  const bool colwise = !is_empty(output_colwise);
  if (colwise) {
    if (int rc = check_tensor(output_colwise, "output_colwise")) return rc;
    if (output_colwise->dtype != MXFP8_DTYPE_U8) return fail(MXFP8_ERR_DTYPE, "output_colwise: dtype must be U8");
    if (numel(output_colwise) - len < out_offset)
      return fail(MXFP8_ERR_SHAPE, "output_colwise holds %lld bytes, needs out_offset + len = %lld",
                  (long long)numel(output_colwise), (long long)(out_offset + len));
    if (is_empty(scale_inv_colwise))
      return fail(MXFP8_ERR_MISSING, "scale_inv_colwise is required when output_colwise is present");
    if (int rc = check_grid(scale_inv_colwise, "scale_inv_colwise", nbc, cols, MXFP8_DTYPE_U8)) return rc;
  }
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;

  const int64_t eb = elem_bytes(dt);
  const int V = int(16 / eb);
  const int64_t shift = out_offset - start_offset;
  CastParams p{};
  p.g = make_geom(rows, cols, start_offset, len, mxfp8::tile_width_for(dt));
  p.in = input->data;
  p.s_r = static_cast<const uint8_t*>(scale_inv_rowwise->data);
  p.ld_sr = scale_inv_rowwise->shape[1];
  p.out_r = static_cast<uint8_t*>(output_rowwise->data);
  p.out_shift = shift;
  bool fast = (virtual_base(input->data, start_offset, eb) % 16 == 0) && (cols % V == 0) &&
              ((reinterpret_cast<uintptr_t>(p.out_r) + uintptr_t(shift)) % uintptr_t(V) == 0);
  if (colwise) {
    p.s_c = static_cast<const uint8_t*>(scale_inv_colwise->data);
    p.ld_sc = scale_inv_colwise->shape[1];
    p.out_c = static_cast<uint8_t*>(output_colwise->data);
    fast = fast && ((reinterpret_cast<uintptr_t>(p.out_c) + uintptr_t(shift)) % uintptr_t(V) == 0);
    p.vec_sc = (reinterpret_cast<uintptr_t>(p.s_c) % uintptr_t(V) == 0) && (p.ld_sc % V == 0);
  }
  p.g.fast_ok = fast;
  return cuda_status(mxfp8::launch_partial_cast(p, dt == MXFP8_DTYPE_F32 ? 0 : 1, colwise, dev,
                                                static_cast<cudaStream_t>(stream)),
                     "partial cast launch");
}

}  // extern "C"
