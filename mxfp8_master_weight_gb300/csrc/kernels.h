// Internal interface between the C ABI (capi.cu) and the kernel translation units.
// Host-side parameter blocks are validated by capi.cu before any launch.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "mxfp8_partial.h"

namespace mxfp8 {

// Geometry of one fragment [start, end) of a rows x cols row-major weight, and
// the 32-row x TW-column warp tiles that cover it.
struct FragGeom {
  int64_t rows, cols;
  int64_t start, end;   // flat element range of the fragment
  int64_t rs, cs;       // (row, col) of the fragment's first element
  int64_t re, ce;       // (row, col) of its last element
  int64_t band0;        // first 32-row band the fragment touches
  int64_t ntiles;       // bands x coltiles
  int32_t coltiles;     // ceil(cols / TW)
  int32_t fast_ok;      // cols % V == 0: whole tiles may take the 16-byte vector path
  int32_t shift;        // (virtual base address of element 0) mod 16, in bytes; the vector
                        // path then loads aligned chunks and realigns them across lanes
};

struct AmaxParams {
  FragGeom g;
  const void* in;  // fragment base: element `start` of the flattened weight
  void* amax_r;    // [rows][ld_r]
  int64_t ld_r;
  void* amax_c;    // [ceil(rows/32)][ld_c]; unused when the colwise kernel is not chosen
  int64_t ld_c;
  int32_t vec_c;   // colwise amax row stores may be 16-byte vectors
};

struct CastParams {
  FragGeom g;
  const void* in;
  const uint8_t* s_r;  // [rows][ld_sr] E8M0
  int64_t ld_sr;
  const uint8_t* s_c;  // [ceil(rows/32)][ld_sc] E8M0 (colwise kernel only)
  int64_t ld_sc;
  uint8_t* out_r;      // byte of flat element f lives at out + (f + out_shift)
  uint8_t* out_c;
  int64_t out_shift;   // out_offset - start
  int32_t vec_sc;      // colwise scale rows may be read as V-byte words
  int32_t vec_out;     // both outputs' virtual bases are V-byte aligned: word stores
};

// One-pass quantisation of a fragment made of whole blocks: block maxima, E8M0
// scales and E4M3 data from one kernel (amax outputs optional).
struct FusedParams {
  FragGeom g;
  const void* in;
  void* amax_r;        // [rows][ld_r] or nullptr
  int64_t ld_r;
  void* amax_c;        // [ceil(rows/32)][ld_c] or nullptr
  int64_t ld_c;
  uint8_t* s_r;        // [rows][ld_sr] E8M0
  int64_t ld_sr;
  uint8_t* s_c;        // [ceil(rows/32)][ld_sc] E8M0 (colwise kernel only)
  int64_t ld_sc;
  uint8_t* out_r;      // byte of flat element f lives at out + (f + out_shift)
  uint8_t* out_c;
  int64_t out_shift;
  int32_t vec_c;       // colwise amax rows may take 16-byte stores
  int32_t vec_sc;      // colwise scale rows may take V-byte stores
  int32_t vec_out;     // outputs' virtual bases are V-byte aligned
};

// One direction of a scale update: scale[r][c] = E8M0(amax[r][c]), r < nrows, c < ncols.
struct ScaleSegment {
  const void* amax;
  uint8_t* scale;
  int64_t nrows, ncols, ld_a, ld_s;
  int32_t vec;  // dense (ld == ncols), 4 | nrows*ncols and aligned: 4 entries per thread
};

// E8M0 grid -> the 128x4-tile layout block-scaled tensor-core GEMMs read.
struct SwizzleParams {
  const uint8_t* s;     // grid [nr][ld]
  int64_t ld;
  uint8_t* out;         // PR * PC bytes
  int64_t lr, lc;       // logical matrix (the grid or its transpose)
  int64_t pr, pc;       // padded to multiples of 128 rows and 4 columns
  int32_t transpose;
  int32_t vec;          // out is 16-byte aligned
};

// Fused MAX reduction + scale update of a run of entries of one block grid that is a
// view into the packed reduced buffer: for linear entries e = r * ld_a + c in [e0, e1)
// (padding columns c >= ncols skipped), reduced[r][c] = max over the contributing slots
// of |slot_s[r][c]| (+0 when none contributes) and scale[r][c] = E8M0(reduced).  The
// contributing slots are slots 0 .. nslots-1 (all_slots) or the set bits of `slots`.
struct ReduceScaleSegment {
  const void* slot0;     // the grid's first entry inside slot 0 of the packed slots
  int64_t slot_stride;   // entries between consecutive slots
  uint64_t slots;        // contributing slots when !all_slots (bit s = slot s)
  int32_t nslots;
  int32_t all_slots;
  int32_t vec;           // dense grid, 4 | e0 and e1, 16-byte (F32) / 8-byte (BF16) aligned:
                         // one work item = 4 entries; otherwise one item = one entry
  void* reduced;         // the grid's view inside the reduced buffer [nrows][ld_a]
  uint8_t* scale;        // [nrows][ld_s]
  int64_t nrows, ncols, ld_a, ld_s;
  int64_t e0, e1;
};

// NVFP4 (E2M1 data, 16-value blocks with E4M3 scales, one FP32 tensor scale).
// Partial amax of one fragment: FP32 1x16 row-block and 16x1 column-block maxima, and
// the fragment's largest |x| max-accumulated into the tensor amax (FP32 bits).
struct Nvfp4AmaxParams {
  FragGeom g;
  const void* in;
  float* amax_r;       // [rows][ld_r], ld_r >= ceil(cols/16)
  int64_t ld_r;
  float* amax_c;       // [ceil(rows/16)][ld_c] (colwise kernel only)
  int64_t ld_c;
  uint32_t* amax_t;    // one FP32, max-accumulated
  int32_t vec_c;       // colwise amax rows may take 16-byte stores
};

// E4M3 block scales of up to two grids under one tensor amax.
struct Nvfp4ScaleSegment {
  const float* amax;
  uint8_t* scale;
  int64_t nrows, ncols, ld_a, ld_s;
  int32_t vec;         // dense (ld == ncols), 4 | nrows*ncols, aligned: 4 entries per thread
};
struct Nvfp4ScaleParams {
  const float* amax_t;
  int32_t nseg;
  Nvfp4ScaleSegment seg[2];
};

// Partial cast of one fragment to packed E2M1 (element f in nibble f + out_shift; the
// low nibble of a byte holds the even position).
struct Nvfp4CastParams {
  FragGeom g;
  const void* in;
  const uint8_t* s_r;  // [rows][ld_sr] E4M3
  int64_t ld_sr;
  const uint8_t* s_c;  // [ceil(rows/16)][ld_sc] E4M3 (colwise kernel only)
  int64_t ld_sc;
  const float* amax_t;
  uint8_t* out_r;
  uint8_t* out_c;
  int64_t out_shift;   // out_offset - start (even)
  int32_t vec_out;     // a lane's V/2 output bytes may leave as one 2- (FP32) or 4-byte store
};

struct DeviceInfo {
  int device;
  int sms;
};

// Direction sets a kernel instantiation handles: only rowwise, rowwise + columnwise,
// or a mix (each job's columnwise pointer picks, per tile, one of the two
// compile-time specialisations, so the inner loops stay specialised).
enum Dirs { kRowOnly = 0, kBidir = 1, kMixed = 2 };

// A batch of fragments launched as one kernel: the warp tiles of every job's first
// and last 32-row bands (the only bands a fragment boundary can cut) come first,
// numbered by prefix_a, then every job's interior bands, numbered by prefix_b.
// The table travels in kernel parameter space (no device allocation): 64 jobs take 10-15 KB
// of the 32 KB parameter space kernels have since CUDA 12.1, so a batch of many small
// weights is a few launches, not one per 16 fragments.
constexpr int kMaxBatchJobs = 64;

template <class P, int N>
struct JobBatch {
  int32_t njobs;
  int64_t prefix_a[N + 1];
  int64_t prefix_b[N + 1];
  P job[N];
};

// Boundary-band and interior-band tile counts of one fragment.
inline void band_tiles(const FragGeom& g, int64_t* boundary, int64_t* interior) {
  const int64_t nbands = g.coltiles > 0 ? g.ntiles / g.coltiles : 0;
  *boundary = (nbands >= 2 ? 2 : nbands) * int64_t(g.coltiles);
  *interior = (nbands > 2 ? nbands - 2 : 0) * int64_t(g.coltiles);
}

template <class P, int N>
inline int64_t fill_batch(JobBatch<P, N>& b, const P* jobs, int n) {
  b.njobs = n;
  b.prefix_a[0] = b.prefix_b[0] = 0;
  for (int k = 0; k < n; ++k) {
    int64_t ta, tb;
    band_tiles(jobs[k].g, &ta, &tb);
    b.prefix_a[k + 1] = b.prefix_a[k] + ta;
    b.prefix_b[k + 1] = b.prefix_b[k] + tb;
    b.job[k] = jobs[k];
  }
  return b.prefix_a[n] + b.prefix_b[n];
}

// dtype: 0 = FP32, 1 = BF16.  Each launcher takes n validated jobs that share the
// dtype and the template choices (virtual base shifted, output word-aligned, model
// dtype), launches them in batches of at most kMaxBatchJobs -- each batch with the
// kernel for its direction set (row-only, bidirectional or mixed) -- and returns the
// CUDA launch status.
cudaError_t launch_partial_amax(const AmaxParams* jobs, int n, int dtype, bool shifted,
                                const DeviceInfo& dev, cudaStream_t stream);
// model: 0 = round through BF16, 1 = round through FP16.
cudaError_t launch_partial_cast(const CastParams* jobs, int n, int dtype, bool shifted,
                                bool vec_out, int model, const DeviceInfo& dev,
                                cudaStream_t stream);
cudaError_t launch_fused_quantize(const FusedParams* jobs, int n, int dtype, bool shifted,
                                  bool vec_out, int model, const DeviceInfo& dev,
                                  cudaStream_t stream);

// Parts of the two launchers above in separate translation units: the cast per input
// dtype and output alignment (word-aligned outputs, or not), the one-pass kernel per
// input dtype.
cudaError_t launch_partial_cast_f32(const CastParams* jobs, int n, bool shifted, int model,
                                    const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_partial_cast_f32_unaligned(const CastParams* jobs, int n, bool shifted, int model,
                                              const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_partial_cast_bf16(const CastParams* jobs, int n, bool shifted, int model,
                                     const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_partial_cast_bf16_unaligned(const CastParams* jobs, int n, bool shifted, int model,
                                               const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_partial_cast_bf16_unaligned_f16(const CastParams* jobs, int n, bool shifted,
                                                  const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_fused_quantize_f32(const FusedParams* jobs, int n, bool shifted, bool vec_out,
                                      int model, const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_fused_quantize_bf16(const FusedParams* jobs, int n, bool shifted,
                                       bool vec_out, int model, const DeviceInfo& dev,
                                       cudaStream_t stream);

// Direction set of a batch of jobs (colwise(job) tells whether a job has one).
template <class P, class F>
inline int batch_dirs(const P* jobs, int n, F colwise) {
  int col = 0;
  for (int k = 0; k < n; ++k) col += colwise(jobs[k]) ? 1 : 0;
  return col == 0 ? kRowOnly : (col == n ? kBidir : kMixed);
}
cudaError_t launch_update_scales(const ScaleSegment* segs, int nseg, int dtype,
                                 const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_reduce_update_scales(const ReduceScaleSegment* segs, int nseg, int dtype,
                                       const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_swizzle_scales(const SwizzleParams& p, const DeviceInfo& dev,
                                  cudaStream_t stream);
cudaError_t launch_max_reduce(const void* slots, void* out, int64_t slot_elems, int num_slots,
                              int dtype, const DeviceInfo& dev, cudaStream_t stream);

cudaError_t launch_nvfp4_amax(const Nvfp4AmaxParams& p, int dtype, bool shifted,
                              const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_nvfp4_scales(const Nvfp4ScaleParams& p, const DeviceInfo& dev,
                                cudaStream_t stream);
cudaError_t launch_nvfp4_cast(const Nvfp4CastParams& p, int dtype, bool shifted,
                              const DeviceInfo& dev, cudaStream_t stream);

// Record `msg` as the calling thread's last error (returned by mxfp8_last_error) and
// return `code`.  For entry points defined outside capi.cu.
int report_error(int code, const char* msg);

// Validate cast jobs exactly as mxfp8_partial_cast_batched does, without launching
// anything (status and last-error message as that entry point would give them).
int validate_cast_jobs(const mxfp8_cast_job* jobs, int njobs);

// Tile width (columns per warp tile) for a dtype.
inline int tile_width_for(int dtype) { return dtype == 0 ? 128 : 256; }

}  // namespace mxfp8
