// Internal interface between the C ABI (capi.cu) and the kernel translation units.
// Host-side parameter blocks are validated by capi.cu before any launch.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mxfp8 {

// Geometry of one fragment [start, end) of a rows x cols row-major weight, and
// the 32-row x TW-column warp tiles that cover it.
struct FragGeom {
  int64_t rows, cols;
  int64_t start, end;   // flat element range of the fragment
  int64_t band0;        // first 32-row band the fragment touches
  int64_t ntiles;       // bands x coltiles
  int32_t coltiles;     // ceil(cols / TW)
  int32_t fast_ok;      // 16-byte vector paths are legal for whole tiles
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
};

// One direction of a scale update: scale[r][c] = E8M0(amax[r][c]), r < nrows, c < ncols.
struct ScaleSegment {
  const void* amax;
  uint8_t* scale;
  int64_t nrows, ncols, ld_a, ld_s;
  int32_t vec;  // dense (ld == ncols), 4 | nrows*ncols and aligned: 4 entries per thread
};

struct DeviceInfo {
  int device;
  int sms;
};

// dtype: 0 = FP32, 1 = BF16.  Each launcher returns the CUDA launch status.
cudaError_t launch_partial_amax(const AmaxParams& p, int dtype, bool colwise,
                                const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_partial_cast(const CastParams& p, int dtype, bool colwise,
                                const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_update_scales(const ScaleSegment* segs, int nseg, int dtype,
                                 const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_max_reduce(const void* slots, void* out, int64_t slot_elems, int num_slots,
                              int dtype, const DeviceInfo& dev, cudaStream_t stream);

// Tile width (columns per warp tile) for a dtype.
inline int tile_width_for(int dtype) { return dtype == 0 ? 128 : 256; }

}  // namespace mxfp8
