/*
 * mxfp8_partial.h -- C ABI of the GB300 partial MXFP8 cast of master weights.
 *
 * The operation is the distributed master-weight writeback described on the page
 * "Support row-only MXFP8 distributed master-weight casts" (TransformerEngine
 * pull request 3488), sections "Changes" and the flow diagram: each rank holds a
 * contiguous fragment of a flattened rows x cols FP32 (or BF16) master weight;
 *   1. partial amax   -- 1x32 row-block and 32x1 column-block maxima of |x| over
 *                        the fragment, for the directions the weight has;
 *   2. packed MAX reduce of those amaxes over all ranks (here: over shard slots
 *                        of one device buffer);
 *   3. scale update   -- E8M0 block scales from the reduced amaxes;
 *   4. partial cast   -- master -> BF16 (nearest-even) -> E4M3 (nearest-even,
 *                        saturating at 448), written in place into the rowwise and,
 *                        when present, columnwise outputs.
 * Scale convention (the pages print none): scale exponent
 * e = floor(log2(amax)) - 8, clamped to [-127, 127], amax 0 -> -127; the stored
 * E8M0 byte is e + 127 (0xFF for a NaN/infinite amax).  Data byte =
 * E4M3(bf16(x) * 2^-e).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer inside an mxfp8_tensor is a DEVICE pointer (global memory of
 *   the current CUDA device), or page-locked host memory that the device can
 *   address directly (see mxfp8_device_can_access).  The caller owns all memory;
 *   the library never allocates, frees or keeps a pointer after the call returns.
 * - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = the
 *   legacy default stream).  A return of 0 means "validated and launched".
 *   Kernels are launched as programmatic dependents of the kernel before them in
 *   the stream: they may be scheduled while that kernel's last blocks run, but
 *   read and write nothing until it has completed, so stream order holds.
 * - Tensors are dense and row-major: a 2-D tensor's row stride is shape[1].
 * - An EMPTY handle (data == NULL, or any shape entry == 0, or a NULL handle
 *   pointer) means "this direction is absent" (section "Changes": omission uses
 *   empty tensor handles, not a magic shape).
 * - Return status: 0 ok; 1 invalid argument; 2 shape/padding mismatch;
 *   3 dtype mismatch; 4 missing required tensor; 6 CUDA launch error.
 *   (5, non-contiguous, is raised by language bindings that can see strides.)
 *   mxfp8_last_error() gives a message for the calling thread's last failure.
 * - Thread safety: entry points may be called concurrently from several host
 *   threads; results written by two launches to the same buffer race.
 */
#ifndef MXFP8_PARTIAL_H_
#define MXFP8_PARTIAL_H_

#include <stdint.h>

/* Every entry point below is exported; everything else in the library is hidden. */
#if defined(__GNUC__)
#define MXFP8_API __attribute__((visibility("default")))
#else
#define MXFP8_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MXFP8_DTYPE_F32 = 0,  /* float                              */
  MXFP8_DTYPE_BF16 = 1, /* bfloat16 (16-bit patterns)         */
  MXFP8_DTYPE_U8 = 2    /* uint8: E8M0 scales and E4M3 data   */
} mxfp8_dtype;

typedef struct {
  void* data;       /* device pointer, element-aligned; NULL => empty      */
  int32_t dtype;    /* mxfp8_dtype                                         */
  int32_t ndim;     /* 1 or 2                                              */
  int64_t shape[2]; /* shape[1] ignored when ndim == 1                     */
} mxfp8_tensor;

/* Size limits of every entry point taking rows x cols: 1 <= cols <= 2^37 and
 * rows * cols <= 2^40 elements; outside them the call returns MXFP8_ERR_INVALID. */
enum {
  MXFP8_OK = 0,
  MXFP8_ERR_INVALID = 1,
  MXFP8_ERR_SHAPE = 2,
  MXFP8_ERR_DTYPE = 3,
  MXFP8_ERR_MISSING = 4,
  MXFP8_ERR_NONCONTIGUOUS = 5,
  MXFP8_ERR_CUDA = 6
};

/*
 * Partial amax (page "Support row-only MXFP8 distributed master-weight casts",
 * review thread: documentation of the partial amax entry point).
 *
 * input         [in]     fragment: numel(input) = len contiguous F32 or BF16
 *                        values, element k of the fragment is element
 *                        start_offset + k of the flattened rows x cols weight.
 * amax_rowwise  [in,out] REQUIRED, 2-D [>= rows][>= ceil(cols/32)], dtype of the
 *                        input.  Entry (i, b) = max |x| over the fragment's
 *                        elements of row i, columns [32b, 32b+32).
 * amax_colwise  [in,out] OPTIONAL (empty => the columnwise direction is skipped
 *                        entirely, at compile time in the kernel), 2-D
 *                        [>= ceil(rows/32)][>= cols], dtype of the input.
 *                        Entry (c, j) = max |x| over the fragment's elements of
 *                        column j, rows [32c, 32c+32).
 * Only entries of blocks that contain at least one fragment element are written
 * (overwritten, not max-accumulated); every other entry keeps its value, so a
 * caller that reduces across fragments zeroes its buffers first.  An empty
 * fragment (len 0) writes nothing and returns 0.  NaN members make the entry NaN,
 * stored as the canonical quiet NaN (F32 0x7FC00000, BF16 0x7FC0) whatever their
 * NaN patterns.
 * Errors: 1 if start_offset < 0, rows/cols out of the size limits, start_offset + len > rows*cols,
 * or a pointer is not element-aligned; 2 on a too-small amax shape;
 * 3 if an amax dtype differs from the input dtype or the input is not F32/BF16;
 * 4 if amax_rowwise is empty (and len > 0).
 */
MXFP8_API int mxfp8_partial_amax(const mxfp8_tensor* input, mxfp8_tensor* amax_rowwise,
                       mxfp8_tensor* amax_colwise, int64_t rows, int64_t cols,
                       int64_t start_offset, void* stream);

/*
 * Packed MAX reduction (page "Support row-only MXFP8 distributed master-weight
 * casts", section "Changes": one packed-amax MAX all-reduce; here the ranks are
 * emulated as slots of one device buffer).
 *
 * slots  [in]  2-D [S][E] F32 or BF16: S packed amax buffers of E entries each.
 * out    [out] E entries (any shape with numel == E), same dtype.
 * out[k] = max over s of |slots[s][k]|; NaN propagates as the canonical quiet NaN
 * (F32 0x7FC00000, BF16 0x7FC0).  S == 1 copies |.|.
 * out may not overlap slots.  Errors: 2 numel mismatch, 3 dtype, 4 empty out.
 */
MXFP8_API int mxfp8_amax_max_reduce(const mxfp8_tensor* slots, mxfp8_tensor* out, void* stream);

/*
 * Scale update (page "Support row-only MXFP8 distributed master-weight casts",
 * flow diagram: "update scales for present directions").
 *
 * amax_rowwise      [in]  REQUIRED, [>= rows][>= ceil(cols/32)], F32 or BF16.
 * amax_colwise      [in]  OPTIONAL, [>= ceil(rows/32)][>= cols], same dtype;
 *                         empty => no columnwise scales are computed.
 * scale_inv_rowwise [out] REQUIRED, U8 [>= rows][>= ceil(cols/32)].
 * scale_inv_colwise [out] U8 [>= ceil(rows/32)][>= cols]; required iff
 *                         amax_colwise is present, ignored otherwise.
 * Writes the E8M0 byte of every entry of the compact block grid
 * (rows x ceil(cols/32) and ceil(rows/32) x cols); padding is left untouched.
 */
MXFP8_API int mxfp8_update_scales(const mxfp8_tensor* amax_rowwise, const mxfp8_tensor* amax_colwise,
                        mxfp8_tensor* scale_inv_rowwise, mxfp8_tensor* scale_inv_colwise,
                        int64_t rows, int64_t cols, void* stream);

/*
 * Partial cast (page "Support row-only MXFP8 distributed master-weight casts",
 * sections "Changes" and the review thread's documentation of the partial cast:
 * rowwise outputs are required; columnwise scales are required when the
 * columnwise output is present and ignored when it is omitted).
 *
 * input             [in]  fragment as for mxfp8_partial_amax.
 * scale_inv_rowwise [in]  REQUIRED U8 [>= rows][>= ceil(cols/32)] E8M0 bytes.
 * scale_inv_colwise [in]  U8 [>= ceil(rows/32)][>= cols]; required iff
 *                         output_colwise is present, ignored otherwise.
 * output_rowwise    [out] REQUIRED U8, numel >= out_offset + len.
 * output_colwise    [out] OPTIONAL U8 (empty => no columnwise reads or writes),
 *                         numel >= out_offset + len.
 * For fragment element k (weight element (i, j)): y = BF16 rounding of x
 * (identity for BF16 input); output_rowwise[out_offset + k] = E4M3(y * 2^-e_r),
 * e_r from scale_inv_rowwise[i][j/32]; output_colwise likewise with
 * scale_inv_colwise[i/32][j].  Outputs hold E4M3 bytes in the weight's own
 * row-major layout (the columnwise copy is not transposed).  out_offset =
 * start_offset writes into a full-size rows*cols output in place; out_offset = 0
 * writes a fragment-sized output.  Bytes outside the fragment are not touched.
 * Errors: 1 bad offsets/sizes; 2 output or scale too small; 3 dtype;
 * 4 rowwise scale/output missing, or columnwise output without columnwise scales.
 */
MXFP8_API int mxfp8_partial_cast(const mxfp8_tensor* input, const mxfp8_tensor* scale_inv_rowwise,
                       const mxfp8_tensor* scale_inv_colwise, mxfp8_tensor* output_rowwise,
                       mxfp8_tensor* output_colwise, int64_t rows, int64_t cols,
                       int64_t start_offset, int64_t out_offset, void* stream);

/*
 * Batched entry points: many fragments (of one or several weights) per call, e.g. all
 * fragments a rank holds for a batch of weights (page "Support row-only MXFP8
 * distributed master-weight casts", section "Changes": mixed row-only and
 * bidirectional batches).  Each job means exactly what the single-fragment call with
 * the same arguments means; the jobs are validated first (a failure launches nothing
 * and names the job), then run as few kernels as possible: jobs that share the input
 * dtype, the model dtype and (cast) whether the outputs allow word stores go into one
 * launch (at most 64 jobs each; row-only and bidirectional jobs, and fragments whose
 * virtual base is or is not 16-byte aligned, together, each tile taking its job's
 * specialisation), with the tiles of all jobs scheduled together.  Jobs may run concurrently:
 * jobs whose written entries overlap (two fragments of one weight writing the SAME
 * amax buffer, whose boundary blocks both jobs overwrite) race -- give each fragment
 * its own amax buffer, as a packed per-rank slot does.  Fragments of one weight write
 * disjoint output bytes and may share the outputs.  F32 and BF16 jobs may be mixed
 * in one call.  njobs may be 0; jobs with empty fragments are skipped.
 */
typedef struct {
  mxfp8_tensor input;
  mxfp8_tensor amax_rowwise;
  mxfp8_tensor amax_colwise; /* empty => row-only */
  int64_t rows, cols, start_offset;
} mxfp8_amax_job;

/* Model dtype the master values are rounded through before quantisation ("rounding
 * through the model dtype", section "Changes").  The single-fragment entry points
 * use BF16; jobs carry the choice (a zero-initialised job means BF16). */
enum { MXFP8_MODEL_BF16 = 0, MXFP8_MODEL_F16 = 1 };

typedef struct {
  mxfp8_tensor input;
  mxfp8_tensor scale_inv_rowwise;
  mxfp8_tensor scale_inv_colwise;
  mxfp8_tensor output_rowwise;
  mxfp8_tensor output_colwise; /* empty => row-only */
  int64_t rows, cols, start_offset, out_offset;
  int32_t model_dtype;         /* MXFP8_MODEL_BF16 (0) or MXFP8_MODEL_F16 */
} mxfp8_cast_job;

typedef struct {
  mxfp8_tensor amax_rowwise;
  mxfp8_tensor amax_colwise; /* empty => row-only */
  mxfp8_tensor scale_inv_rowwise;
  mxfp8_tensor scale_inv_colwise;
  int64_t rows, cols;
} mxfp8_scale_job;

MXFP8_API int mxfp8_partial_amax_batched(const mxfp8_amax_job* jobs, int32_t njobs, void* stream);
MXFP8_API int mxfp8_update_scales_batched(const mxfp8_scale_job* jobs, int32_t njobs, void* stream);

/*
 * Packed MAX reduction fused with the scale update (the reduction of
 * mxfp8_amax_max_reduce and the scale update of mxfp8_update_scales_batched in one
 * pass over the packed buffer, for the slots of ranks emulated on one GPU).
 *
 * slots   [in]  2-D [S][P] F32 or BF16 packed amax buffers.
 * reduced [out] P entries, same dtype.
 * jobs    [in]  njobs scale jobs (see mxfp8_scale_job) whose amax grids are views
 *               INTO `reduced`; entry (r, c) of such a view at reduced offset o is
 *               reduced[o] = max_s |slots[s][o]|, and its E8M0 byte goes to the job's
 *               scale grid.  Entries of `reduced` outside every view are not written.
 * Results equal mxfp8_amax_max_reduce followed by mxfp8_update_scales_batched.
 * Errors: as those two; 1 if a view does not lie inside `reduced`.
 */
MXFP8_API int mxfp8_amax_max_reduce_update_scales(const mxfp8_tensor* slots, mxfp8_tensor* reduced,
                                        const mxfp8_scale_job* jobs, int32_t njobs,
                                        void* stream);

/*
 * The same reduction when each slot holds amaxes only where its rank's fragments are.
 * A rank's partial amax writes exactly the entries of the blocks its fragments touch;
 * every other entry of its slot is never written.  Rather than zeroing those entries
 * before every step and reading them back in the reduction, the caller names, per slot,
 * the packed entries it holds, and the reduction reads only those (the emulated MAX
 * all-reduce of section "Changes" then moves only the bytes the ranks produced).
 *
 * slot_ranges [in] nranges triples (slot, begin, end): slot `slot` (< S <= 64) holds
 *                  valid amaxes for packed entries [begin, end) (0 <= begin <= end <= P).
 *                  Entries of a slot outside all of its ranges count as zero and are
 *                  not read (their contents are irrelevant); an entry no slot holds
 *                  reduces to +0.  Ranges of one slot may touch or overlap.
 * nranges == 0 (slot_ranges may be NULL): every slot holds every entry, exactly as
 * mxfp8_amax_max_reduce_update_scales.
 * Other arguments, results and errors as mxfp8_amax_max_reduce_update_scales; 1 also
 * for a malformed range or more than 64 slots with ranges.
 */
MXFP8_API int mxfp8_amax_max_reduce_update_scales_ranged(const mxfp8_tensor* slots,
                                               mxfp8_tensor* reduced,
                                               const mxfp8_scale_job* jobs, int32_t njobs,
                                               const int64_t* slot_ranges, int32_t nranges,
                                               void* stream);

MXFP8_API int mxfp8_partial_cast_batched(const mxfp8_cast_job* jobs, int32_t njobs, void* stream);

/*
 * One-pass quantisation of a fragment made of WHOLE blocks.  When every row block
 * (and, with a columnwise output, every column block) that the fragment touches lies
 * wholly inside it -- a rank that owns whole weights or whole 32-row bands, or a
 * single rank -- no cross-rank MAX reduction is needed (the MAX over one rank is the
 * identity), and amax, scale update and cast of the page "Support row-only MXFP8
 * distributed master-weight casts" (flow diagram) run as ONE kernel that reads the
 * input from HBM once.  Results are bit-identical to mxfp8_partial_amax ->
 * mxfp8_update_scales -> mxfp8_partial_cast on the same fragment.
 *
 * input, output_rowwise, output_colwise, rows, cols, start_offset, out_offset: as for
 *                   mxfp8_partial_cast; the columnwise direction is present iff
 *                   output_colwise is.
 * amax_rowwise / amax_colwise [out] OPTIONAL grids as for mxfp8_partial_amax; when
 *                   given, the block maxima are stored too (a columnwise amax grid is
 *                   ignored without a columnwise output).
 * scale_inv_rowwise [out] REQUIRED; scale_inv_colwise [out] required iff
 *                   output_colwise is present.  Entries of blocks the fragment touches
 *                   are written; others are left untouched.
 * Precondition (status 1 otherwise): start_offset % cols and (start_offset + len) %
 * cols are multiples of 32, and with a columnwise output start_offset and
 * start_offset + len are multiples of 32*cols (the end may also be rows*cols).
 */
MXFP8_API int mxfp8_quantize_whole_blocks(const mxfp8_tensor* input, mxfp8_tensor* amax_rowwise,
                                mxfp8_tensor* amax_colwise, mxfp8_tensor* scale_inv_rowwise,
                                mxfp8_tensor* scale_inv_colwise, mxfp8_tensor* output_rowwise,
                                mxfp8_tensor* output_colwise, int64_t rows, int64_t cols,
                                int64_t start_offset, int64_t out_offset, void* stream);

typedef struct {
  mxfp8_tensor input;
  mxfp8_tensor amax_rowwise;      /* optional */
  mxfp8_tensor amax_colwise;      /* optional */
  mxfp8_tensor scale_inv_rowwise;
  mxfp8_tensor scale_inv_colwise;
  mxfp8_tensor output_rowwise;
  mxfp8_tensor output_colwise;    /* empty => row-only */
  int64_t rows, cols, start_offset, out_offset;
  int32_t model_dtype;            /* MXFP8_MODEL_BF16 (0) or MXFP8_MODEL_F16 */
} mxfp8_quantize_job;

/* Batched form of mxfp8_quantize_whole_blocks, with the conventions of the other
 * batched entry points. */
MXFP8_API int mxfp8_quantize_whole_blocks_batched(const mxfp8_quantize_job* jobs, int32_t njobs,
                                        void* stream);

/*
 * Scale layout for GEMM consumers.  Rearranges a compact E8M0 grid into the layout in
 * which block-scaled tensor-core GEMMs read scale factors: the logical matrix L (the
 * grid when transpose == 0; its transpose when transpose == 1, e.g. a columnwise
 * [ceil(rows/32)][cols] grid consumed as [cols][ceil(rows/32)]) is padded with zero
 * bytes to multiples of 128 rows and 4 columns and cut into 128x4 tiles, stored in
 * row-major tile order, 512 bytes each; inside a tile element (r, c) sits at byte
 * (r % 32) * 16 + (r / 32) * 4 + c.  (An output format next to the path: the pages
 * only require padded scale grids.)
 *
 * scale_inv [in]  U8 2-D [>= nrows][>= ncols] (row stride shape[1]).
 * out       [out] U8, numel >= mxfp8_swizzled_scales_size(nrows, ncols, transpose).
 * Errors: 1 bad sizes or transpose flag, 2 out too small, 3 dtype, 4 missing tensor.
 */
MXFP8_API int mxfp8_swizzle_scales(const mxfp8_tensor* scale_inv, mxfp8_tensor* out, int64_t nrows,
                         int64_t ncols, int32_t transpose, void* stream);

/* Bytes of the GEMM layout of an nrows x ncols grid (transpose as above). */
MXFP8_API int64_t mxfp8_swizzled_scales_size(int64_t nrows, int64_t ncols, int32_t transpose);

/*
 * Host memory.  Every entry point takes device-accessible pointers.  On this platform
 * (unified virtual addressing; Grace-Blackwell's coherent CPU-GPU link) page-locked
 * host memory from cudaHostAlloc / cudaHostRegister is device-accessible through the
 * same pointer, so the kernels can read master weights from, and write E4M3 data to,
 * host memory directly.  mxfp8_device_can_access returns 1 when the current device can
 * dereference [ptr, ptr + bytes) (device, managed, or mapped page-locked host memory)
 * and 0 otherwise (e.g. pageable host memory); language bindings check host buffers
 * with it before passing them.  It enqueues nothing.
 */
MXFP8_API int mxfp8_device_can_access(const void* ptr, int64_t bytes);

/*
 * Sharded update of one weight without any device allocation.  The source pages have
 * no counterpart of this entry point.
 *
 * It is for callers that cannot allocate device memory at the moment they need the
 * update -- a memory-pool allocator running its own maintenance, a framework that has
 * reserved all device memory up front, or code where a cudaMalloc would synchronise
 * the device.  The update needs working memory for one amax slot per fragment and for
 * the reduced amax; here that memory is one file-scope device array of 64 MiB, which
 * every GPU that loads this library holds until the process exits.
 *
 * fragments[f]      [in]  fragment f of the rows x cols weight (F32 or BF16, one dtype
 *                         for all; empty fragments are skipped), starting at flat
 *                         element start_offsets[f].  Fragments must not overlap
 *                         (status 1 when two non-empty fragments do).
 * scale_inv_rowwise [out] REQUIRED U8 [>= rows][>= ceil(cols/32)].
 * scale_inv_colwise [out] U8 [>= ceil(rows/32)][>= cols]; required iff output_colwise.
 * output_rowwise    [out] REQUIRED U8, full size (rows*cols), written where the
 *                         fragments are.
 * output_colwise    [out] OPTIONAL U8 full size; empty => row-only.
 * Results equal mxfp8_partial_amax of every fragment into its own zeroed slot,
 * mxfp8_amax_max_reduce over the slots, mxfp8_update_scales and mxfp8_partial_cast of
 * every fragment (it runs exactly those entry points), with BF16 as the model dtype.
 * Limits: 1..64 fragments and (nfrags + 1) amax slots of rows*ceil(cols/32) (+
 * ceil(rows/32)*cols when columnwise) entries, each rounded up to 256 bytes, within
 * the 64 MiB; a larger request fails with status 2 and a message giving the bytes
 * needed.  Every argument is checked before anything is launched: a non-zero status
 * leaves every caller buffer untouched.  The first call on a device looks up the
 * array's device address (with that device current); make that first call before any
 * stream capture.  Every call uses
 * the same array and leaves its contents behind (slots are cleared at the start of
 * each call); calls that overlap on the GPU -- on different streams or from
 * different threads -- race on it.
 */
MXFP8_API int mxfp8_sharded_update_noalloc(const mxfp8_tensor* fragments, const int64_t* start_offsets,
                                 int32_t nfrags, mxfp8_tensor* scale_inv_rowwise,
                                 mxfp8_tensor* scale_inv_colwise, mxfp8_tensor* output_rowwise,
                                 mxfp8_tensor* output_colwise, int64_t rows, int64_t cols,
                                 void* stream);

/*
 * NVFP4 partial cast.  The same distributed steps as the MXFP8 entry points above (partial
 * amax of a fragment, MAX reduction of the packed amaxes over ranks with
 * mxfp8_amax_max_reduce on F32 slots, scale update, partial cast in place) for the NVFP4
 * format.  The page "Support row-only MXFP8 distributed master-weight casts" leaves NVFP4
 * out of its scope (section "Scope") and gives no rule for it; the convention is:
 *   blocks   1x16 along rows (rowwise), 16x1 along columns (columnwise);
 *   G        tensor amax: max |x| over the whole weight, F32;
 *   S        tensor encode scale 2688 / G in F32 (448 * 6); 1 when G == 0; the largest
 *            finite float when the quotient overflows;
 *   s        block scale byte: E4M3(fp32(fp32(A / 6) * S)), A the block amax
 *            (nearest-even, saturating at 448);
 *   data     E2M1(fp32(y * fp32(S / decode(s)))) (0 when s decodes to 0), y = x rounded
 *            to BF16 (nearest-even; identity for BF16 input); E2M1 has magnitudes 0,
 *            0.5, 1, 1.5, 2, 3, 4, 6 (codes 0-7, sign in bit 3), nearest-even,
 *            saturating at 6.  Two codes per byte: element at nibble position p sits in
 *            byte p / 2, the low nibble holding even p.
 * Each F32 step is one correctly rounded operation.  Non-finite inputs are outside the
 * convention (E2M1 has no NaN or infinity): their codes are unspecified.  A consumer
 * dequantises a code q of block scale s as decode(q) * decode(s) / S.
 */

/*
 * input         [in]     fragment as for mxfp8_partial_amax (F32 or BF16).
 * amax_rowwise  [in,out] REQUIRED F32 [>= rows][>= ceil(cols/16)]: entry (i, b) = max |x|
 *                        over the fragment's elements of row i, columns [16b, 16b+16).
 * amax_colwise  [in,out] OPTIONAL F32 [>= ceil(rows/16)][>= cols]: entry (c, j) over
 *                        rows [16c, 16c+16) of column j; empty => row-only.
 * amax_tensor   [in,out] REQUIRED F32, at least 1 element: element 0 is max-accumulated
 *                        with the fragment's largest |x| (it must hold +0 or a previous
 *                        maximum: initialise it to +0 before the first fragment).
 * Entries of blocks the fragment touches are overwritten, others untouched; NaN
 * members give the canonical quiet NaN.  Errors as mxfp8_partial_amax; 4 also for a
 * missing amax_tensor; 3 if an amax tensor is not F32.
 */
MXFP8_API int nvfp4_partial_amax(const mxfp8_tensor* input, mxfp8_tensor* amax_rowwise,
                       mxfp8_tensor* amax_colwise, mxfp8_tensor* amax_tensor, int64_t rows,
                       int64_t cols, int64_t start_offset, void* stream);

/*
 * amax_rowwise [in] REQUIRED F32 [>= rows][>= ceil(cols/16)] (reduced over ranks);
 * amax_colwise [in] OPTIONAL F32 [>= ceil(rows/16)][>= cols]; empty => no columnwise scales;
 * amax_tensor  [in] REQUIRED F32: element 0 is G;
 * scale_rowwise [out] REQUIRED U8 [>= rows][>= ceil(cols/16)] E4M3 block scales;
 * scale_colwise [out] U8 [>= ceil(rows/16)][>= cols]; required iff amax_colwise present.
 * Writes every entry of the compact grids; padding untouched.
 */
MXFP8_API int nvfp4_update_scales(const mxfp8_tensor* amax_rowwise, const mxfp8_tensor* amax_colwise,
                        const mxfp8_tensor* amax_tensor, mxfp8_tensor* scale_rowwise,
                        mxfp8_tensor* scale_colwise, int64_t rows, int64_t cols, void* stream);

/*
 * input          [in]  fragment as for mxfp8_partial_cast.
 * scale_rowwise  [in]  REQUIRED U8 [>= rows][>= ceil(cols/16)].
 * scale_colwise  [in]  U8 [>= ceil(rows/16)][>= cols]; required iff output_colwise.
 * amax_tensor    [in]  REQUIRED F32: element 0 is G (the same G the scales came from).
 * output_rowwise [out] REQUIRED U8 packed codes, numel >= (out_offset + len) / 2.
 * output_colwise [out] OPTIONAL U8 packed codes (empty => row-only), same size rule.
 * Element k of the fragment goes to nibble position out_offset + k (out_offset =
 * start_offset: full-size output of ceil(rows*cols/2) bytes, in place; 0: fragment-
 * size output).  Two codes share a byte, so cols, start_offset, the fragment length and
 * out_offset must be even (status 1 otherwise); then every byte a fragment writes
 * belongs to it alone.  Other errors as mxfp8_partial_cast.
 */
MXFP8_API int nvfp4_partial_cast(const mxfp8_tensor* input, const mxfp8_tensor* scale_rowwise,
                       const mxfp8_tensor* scale_colwise, const mxfp8_tensor* amax_tensor,
                       mxfp8_tensor* output_rowwise, mxfp8_tensor* output_colwise, int64_t rows,
                       int64_t cols, int64_t start_offset, int64_t out_offset, void* stream);

/* Message describing the calling thread's most recent non-zero status ("" if none). */
MXFP8_API const char* mxfp8_last_error(void);

/* Library version as major*10000 + minor*100 + patch. */
MXFP8_API int mxfp8_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MXFP8_PARTIAL_H_ */
