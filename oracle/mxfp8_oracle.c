/*
 * CPU ORACLE for the partial MXFP8 cast of high-precision master weights.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline leg
 * do.  It shares no code, header, table or constant with the CUDA library.
 *
 * Plain, slow, scalar C.  Floating point is carried in double (every operation
 * used here is exact in double: max, power-of-two scaling, and the two
 * roundings, which are done by an explicit nearest-integer step).
 *
 * What it computes follows the page "Support row-only MXFP8 distributed
 * master-weight casts" (TransformerEngine pull request 3488):
 *   - section "Changes": amax is packed and MAX-reduced only for the directions
 *     that exist; scale updates and columnwise writes are skipped when the
 *     columnwise output is absent; values are rounded through the model dtype
 *     before quantisation; writes go in place into full-size outputs, or into a
 *     fragment-sized output (the helper's fragment-output interface);
 *   - the review thread's API documentation: the input is a contiguous segment of
 *     the flattened original tensor; amax_rowwise / amax_colwise are in/out
 *     tensors of row-wise (1x32) and column-wise (32x1) block maxima of |x| in the
 *     input dtype; columnwise scales are required iff the columnwise output is
 *     present and ignored otherwise;
 *   - the flow diagram: amax for present directions, one packed MAX all-reduce,
 *     scale update for present directions, rowwise write, optional columnwise
 *     write.
 * The pages print no formula for the E8M0 scale.  The convention used is:
 * scale exponent e = floor(log2(block amax)) - 8, clamped to [-127, 127],
 * amax 0 -> e = -127; stored as the biased E8M0 byte e + 127; the data byte is
 * E4M3 (bias 7, max 448, no infinities) of y * 2^-e, y = master value rounded
 * to BF16 (nearest, ties to even), with round-to-nearest-even and saturation
 * to +-448.  Non-finite handling (not a parity target of any workload): a block
 * with a NaN member has a NaN amax, stored as the canonical quiet NaN whatever
 * the members' NaN payloads; a NaN or infinite amax gives scale byte 0xFF; a
 * scale byte 0xFF casts every element of its block to 0x7F; a NaN value casts to
 * 0x7F; an infinite value saturates.
 *
 * dtype codes: 0 = FP32 (float), 1 = BF16 (uint16_t bit patterns).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_MODEL_BF16 0
#define ORACLE_MODEL_F16 1

/* ---------- element access ---------------------------------------------------- */

/* Value of element k (0-based) of a fragment buffer, widened exactly to double. */
static double load_value(const void *buf, int dtype, int64_t k) {
    if (dtype == ORACLE_F32) {
        return (double)((const float *)buf)[k];
    } else {
        uint32_t bits = (uint32_t)((const uint16_t *)buf)[k] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
}

/* Store a double that is exactly representable in the dtype (amax values are).
 * A NaN amax is stored as the canonical quiet NaN: FP32 bits 0x7FC00000, BF16
 * bits 0x7FC0 (the pages print no NaN rule; one fixed pattern is the plainest). */
static void store_value(void *buf, int dtype, int64_t k, double v) {
    uint32_t bits;
    if (isnan(v)) {
        bits = 0x7FC00000u;
    } else {
        float f = (float)v;
        memcpy(&bits, &f, sizeof bits);
    }
    if (dtype == ORACLE_F32) {
        memcpy((char *)buf + 4 * k, &bits, sizeof bits);
    } else {
        ((uint16_t *)buf)[k] = (uint16_t)(bits >> 16);
    }
}

/* ---------- the three roundings / encodings ---------------------------------- */

/* floor(log2(a)) for finite a > 0, from frexp (a = f * 2^e, f in [0.5, 1)). */
static int floor_log2(double a) {
    int e;
    frexp(a, &e);
    return e - 1;
}

/* Round an FP32 value to BF16 (8 significant bits, FP32 exponent range),
 * nearest with ties to even; returns the BF16 value as a double.
 * "rounding through the model dtype" (section "Changes"). */
double oracle_bf16_round(float x) {
    double v = (double)x;
    if (isnan(v) || isinf(v) || v == 0.0) return v;
    double a = fabs(v);
    int p = floor_log2(a);
    if (p < -126) p = -126;               /* BF16 subnormals share the spacing 2^-133 */
    double quantum = ldexp(1.0, p - 7);   /* 8 significant bits */
    double r = nearbyint(a / quantum) * quantum;  /* a/quantum is exact in double */
    if (r >= ldexp(1.0, 128)) r = INFINITY;       /* past the largest finite BF16 */
    return v < 0 ? -r : r;
}

/* Round a value to IEEE FP16 (11 significant bits, normal exponents -14..15,
 * subnormal spacing 2^-24), nearest with ties to even; past the largest finite
 * value 65504 by half a unit (65520) the result is infinite.  Returns a double.
 * The model dtype may be FP16 instead of BF16 ("rounding through the model dtype",
 * section "Changes"). */
double oracle_f16_round(double v) {
    if (isnan(v) || isinf(v) || v == 0.0) return v;
    double a = fabs(v);
    int p = floor_log2(a);
    if (p < -14) p = -14;                 /* subnormals share the spacing 2^-24 */
    double quantum = ldexp(1.0, p - 10);  /* 11 significant bits */
    double r = nearbyint(a / quantum) * quantum;
    if (r > 65504.0) r = INFINITY;
    return v < 0 ? -r : r;
}

/* FP16 bit pattern of oracle_f16_round(x) (for the pins). */
uint16_t oracle_f16_bits(double v) {
    double r = oracle_f16_round(v);
    uint16_t sign = signbit(r) ? 0x8000 : 0;
    double a = fabs(r);
    if (isnan(r)) return 0x7E00;
    if (isinf(a)) return sign | 0x7C00;
    if (a == 0.0) return sign;
    int p = floor_log2(a);
    if (p < -14) return sign | (uint16_t)(a / ldexp(1.0, -24));            /* subnormal */
    return sign | (uint16_t)(((p + 15) << 10) | (int)(ldexp(a, -p) * 1024.0 - 1024.0));
}

/* BF16 bit pattern of oracle_bf16_round(x). */
uint16_t oracle_bf16_rne_bits(float x) {
    double r = oracle_bf16_round(x);
    float f = (float)r;
    if (isnan(r)) f = NAN;
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    if (isnan(r)) bits = (bits & 0x80000000u) | 0x7fc00000u;
    return (uint16_t)(bits >> 16);
}

/* E8M0 scale byte of a block amax: e = floor(log2(amax)) - 8 clamped to
 * [-127, 127], amax 0 -> -127, byte = e + 127; NaN / infinite amax -> 0xFF. */
uint8_t oracle_e8m0_from_amax(double amax) {
    if (isnan(amax) || isinf(amax)) return 0xFF;
    double a = fabs(amax);
    int e;
    if (a == 0.0) {
        e = -127;
    } else {
        e = floor_log2(a) - 8;
        if (e < -127) e = -127;
        if (e > 127) e = 127;
    }
    return (uint8_t)(e + 127);
}

/* OCP E4M3 ("fn" variant: bias 7, 3 mantissa bits, no infinities, 0x7F/0xFF NaN,
 * largest finite 448, smallest subnormal 2^-9).  Round to nearest, ties to even,
 * then saturate to +-448.  NaN -> 0x7F. */
uint8_t oracle_e4m3_encode(double v) {
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a >= 448.0) return sign | 0x7E;          /* everything at or past 448 saturates */
    int p = (a < ldexp(1.0, -6)) ? -6 : floor_log2(a);  /* subnormals: spacing 2^-9 */
    double quantum = ldexp(1.0, p - 3);
    double r = nearbyint(a / quantum);            /* ties to even (default mode) */
    double q = r * quantum;
    if (q < ldexp(1.0, -6)) {
        /* subnormal code r in 0..8 (r == 8 is 2^-6, the first normal, code 0x08) */
        return sign | (uint8_t)r;
    }
    int pe = floor_log2(q);
    int mant = (int)(ldexp(q, -pe) * 8.0) - 8;
    return sign | (uint8_t)(((pe + 7) << 3) | mant);
}

/* Value of an E4M3 byte (for the error-bound pins). */
double oracle_e4m3_decode(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* y * 2^(127 - s): the quantity that is encoded to E4M3 for scale byte s. */
static double scaled_value(double y, uint8_t s) {
    return ldexp(y, 127 - (int)s);
}

uint8_t oracle_quantize(double y, uint8_t s) {
    if (s == 0xFF) return 0x7F;
    return oracle_e4m3_encode(scaled_value(y, s));
}

/* ---------- step 1: partial amax -------------------------------------------- */

/* Row-wise (1x32) and column-wise (32x1) block maxima of |x| over the elements of
 * the fragment [start, start+len) of a rows x cols row-major weight.  frag points
 * at element `start`.  Every block that holds at least one fragment element is
 * overwritten with the maximum over those elements; all other entries are left
 * as they were.  A NaN member makes the block amax NaN.
 * amax_r: [rows][ld_r] (ld_r >= ceil(cols/32)), amax_c: [ceil(rows/32)][ld_c]
 * (ld_c >= cols) or NULL when the weight has no columnwise direction. */
int oracle_partial_amax(const void *frag, int dtype, int64_t rows, int64_t cols,
                        int64_t start, int64_t len, void *amax_r, int64_t ld_r,
                        void *amax_c, int64_t ld_c) {
    (void)rows;
    if (len == 0) return 0;
    /* accumulators cover only the rows the fragment spans: r0 .. r1 */
    int64_t r0 = start / cols, r1 = (start + len - 1) / cols;
    int64_t c0 = r0 / 32, c1 = r1 / 32;
    int64_t nbr = (cols + 31) / 32;
    int64_t nr = r1 - r0 + 1, nc = c1 - c0 + 1;
    double *acc_r = calloc((size_t)(nr * nbr), sizeof(double));
    unsigned char *hit_r = calloc((size_t)(nr * nbr), 1);
    double *acc_c = amax_c ? calloc((size_t)(nc * cols), sizeof(double)) : NULL;
    unsigned char *hit_c = amax_c ? calloc((size_t)(nc * cols), 1) : NULL;
    if (!acc_r || !hit_r || (amax_c && (!acc_c || !hit_c))) {
        free(acc_r); free(hit_r); free(acc_c); free(hit_c);
        return 1;
    }
    for (int64_t k = start; k < start + len; ++k) {
        int64_t i = k / cols, j = k % cols;
        double a = fabs(load_value(frag, dtype, k - start));
        int64_t br = (i - r0) * nbr + j / 32;          /* row block (i, j/32) */
        hit_r[br] = 1;
        if (isnan(a) || isnan(acc_r[br])) acc_r[br] = NAN;
        else if (a > acc_r[br]) acc_r[br] = a;
        if (amax_c) {
            int64_t bc = (i / 32 - c0) * cols + j;     /* column block (i/32, j) */
            hit_c[bc] = 1;
            if (isnan(a) || isnan(acc_c[bc])) acc_c[bc] = NAN;
            else if (a > acc_c[bc]) acc_c[bc] = a;
        }
    }
    for (int64_t i = r0; i <= r1; ++i)
        for (int64_t b = 0; b < nbr; ++b)
            if (hit_r[(i - r0) * nbr + b])
                store_value(amax_r, dtype, i * ld_r + b, acc_r[(i - r0) * nbr + b]);
    if (amax_c)
        for (int64_t c = c0; c <= c1; ++c)
            for (int64_t j = 0; j < cols; ++j)
                if (hit_c[(c - c0) * cols + j])
                    store_value(amax_c, dtype, c * ld_c + j, acc_c[(c - c0) * cols + j]);
    free(acc_r); free(hit_r); free(acc_c); free(hit_c);
    return 0;
}

/* ---------- step 2: packed MAX reduction over shards ------------------------- */

/* out[k] = max over s of |slots[s*slot_elems + k]| (the MAX all-reduce of the
 * packed amax buffer, here over num_slots emulated ranks).  NaN propagates. */
int oracle_max_reduce(const void *slots, int dtype, int64_t slot_elems, int num_slots, void *out) {
    for (int64_t k = 0; k < slot_elems; ++k) {
        double m = 0.0;
        for (int s = 0; s < num_slots; ++s) {
            double a = fabs(load_value(slots, dtype, (int64_t)s * slot_elems + k));
            if (isnan(a) || isnan(m)) m = NAN;
            else if (a > m) m = a;
        }
        store_value(out, dtype, k, m);
    }
    return 0;
}

/* ---------- step 3: scale update --------------------------------------------- */

/* scale[r][c] = E8M0 byte of amax[r][c] for r < nrows, c < ncols. */
int oracle_update_scales(const void *amax, int dtype, int64_t nrows, int64_t ncols,
                         int64_t ld_a, uint8_t *scale, int64_t ld_s) {
    for (int64_t r = 0; r < nrows; ++r)
        for (int64_t c = 0; c < ncols; ++c)
            scale[r * ld_s + c] = oracle_e8m0_from_amax(load_value(amax, dtype, r * ld_a + c));
    return 0;
}

/* ---------- step 4: partial cast --------------------------------------------- */

/* For every fragment element k (element (i, j) of the weight): y = the master value
 * rounded to the model dtype (BF16: identity for BF16 input; FP16: IEEE half); rowwise byte = E4M3 of
 * y * 2^-e with the scale of row block (i, j/32); columnwise byte (only when
 * out_c is non-NULL) with the scale of column block (i/32, j).  Byte k is
 * written at out_offset + (k - start); nothing else is written.
 * scale_c is ignored when out_c is NULL. */
int oracle_partial_cast_model(const void *frag, int dtype, int model, int64_t rows, int64_t cols,
                              int64_t start, int64_t len,
                              const uint8_t *scale_r, int64_t ld_sr,
                              const uint8_t *scale_c, int64_t ld_sc,
                              uint8_t *out_r, uint8_t *out_c, int64_t out_offset) {
    (void)rows;
    for (int64_t k = start; k < start + len; ++k) {
        int64_t i = k / cols, j = k % cols;
        double x = load_value(frag, dtype, k - start);
        double y;
        if (model == ORACLE_MODEL_F16) y = oracle_f16_round(x);
        else y = (dtype == ORACLE_F32) ? oracle_bf16_round((float)x) : x;
        int64_t o = out_offset + (k - start);
        out_r[o] = oracle_quantize(y, scale_r[i * ld_sr + j / 32]);
        if (out_c) out_c[o] = oracle_quantize(y, scale_c[(i / 32) * ld_sc + j]);
    }
    return 0;
}

int oracle_partial_cast(const void *frag, int dtype, int64_t rows, int64_t cols,
                        int64_t start, int64_t len,
                        const uint8_t *scale_r, int64_t ld_sr,
                        const uint8_t *scale_c, int64_t ld_sc,
                        uint8_t *out_r, uint8_t *out_c, int64_t out_offset) {
    return oracle_partial_cast_model(frag, dtype, ORACLE_MODEL_BF16, rows, cols, start, len,
                                     scale_r, ld_sr, scale_c, ld_sc, out_r, out_c, out_offset);
}

/* ---------- scale layout for GEMM consumers ---------------------------------- */

/* Rearrange an E8M0 grid into the layout block-scaled tensor-core GEMMs read.  The
 * logical matrix L is the grid itself (transpose == 0, L[r][c] = S[r][c], LR = nr,
 * LC = nc) or its transpose (transpose == 1, L[r][c] = S[c][r], LR = nc, LC = nr).
 * L is padded with zero bytes to PR = ceil(LR/128)*128 rows and PC = ceil(LC/4)*4
 * columns and cut into 128x4 tiles stored in row-major tile order, 512 bytes each;
 * inside a tile, element (r, c) sits at (r % 32) * 16 + (r / 32) * 4 + c. */
int oracle_swizzle_scales(const uint8_t *S, int64_t nr, int64_t nc, int64_t ld, int transpose,
                          uint8_t *out) {
    int64_t LR = transpose ? nc : nr, LC = transpose ? nr : nc;
    int64_t PR = (LR + 127) / 128 * 128, PC = (LC + 3) / 4 * 4;
    int64_t tiles_per_row = PC / 4;
    for (int64_t r = 0; r < PR; ++r) {
        for (int64_t c = 0; c < PC; ++c) {
            uint8_t v = 0;
            if (r < LR && c < LC) v = transpose ? S[c * ld + r] : S[r * ld + c];
            int64_t tile = (r / 128) * tiles_per_row + c / 4;
            int64_t rr = r % 128, cc = c % 4;
            out[tile * 512 + (rr % 32) * 16 + (rr / 32) * 4 + cc] = v;
        }
    }
    return 0;
}

/* ---------- element-wise batch helpers for the pins -------------------------- */

void oracle_bf16_rne_bits_array(const float *x, uint16_t *out, int64_t n) {
    for (int64_t k = 0; k < n; ++k) out[k] = oracle_bf16_rne_bits(x[k]);
}

void oracle_e4m3_encode_array(const double *v, uint8_t *out, int64_t n) {
    for (int64_t k = 0; k < n; ++k) out[k] = oracle_e4m3_encode(v[k]);
}

void oracle_f16_bits_array(const double *v, uint16_t *out, int64_t n) {
    for (int64_t k = 0; k < n; ++k) out[k] = oracle_f16_bits(v[k]);
}

void oracle_e8m0_array(const double *amax, uint8_t *out, int64_t n) {
    for (int64_t k = 0; k < n; ++k) out[k] = oracle_e8m0_from_amax(amax[k]);
}

/* ======================================================================== *
 * NVFP4 partial cast.                                                       *
 *                                                                           *
 * The subject page excludes NVFP4 from its scope and prints no rule for it; *
 * this section follows one stated convention (the NVFP4 format as NVIDIA    *
 * defines it: E2M1 data, 16-value blocks with E4M3 scales, one FP32 scale   *
 * per tensor), taking the same distributed steps as the MXFP8 path: partial *
 * block maxima of each fragment, MAX reduction, scale update, partial cast. *
 *                                                                           *
 *   blocks   1x16 along rows (rowwise), 16x1 along columns (columnwise);    *
 *   G        tensor amax = max |x| over the whole weight (FP32);            *
 *   S        tensor encode scale = 2688 / G in FP32 (2688 = 448 * 6, the   *
 *            largest E4M3 value times the largest E2M1 value); G == 0 gives *
 *            S = 1, a quotient past the largest finite float gives that     *
 *            largest finite float;                                          *
 *   s        block scale = E4M3(fp32(fp32(A / 6) * S)) for block amax A,    *
 *            nearest-even, saturating at 448;                               *
 *   M        block multiplier = fp32(S / decode(s)), 0 when s decodes to 0; *
 *   q        data = E2M1(fp32(y * M)), y the master value rounded to BF16,  *
 *            nearest-even, saturating at 6.                                 *
 * Every FP32 operation here is one correctly rounded IEEE single-precision *
 * operation (float arithmetic, no contraction), so the integer codes are    *
 * decided in the same precision as on the GPU.  Non-finite inputs are       *
 * outside this convention (E2M1 has no NaN or infinity).                    *
 * ======================================================================== */

/* E2M1: sign bit, 2 exponent bits (bias 1), 1 mantissa bit.  Magnitudes 0, 0.5
 * (subnormal), 1, 1.5, 2, 3, 4, 6; code = sign << 3 | exponent << 1 | mantissa.
 * Round to nearest, ties to the even code, then saturate to 6. */
uint8_t oracle_e2m1_encode(double v) {
    if (isnan(v)) return 0x7;                  /* outside the convention; any fixed code */
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    double a = fabs(v);
    double quantum = a < 2.0 ? 0.5 : (a < 4.0 ? 1.0 : 2.0);   /* spacing of the binade */
    double r = nearbyint(a / quantum) * quantum;
    if (r > 6.0) r = 6.0;
    uint8_t mag;
    if (r < 1.0) mag = (uint8_t)(r * 2.0);                      /* 0 -> 0, 0.5 -> 1 */
    else {
        int e = floor_log2(r);                                   /* 0, 1 or 2 */
        int m = (int)(ldexp(r, -e) * 2.0) - 2;                   /* 0 or 1 */
        mag = (uint8_t)(((e + 1) << 1) | m);
    }
    return sign | mag;
}

double oracle_e2m1_decode(uint8_t c) {
    int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

float oracle_nvfp4_tensor_scale(float g) {
    if (g == 0.0f) return 1.0f;
    float s = 2688.0f / g;
    if (isinf(s)) s = FLT_MAX;
    return s;
}

uint8_t oracle_nvfp4_block_scale(float amax, float s_enc) {
    float t = amax / 6.0f;
    float u = t * s_enc;
    return oracle_e4m3_encode((double)u);
}

float oracle_nvfp4_multiplier(uint8_t s, float s_enc) {
    float d = (float)oracle_e4m3_decode(s);   /* exact: every E4M3 value is a float */
    if (d == 0.0f) return 0.0f;
    return s_enc / d;
}

uint8_t oracle_nvfp4_quantize(float y, float m) {
    float p = y * m;
    return oracle_e2m1_encode((double)p);
}

/* Row-wise (1x16) and column-wise (16x1) block maxima of |x| over the fragment
 * [start, start+len) of a rows x cols weight, in FP32; blocks with at least one
 * fragment element are overwritten, others untouched (as the MXFP8 partial amax).
 * amax_t (one float) is max-accumulated with the fragment's largest |x|.
 * amax_r: [rows][ld_r] (ld_r >= ceil(cols/16)); amax_c: [ceil(rows/16)][ld_c] or
 * NULL. */
int oracle_nvfp4_partial_amax(const void *frag, int dtype, int64_t rows, int64_t cols,
                              int64_t start, int64_t len, float *amax_r, int64_t ld_r,
                              float *amax_c, int64_t ld_c, float *amax_t) {
    (void)rows;
    if (len == 0) return 0;
    int64_t r0 = start / cols, r1 = (start + len - 1) / cols;
    int64_t c0 = r0 / 16, c1 = r1 / 16;
    int64_t nbr = (cols + 15) / 16;
    int64_t nr = r1 - r0 + 1, nc = c1 - c0 + 1;
    double *acc_r = calloc((size_t)(nr * nbr), sizeof(double));
    unsigned char *hit_r = calloc((size_t)(nr * nbr), 1);
    double *acc_c = amax_c ? calloc((size_t)(nc * cols), sizeof(double)) : NULL;
    unsigned char *hit_c = amax_c ? calloc((size_t)(nc * cols), 1) : NULL;
    if (!acc_r || !hit_r || (amax_c && (!acc_c || !hit_c))) {
        free(acc_r); free(hit_r); free(acc_c); free(hit_c);
        return 1;
    }
    double tmax = 0.0;
    for (int64_t k = start; k < start + len; ++k) {
        int64_t i = k / cols, j = k % cols;
        double a = fabs(load_value(frag, dtype, k - start));
        if (isnan(a) || isnan(tmax)) tmax = NAN;
        else if (a > tmax) tmax = a;
        int64_t br = (i - r0) * nbr + j / 16;          /* row block (i, j/16) */
        hit_r[br] = 1;
        if (isnan(a) || isnan(acc_r[br])) acc_r[br] = NAN;
        else if (a > acc_r[br]) acc_r[br] = a;
        if (amax_c) {
            int64_t bc = (i / 16 - c0) * cols + j;     /* column block (i/16, j) */
            hit_c[bc] = 1;
            if (isnan(a) || isnan(acc_c[bc])) acc_c[bc] = NAN;
            else if (a > acc_c[bc]) acc_c[bc] = a;
        }
    }
    for (int64_t i = r0; i <= r1; ++i)
        for (int64_t b = 0; b < nbr; ++b)
            if (hit_r[(i - r0) * nbr + b])
                store_value(amax_r, ORACLE_F32, i * ld_r + b, acc_r[(i - r0) * nbr + b]);
    if (amax_c)
        for (int64_t c = c0; c <= c1; ++c)
            for (int64_t j = 0; j < cols; ++j)
                if (hit_c[(c - c0) * cols + j])
                    store_value(amax_c, ORACLE_F32, c * ld_c + j, acc_c[(c - c0) * cols + j]);
    double prev = (double)*amax_t;
    if (isnan(prev) || isnan(tmax)) store_value(amax_t, ORACLE_F32, 0, NAN);
    else if (tmax > prev) store_value(amax_t, ORACLE_F32, 0, tmax);
    free(acc_r); free(hit_r); free(acc_c); free(hit_c);
    return 0;
}

/* scale[r][c] = E4M3 block scale of amax[r][c] under tensor amax g, r < nrows, c < ncols. */
int oracle_nvfp4_update_scales(const float *amax, int64_t nrows, int64_t ncols, int64_t ld_a,
                               float g, uint8_t *scale, int64_t ld_s) {
    float s_enc = oracle_nvfp4_tensor_scale(g);
    for (int64_t r = 0; r < nrows; ++r)
        for (int64_t c = 0; c < ncols; ++c)
            scale[r * ld_s + c] = oracle_nvfp4_block_scale(amax[r * ld_a + c], s_enc);
    return 0;
}

/* Write E2M1 code q into nibble p of a packed buffer (low nibble = even position). */
static void put_nibble(uint8_t *buf, int64_t p, uint8_t q) {
    uint8_t *b = buf + p / 2;
    if (p % 2 == 0) *b = (uint8_t)((*b & 0xF0) | q);
    else *b = (uint8_t)((*b & 0x0F) | (q << 4));
}

/* For every fragment element k (element (i, j)): y = BF16 rounding of x (identity for
 * BF16 input); rowwise code with the scale of row block (i, j/16), columnwise code
 * (when out_c is non-NULL) with the scale of column block (i/16, j); each written to
 * nibble out_offset + (k - start) of its output; nothing else is written. */
int oracle_nvfp4_partial_cast(const void *frag, int dtype, int64_t rows, int64_t cols,
                              int64_t start, int64_t len, const uint8_t *scale_r, int64_t ld_sr,
                              const uint8_t *scale_c, int64_t ld_sc, float g,
                              uint8_t *out_r, uint8_t *out_c, int64_t out_offset) {
    (void)rows;
    float s_enc = oracle_nvfp4_tensor_scale(g);
    for (int64_t k = start; k < start + len; ++k) {
        int64_t i = k / cols, j = k % cols;
        double x = load_value(frag, dtype, k - start);
        float y = (float)((dtype == ORACLE_F32) ? oracle_bf16_round((float)x) : x);
        int64_t p = out_offset + (k - start);
        put_nibble(out_r, p, oracle_nvfp4_quantize(y, oracle_nvfp4_multiplier(scale_r[i * ld_sr + j / 16], s_enc)));
        if (out_c)
            put_nibble(out_c, p, oracle_nvfp4_quantize(y, oracle_nvfp4_multiplier(scale_c[(i / 16) * ld_sc + j], s_enc)));
    }
    return 0;
}

void oracle_e2m1_encode_array(const double *v, uint8_t *out, int64_t n) {
    for (int64_t k = 0; k < n; ++k) out[k] = oracle_e2m1_encode(v[k]);
}

void oracle_nvfp4_block_scale_array(const float *amax, float s_enc, uint8_t *out, int64_t n) {
    for (int64_t k = 0; k < n; ++k) out[k] = oracle_nvfp4_block_scale(amax[k], s_enc);
}
