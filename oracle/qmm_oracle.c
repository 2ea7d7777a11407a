/*
 * qmm_oracle.c -- plain, slow, scalar CPU oracle for the quantized matmul path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or constant
 * generator with the CUDA library: every step is written out here again, in
 * the order the pages define it, as straight loops over one element at a time.
 *
 * Build: plain C99, -O2 -ffp-contract=off (no fused multiply-add except where
 * written as fmaf(), no fast-math), so x86-64 and aarch64 give the same bits.
 *
 * Sources (cited by page and section):
 *   [LCG31]  llama.cpp visual guide, lesson 31 "The CPU backend", section
 *            "How the quantized dot product works": the block_q4_0 layout (one
 *            fp16 scale d plus qs[16] holding 32 four-bit values), the Q8_0
 *            activation blocks, and the per-block chain unpack -> subtract 8 ->
 *            int8 dot -> multiply by dx*dy -> fused multiply-add into acc.
 *   [LOOM]   Loom docs, "Plan 9 SIMD Forward", section "BitNet ternary MAD
 *            kernel": ternary weights packed 16 per uint32 as 2-bit codes
 *            (code = w + 1), the identity dot = sum(code*act) - sum(act), the
 *            per-row activation scale 127/max|x| and y = dot*absmean/scale.
 *   [FUC06]  Fucina course, chapter 06 "Going fast on CPUs", section 6.4 "The
 *            scalar backend is the specification": the referee is the plain
 *            triple loop, serial, in the order the definition suggests.
 *   [WORKLOAD] the quantizer recipe of the benchmark workloads: Q4_0 with
 *            d = (signed absmax)/-8 and q = clamp(round(w/d)+8, 0, 15);
 *            Q8_0 with d = absmax/127 and q = round(x/d).
 *   [FUC09]  Fucina reference, "9. Backends: CPU SIMD, BLAS, threading, and
 *            GPU offload": Q8_0 also serves as a weight (right-hand side)
 *            format next to Q4_0 (9.2 quantizeMatmulRhsQ8_0, 9.7 the Q8_0 arm
 *            and its packed layout, 9.9.2 Q8_0 decode and prefill).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   R1 "round" is round-half-away-from-zero (C roundf).
 *   R2 Q8_0 and Q4_0 divide (x/d, w/d); the BitNet quantizer multiplies (x*s),
 *      because the Loom page defines s as a multiplier 127/max|x|.
 *   R3 q values use the f32 d; the stored scale is fp16(d), round-to-nearest-
 *      even, and dequantization / the dot use the stored fp16 scale.
 *   R4 nibble order: element j (0..15) of a block is the low nibble of byte j,
 *      element j+16 the high nibble of byte j.
 *   R5 ternary code of element i (0..15) of a word sits at bits [2i, 2i+1].
 *   R6 Q4_0 "signed absmax": the element with the largest |w|, the first one on
 *      ties, keeps its sign; it maps to q = 0.
 *   R7 activations clamp to [-127, 127] (never -128).
 *   R8 an all-zero block/row: Q8_0 d = 0 and q = 0; Q4_0 d = 0 and q = 8;
 *      BitNet scale = 0, q = 0, sum = 0 and y = 0.
 *   R9 the f32 output accumulates blocks in ascending order:
 *      acc = fmaf((float)sumi, f32(dw)*f32(da), acc), acc starting at +0.
 *  R10 BitNet y = ((float)dot * absmean) / scale, left to right in f32.
 *  R18 the load-time repack of Q4_0 nibbles for the tensor-core GEMM is a
 *      pure byte/nibble permutation (no value changes): tiles of 128 rows x
 *      2 blocks, each 4096 contiguous bytes; inside a tile, unit u = 2*r +
 *      blk (row r, block blk) holds the block's 32 nibbles in 16 bytes as 4
 *      words; word c carries elements 8c..8c+7, element 8c + 2i + h at bits
 *      4i + 16h (i = 0..3, h = 0..1).  Rows past n and blocks past k/32 are
 *      nibble 8 (value 0).
 *  R16 Q8_0 weights use the Q8_0 activation block and recipe unchanged: per
 *      32-block d = absmax/127, q = clamp(round(w/d), -127, 127), fp16(d)
 *      stored; the block dot is sum_j q_w * q_a (no offset) and y follows R9.
 *
 * Layouts (row-major throughout):
 *   x   f32  [m, k] with row stride ldx elements
 *   aq  int8 [m, k]            ad fp16 bits [m, k/32]
 *   wq  u8   [n, k/2]          wd fp16 bits [n, k/32]   (two planes of block_q4_0)
 *   w8  int8 [n, k]            wd fp16 bits [n, k/32]   (two planes of Q8_0 weight blocks)
 *   wr  u8   [ceil(n/128), ceil(k/64), 4096]   (Q4_0 nibbles in GEMM tile order, R18)
 *   y   f32  [m, n]
 *   sumi int32 [m, n, k/32]
 *   tw  u32  [n, k/16]         (ternary, 16 codes per word)
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_QK 32 /* elements per quantization block [LCG31] */

/* ---------------------------------------------------------------------- */
/* IEEE-754 binary16 <-> binary32, written from the format definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; subnormals have
 * exponent field 0 and value frac * 2^-24.                                 */

static uint32_t orc_bits_f32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float orc_f32_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

float orc_fp16_to_fp32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h >> 15) << 31;
    uint32_t e = (h >> 10) & 0x1f;
    uint32_t frac = h & 0x3ff;
    if (e == 0x1f) /* inf / nan: keep the payload in the top fraction bits */
        return orc_f32_bits(sign | 0x7f800000u | (frac << 13));
    if (e == 0) {
        /* zero or subnormal: frac * 2^-24, exact in f32 */
        float mag = (float)frac * 0x1p-24f;
        return sign ? -mag : mag;
    }
    return orc_f32_bits(sign | ((e - 15 + 127) << 23) | (frac << 13));
}

/* round-to-nearest, ties to even */
uint16_t orc_fp32_to_fp16(float f)
{
    uint32_t x = orc_bits_f32(f);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ax = x & 0x7fffffffu;
    if (ax >= 0x7f800000u) { /* inf or nan */
        if (ax == 0x7f800000u) return sign | 0x7c00u;
        return sign | 0x7c00u | 0x200u | (uint16_t)((ax >> 13) & 0x3ffu);
    }
    if (ax >= 0x477ff000u) /* >= 65520 = halfway between 65504 and 2^16 */
        return sign | 0x7c00u;
    if (ax >= 0x38800000u) { /* result is a normal binary16 (>= 2^-14) */
        uint32_t e = (ax >> 23) - 127 + 15;
        uint32_t mant = ax & 0x7fffffu;
        uint32_t h = (e << 10) | (mant >> 13);
        uint32_t rem = mant & 0x1fffu;
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u)))
            h += 1; /* a carry into the exponent is the correct next value */
        return sign | (uint16_t)h;
    }
    if (ax <= 0x33000000u) /* <= 2^-25: rounds to zero (2^-25 is a tie, even = 0) */
        return sign;
    {
        /* subnormal result: value / 2^-24 rounded to an integer */
        uint32_t e = ax >> 23; /* 102..112 */
        uint32_t mant = (ax & 0x7fffffu) | 0x800000u;
        uint32_t shift = 126 - e; /* value = mant * 2^(e-150) = (mant >> shift) * 2^-24 */
        uint32_t h = mant >> shift;
        uint32_t rem = mant & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1);
        if (rem > half || (rem == half && (h & 1u)))
            h += 1;
        return sign | (uint16_t)h;
    }
}

/* Array forms of the two conversions above (same code, one call per array). */
void orc_fp16_to_fp32_array(const uint16_t *h, int64_t count, float *out)
{
    for (int64_t i = 0; i < count; i++) out[i] = orc_fp16_to_fp32(h[i]);
}

void orc_fp32_to_fp16_array(const float *f, int64_t count, uint16_t *out)
{
    for (int64_t i = 0; i < count; i++) out[i] = orc_fp32_to_fp16(f[i]);
}

/* ---------------------------------------------------------------------- */
/* Q8_0 activation quantization [LCG31] [WORKLOAD], readings R1 R2 R3 R7 R8.
 * Per row and 32-block: amax = max|x|, d = amax/127 (f32), q = clamp(round(x/d)). */
void orc_quantize_q8_0(const float *x, int64_t m, int64_t k, int64_t ldx,
                       int8_t *aq, uint16_t *ad)
{
    int64_t kb = k / ORC_QK;
    for (int64_t i = 0; i < m; i++) {
        for (int64_t b = 0; b < kb; b++) {
            const float *xb = x + i * ldx + b * ORC_QK;
            float amax = 0.0f;
            for (int j = 0; j < ORC_QK; j++) {
                float a = fabsf(xb[j]);
                if (a > amax) amax = a;
            }
            float d = amax / 127.0f;
            ad[i * kb + b] = orc_fp32_to_fp16(d);
            for (int j = 0; j < ORC_QK; j++) {
                float q = 0.0f;
                if (d != 0.0f) {
                    q = roundf(xb[j] / d);
                    if (q > 127.0f) q = 127.0f;
                    if (q < -127.0f) q = -127.0f;
                }
                aq[i * k + b * ORC_QK + j] = (int8_t)q;
            }
        }
    }
}

/* ---------------------------------------------------------------------- */
/* Q4_0 weight quantization [WORKLOAD] (block layout [LCG31]), readings R1 R2
 * R3 R4 R6 R8.  Weights are row-major [n, k]; output planes wq [n, k/2] and
 * wd [n, k/32]. */
void orc_quantize_q4_0(const float *w, int64_t n, int64_t k,
                       uint8_t *wq, uint16_t *wd)
{
    int64_t kb = k / ORC_QK;
    for (int64_t r = 0; r < n; r++) {
        for (int64_t b = 0; b < kb; b++) {
            const float *wb = w + r * k + b * ORC_QK;
            float amax = 0.0f, maxv = 0.0f;
            for (int j = 0; j < ORC_QK; j++) {
                float a = fabsf(wb[j]);
                if (a > amax) { amax = a; maxv = wb[j]; } /* strict: first index wins ties */
            }
            float d = maxv / -8.0f;
            wd[r * kb + b] = orc_fp32_to_fp16(d);
            uint8_t q[ORC_QK];
            for (int j = 0; j < ORC_QK; j++) {
                float v = 8.0f;
                if (d != 0.0f) {
                    v = roundf(wb[j] / d) + 8.0f;
                    if (v > 15.0f) v = 15.0f;
                    if (v < 0.0f) v = 0.0f;
                }
                q[j] = (uint8_t)v;
            }
            uint8_t *dst = wq + r * (k / 2) + b * (ORC_QK / 2);
            for (int j = 0; j < ORC_QK / 2; j++)
                dst[j] = (uint8_t)(q[j] | (q[j + ORC_QK / 2] << 4));
        }
    }
}

/* The 4-bit value of element j (0..31) of the block starting at qs, R4. */
static int orc_q4_nibble(const uint8_t *qs, int j)
{
    return j < ORC_QK / 2 ? (qs[j] & 0x0f) : (qs[j - ORC_QK / 2] >> 4);
}

/* ---------------------------------------------------------------------- */
/* Per-block integer dot [LCG31]: sumi[i, r, b] = sum_j (q_w - 8) * q_a. */
void orc_block_sums_q4_0_q8_0(const uint8_t *wq, const int8_t *aq,
                              int64_t m, int64_t n, int64_t k, int32_t *sumi)
{
    int64_t kb = k / ORC_QK;
    for (int64_t i = 0; i < m; i++)
        for (int64_t r = 0; r < n; r++)
            for (int64_t b = 0; b < kb; b++) {
                const uint8_t *qs = wq + r * (k / 2) + b * (ORC_QK / 2);
                const int8_t *qa = aq + i * k + b * ORC_QK;
                int32_t s = 0;
                for (int j = 0; j < ORC_QK; j++)
                    s += (orc_q4_nibble(qs, j) - 8) * (int32_t)qa[j];
                sumi[(i * n + r) * kb + b] = s;
            }
}

/* ---------------------------------------------------------------------- */
/* Q4_0 x Q8_0 product in f32 [LCG31], reading R9: per output, blocks in
 * ascending order, acc = fma((float)sumi, dw*da, acc).  dw*da is exact in f32
 * (two 11-bit significands). */
void orc_gemm_q4_0_q8_0(const uint8_t *wq, const uint16_t *wd,
                        const int8_t *aq, const uint16_t *ad,
                        int64_t m, int64_t n, int64_t k, float *y)
{
    int64_t kb = k / ORC_QK;
    for (int64_t i = 0; i < m; i++)
        for (int64_t r = 0; r < n; r++) {
            float acc = 0.0f;
            for (int64_t b = 0; b < kb; b++) {
                const uint8_t *qs = wq + r * (k / 2) + b * (ORC_QK / 2);
                const int8_t *qa = aq + i * k + b * ORC_QK;
                int32_t s = 0;
                for (int j = 0; j < ORC_QK; j++)
                    s += (orc_q4_nibble(qs, j) - 8) * (int32_t)qa[j];
                float scale = orc_fp16_to_fp32(wd[r * kb + b]) * orc_fp16_to_fp32(ad[i * kb + b]);
                acc = fmaf((float)s, scale, acc);
            }
            y[i * n + r] = acc;
        }
}

/* Same product in double precision: every term sumi*dw*da is exact in double
 * (15 + 11 + 11 significant bits); only the sum over blocks rounds.  Used to
 * judge the f32 result, never as a gate on the GPU directly. */
void orc_gemm_q4_0_q8_0_f64(const uint8_t *wq, const uint16_t *wd,
                            const int8_t *aq, const uint16_t *ad,
                            int64_t m, int64_t n, int64_t k, double *y)
{
    int64_t kb = k / ORC_QK;
    for (int64_t i = 0; i < m; i++)
        for (int64_t r = 0; r < n; r++) {
            double acc = 0.0;
            for (int64_t b = 0; b < kb; b++) {
                const uint8_t *qs = wq + r * (k / 2) + b * (ORC_QK / 2);
                const int8_t *qa = aq + i * k + b * ORC_QK;
                int64_t s = 0;
                for (int j = 0; j < ORC_QK; j++)
                    s += (int64_t)(orc_q4_nibble(qs, j) - 8) * qa[j];
                acc += (double)s * (double)orc_fp16_to_fp32(wd[r * kb + b])
                                 * (double)orc_fp16_to_fp32(ad[i * kb + b]);
            }
            y[i * n + r] = acc;
        }
}

/* Per-output sum of |sumi * dw * da| in double: the scale of the f32
 * rounding-error bound used by the parity tolerance. */
void orc_gemm_q4_0_q8_0_absterms(const uint8_t *wq, const uint16_t *wd,
                                 const int8_t *aq, const uint16_t *ad,
                                 int64_t m, int64_t n, int64_t k, double *y)
{
    int64_t kb = k / ORC_QK;
    for (int64_t i = 0; i < m; i++)
        for (int64_t r = 0; r < n; r++) {
            double acc = 0.0;
            for (int64_t b = 0; b < kb; b++) {
                const uint8_t *qs = wq + r * (k / 2) + b * (ORC_QK / 2);
                const int8_t *qa = aq + i * k + b * ORC_QK;
                int64_t s = 0;
                for (int j = 0; j < ORC_QK; j++)
                    s += (int64_t)(orc_q4_nibble(qs, j) - 8) * qa[j];
                acc += fabs((double)s * (double)orc_fp16_to_fp32(wd[r * kb + b])
                                      * (double)orc_fp16_to_fp32(ad[i * kb + b]));
            }
            y[i * n + r] = acc;
        }
}

/* ---------------------------------------------------------------------- */
/* Q8_0 weights x Q8_0 activations [LCG31] [FUC09], reading R16.  Weights are
 * quantized by orc_quantize_q8_0 like activations; the two planes are the
 * int8 codes w8 [n, k] and the fp16 scales wd [n, k/32]. */

/* Per-block integer dot: sumi[i, r, b] = sum_j q_w * q_a. */
void orc_block_sums_q8_0_q8_0(const int8_t *w8, const int8_t *aq,
                              int64_t m, int64_t n, int64_t k, int32_t *sumi)
{
    int64_t kb = k / ORC_QK;
    for (int64_t i = 0; i < m; i++)
        for (int64_t r = 0; r < n; r++)
            for (int64_t b = 0; b < kb; b++) {
                const int8_t *qw = w8 + r * k + b * ORC_QK;
                const int8_t *qa = aq + i * k + b * ORC_QK;
                int32_t s = 0;
                for (int j = 0; j < ORC_QK; j++)
                    s += (int32_t)qw[j] * (int32_t)qa[j];
                sumi[(i * n + r) * kb + b] = s;
            }
}

/* The f32 product, reading R9: blocks ascending, acc = fma((float)sumi,
 * dw*da, acc), dw*da exact in f32. */
void orc_gemm_q8_0_q8_0(const int8_t *w8, const uint16_t *wd,
                        const int8_t *aq, const uint16_t *ad,
                        int64_t m, int64_t n, int64_t k, float *y)
{
    int64_t kb = k / ORC_QK;
    for (int64_t i = 0; i < m; i++)
        for (int64_t r = 0; r < n; r++) {
            float acc = 0.0f;
            for (int64_t b = 0; b < kb; b++) {
                const int8_t *qw = w8 + r * k + b * ORC_QK;
                const int8_t *qa = aq + i * k + b * ORC_QK;
                int32_t s = 0;
                for (int j = 0; j < ORC_QK; j++)
                    s += (int32_t)qw[j] * (int32_t)qa[j];
                float scale = orc_fp16_to_fp32(wd[r * kb + b]) * orc_fp16_to_fp32(ad[i * kb + b]);
                acc = fmaf((float)s, scale, acc);
            }
            y[i * n + r] = acc;
        }
}

/* Double-precision product (|sumi| <= 32*127*127 < 2^19, so each term
 * sumi*dw*da is exact in double) and the per-output sum of |terms|, as for
 * Q4_0. */
void orc_gemm_q8_0_q8_0_f64(const int8_t *w8, const uint16_t *wd,
                            const int8_t *aq, const uint16_t *ad,
                            int64_t m, int64_t n, int64_t k, double *y, double *absterms)
{
    int64_t kb = k / ORC_QK;
    for (int64_t i = 0; i < m; i++)
        for (int64_t r = 0; r < n; r++) {
            double acc = 0.0, abs_acc = 0.0;
            for (int64_t b = 0; b < kb; b++) {
                const int8_t *qw = w8 + r * k + b * ORC_QK;
                const int8_t *qa = aq + i * k + b * ORC_QK;
                int64_t s = 0;
                for (int j = 0; j < ORC_QK; j++)
                    s += (int64_t)qw[j] * qa[j];
                double t = (double)s * (double)orc_fp16_to_fp32(wd[r * kb + b])
                                     * (double)orc_fp16_to_fp32(ad[i * kb + b]);
                acc += t;
                abs_acc += fabs(t);
            }
            y[i * n + r] = acc;
            absterms[i * n + r] = abs_acc;
        }
}

/* ---------------------------------------------------------------------- */
/* Load-time repack of Q4_0 nibbles into the GEMM's tile order, reading R18
 * (Fucina reference, section 9.7: weights packed once at load time into the
 * kernel's interleaved layout).  wr holds ceil(n/128) * ceil(k/64) tiles of
 * 4096 bytes. */
static int64_t orc_repack_offset(int64_t n_tiles_k, int64_t r, int64_t b, int e, int *shift)
{
    int64_t g = r / 128, rr = r % 128, j = b / 2;
    int blk = (int)(b % 2);
    int64_t unit = 2 * rr + blk;
    int c = e / 8, i = (e % 8) / 2, h = e % 2;
    int bit = 4 * i + 16 * h;        /* bit inside word c */
    *shift = bit % 8;
    return (g * n_tiles_k + j) * 4096 + unit * 16 + c * 4 + bit / 8;
}

void orc_repack_q4_0_gemm(const uint8_t *wq, int64_t n, int64_t k, uint8_t *wr)
{
    int64_t kb = k / ORC_QK;
    int64_t tiles_n = (n + 127) / 128, tiles_k = (kb + 1) / 2;
    int64_t bytes = tiles_n * tiles_k * 4096;
    for (int64_t i = 0; i < bytes; i++) wr[i] = 0x88;  /* nibble 8 everywhere */
    for (int64_t r = 0; r < n; r++)
        for (int64_t b = 0; b < kb; b++)
            for (int e = 0; e < ORC_QK; e++) {
                int shift;
                int64_t off = orc_repack_offset(tiles_k, r, b, e, &shift);
                int v = orc_q4_nibble(wq + r * (k / 2) + b * (ORC_QK / 2), e);
                wr[off] = (uint8_t)((wr[off] & ~(0x0f << shift)) | (v << shift));
            }
}

/* The inverse, for the round-trip pin: planes wq [n, k/2] from wr. */
void orc_unrepack_q4_0_gemm(const uint8_t *wr, int64_t n, int64_t k, uint8_t *wq)
{
    int64_t kb = k / ORC_QK;
    int64_t tiles_k = (kb + 1) / 2;
    for (int64_t r = 0; r < n; r++)
        for (int64_t b = 0; b < kb; b++) {
            uint8_t *qs = wq + r * (k / 2) + b * (ORC_QK / 2);
            for (int e = 0; e < ORC_QK; e++) {
                int shift;
                int64_t off = orc_repack_offset(tiles_k, r, b, e, &shift);
                int v = (wr[off] >> shift) & 0x0f;
                if (e < ORC_QK / 2)
                    qs[e] = (uint8_t)((qs[e] & 0xf0) | v);
                else
                    qs[e - ORC_QK / 2] = (uint8_t)((qs[e - ORC_QK / 2] & 0x0f) | (v << 4));
            }
        }
}

/* ---------------------------------------------------------------------- */
/* block_q4_0 array-of-structs (18 bytes: fp16 d little-endian, then qs[16])
 * <-> the two planes used everywhere else.  A pure byte shuffle [LCG31]. */
void orc_q4_0_blocks_to_planes(const uint8_t *blocks, int64_t n, int64_t k,
                               uint8_t *wq, uint16_t *wd)
{
    int64_t kb = k / ORC_QK;
    for (int64_t r = 0; r < n; r++)
        for (int64_t b = 0; b < kb; b++) {
            const uint8_t *blk = blocks + (r * kb + b) * 18;
            wd[r * kb + b] = (uint16_t)(blk[0] | (blk[1] << 8));
            for (int j = 0; j < 16; j++)
                wq[r * (k / 2) + b * 16 + j] = blk[2 + j];
        }
}

void orc_q4_0_planes_to_blocks(const uint8_t *wq, const uint16_t *wd,
                               int64_t n, int64_t k, uint8_t *blocks)
{
    int64_t kb = k / ORC_QK;
    for (int64_t r = 0; r < n; r++)
        for (int64_t b = 0; b < kb; b++) {
            uint8_t *blk = blocks + (r * kb + b) * 18;
            blk[0] = (uint8_t)(wd[r * kb + b] & 0xff);
            blk[1] = (uint8_t)(wd[r * kb + b] >> 8);
            for (int j = 0; j < 16; j++)
                blk[2 + j] = wq[r * (k / 2) + b * 16 + j];
        }
}

/* ---------------------------------------------------------------------- */
/* BitNet activation quantization [LOOM], readings R1 R2 R7 R8:
 * per row s = 127/max|x|, q = clamp(round(x*s), -127, 127), asum = sum q. */
void orc_quantize_act_bitnet(const float *x, int64_t m, int64_t k,
                             int8_t *aq, float *act_scale, int32_t *act_sum)
{
    for (int64_t i = 0; i < m; i++) {
        const float *xr = x + i * k;
        float amax = 0.0f;
        for (int64_t j = 0; j < k; j++) {
            float a = fabsf(xr[j]);
            if (a > amax) amax = a;
        }
        float s = 0.0f;
        if (amax != 0.0f) s = 127.0f / amax;
        int32_t sum = 0;
        for (int64_t j = 0; j < k; j++) {
            float q = 0.0f;
            if (s != 0.0f) {
                q = roundf(xr[j] * s);
                if (q > 127.0f) q = 127.0f;
                if (q < -127.0f) q = -127.0f;
            }
            aq[i * k + j] = (int8_t)q;
            sum += (int32_t)q;
        }
        act_scale[i] = s;
        act_sum[i] = sum;
    }
}

/* Pack ternary weights t in {-1, 0, +1} (int8 [n, k]) as code = t + 1,
 * 16 codes per uint32, element i of a word at bits [2i, 2i+1] [LOOM], R5. */
void orc_pack_ternary(const int8_t *t, int64_t n, int64_t k, uint32_t *tw)
{
    int64_t kw = k / 16;
    for (int64_t r = 0; r < n; r++)
        for (int64_t wi = 0; wi < kw; wi++) {
            uint32_t word = 0;
            for (int i = 0; i < 16; i++) {
                uint32_t code = (uint32_t)(t[r * k + wi * 16 + i] + 1);
                word |= code << (2 * i);
            }
            tw[r * kw + wi] = word;
        }
}

/* Ternary dot through the identity [LOOM]: dot = sum(code*q) - sum(q),
 * codes decoded two bits at a time. */
void orc_bitnet_dot(const uint32_t *tw, const int8_t *aq, const int32_t *act_sum,
                    int64_t m, int64_t n, int64_t k, int32_t *dot)
{
    int64_t kw = k / 16;
    for (int64_t i = 0; i < m; i++)
        for (int64_t r = 0; r < n; r++) {
            int32_t acc = 0;
            for (int64_t j = 0; j < k; j++) {
                uint32_t word = tw[r * kw + j / 16];
                int32_t code = (int32_t)((word >> (2 * (j % 16))) & 3u);
                acc += code * (int32_t)aq[i * k + j];
            }
            dot[i * n + r] = acc - act_sum[i];
        }
}

/* BitNet output [LOOM], readings R8 R10: y = (dot * absmean) / scale. */
void orc_bitnet_gemv(const uint32_t *tw, float weight_absmean,
                     const int8_t *aq, const float *act_scale, const int32_t *act_sum,
                     int64_t m, int64_t n, int64_t k, float *y)
{
    int64_t kw = k / 16;
    for (int64_t i = 0; i < m; i++)
        for (int64_t r = 0; r < n; r++) {
            int32_t acc = 0;
            for (int64_t j = 0; j < k; j++) {
                uint32_t word = tw[r * kw + j / 16];
                int32_t code = (int32_t)((word >> (2 * (j % 16))) & 3u);
                acc += code * (int32_t)aq[i * k + j];
            }
            int32_t d = acc - act_sum[i];
            float out = 0.0f;
            if (act_scale[i] != 0.0f)
                out = ((float)d * weight_absmean) / act_scale[i];
            y[i * n + r] = out;
        }
}
