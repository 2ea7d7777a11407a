// Decode-shaped products (m <= 16): Q4_0 x Q8_0 and BitNet ternary GEMV.
//
// Q4_0 x Q8_0 (llama.cpp visual guide, lesson 31 "The CPU backend", section
// "How the quantized dot product works"): per block, sumi = sum_j
// (nibble_j - 8) * q_j exactly in int32, then acc += sumi * (dw * da) in f32.
// On the GPU a warp owns ROWS weight rows; lane l takes blocks l, l+32, ...
// of every row, so each warp-wide 128-bit load reads 512 contiguous bytes of
// one row (coalesced streaming, no reuse, L1 bypassed).  The 16 nibble bytes
// of a block are one uint4; the low nibbles of word i are elements 4i..4i+3
// and the high nibbles elements 16+4i..16+4i+3, which line up with
// activation words i and 4+i, so each block is 8 dp4a (unsigned nibble x
// signed int8) plus the -8 offset applied once per block as -8 * sum(q)
// (computed with dp4a against 0x01010101 and shared by all ROWS rows).  The
// per-lane f32 partials are summed by an xor-shuffle tree.  An optional
// split over k writes f32 partials [S, m, n] to the workspace and a second
// kernel adds them in slice order (deterministic; the prefill page of the
// Fucina reference section 9.9.2 does the same for its split-K).
//
// BitNet (Loom docs, "Plan 9 SIMD Forward", section "BitNet ternary MAD
// kernel"): dot = sum(code * q) - sum(q), exact in int32.  Codes are unpacked
// in registers, four at a time: (word >> 2s) & 0x03030303 holds the codes of
// elements s, s+4, s+8, s+12, and the matching activation bytes are gathered
// with byte permutes, so each 16 weights cost four dp4a.
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "qmm_internal.h"

namespace qmm {
namespace {

// Warps per CTA.  Small CTAs start and finish in finer steps: against 4
// warps, 2 measured 1% faster for the single 4096x4096 GEMV, 2% for the BitNet
// GEMV and the same for the vocabulary GEMV; against 8, 4 was 4.7% faster at
// vocabulary size.
constexpr int kWarps = 2;
// warps per CTA of the grouped GEMV (2 at 4 rows: 5178 against 5124 GB/s for 4)
constexpr int kGroupedWarps = 2;
constexpr int kUnroll = 4;       // blocks (per lane, per row) loaded before use

__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// unsigned bytes of a times signed bytes of b, summed into c
__device__ __forceinline__ int dp4a_us(unsigned a, int b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ float h2f(unsigned short h) {
    return __half2float(__ushort_as_half(h));
}

// Sum of a block's 32 int8 activation codes (a0: codes 0-15, a1: 16-31).
__device__ __forceinline__ int block_code_sum(const int4 &a0, const int4 &a1) {
    int s = dp4a_us(0x01010101u, a0.x, 0);
    s = dp4a_us(0x01010101u, a0.y, s);
    s = dp4a_us(0x01010101u, a0.z, s);
    s = dp4a_us(0x01010101u, a0.w, s);
    s = dp4a_us(0x01010101u, a1.x, s);
    s = dp4a_us(0x01010101u, a1.y, s);
    s = dp4a_us(0x01010101u, a1.z, s);
    return dp4a_us(0x01010101u, a1.w, s);
}

// s + the dot of a Q4_0 block's raw nibbles (16 bytes: element j in the low
// nibble of byte j, element j + 16 in its high nibble) with its activation
// codes; with s = -8 * block_code_sum this is the block sum of (v - 8) * q.
__device__ __forceinline__ int q4_block_dot(const uint4 &w, const int4 &a0, const int4 &a1, int s) {
    s = dp4a_us(w.x & 0x0F0F0F0Fu, a0.x, s);
    s = dp4a_us(w.y & 0x0F0F0F0Fu, a0.y, s);
    s = dp4a_us(w.z & 0x0F0F0F0Fu, a0.z, s);
    s = dp4a_us(w.w & 0x0F0F0F0Fu, a0.w, s);
    s = dp4a_us((w.x >> 4) & 0x0F0F0F0Fu, a1.x, s);
    s = dp4a_us((w.y >> 4) & 0x0F0F0F0Fu, a1.y, s);
    s = dp4a_us((w.z >> 4) & 0x0F0F0F0Fu, a1.z, s);
    return dp4a_us((w.w >> 4) & 0x0F0F0F0Fu, a1.w, s);
}

// ---------------------------------------------------------------------------
// Q4_0 x Q8_0

// The weight blocks bb + 32 u (u < kUnroll) of rows row0 .. row0 + ROWS - 1,
// up to block kb1: nibbles with streaming 16-byte loads, scales through the
// read-only path (none when emitting block sums).  Blocks past the end read
// as nibbles 8 (value 0) with scale 0.
template <int ROWS, bool EMIT>
__device__ __forceinline__ void load_q4_batch(uint4 (&wv)[kUnroll][ROWS],
                                              unsigned short (&dwv)[kUnroll][ROWS],
                                              const uint8_t *__restrict__ wq,
                                              const unsigned short *__restrict__ wd, int64_t row0,
                                              int64_t n, int64_t kb, int64_t kb1, int64_t bb) {
    const int64_t wrow = kb * 16;  // bytes per weight row
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int64_t b = bb + 32 * u;
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const int64_t row = row0 + r;
            if (b < kb1 && row < n) {
                wv[u][r] = ld_stream_v4(wq + row * wrow + b * 16);
                dwv[u][r] = EMIT ? (unsigned short)0 : __ldg(wd + row * kb + b);
            } else {
                wv[u][r] = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
                dwv[u][r] = 0;
            }
        }
    }
}

// One CTA's share of the GEMV: row group `group` (WARPS * ROWS rows), k
// slice `slice`.  PDL: the warp loads its first batch of weight blocks and
// scales (model parameters, never written by the preceding kernels), then
// waits for the predecessor (the activation quantizer) before it reads aq/ad
// or writes out.
template <int MT, int ROWS, bool EMIT, bool PDL, int WARPS = kWarps>
__device__ __forceinline__ void gemv_cta(const uint8_t *__restrict__ wq,
                                         const unsigned short *__restrict__ wd,
                                         const int8_t *__restrict__ aq,
                                         const unsigned short *__restrict__ ad,
                                         float *__restrict__ out, int32_t *__restrict__ sumi,
                                         int m, int64_t n, int64_t k, int64_t kb_per_split,
                                         int64_t group, int64_t slice) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t kb = k / kQK;
    const int64_t row0 = (group * WARPS + warp) * ROWS;
    if (row0 >= n) return;
    const int64_t kb0 = slice * kb_per_split;
    const int64_t kb1 = min(kb, kb0 + kb_per_split);

    float acc[ROWS][MT];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[r][t] = 0.0f;

    uint4 wv[kUnroll][ROWS];
    unsigned short dwv[kUnroll][ROWS];
    auto load_batch = [&](int64_t bb) {
        load_q4_batch<ROWS, EMIT>(wv, dwv, wq, wd, row0, n, kb, kb1, bb);
    };
    const int64_t first = kb0 + lane;
    if (PDL) {
        load_batch(first);
        pdl_wait();
        pdl_launch_dependents();
    }
    for (int64_t bb = first; bb < kb1; bb += 32 * kUnroll) {
        if (!PDL || bb != first) load_batch(bb);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t b = bb + 32 * u;
            if (b >= kb1) break;
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                if (t >= m) break;
                const int4 a0 = __ldg(reinterpret_cast<const int4 *>(aq + t * k + b * kQK));
                const int4 a1 = __ldg(reinterpret_cast<const int4 *>(aq + t * k + b * kQK + 16));
                const float da = EMIT ? 0.0f : h2f(__ldg(ad + t * kb + b));
                const int asum = block_code_sum(a0, a1);
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const int s = q4_block_dot(wv[u][r], a0, a1, -8 * asum);
                    if (EMIT) {
                        if (row0 + r < n) sumi[((int64_t)t * n + row0 + r) * kb + b] = s;
                    } else {
                        const float sc = __fmul_rn(h2f(dwv[u][r]), da);
                        acc[r][t] = fmaf((float)s, sc, acc[r][t]);
                    }
                }
            }
        }
    }
    if constexpr (!EMIT) {  // the emitting variant stores block sums only
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                float v = acc[r][t];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                acc[r][t] = v;
            }
        if (lane == 0) {
            float *dst = out + slice * m * n;  // split slice (0 when unsplit)
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                if (row0 + r >= n) break;
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    if (t >= m) break;
                    dst[(int64_t)t * n + row0 + r] = acc[r][t];
                }
            }
        }
    }
}

template <int MT, int ROWS, bool EMIT, bool PDL>
__global__ void __launch_bounds__(kWarps * 32)
gemv_q4_0_q8_0_kernel(const uint8_t *__restrict__ wq, const unsigned short *__restrict__ wd,
                      const int8_t *__restrict__ aq, const unsigned short *__restrict__ ad,
                      float *__restrict__ out, int32_t *__restrict__ sumi, int m, int64_t n,
                      int64_t k, int64_t kb_per_split) {
    gemv_cta<MT, ROWS, EMIT, PDL>(wq, wd, aq, ad, out, sumi, m, n, k, kb_per_split, blockIdx.x,
                                  blockIdx.y);
}

// Several independent GEMVs in one launch: CTA c serves the problem whose
// range of CTAs holds c (the table is a kernel parameter, read in place).
template <int MT, int ROWS, bool PDL>
__global__ void __launch_bounds__(kGroupedWarps * 32)
gemv_grouped_kernel(const __grid_constant__ LinearGroup tab) {
    int p = 0;
    while (p + 1 < tab.count && (int64_t)blockIdx.x >= tab.cta_end[p]) ++p;
    const int64_t group = (int64_t)blockIdx.x - (p ? tab.cta_end[p - 1] : 0);
    const LinearProblem &P = tab.p[p];
    gemv_cta<MT, ROWS, false, PDL, kGroupedWarps>(P.wq, reinterpret_cast<const unsigned short *>(P.wd),
                                                  P.aq, reinterpret_cast<const unsigned short *>(P.ad),
                                                  P.y, nullptr, tab.m, P.n, P.k, P.k / kQK, group, 0);
}

// One token (m = 1), the activation slice staged once per CTA.  At m = 1 a
// row's int8 activations (k bytes) outweigh its weights (k/2 + k/16 bytes),
// so warps that each read them from L2 (gemv_cta) move more bytes between
// L2 and the SMs than the weight stream; here the CTA's threads read the
// slice once into shared memory as one 48-byte record per block, {codes
// 0-15, codes 16-31, {da as f32, -8 * (sum of the 32 codes), 0, 0}}, whose
// 16-byte parts lanes reading consecutive blocks find in distinct banks.
// The block sum, the scale product and the accumulation are gemv_cta's, in
// the same lane order (lane l takes blocks l, l + 32, ...), so y has the
// same bits.  The weight words of the first batch are requested before the
// staging (and, with PDL, before the wait for the quantizer).  EMIT stores
// the block sums instead (sumi [n, k/32]).
template <int ROWS, bool PDL, int WARPS, bool EMIT = false>
__device__ __forceinline__ void gemv_cta_m1_staged(const uint8_t *__restrict__ wq,
                                                   const unsigned short *__restrict__ wd,
                                                   const int8_t *__restrict__ aq,
                                                   const unsigned short *__restrict__ ad,
                                                   float *__restrict__ out,
                                                   int32_t *__restrict__ sumi, int64_t n,
                                                   int64_t k, int64_t kb_per_split,
                                                   int64_t group, int64_t slice) {
    extern __shared__ uint4 stg[];  // 3 x 16 bytes per block of the slice
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t kb = k / kQK;
    const int64_t row0 = (group * WARPS + warp) * ROWS;
    const int64_t kb0 = slice * kb_per_split;
    const int64_t kb1 = min(kb, kb0 + kb_per_split);
    float acc[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) acc[r] = 0.0f;
    uint4 wv[kUnroll][ROWS];
    unsigned short dwv[kUnroll][ROWS];
    auto load_batch = [&](int64_t bb) {
        load_q4_batch<ROWS, EMIT>(wv, dwv, wq, wd, row0, n, kb, kb1, bb);
    };
    const int64_t first = kb0 + lane;
    load_batch(first);
    if (PDL) {
        pdl_wait();
        pdl_launch_dependents();
    }
    for (int64_t b = kb0 + threadIdx.x; b < kb1; b += WARPS * 32) {
        const int4 a0 = __ldg(reinterpret_cast<const int4 *>(aq + b * kQK));
        const int4 a1 = __ldg(reinterpret_cast<const int4 *>(aq + b * kQK + 16));
        const float da = EMIT ? 0.0f : h2f(__ldg(ad + b));
        const int asum = block_code_sum(a0, a1);
        uint4 *rec = stg + 3 * (b - kb0);
        rec[0] = make_uint4(a0.x, a0.y, a0.z, a0.w);
        rec[1] = make_uint4(a1.x, a1.y, a1.z, a1.w);
        rec[2] = make_uint4(__float_as_uint(da), (uint32_t)(-8 * asum), 0u, 0u);
    }
    __syncthreads();
    if (row0 >= n) return;
    for (int64_t bb = first; bb < kb1; bb += 32 * kUnroll) {
        if (bb != first) load_batch(bb);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t b = bb + 32 * u;
            if (b >= kb1) break;
            const uint4 *rec = stg + 3 * (b - kb0);
            const uint4 r0 = rec[0], r1 = rec[1], e = rec[2];
            const int4 a0 = make_int4((int)r0.x, (int)r0.y, (int)r0.z, (int)r0.w);
            const int4 a1 = make_int4((int)r1.x, (int)r1.y, (int)r1.z, (int)r1.w);
            const float da = __uint_as_float(e.x);
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                const int s = q4_block_dot(wv[u][r], a0, a1, (int)e.y);
                if (EMIT) {
                    if (row0 + r < n) sumi[(row0 + r) * kb + b] = s;
                } else {
                    const float sc = __fmul_rn(h2f(dwv[u][r]), da);
                    acc[r] = fmaf((float)s, sc, acc[r]);
                }
            }
        }
    }
    if constexpr (!EMIT) {  // the emitting variant stores block sums only
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            float v = acc[r];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            acc[r] = v;
        }
        if (lane == 0) {
            float *dst = out + slice * n;  // split slice (0 when unsplit)
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                if (row0 + r >= n) break;
                dst[row0 + r] = acc[r];
            }
        }
    }
}

// CTA shapes of the staged one-token GEMVs (rows per warp, warps per CTA).
// Grouped (layer set): 2 x 4, 5477 GB/s against 5386 for the per-warp reads
// (2 x 8: 5412, 4 x 4: 5344, 3 x 4: 5330, 4 x 8: 5166, 4 x 2: 5098, 2 x 2:
// 4661, 1 x 8: 4560, 1 x 4: 4490, 1 x 16: 4187, 2 x 16: 3591).
// Single matrix: each CTA stages the row once however few rows it has, so
// the staging pays off with 8-row CTAs when there are many rows (vocabulary,
// 128256 x 4096: 40.5 against 41.3 us per-warp, 52.5 with 4-row CTAs), and
// 4-row CTAs are best for a few thousand rows (4096 x 4096: 3.69 against
// 3.75 per-warp, 3.82 with 8-row CTAs).
constexpr int kM1GroupRows = 2, kM1GroupWarps = 4;
constexpr int kM1Warps = 4;
// The grouped kernel's registers are capped so that six 4-warp CTAs fit an
// SM (80 registers, no spills; left free, the 2-row form took 96 and five
// CTAs): more weight bytes in flight per SM. Layer set: 5619 against 5437
// GB/s; seven CTAs (72 registers, spills) 5342, eight (64) 4285.  The same
// cap on the single-matrix kernel let its 1-row form grow from 56 to 79
// registers, and 4096 x 4096 took two waves: 4.22 against 3.70 us.
constexpr int kM1CtasPerSm = 6;
constexpr int64_t kM1ManyRows = 16384;  // from here on 2 rows per warp, else 1

template <int ROWS, bool PDL, int WARPS, bool EMIT>
__global__ void __launch_bounds__(WARPS * 32)
gemv_m1_staged_kernel(const uint8_t *__restrict__ wq, const unsigned short *__restrict__ wd,
                      const int8_t *__restrict__ aq, const unsigned short *__restrict__ ad,
                      float *__restrict__ out, int32_t *__restrict__ sumi, int64_t n, int64_t k,
                      int64_t kb_per_split) {
    gemv_cta_m1_staged<ROWS, PDL, WARPS, EMIT>(wq, wd, aq, ad, out, sumi, n, k, kb_per_split,
                                               blockIdx.x, blockIdx.y);
}

template <int ROWS, bool PDL, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, kM1CtasPerSm)
gemv_grouped_m1_staged_kernel(const __grid_constant__ LinearGroup tab) {
    int p = 0;
    while (p + 1 < tab.count && (int64_t)blockIdx.x >= tab.cta_end[p]) ++p;
    const int64_t group = (int64_t)blockIdx.x - (p ? tab.cta_end[p - 1] : 0);
    const LinearProblem &P = tab.p[p];
    gemv_cta_m1_staged<ROWS, PDL, WARPS>(P.wq, reinterpret_cast<const unsigned short *>(P.wd), P.aq,
                                         reinterpret_cast<const unsigned short *>(P.ad), P.y,
                                         nullptr, P.n, P.k, P.k / kQK, group, 0);
}

// y[i] = sum over slices s = 0..S-1 of partials[s][i], in that order.
template <bool PDL>
__global__ void splitk_reduce_kernel(const float *__restrict__ partials, float *__restrict__ y,
                                     int64_t count, int splits) {
    if (PDL) {
        pdl_launch_dependents();
        pdl_wait();
    }
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= count) return;
    float v = partials[i];
    for (int s = 1; s < splits; ++s) v += partials[(int64_t)s * count + i];
    y[i] = v;
}

template <int MT, int ROWS>
cudaError_t launch_q4(const uint8_t *wq, const uint16_t *wd, const int8_t *aq, const uint16_t *ad,
                      float *out, int32_t *sumi, int64_t m, int64_t n, int64_t k, int split,
                      cudaStream_t s, bool pdl) {
    const int64_t kb = k / kQK;
    const int64_t per = (kb + split - 1) / split;
    const int64_t rows_per_cta = (int64_t)kWarps * ROWS;
    dim3 grid((unsigned)((n + rows_per_cta - 1) / rows_per_cta), (unsigned)split);
    const auto *wdp = reinterpret_cast<const unsigned short *>(wd);
    const auto *adp = reinterpret_cast<const unsigned short *>(ad);
    if (pdl)
        return launch_kernel(gemv_q4_0_q8_0_kernel<MT, ROWS, false, true>, grid, dim3(kWarps * 32),
                             0, s, true, wq, wdp, aq, adp, out, sumi, (int)m, n, k, per);
    if (sumi)
        gemv_q4_0_q8_0_kernel<MT, ROWS, true, false><<<grid, kWarps * 32, 0, s>>>(
            wq, wdp, aq, adp, out, sumi, (int)m, n, k, per);
    else
        gemv_q4_0_q8_0_kernel<MT, ROWS, false, false><<<grid, kWarps * 32, 0, s>>>(
            wq, wdp, aq, adp, out, sumi, (int)m, n, k, per);
    return cudaPeekAtLastError();
}

// ---------------------------------------------------------------------------
// BitNet ternary

// Gather byte s of each of the four words into one word:
// out_s = (a.byte s, b.byte s, c.byte s, d.byte s).
__device__ __forceinline__ void transpose4x4(int a, int b, int c, int d, int out[4]) {
    const int t0 = __byte_perm(a, b, 0x5140);  // a0 b0 a1 b1
    const int t1 = __byte_perm(c, d, 0x5140);  // c0 d0 c1 d1
    const int t2 = __byte_perm(a, b, 0x7362);  // a2 b2 a3 b3
    const int t3 = __byte_perm(c, d, 0x7362);  // c2 d2 c3 d3
    out[0] = __byte_perm(t0, t1, 0x5410);      // a0 b0 c0 d0
    out[1] = __byte_perm(t0, t1, 0x7632);      // a1 b1 c1 d1
    out[2] = __byte_perm(t2, t3, 0x5410);
    out[3] = __byte_perm(t2, t3, 0x7632);
}

// 16 codes of `word` against 16 activations (int4 a = elements 0..15).
__device__ __forceinline__ int ternary_dot16(uint32_t word, const int act_t[4], int acc) {
#pragma unroll
    for (int s = 0; s < 4; ++s) acc = dp4a_us((word >> (2 * s)) & 0x03030303u, act_t[s], acc);
    return acc;
}

// PDL: the warp loads its first weight words (model parameters, never
// written by the preceding kernels), then waits for the predecessor (the
// activation quantizer) before it reads aq, scale and asum or writes y.
template <int MT, int ROWS, bool VEC, bool EMIT, bool PDL>
__global__ void __launch_bounds__(kWarps * 32)
bitnet_gemv_kernel(const uint32_t *__restrict__ w, float absmean, const int8_t *__restrict__ aq,
                   const float *__restrict__ scale, const int32_t *__restrict__ asum,
                   float *__restrict__ y, int32_t *__restrict__ dot_out, int m, int64_t n,
                   int64_t k) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t row0 = ((int64_t)blockIdx.x * kWarps + warp) * ROWS;
    if (row0 >= n) return;
    const int64_t kw = k / 16;  // words per row
    int acc[ROWS][MT];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[r][t] = 0;

    if (VEC) {
        // 4 words (64 weights) per lane per step, 128-bit loads
        const int64_t kv = kw / 4;
        uint4 wv[kUnroll][ROWS];
        auto load_batch = [&](int64_t jj) {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t j = jj + 32 * u;
#pragma unroll
                for (int r = 0; r < ROWS; ++r)
                    wv[u][r] = (j < kv && row0 + r < n)
                                   ? ld_stream_v4(w + (row0 + r) * kw + j * 4)
                                   : make_uint4(0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u);
            }
        };
        if (PDL) {
            load_batch(lane);
            pdl_wait();
            pdl_launch_dependents();
        }
        for (int64_t jj = lane; jj < kv; jj += 32 * kUnroll) {
            if (!PDL || jj != lane) load_batch(jj);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t j = jj + 32 * u;
                if (j >= kv) break;
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    if (t >= m) break;
                    const int4 *ap = reinterpret_cast<const int4 *>(aq + t * k + j * 64);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int4 a = __ldg(ap + q);
                        int at[4];
                        transpose4x4(a.x, a.y, a.z, a.w, at);
#pragma unroll
                        for (int r = 0; r < ROWS; ++r) {
                            const uint32_t word = q == 0 ? wv[u][r].x
                                                : q == 1 ? wv[u][r].y
                                                : q == 2 ? wv[u][r].z
                                                         : wv[u][r].w;
                            acc[r][t] = ternary_dot16(word, at, acc[r][t]);
                        }
                    }
                }
            }
        }
    } else {
        if (PDL) {
            pdl_wait();
            pdl_launch_dependents();
        }
        // one word (16 weights) per lane per step
        for (int64_t j = lane; j < kw; j += 32) {
            uint32_t wv[ROWS];
#pragma unroll
            for (int r = 0; r < ROWS; ++r) wv[r] = (row0 + r < n) ? __ldg(w + (row0 + r) * kw + j) : 0x55555555u;
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                if (t >= m) break;
                const int *ap = reinterpret_cast<const int *>(aq + t * k + j * 16);
                int at[4];
                transpose4x4(__ldg(ap), __ldg(ap + 1), __ldg(ap + 2), __ldg(ap + 3), at);
#pragma unroll
                for (int r = 0; r < ROWS; ++r) acc[r][t] = ternary_dot16(wv[r], at, acc[r][t]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            int v = acc[r][t];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            acc[r][t] = v;
        }
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            if (row0 + r >= n) break;
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                if (t >= m) break;
                const int d = acc[r][t] - asum[t];
                if (EMIT) {
                    dot_out[(int64_t)t * n + row0 + r] = d;
                } else {
                    const float st = scale[t];
                    y[(int64_t)t * n + row0 + r] =
                        st != 0.0f ? __fdiv_rn(__fmul_rn((float)d, absmean), st) : 0.0f;
                }
            }
        }
    }
}

// The ternary GEMV for one token (m = 1, k % 64 == 0): the same dot and
// output rule as bitnet_gemv_kernel, but the activation row is read from L2
// once per CTA into shared memory, already transposed for the ternary dot
// (word i, 16 elements, as the four ints t_s of ternary_dot16 at slot
// [i % 4][i / 4], so that lanes reading consecutive 64-element chunks read
// consecutive 16-byte slots), instead of once per warp: with one row per
// warp the warps of a CTA share one copy.  The weight words are requested
// before the row (and, with PDL, before the wait for the predecessor).
template <int ROWS, int WARPS, bool EMIT, bool PDL>
__global__ void __launch_bounds__(WARPS * 32, 6)
bitnet_gemv_m1_kernel(const uint32_t *__restrict__ w, float absmean, const int8_t *__restrict__ aq,
                      const float *__restrict__ scale, const int32_t *__restrict__ asum,
                      float *__restrict__ y, int32_t *__restrict__ dot_out, int64_t n, int64_t k) {
    extern __shared__ int4 act_t[];  // k / 16 slots
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t row0 = ((int64_t)blockIdx.x * WARPS + warp) * ROWS;
    const int64_t kw = k / 16, kv = k / 64;
    // two 64-element chunks per lane and row in flight: at 40 registers six
    // 8-warp CTAs fit an SM, so the 864 CTAs of a 6912-row matrix run in one
    // wave (four chunks: 48 registers, five CTAs, 4.15 against 3.35 us)
    constexpr int kU = 2;
    uint4 wv[kU][ROWS];
    auto load_batch = [&](int64_t jj) {
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t j = jj + 32 * u;
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
                wv[u][r] = (j < kv && row0 + r < n)
                               ? ld_stream_v4(w + (row0 + r) * kw + j * 4)
                               : make_uint4(0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u);
        }
    };
    load_batch(lane);
    if (PDL) {
        pdl_wait();
        pdl_launch_dependents();
    }
    for (int64_t i = threadIdx.x; i < kw; i += WARPS * 32) {
        const int4 a = __ldg(reinterpret_cast<const int4 *>(aq) + i);
        int at[4];
        transpose4x4(a.x, a.y, a.z, a.w, at);
        act_t[(i & 3) * kv + (i >> 2)] = make_int4(at[0], at[1], at[2], at[3]);
    }
    __syncthreads();
    if (row0 >= n) return;
    int acc[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) acc[r] = 0;
    for (int64_t jj = lane; jj < kv; jj += 32 * kU) {
        if (jj != lane) load_batch(jj);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t j = jj + 32 * u;
            if (j >= kv) break;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int4 t = act_t[q * kv + j];
                const int at[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const uint32_t word = q == 0 ? wv[u][r].x
                                        : q == 1 ? wv[u][r].y
                                        : q == 2 ? wv[u][r].z
                                                 : wv[u][r].w;
                    acc[r] = ternary_dot16(word, at, acc[r]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        int v = acc[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        acc[r] = v;
    }
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            if (row0 + r >= n) break;
            const int d = acc[r] - asum[0];
            if (EMIT) {
                dot_out[row0 + r] = d;
            } else {
                const float st = scale[0];
                y[row0 + r] = st != 0.0f ? __fdiv_rn(__fmul_rn((float)d, absmean), st) : 0.0f;
            }
        }
    }
}

// The BitNet decode step for one token (m = 1, k % 64 == 0) in one kernel.
// Every CTA quantizes the activation row itself: the per-row scale needs
// the whole row's maximum, and the row (k floats, read from L2) is small
// next to the CTA's weights, so this costs each CTA well under a
// microsecond and takes the separate quantizer launch, and its latency, out
// of the step.  The operations are the quantizer's (max of |x|, s =
// 127 / max, q = clamp(round(x * s), -127, 127), sum q), so codes, scale, sum
// and y are bit for bit those of the two-kernel step; CTA 0 also writes them
// out.  The codes go to shared memory already transposed for the ternary
// dot: for 16-element group j, int t_s = bytes of elements 16j + s, s+4, s+8,
// s+12, stored at [s][j] so that a warp's 16-byte reads are contiguous.
// PDL: the weight words are loaded before the wait, x after it.
template <int ROWS, int WARPS, bool PDL>
__global__ void __launch_bounds__(WARPS * 32)
bitnet_linear_m1_kernel(const uint32_t *__restrict__ w, float absmean, const float *__restrict__ x,
                        int8_t *__restrict__ aq, float *__restrict__ scale_out,
                        int32_t *__restrict__ sum_out, float *__restrict__ y, int64_t n, int64_t k) {
    extern __shared__ int4 s_act[];  // [4 byte planes][k / 64 vectors], 16 bytes each
    __shared__ float s_max[WARPS];
    __shared__ int s_sum[WARPS];
    constexpr int kThreads = WARPS * 32;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t row0 = ((int64_t)blockIdx.x * WARPS + warp) * ROWS;
    const int64_t kw = k / 16, kv = k / 64;

    uint4 wv[kUnroll][ROWS];
    auto load_batch = [&](int64_t jj) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t j = jj + 32 * u;
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
                wv[u][r] = (j < kv && row0 + r < n)
                               ? ld_stream_v4(w + (row0 + r) * kw + j * 4)
                               : make_uint4(0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u);
        }
    };
    load_batch(lane);
    if (PDL) {
        pdl_wait();
        pdl_launch_dependents();
    }
    // the row's maximum magnitude.  With at most one 16-element group per
    // thread (k <= 16 * threads) each thread reads its group once and keeps
    // it in registers for the quantization below, so x crosses from L2 once
    // instead of twice (the maximum is the same whatever the order)
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    const bool one_group = kw <= kThreads;
    float4 xg[4] = {};
    float amax = 0.0f;
    if (one_group) {
        if (threadIdx.x < kw) {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                xg[h] = __ldg(x4 + threadIdx.x * 4 + h);
                const float4 v = xg[h];
                amax = fmaxf(fmaxf(amax, fmaxf(fabsf(v.x), fabsf(v.y))), fmaxf(fabsf(v.z), fabsf(v.w)));
            }
        }
    } else {
        for (int64_t i = threadIdx.x; i < k / 4; i += kThreads) {
            const float4 v = __ldg(x4 + i);
            amax = fmaxf(fmaxf(amax, fmaxf(fabsf(v.x), fabsf(v.y))), fmaxf(fabsf(v.z), fabsf(v.w)));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) s_max[warp] = amax;
    __syncthreads();
    float mx = s_max[0];
#pragma unroll
    for (int i = 1; i < WARPS; ++i) mx = fmaxf(mx, s_max[i]);
    const float sc = (mx != 0.0f) ? __fdiv_rn(127.0f, mx) : 0.0f;
    // codes of 16-element groups: natural order to aq (CTA 0), transposed to
    // shared memory
    int part = 0;
    for (int64_t gi = threadIdx.x; gi < kw; gi += kThreads) {
        uint32_t q4[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const float4 v = one_group ? xg[h] : __ldg(x4 + gi * 4 + h);
            const float f[4] = {v.x, v.y, v.z, v.w};
            uint32_t packed = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float q = 0.0f;
                if (sc != 0.0f) q = fminf(fmaxf(roundf(__fmul_rn(f[e], sc)), -127.0f), 127.0f);
                const int qi = (int)q;
                part += qi;
                packed |= (uint32_t)(qi & 0xff) << (8 * e);
            }
            q4[h] = packed;
        }
        if (blockIdx.x == 0)
            reinterpret_cast<int4 *>(aq)[gi] = make_int4((int)q4[0], (int)q4[1], (int)q4[2], (int)q4[3]);
        int t[4];
        transpose4x4((int)q4[0], (int)q4[1], (int)q4[2], (int)q4[3], t);
        // group gi is word (gi % 4) of vector gi / 4; plane s holds t_s
        int *plane = reinterpret_cast<int *>(s_act);
#pragma unroll
        for (int sp = 0; sp < 4; ++sp) plane[(sp * kv + gi / 4) * 4 + (gi & 3)] = t[sp];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) s_sum[warp] = part;
    __syncthreads();
    int asum = 0;
#pragma unroll
    for (int i = 0; i < WARPS; ++i) asum += s_sum[i];
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        scale_out[0] = sc;
        sum_out[0] = asum;
    }
    if (row0 >= n) return;
    int acc[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) acc[r] = 0;
    for (int64_t jj = lane; jj < kv; jj += 32 * kUnroll) {
        if (jj != lane) load_batch(jj);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t j = jj + 32 * u;
            if (j >= kv) break;
            // the activations of vector j: planes s = 0..3, word q = 0..3
            int4 ta[4];
#pragma unroll
            for (int sp = 0; sp < 4; ++sp) ta[sp] = s_act[sp * kv + j];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int at[4] = {(&ta[0].x)[q], (&ta[1].x)[q], (&ta[2].x)[q], (&ta[3].x)[q]};
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const uint32_t word = q == 0 ? wv[u][r].x
                                        : q == 1 ? wv[u][r].y
                                        : q == 2 ? wv[u][r].z
                                                 : wv[u][r].w;
                    acc[r] = ternary_dot16(word, at, acc[r]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        int v = acc[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        acc[r] = v;
    }
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            if (row0 + r >= n) break;
            const int d = acc[r] - asum;
            y[row0 + r] = sc != 0.0f ? __fdiv_rn(__fmul_rn((float)d, absmean), sc) : 0.0f;
        }
    }
}

template <int MT, int ROWS>
cudaError_t launch_bitnet(const uint32_t *w, float absmean, const int8_t *aq, const float *scale,
                          const int32_t *asum, float *y, int32_t *dot, int64_t m, int64_t n,
                          int64_t k, cudaStream_t s, bool pdl) {
    const int64_t rows_per_cta = (int64_t)kWarps * ROWS;
    const dim3 grid((unsigned)((n + rows_per_cta - 1) / rows_per_cta));
    const bool vec = (k % 64) == 0;
    if (dot) {
        if (vec)
            bitnet_gemv_kernel<MT, ROWS, true, true, false><<<grid, kWarps * 32, 0, s>>>(
                w, absmean, aq, scale, asum, y, dot, (int)m, n, k);
        else
            bitnet_gemv_kernel<MT, ROWS, false, true, false><<<grid, kWarps * 32, 0, s>>>(
                w, absmean, aq, scale, asum, y, dot, (int)m, n, k);
        return cudaPeekAtLastError();
    }
    if (pdl)
        return vec ? launch_kernel(bitnet_gemv_kernel<MT, ROWS, true, false, true>, grid,
                                   dim3(kWarps * 32), 0, s, true, w, absmean, aq, scale, asum, y,
                                   dot, (int)m, n, k)
                   : launch_kernel(bitnet_gemv_kernel<MT, ROWS, false, false, true>, grid,
                                   dim3(kWarps * 32), 0, s, true, w, absmean, aq, scale, asum, y,
                                   dot, (int)m, n, k);
    if (vec)
        bitnet_gemv_kernel<MT, ROWS, true, false, false><<<grid, kWarps * 32, 0, s>>>(
            w, absmean, aq, scale, asum, y, dot, (int)m, n, k);
    else
        bitnet_gemv_kernel<MT, ROWS, false, false, false><<<grid, kWarps * 32, 0, s>>>(
            w, absmean, aq, scale, asum, y, dot, (int)m, n, k);
    return cudaPeekAtLastError();
}

template <int R>
cudaError_t launch_m1_staged(const uint8_t *wq, const uint16_t *wd, const int8_t *aq,
                             const uint16_t *ad, float *out, int32_t *sumi, int64_t n, int64_t k,
                             int split, int64_t per, cudaStream_t s, bool pdl) {
    constexpr int W = kM1Warps;
    const dim3 grid((unsigned)((n + W * R - 1) / (W * R)), (unsigned)split);
    const size_t smem = (size_t)per * 48;
    const auto *wdp = reinterpret_cast<const unsigned short *>(wd);
    const auto *adp = reinterpret_cast<const unsigned short *>(ad);
    if (sumi) {
        gemv_m1_staged_kernel<R, false, W, true><<<grid, W * 32, smem, s>>>(wq, wdp, aq, adp, out,
                                                                            sumi, n, k, per);
        return cudaPeekAtLastError();
    }
    if (pdl)
        return launch_kernel(gemv_m1_staged_kernel<R, true, W, false>, grid, dim3(W * 32), smem, s,
                             true, wq, wdp, aq, adp, out, sumi, n, k, per);
    gemv_m1_staged_kernel<R, false, W, false><<<grid, W * 32, smem, s>>>(wq, wdp, aq, adp, out,
                                                                         sumi, n, k, per);
    return cudaPeekAtLastError();
}

template <int MT, int ROWS>
cudaError_t launch_grouped(LinearGroup tab, bool pdl, cudaStream_t s) {
    // m = 1: the staged form, while the longest row's records fit the 48 KB
    // of shared memory a launch gets without opting in (k <= 32768)
    int64_t kmax = 0;
    for (int p = 0; p < tab.count; ++p) kmax = std::max(kmax, tab.p[p].k);
    const bool staged = MT == 1 && kmax / kQK * 48 <= 48 * 1024;
    const int64_t rows_per_cta =
        staged ? (int64_t)kM1GroupWarps * kM1GroupRows : (int64_t)kGroupedWarps * ROWS;
    // Longest CTAs first: a CTA's time grows with its problem's k, and CTAs
    // start in index order, so the long ones must not form the last wave.
    // (The problems are independent; their order changes no result.)
    std::stable_sort(tab.p, tab.p + tab.count,
                     [](const LinearProblem &a, const LinearProblem &b) { return a.k > b.k; });
    int64_t total = 0;
    for (int p = 0; p < tab.count; ++p) {
        total += (tab.p[p].n + rows_per_cta - 1) / rows_per_cta;
        tab.cta_end[p] = total;
    }
    if (staged) {
        const size_t smem = (size_t)(kmax / kQK) * 48;
        constexpr int R = kM1GroupRows, W = kM1GroupWarps;
        if (pdl)
            return launch_kernel(gemv_grouped_m1_staged_kernel<R, true, W>, dim3((unsigned)total),
                                 dim3(W * 32), smem, s, true, tab);
        gemv_grouped_m1_staged_kernel<R, false, W><<<(unsigned)total, W * 32, smem, s>>>(tab);
        return cudaPeekAtLastError();
    }
    if (pdl)
        return launch_kernel(gemv_grouped_kernel<MT, ROWS, true>, dim3((unsigned)total),
                             dim3(kGroupedWarps * 32), 0, s, true, tab);
    gemv_grouped_kernel<MT, ROWS, false><<<(unsigned)total, kGroupedWarps * 32, 0, s>>>(tab);
    return cudaPeekAtLastError();
}

}  // namespace

// ---------------------------------------------------------------------------

int gemv_auto_split(int64_t m, int64_t n, int64_t k) {
    // Aim for at least two CTAs per SM (152 SMs) without slices shorter than
    // 32 blocks per lane group.
    const int64_t kb = k / kQK;
    const int rows_per_cta = kWarps * (m <= 2 ? 2 : 1);
    const int64_t ctas = (n + rows_per_cta - 1) / rows_per_cta;
    const int64_t want = 2 * 152;
    if (ctas >= want) return 1;
    int64_t s = (want + ctas - 1) / ctas;
    s = std::min<int64_t>(s, std::max<int64_t>(1, kb / 64));
    s = std::min<int64_t>(s, 32);
    return (int)std::max<int64_t>(1, s);
}

size_t gemv_workspace_bytes(int64_t m, int64_t n, int64_t /*k*/, int split) {
    return split > 1 ? (size_t)split * (size_t)m * (size_t)n * sizeof(float) : 0;
}

cudaError_t launch_gemv_q4_0_q8_0(const uint8_t *wq, const uint16_t *wd, const int8_t *aq,
                                  const uint16_t *ad, float *y, int32_t *sumi, int64_t m,
                                  int64_t n, int64_t k, int split, float *partials,
                                  cudaStream_t s, bool pdl) {
    if (sumi) pdl = false;
    if (!sumi && split <= 1) {
        LinearGroup tab = {};
        tab.p[0] = {wq, wd, nullptr, 0, const_cast<int8_t *>(aq), const_cast<uint16_t *>(ad),
                    y, n, k};
        tab.count = 1;
        tab.m = (int)m;
        if (stream_gemv_supported(tab)) return launch_stream_gemv(tab, pdl, s);
    }
    float *out = split > 1 ? partials : y;
    cudaError_t e;
    const int64_t per = (k / kQK + split - 1) / split;  // blocks per slice
    if (m == 1 && per * 48 <= 48 * 1024) {
        // one token: the staged form (also for the block sums)
        e = n >= kM1ManyRows ? launch_m1_staged<2>(wq, wd, aq, ad, out, sumi, n, k, split, per, s, pdl)
                             : launch_m1_staged<1>(wq, wd, aq, ad, out, sumi, n, k, split, per, s, pdl);
    } else if (m == 1) e = launch_q4<1, 2>(wq, wd, aq, ad, out, sumi, m, n, k, split, s, pdl);
    else if (m == 2) e = launch_q4<2, 2>(wq, wd, aq, ad, out, sumi, m, n, k, split, s, pdl);
    else if (m <= 4) e = launch_q4<4, 1>(wq, wd, aq, ad, out, sumi, m, n, k, split, s, pdl);
    else if (m <= 8) e = launch_q4<8, 1>(wq, wd, aq, ad, out, sumi, m, n, k, split, s, pdl);
    else e = launch_q4<16, 1>(wq, wd, aq, ad, out, sumi, m, n, k, split, s, pdl);
    if (e != cudaSuccess || split <= 1 || sumi) return e;
    const int64_t count = m * n;
    const int threads = 256;
    const dim3 grid((unsigned)((count + threads - 1) / threads));
    if (pdl)
        return launch_kernel(splitk_reduce_kernel<true>, grid, dim3(threads), 0, s, true,
                             (const float *)partials, y, count, split);
    splitk_reduce_kernel<false><<<grid, threads, 0, s>>>(partials, y, count, split);
    return cudaPeekAtLastError();
}

cudaError_t launch_splitk_reduce(const float *partials, float *y, int64_t count, int split,
                                 cudaStream_t s) {
    const int threads = 256;
    const dim3 grid((unsigned)((count + threads - 1) / threads));
    splitk_reduce_kernel<false><<<grid, threads, 0, s>>>(partials, y, count, split);
    return cudaPeekAtLastError();
}

cudaError_t launch_bitnet_gemv(const uint32_t *w, float absmean, const int8_t *aq,
                               const float *scale, const int32_t *sum, float *y, int32_t *dot,
                               int64_t m, int64_t n, int64_t k, cudaStream_t s, bool pdl) {
    // m = 1: the row staged once per CTA, one row per warp and 8 warps (at
    // N=6912, K=2560: 3.35 us; rows x warps 2x8: 3.48, 1x16: 3.49, 4x4: 3.52,
    // 2x2: 3.53, 1x4: 3.58, 4x2: 3.58, 2x4: 3.59, 4x8: 3.78, 2x16: 3.89; each
    // warp reading the row from L2 itself, four rows per warp and 2 warps: 3.66)
    if (m == 1 && k % 64 == 0 && k <= 32768) {
        constexpr int kRows = 1, kW = 8;
        const dim3 grid((unsigned)((n + kW * kRows - 1) / (kW * kRows)));
        const size_t smem = (size_t)k;  // one byte per activation
        if (dot) {
            bitnet_gemv_m1_kernel<kRows, kW, true, false><<<grid, kW * 32, smem, s>>>(
                w, absmean, aq, scale, sum, y, dot, n, k);
            return cudaPeekAtLastError();
        }
        if (pdl)
            return launch_kernel(bitnet_gemv_m1_kernel<kRows, kW, false, true>, grid, dim3(kW * 32),
                                 smem, s, true, w, absmean, aq, scale, sum, y, dot, n, k);
        bitnet_gemv_m1_kernel<kRows, kW, false, false><<<grid, kW * 32, smem, s>>>(
            w, absmean, aq, scale, sum, y, dot, n, k);
        return cudaPeekAtLastError();
    }
    if (m == 1) return launch_bitnet<1, 4>(w, absmean, aq, scale, sum, y, dot, m, n, k, s, pdl);
    if (m == 2) return launch_bitnet<2, 2>(w, absmean, aq, scale, sum, y, dot, m, n, k, s, pdl);
    if (m <= 4) return launch_bitnet<4, 1>(w, absmean, aq, scale, sum, y, dot, m, n, k, s, pdl);
    if (m <= 8) return launch_bitnet<8, 1>(w, absmean, aq, scale, sum, y, dot, m, n, k, s, pdl);
    return launch_bitnet<16, 1>(w, absmean, aq, scale, sum, y, dot, m, n, k, s, pdl);
}

bool bitnet_linear_fused_supported(int64_t m, int64_t k, int64_t ldx, const void *x, const void *aq) {
    return m == 1 && k % 64 == 0 && k <= 32768 && ldx >= k &&
           (reinterpret_cast<uintptr_t>(x) & 15) == 0 && (reinterpret_cast<uintptr_t>(aq) & 15) == 0;
}

cudaError_t launch_bitnet_linear_fused(const uint32_t *w, float absmean, const float *x, int8_t *aq,
                                       float *scale, int32_t *sum, float *y, int64_t n, int64_t k,
                                       cudaStream_t s, bool pdl) {
    // 3 rows per warp, 8 warps: 3.71 us per step at N=6912, K=2560 with the
    // row read from L2 once (rows x warps 3x16: 3.79, 4x8: 3.89, 2x8: 4.10,
    // 4x4: 4.61, 2x16: 5.84).  Reading it twice, 3x8 took 3.96-4.05 (2x8:
    // 4.01, 4x16: 4.12, 4x8: 4.36, 2x6: 4.48, 4x4: 4.63, 8x8: 4.63, 2x4: 5.39,
    // 4x2: 5.87, 1x16: 6.05, 1x8: 6.47, 16x4: 8.57); two launches, quantizer
    // then GEMV: 5.03)
    constexpr int kRows = 3, kW = 8;
    const dim3 grid((unsigned)((n + kW * kRows - 1) / (kW * kRows)));
    const size_t smem = (size_t)k;  // one byte per code
    if (pdl)
        return launch_kernel(bitnet_linear_m1_kernel<kRows, kW, true>, grid, dim3(kW * 32), smem, s,
                             true, w, absmean, x, aq, scale, sum, y, n, k);
    bitnet_linear_m1_kernel<kRows, kW, false><<<grid, kW * 32, smem, s>>>(w, absmean, x, aq, scale,
                                                                          sum, y, n, k);
    return cudaPeekAtLastError();
}

cudaError_t launch_linear_grouped(const LinearGroup &tab, bool pdl, cudaStream_t s) {
    cudaError_t e = launch_quantize_grouped(tab, s, pdl);
    if (e != cudaSuccess) return e;
    if (stream_gemv_supported(tab)) return launch_stream_gemv(tab, pdl, s);
    const int m = tab.m;
    // m = 1: four rows per warp in the grouped step (5100 against 5008 GB/s
    // for two); the single GEMV keeps two (3.61 against 3.74 us)
    if (m == 1) return launch_grouped<1, 4>(tab, pdl, s);
    if (m == 2) return launch_grouped<2, 2>(tab, pdl, s);
    if (m <= 4) return launch_grouped<4, 1>(tab, pdl, s);
    if (m <= 8) return launch_grouped<8, 1>(tab, pdl, s);
    return launch_grouped<16, 1>(tab, pdl, s);
}

// ---------------------------------------------------------------------------
// Split-K GEMV without caller-provided memory.
//
// Some callers cannot allocate device memory at the point where they run the
// product: code running where cudaMalloc is off limits (a real-time or
// latency-critical loop that must not take the allocator's locks or risk
// an implicit synchronization, or a host process that was handed device
// pointers by another component and owns no allocator at all).  For them the
// split-K partials live in this library-owned array, reserved once per GPU
// when the library is loaded on it and held until the process exits.

static __device__ __align__(256) float g_gemv_scratch[kGemvNoAllocScratchFloats];

namespace {
std::mutex g_scratch_mu;
float *g_scratch_ptr[64] = {};  // device address of g_gemv_scratch, per device
}  // namespace

cudaError_t launch_gemv_q4_0_q8_0_noalloc(const uint8_t *wq, const uint16_t *wd, const int8_t *aq,
                                          const uint16_t *ad, float *y, int64_t m, int64_t n,
                                          int64_t k, int split, cudaStream_t s) {
    float *scratch = nullptr;
    if (split > 1) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (!g_scratch_ptr[dev]) {
            // host code only knows a stand-in for the array: ask the runtime
            // for its address on the current device (first call per device)
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_gemv_scratch);
            if (e != cudaSuccess) return e;
            g_scratch_ptr[dev] = static_cast<float *>(p);
        }
        scratch = g_scratch_ptr[dev];
    }
    // every slice writes all of its m * n partials, so nothing needs clearing
    return launch_gemv_q4_0_q8_0(wq, wd, aq, ad, y, nullptr, m, n, k, split, scratch, s);
}

}  // namespace qmm
