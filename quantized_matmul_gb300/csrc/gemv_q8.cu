// Decode-shaped product with Q8_0 weights: Q8_0 x Q8_0 GEMV (m <= 16).
//
// The Q8_0 block (llama.cpp visual guide, lesson 31 "The CPU backend",
// section "How the quantized dot product works": 32 int8 values and one fp16
// scale) serves here as the weight format too, as in the Fucina reference,
// section 9 (the Q8_0 right-hand side of 9.2 / 9.7, and the Q8_0 decode of
// 9.9.2).  Per block, sumi = sum_j q_w * q_a exactly in int32 (eight signed
// dp4a), then acc += sumi * (dw * da) in f32, as for Q4_0.
//
// Layout: weight codes int8 [n, k] and scales fp16 [n, k/32] (two planes).
// A warp owns ROWS rows; lane l takes blocks l, l+32, ... of every row, so a
// block is two 16-byte loads and each warp-wide pair reads 1 KB of one row
// contiguously (coalesced, no reuse, L1 bypassed).  The per-lane partials are
// summed by the xor-shuffle tree.  A split over k writes f32 partials
// [S, m, n] that a second kernel adds in slice order.
#include <cuda_fp16.h>

#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr int kWarps = 4;   // warps per CTA (4: 2.7% faster than 8 at 4096x4096)
constexpr int kUnroll = 2;  // blocks (per lane, per row) loaded before use: 64 bytes

__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// signed bytes of a times signed bytes of b, summed into c
__device__ __forceinline__ int dp4a_ss(int a, int b, int c) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ float h2f(unsigned short h) {
    return __half2float(__ushort_as_half(h));
}

template <int MT, int ROWS, bool EMIT>
__global__ void __launch_bounds__(kWarps * 32)
gemv_q8_0_q8_0_kernel(const int8_t *__restrict__ w8, const unsigned short *__restrict__ wd,
                      const int8_t *__restrict__ aq, const unsigned short *__restrict__ ad,
                      float *__restrict__ out, int32_t *__restrict__ sumi, int m, int64_t n,
                      int64_t k, int64_t kb_per_split) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t kb = k / kQK;
    const int64_t row0 = ((int64_t)blockIdx.x * kWarps + warp) * ROWS;
    if (row0 >= n) return;
    const int64_t slice = blockIdx.y;
    const int64_t kb0 = slice * kb_per_split;
    const int64_t kb1 = min(kb, kb0 + kb_per_split);

    float acc[ROWS][MT];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[r][t] = 0.0f;

    for (int64_t bb = kb0 + lane; bb < kb1; bb += 32 * kUnroll) {
        uint4 wv[kUnroll][ROWS][2];
        unsigned short dwv[kUnroll][ROWS];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t b = bb + 32 * u;
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                const int64_t row = row0 + r;
                if (b < kb1 && row < n) {
                    const int8_t *p = w8 + row * k + b * kQK;
                    wv[u][r][0] = ld_stream_v4(p);
                    wv[u][r][1] = ld_stream_v4(p + 16);
                    dwv[u][r] = EMIT ? (unsigned short)0 : __ldg(wd + row * kb + b);
                } else {
                    wv[u][r][0] = make_uint4(0u, 0u, 0u, 0u);
                    wv[u][r][1] = make_uint4(0u, 0u, 0u, 0u);
                    dwv[u][r] = 0;
                }
            }
        }
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
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const uint4 w0 = wv[u][r][0], w1 = wv[u][r][1];
                    int s = dp4a_ss((int)w0.x, a0.x, 0);
                    s = dp4a_ss((int)w0.y, a0.y, s);
                    s = dp4a_ss((int)w0.z, a0.z, s);
                    s = dp4a_ss((int)w0.w, a0.w, s);
                    s = dp4a_ss((int)w1.x, a1.x, s);
                    s = dp4a_ss((int)w1.y, a1.y, s);
                    s = dp4a_ss((int)w1.z, a1.z, s);
                    s = dp4a_ss((int)w1.w, a1.w, s);
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
    if constexpr (!EMIT) {
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

template <int MT, int ROWS>
cudaError_t launch_q8(const int8_t *w8, const uint16_t *wd, const int8_t *aq, const uint16_t *ad,
                      float *out, int32_t *sumi, int64_t m, int64_t n, int64_t k, int split,
                      cudaStream_t s) {
    const int64_t kb = k / kQK;
    const int64_t per = (kb + split - 1) / split;
    const int64_t rows_per_cta = (int64_t)kWarps * ROWS;
    dim3 grid((unsigned)((n + rows_per_cta - 1) / rows_per_cta), (unsigned)split);
    const auto *wdp = reinterpret_cast<const unsigned short *>(wd);
    const auto *adp = reinterpret_cast<const unsigned short *>(ad);
    if (sumi)
        gemv_q8_0_q8_0_kernel<MT, ROWS, true><<<grid, kWarps * 32, 0, s>>>(
            w8, wdp, aq, adp, out, sumi, (int)m, n, k, per);
    else
        gemv_q8_0_q8_0_kernel<MT, ROWS, false><<<grid, kWarps * 32, 0, s>>>(
            w8, wdp, aq, adp, out, sumi, (int)m, n, k, per);
    return cudaPeekAtLastError();
}

}  // namespace

cudaError_t launch_gemv_q8_0_q8_0(const int8_t *w8, const uint16_t *wd, const int8_t *aq,
                                  const uint16_t *ad, float *y, int32_t *sumi, int64_t m,
                                  int64_t n, int64_t k, int split, float *partials,
                                  cudaStream_t s) {
    float *out = split > 1 ? partials : y;
    cudaError_t e;
    if (m == 1) e = launch_q8<1, 2>(w8, wd, aq, ad, out, sumi, m, n, k, split, s);
    else if (m == 2) e = launch_q8<2, 2>(w8, wd, aq, ad, out, sumi, m, n, k, split, s);
    else if (m <= 4) e = launch_q8<4, 1>(w8, wd, aq, ad, out, sumi, m, n, k, split, s);
    else if (m <= 8) e = launch_q8<8, 1>(w8, wd, aq, ad, out, sumi, m, n, k, split, s);
    else e = launch_q8<16, 1>(w8, wd, aq, ad, out, sumi, m, n, k, split, s);
    if (e != cudaSuccess || split <= 1 || sumi) return e;
    return launch_splitk_reduce(partials, y, m * n, split, s);
}

}  // namespace qmm
