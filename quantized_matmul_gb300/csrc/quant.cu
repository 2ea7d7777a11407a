// Quantizers: f32 activations -> Q8_0, f32 weights -> Q4_0 (load time),
// f32 activations -> BitNet int8 with a per-row scale, and ternary packing.
//
// Q8_0 / Q4_0 follow llama.cpp visual guide, lesson 31 "The CPU backend",
// section "How the quantized dot product works" (32-element blocks, one fp16
// scale per block, Q4_0 nibbles hold value + 8) with the workload recipe
// d = absmax/127 (activations) and d = signed absmax / -8 (weights).  The
// BitNet steps follow Loom docs, "Plan 9 SIMD Forward", section "BitNet
// ternary MAD kernel".  Every step that decides an integer is taken in IEEE
// f32 with explicit round-to-nearest intrinsics (__fdiv_rn, __fmul_rn) and
// roundf (half away from zero), so the codes are reproducible bit for bit.
//
// One warp owns one 32-element block: lane j holds element j, so the block
// reductions are five xor-shuffles and every load and store is coalesced.
#include <cuda_fp16.h>

#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr int kWarpsPerCta = 4;  // 0.3% faster decode step than 8, 2 or 16

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ unsigned short f32_to_f16_bits(float v) {
    return __half_as_ushort(__float2half_rn(v));
}

// One Q8_0 block (row i, block b) per warp, lane j holding element j.
__device__ __forceinline__ void quantize_q8_0_block(const float *__restrict__ x, int64_t ldx,
                                                    int64_t k, int64_t i, int64_t b, int lane,
                                                    int8_t *__restrict__ aq,
                                                    unsigned short *__restrict__ ad) {
    const int64_t kb = k / kQK;
    const float v = x[i * ldx + b * kQK + lane];
    const float amax = warp_max(fabsf(v));
    const float d = __fdiv_rn(amax, 127.0f);
    float q = 0.0f;
    if (d != 0.0f) q = fminf(fmaxf(roundf(__fdiv_rn(v, d)), -127.0f), 127.0f);
    aq[i * k + b * kQK + lane] = (int8_t)(int)q;
    if (lane == 0) ad[i * kb + b] = f32_to_f16_bits(d);
}

// Q8_0: grid covers m * (k/32) blocks, one warp each.  With PDL the next
// kernel (the GEMV) may launch at once and stream its weights while this
// grid waits for x from its own predecessor.
template <bool PDL>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
quantize_act_q8_0_kernel(const float *__restrict__ x, int64_t m, int64_t k, int64_t ldx,
                         int8_t *__restrict__ aq, unsigned short *__restrict__ ad) {
    if (PDL) {
        pdl_launch_dependents();
        pdl_wait();
    }
    const int64_t kb = k / kQK;
    const int64_t blk = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
    if (blk >= m * kb) return;
    const int64_t i = blk / kb;
    quantize_q8_0_block(x, ldx, k, i, blk - i * kb, threadIdx.x & 31, aq, ad);
}

// The same over a group of problems: warp w serves the problem whose range
// of blocks holds w (cta_end here counts blocks, filled by the launcher).
template <bool PDL>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
quantize_grouped_kernel(const __grid_constant__ LinearGroup tab) {
    if (PDL) {
        pdl_launch_dependents();
        pdl_wait();
    }
    const int64_t blk = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
    if (blk >= tab.cta_end[tab.count - 1]) return;
    int p = 0;
    while (p + 1 < tab.count && blk >= tab.cta_end[p]) ++p;
    const LinearProblem &P = tab.p[p];
    const int64_t local = blk - (p ? tab.cta_end[p - 1] : 0);
    const int64_t kb = P.k / kQK;
    const int64_t i = local / kb;
    quantize_q8_0_block(P.x, P.ldx, P.k, i, local - i * kb, threadIdx.x & 31, P.aq,
                        reinterpret_cast<unsigned short *>(P.ad));
}

// Q4_0: one warp per block; the signed absmax is the element of largest |w|
// with the lowest index on ties.
__global__ void __launch_bounds__(kWarpsPerCta * 32)
quantize_weight_q4_0_kernel(const float *__restrict__ w, int64_t n, int64_t k,
                            uint8_t *__restrict__ wq, unsigned short *__restrict__ wd) {
    const int lane = threadIdx.x & 31;
    const int64_t kb = k / kQK;
    const int64_t blk = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
    if (blk >= n * kb) return;
    const int64_t r = blk / kb, b = blk - r * kb;
    const float v = w[r * k + b * kQK + lane];
    float a = fabsf(v);
    int idx = lane;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float a2 = __shfl_xor_sync(0xffffffffu, a, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
        if (a2 > a || (a2 == a && i2 < idx)) { a = a2; idx = i2; }
    }
    const float maxv = __shfl_sync(0xffffffffu, v, idx);
    const float d = __fdiv_rn(maxv, -8.0f);
    float q = 8.0f;
    if (d != 0.0f) q = fminf(fmaxf(roundf(__fdiv_rn(v, d)) + 8.0f, 0.0f), 15.0f);
    const unsigned qi = (unsigned)(int)q;
    const unsigned hi = __shfl_down_sync(0xffffffffu, qi, 16);  // element lane+16
    if (lane < 16) wq[r * (k / 2) + b * (kQK / 2) + lane] = (uint8_t)(qi | (hi << 4));
    if (lane == 0) wd[r * kb + b] = f32_to_f16_bits(d);
}

// BitNet activations: one CTA per row; the row max and the integer sum are
// CTA reductions (max and integer addition do not depend on order).
constexpr int kBitnetThreads = 256;

// BitNet per-row quantization, one CTA per row.  With PDL the next kernel
// (the ternary GEMV) may launch at once and stream its weights while this
// grid waits for x from its own predecessor.
template <bool PDL>
__global__ void __launch_bounds__(kBitnetThreads)
quantize_act_bitnet_kernel(const float *__restrict__ x, int64_t k, int64_t ldx, int8_t *__restrict__ aq,
                           float *__restrict__ scale, int32_t *__restrict__ sum) {
    __shared__ float s_max[kBitnetThreads / 32];
    __shared__ int s_sum[kBitnetThreads / 32];
    __shared__ float s_scale;
    if (PDL) {
        pdl_launch_dependents();
        pdl_wait();
    }
    const int64_t i = blockIdx.x;
    const float *xr = x + i * ldx;
    float amax = 0.0f;
    for (int64_t j = threadIdx.x; j < k; j += kBitnetThreads) amax = fmaxf(amax, fabsf(xr[j]));
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = amax;
    __syncthreads();
    if (threadIdx.x == 0) {
        float mx = 0.0f;
        for (int w = 0; w < kBitnetThreads / 32; ++w) mx = fmaxf(mx, s_max[w]);
        s_scale = (mx != 0.0f) ? __fdiv_rn(127.0f, mx) : 0.0f;
    }
    __syncthreads();
    const float s = s_scale;
    int part = 0;
    for (int64_t j = threadIdx.x; j < k; j += kBitnetThreads) {
        float q = 0.0f;
        if (s != 0.0f) q = fminf(fmaxf(roundf(__fmul_rn(xr[j], s)), -127.0f), 127.0f);
        const int qi = (int)q;
        aq[i * k + j] = (int8_t)qi;
        part += qi;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if ((threadIdx.x & 31) == 0) s_sum[threadIdx.x >> 5] = part;
    __syncthreads();
    if (threadIdx.x == 0) {
        int tot = 0;
        for (int w = 0; w < kBitnetThreads / 32; ++w) tot += s_sum[w];
        sum[i] = tot;
        scale[i] = s;
    }
}

// Ternary packing: one thread per output word.
__global__ void pack_ternary_kernel(const int8_t *__restrict__ t, int64_t words,
                                    uint32_t *__restrict__ w) {
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= words) return;
    const int8_t *src = t + g * 16;
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) word |= ((uint32_t)(src[i] + 1) & 3u) << (2 * i);
    w[g] = word;
}

}  // namespace

cudaError_t launch_quantize_act_q8_0(const float *x, int64_t m, int64_t k, int64_t ldx,
                                     int8_t *aq, uint16_t *ad, cudaStream_t s, bool pdl) {
    const int64_t blocks = m * (k / kQK);
    const int64_t grid = (blocks + kWarpsPerCta - 1) / kWarpsPerCta;
    auto *adp = reinterpret_cast<unsigned short *>(ad);
    if (pdl)
        return launch_kernel(quantize_act_q8_0_kernel<true>, dim3((unsigned)grid),
                             dim3(kWarpsPerCta * 32), 0, s, true, x, m, k, ldx, aq, adp);
    quantize_act_q8_0_kernel<false><<<(unsigned)grid, kWarpsPerCta * 32, 0, s>>>(
        x, m, k, ldx, aq, adp);
    return cudaPeekAtLastError();
}

cudaError_t launch_quantize_grouped(const LinearGroup &g, cudaStream_t s, bool pdl) {
    LinearGroup tab = g;
    int64_t total = 0;
    for (int p = 0; p < tab.count; ++p) {
        total += (int64_t)tab.m * (tab.p[p].k / kQK);
        tab.cta_end[p] = total;
    }
    const dim3 grid((unsigned)((total + kWarpsPerCta - 1) / kWarpsPerCta));
    if (pdl)
        return launch_kernel(quantize_grouped_kernel<true>, grid, dim3(kWarpsPerCta * 32), 0, s,
                             true, tab);
    quantize_grouped_kernel<false><<<grid, kWarpsPerCta * 32, 0, s>>>(tab);
    return cudaPeekAtLastError();
}

cudaError_t launch_quantize_weight_q4_0(const float *w, int64_t n, int64_t k, uint8_t *wq,
                                        uint16_t *wd, cudaStream_t s) {
    const int64_t blocks = n * (k / kQK);
    const int64_t grid = (blocks + kWarpsPerCta - 1) / kWarpsPerCta;
    quantize_weight_q4_0_kernel<<<(unsigned)grid, kWarpsPerCta * 32, 0, s>>>(
        w, n, k, wq, reinterpret_cast<unsigned short *>(wd));
    return cudaPeekAtLastError();
}

cudaError_t launch_quantize_act_bitnet(const float *x, int64_t m, int64_t k, int64_t ldx, int8_t *aq,
                                       float *scale, int32_t *sum, cudaStream_t s, bool pdl) {
    if (pdl)
        return launch_kernel(quantize_act_bitnet_kernel<true>, dim3((unsigned)m), dim3(kBitnetThreads),
                             0, s, true, x, k, ldx, aq, scale, sum);
    quantize_act_bitnet_kernel<false><<<(unsigned)m, kBitnetThreads, 0, s>>>(x, k, ldx, aq, scale, sum);
    return cudaPeekAtLastError();
}

cudaError_t launch_pack_ternary(const int8_t *t, int64_t n, int64_t k, uint32_t *w,
                                cudaStream_t s) {
    const int64_t words = n * (k / 16);
    const int threads = 256;
    pack_ternary_kernel<<<(unsigned)((words + threads - 1) / threads), threads, 0, s>>>(t, words, w);
    return cudaPeekAtLastError();
}

}  // namespace qmm
