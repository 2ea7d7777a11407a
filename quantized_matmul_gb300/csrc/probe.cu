// Tensor-pipe peak probes for the measurement harness.
//
// The only int8 tensor-core instruction sm_103a accepts is the warp-level
// mma.sync (m16n8k32, s8 x s8 -> s32); tcgen05.mma kind::i8 is rejected by
// the assembler for this target.  The int8 tensor peak of the GPU is
// therefore what that instruction sustains, which this kernel measures: every
// warp of one CTA per SM issues independent MMAs back to back (eight
// accumulator chains per warp, enough to cover the instruction's latency),
// and the host times the launch with CUDA events.  The same loop with the f16
// form (m16n8k16, f32 accumulators) gives the warp-level f16 rate for
// comparison.  Results are written out only so the loop is not removed.
#include <cuda_runtime.h>

#include <cstdint>

#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr int kProbeThreads = 512;
constexpr int kProbeChains = 8;

__global__ void __launch_bounds__(kProbeThreads) mma_s8_probe_kernel(int iters, int *out) {
    const int a0 = threadIdx.x, a1 = a0 * 3, a2 = a0 ^ 5, a3 = a0 + 7, b0 = a0 * 11, b1 = a0 ^ 9;
    int c[kProbeChains][4];
#pragma unroll
    for (int j = 0; j < kProbeChains; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = j;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < kProbeChains; ++j)
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                "{%8,%9}, {%0,%1,%2,%3};"
                : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    int s = 0;
#pragma unroll
    for (int j = 0; j < kProbeChains; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void __launch_bounds__(kProbeThreads) mma_f16_probe_kernel(int iters, int *out) {
    const uint32_t a0 = 0x3c003c00u + threadIdx.x, a1 = a0 ^ 1u, a2 = a0 ^ 2u, a3 = a0 ^ 3u;
    const uint32_t b0 = a0 ^ 4u, b1 = a0 ^ 5u;
    float c[kProbeChains][4];
#pragma unroll
    for (int j = 0; j < kProbeChains; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = (float)j;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < kProbeChains; ++j)
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                "{%8,%9}, {%0,%1,%2,%3};"
                : "+f"(c[j][0]), "+f"(c[j][1]), "+f"(c[j][2]), "+f"(c[j][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < kProbeChains; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
    out[blockIdx.x * blockDim.x + threadIdx.x] = __float_as_int(s);
}

}  // namespace

int64_t mma_probe_macs_per_iter(int kind, int sms) {
    const int64_t per_mma = kind == 0 ? 16 * 8 * 32 : 16 * 8 * 16;
    return (int64_t)sms * (kProbeThreads / 32) * kProbeChains * per_mma;
}

cudaError_t launch_mma_probe(int kind, int iters, int sms, int *out, cudaStream_t s) {
    if (kind == 0)
        mma_s8_probe_kernel<<<sms, kProbeThreads, 0, s>>>(iters, out);
    else
        mma_f16_probe_kernel<<<sms, kProbeThreads, 0, s>>>(iters, out);
    return cudaPeekAtLastError();
}

}  // namespace qmm
