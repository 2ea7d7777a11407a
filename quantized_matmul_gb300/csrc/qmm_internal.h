// Internal launcher interface between the C ABI (qmm_api.cu) and the kernel
// translation units.  Launchers assume their arguments were validated by the
// C ABI; they enqueue kernels on `stream` and return the launch status.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace qmm {

// The current device's SM count, queried once per device and cached (152,
// a GB300's count, if the query fails).  Safe to call from several host
// threads.
inline int device_sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
        return 152;
    cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

constexpr int kQK = 32;  // elements per quantization block

// Programmatic dependent launch.  A kernel launched with `pdl` set may start
// while the previous kernel on its stream is still running.  pdl_wait()
// returns once that kernel has completed and its writes are visible (at once
// when the launch had no such predecessor), so everything a kernel reads
// from its predecessor comes after it; pdl_launch_dependents() lets the next
// PDL launch on the stream begin once every CTA of this grid has called it
// or exited.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... Params, typename... Args>
cudaError_t launch_kernel(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, bool pdl, Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

// A group of independent decode linear layers sharing m: layer p computes
// y_p = x_p W_p^T (Q8_0 quantization of x_p into aq_p/ad_p, then the GEMV).
// Passed by value as a kernel parameter, so no device copy of the table.
constexpr int kGroupMax = 16;
struct LinearProblem {
    const uint8_t *wq;
    const uint16_t *wd;
    const float *x;
    int64_t ldx;
    int8_t *aq;
    uint16_t *ad;
    float *y;
    int64_t n, k;
};
struct LinearGroup {
    LinearProblem p[kGroupMax];
    int64_t cta_end[kGroupMax];  // cumulative CTA counts (filled by the launchers)
    int count;
    int m;
};

// quant.cu
// The quantizer over every problem of a group in one launch.
cudaError_t launch_quantize_grouped(const LinearGroup &g, cudaStream_t s, bool pdl);
// pdl: launch with programmatic dependent launch (x is read after pdl_wait)
cudaError_t launch_quantize_act_q8_0(const float *x, int64_t m, int64_t k, int64_t ldx,
                                     int8_t *aq, uint16_t *ad, cudaStream_t s, bool pdl = false);
cudaError_t launch_quantize_weight_q4_0(const float *w, int64_t n, int64_t k,
                                        uint8_t *wq, uint16_t *wd, cudaStream_t s);
// x rows ldx floats apart; pdl: launch with programmatic dependent launch
// (x is read after pdl_wait)
cudaError_t launch_quantize_act_bitnet(const float *x, int64_t m, int64_t k, int64_t ldx, int8_t *aq,
                                       float *scale, int32_t *sum, cudaStream_t s, bool pdl = false);
cudaError_t launch_pack_ternary(const int8_t *t, int64_t n, int64_t k, uint32_t *w,
                                cudaStream_t s);

// gemv.cu
int gemv_auto_split(int64_t m, int64_t n, int64_t k);
size_t gemv_workspace_bytes(int64_t m, int64_t n, int64_t k, int split);
// sumi != nullptr selects the block-sum emitting variant (split must be 1).
// pdl: launch with programmatic dependent launch; the GEMV then loads its
// first weight blocks before pdl_wait and everything else after it (sumi
// must be null).
cudaError_t launch_gemv_q4_0_q8_0(const uint8_t *wq, const uint16_t *wd, const int8_t *aq,
                                  const uint16_t *ad, float *y, int32_t *sumi, int64_t m,
                                  int64_t n, int64_t k, int split, float *partials,
                                  cudaStream_t s, bool pdl = false);
// Split-K GEMV whose partials live in a library-owned device array of
// kGemvNoAllocScratchFloats floats (split * m * n must fit).
constexpr int64_t kGemvNoAllocScratchFloats = int64_t(1) << 20;
cudaError_t launch_gemv_q4_0_q8_0_noalloc(const uint8_t *wq, const uint16_t *wd, const int8_t *aq,
                                          const uint16_t *ad, float *y, int64_t m, int64_t n,
                                          int64_t k, int split, cudaStream_t s);
// pdl: launch with programmatic dependent launch; the GEMV then loads its
// first weight words before pdl_wait and reads aq/scale/sum after it (dot
// must be null).
cudaError_t launch_bitnet_gemv(const uint32_t *w, float absmean, const int8_t *aq,
                               const float *scale, const int32_t *sum, float *y, int32_t *dot,
                               int64_t m, int64_t n, int64_t k, cudaStream_t s, bool pdl = false);
// The BitNet decode step for m = 1 in one kernel (every CTA quantizes the
// row itself; CTA 0 writes aq, scale and sum): when m == 1, k % 64 == 0,
// k <= 32768 and x, aq are 16-byte aligned (x's row stride does not matter
// at m = 1).
bool bitnet_linear_fused_supported(int64_t m, int64_t k, int64_t ldx, const void *x, const void *aq);
cudaError_t launch_bitnet_linear_fused(const uint32_t *w, float absmean, const float *x, int8_t *aq,
                                       float *scale, int32_t *sum, float *y, int64_t n, int64_t k,
                                       cudaStream_t s, bool pdl);
// y[i] = sum over slices s of partials[s * count + i], slices in order.
cudaError_t launch_splitk_reduce(const float *partials, float *y, int64_t count, int split,
                                 cudaStream_t s);
// Quantizer then GEMV (unsplit) for every problem of the group: two launches.
cudaError_t launch_linear_grouped(const LinearGroup &g, bool pdl, cudaStream_t s);

// gemv_stream.cu: the decode GEMV (unsplit) with the weights staged through
// shared memory by tensor copies; identical results to the register GEMV.
// Used when 8 <= m <= 16, every problem has k/32 % 8 == 0 and 16-byte
// aligned wq, wd, aq, ad, and the activations fit in shared memory.
bool stream_gemv_supported(const LinearGroup &g);
cudaError_t launch_stream_gemv(const LinearGroup &g, bool pdl, cudaStream_t s);
cudaError_t stream_read_and_clear_error(unsigned int *word, cudaStream_t s);
void stream_set_wait_limit(uint32_t iterations);
void stream_set_withhold_loads(int enable);

// bitnet_gemm.cu: BitNet ternary product on the tensor cores (any m, k % 64
// == 0, k <= 2^17); workspace: fp16 copy of the activations.
size_t bitnet_gemm_workspace_bytes(int64_t m, int64_t k);
cudaError_t launch_bitnet_gemm(const uint32_t *w, float absmean, const int8_t *aq,
                               const float *act_scale, float *y, int64_t m, int64_t n, int64_t k,
                               void *workspace, cudaStream_t s);
void bitnet_gemm_set_wait_limit(uint32_t iterations);
cudaError_t bitnet_gemm_read_and_clear_error(unsigned int *word, cudaStream_t s);
// bitnet_small.cu: the BitNet product for a few tokens (m <= 32, k % 64 == 0,
// k <= 131072) on the warp-level tensor-core MMA; launched by qmm_bitnet_gemm
// for those shapes.  Its workspace holds the activations in the MMA's
// fragment order, the per-group corrections and a row-set counter.
bool bitnet_small_m_supported(int64_t m, int64_t n, int64_t k);
size_t bitnet_small_m_workspace_bytes(int64_t m, int64_t k);
cudaError_t launch_bitnet_small_m(const uint32_t *w, float absmean, const int8_t *aq,
                                  const float *act_scale, float *y, int64_t m, int64_t n,
                                  int64_t k, void *workspace, cudaStream_t s);
void bitnet_small_set_wait_limit(uint32_t iterations);
void bitnet_small_set_withhold_loads(int enable);
cudaError_t bitnet_small_read_and_clear_error(unsigned int *word, cudaStream_t s);

// gemv_q8.cu: Q8_0 weights (int8 [n, k] + fp16 scales [n, k/32]) x Q8_0
// activations, m <= 16; same workspace rule as the Q4_0 GEMV; sumi != nullptr
// selects the block-sum variant (split must be 1).
cudaError_t launch_gemv_q8_0_q8_0(const int8_t *w8, const uint16_t *wd, const int8_t *aq,
                                  const uint16_t *ad, float *y, int32_t *sumi, int64_t m,
                                  int64_t n, int64_t k, int split, float *partials,
                                  cudaStream_t s);

// gemm_small.cu: Q4_0 x Q8_0 (m <= 64) and Q8_0 x Q8_0 (m <= 32) products
// for k % 256 == 0 on the warp-level tensor-core MMA (accumulators in
// registers); launched by the GEMM launchers for those shapes and by the
// decode GEMV entries from three tokens on.  wd / ad may be null when sumi is
// given (block-sum variant).
bool gemm_small_m_supported(int64_t m, int64_t n, int64_t k);
// Q4_0 weights also from 33 to 64 tokens
bool gemm_small_m_supported_q4(int64_t m, int64_t n, int64_t k);
size_t gemm_small_m_workspace_bytes(int64_t m, int64_t k);
cudaError_t launch_gemm_small_m(const uint8_t *wq, const uint16_t *wd, const int8_t *aq,
                                const uint16_t *ad, float *y, int32_t *sumi, int64_t m, int64_t n,
                                int64_t k, void *workspace, cudaStream_t s);
cudaError_t launch_gemm_small_m_q8(const int8_t *w8, const uint16_t *wd, const int8_t *aq,
                                   const uint16_t *ad, float *y, int32_t *sumi, int64_t m, int64_t n,
                                   int64_t k, void *workspace, cudaStream_t s);
void gemm_small_set_wait_limit(uint32_t iterations);
void gemm_small_set_withhold_loads(int enable);
cudaError_t gemm_small_read_and_clear_error(unsigned int *word, cudaStream_t s);
// probe.cu: tensor-pipe peak probes (kind 0: int8 mma.sync m16n8k32; 1: f16
// mma.sync m16n8k16), one CTA of 512 threads per SM; `out` holds sms * 512
// ints.
int64_t mma_probe_macs_per_iter(int kind, int sms);
cudaError_t launch_mma_probe(int kind, int iters, int sms, int *out, cudaStream_t s);
// gemm.cu
size_t gemm_workspace_bytes(int64_t m, int64_t n, int64_t k);
// sumi != nullptr selects the block-sum emitting variant.
cudaError_t launch_gemm_q4_0_q8_0(const uint8_t *wq, const uint16_t *wd, const int8_t *aq,
                                  const uint16_t *ad, float *y, int32_t *sumi, int64_t m,
                                  int64_t n, int64_t k, void *workspace, cudaStream_t s);
// Load-time repack of the Q4_0 nibble plane into the GEMM tile order
// (ceil(n/128) * ceil(k/64) tiles of 4096 bytes), and the GEMM reading it.
size_t repack_q4_0_gemm_bytes(int64_t n, int64_t k);
cudaError_t launch_repack_q4_0_gemm(const uint8_t *wq, int64_t n, int64_t k, uint8_t *wr,
                                    cudaStream_t s);
cudaError_t launch_gemm_q4_0_q8_0_repacked(const uint8_t *wr, const uint16_t *wd, const int8_t *aq,
                                           const uint16_t *ad, float *y, int32_t *sumi, int64_t m,
                                           int64_t n, int64_t k, void *workspace, cudaStream_t s);
// The same product with Q8_0 weights (int8 [n, k]); same workspace.
cudaError_t launch_gemm_q8_0_q8_0(const int8_t *w8, const uint16_t *wd, const int8_t *aq,
                                  const uint16_t *ad, float *y, int32_t *sumi, int64_t m,
                                  int64_t n, int64_t k, void *workspace, cudaStream_t s);
// Reads and clears the GEMM kernels' device error word (after the caller
// synchronized).  Returns the raw word: 0 = no error.
cudaError_t gemm_read_and_clear_error(unsigned int *word, cudaStream_t s);
void gemm_set_wait_limit(uint32_t iterations);
void gemm_set_withhold_loads(int enable);

}  // namespace qmm
