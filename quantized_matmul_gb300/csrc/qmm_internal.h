// Internal launcher interface between the C ABI (qmm_api.cu) and the kernel
// translation units.  Launchers assume their arguments were validated by the
// C ABI; they enqueue kernels on `stream` and return the launch status.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace qmm {

constexpr int kQK = 32;  // elements per quantization block

// quant.cu
cudaError_t launch_quantize_act_q8_0(const float *x, int64_t m, int64_t k, int64_t ldx,
                                     int8_t *aq, uint16_t *ad, cudaStream_t s);
cudaError_t launch_quantize_weight_q4_0(const float *w, int64_t n, int64_t k,
                                        uint8_t *wq, uint16_t *wd, cudaStream_t s);
cudaError_t launch_quantize_act_bitnet(const float *x, int64_t m, int64_t k, int8_t *aq,
                                       float *scale, int32_t *sum, cudaStream_t s);
cudaError_t launch_pack_ternary(const int8_t *t, int64_t n, int64_t k, uint32_t *w,
                                cudaStream_t s);

// gemv.cu
int gemv_auto_split(int64_t m, int64_t n, int64_t k);
size_t gemv_workspace_bytes(int64_t m, int64_t n, int64_t k, int split);
// sumi != nullptr selects the block-sum emitting variant (split must be 1).
cudaError_t launch_gemv_q4_0_q8_0(const uint8_t *wq, const uint16_t *wd, const int8_t *aq,
                                  const uint16_t *ad, float *y, int32_t *sumi, int64_t m,
                                  int64_t n, int64_t k, int split, float *partials,
                                  cudaStream_t s);
// Split-K GEMV whose partials live in a library-owned device array of
// kGemvNoAllocScratchFloats floats (split * m * n must fit).
constexpr int64_t kGemvNoAllocScratchFloats = int64_t(1) << 20;
cudaError_t launch_gemv_q4_0_q8_0_noalloc(const uint8_t *wq, const uint16_t *wd, const int8_t *aq,
                                          const uint16_t *ad, float *y, int64_t m, int64_t n,
                                          int64_t k, int split, cudaStream_t s);
cudaError_t launch_bitnet_gemv(const uint32_t *w, float absmean, const int8_t *aq,
                               const float *scale, const int32_t *sum, float *y, int32_t *dot,
                               int64_t m, int64_t n, int64_t k, cudaStream_t s);

// gemm.cu
size_t gemm_workspace_bytes(int64_t m, int64_t n, int64_t k);
// sumi != nullptr selects the block-sum emitting variant.
cudaError_t launch_gemm_q4_0_q8_0(const uint8_t *wq, const uint16_t *wd, const int8_t *aq,
                                  const uint16_t *ad, float *y, int32_t *sumi, int64_t m,
                                  int64_t n, int64_t k, void *workspace, cudaStream_t s);
// Reads and clears the GEMM kernels' device error word (after the caller
// synchronized).  Returns the raw word: 0 = no error.
cudaError_t gemm_read_and_clear_error(unsigned int *word, cudaStream_t s);
void gemm_set_wait_limit(uint32_t iterations);
void gemm_set_withhold_loads(int enable);

}  // namespace qmm
