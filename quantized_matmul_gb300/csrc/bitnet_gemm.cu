// BitNet ternary matrix product for prefill on the 5th-generation tensor
// cores (Loom docs, "Plan 9 SIMD Forward", section "BitNet ternary MAD
// kernel": dot = sum(code * q) - sum(q), y = dot * absmean / scale).
//
// What it computes: dot[t, r] = sum_j (code[r, j] - 1) * q[t, j], the same
// integer as the identity above, and y[t, r] = scale[t] == 0 ? 0 :
// ((float)dot * absmean) / scale[t] (two IEEE f32 operations), bit for bit
// the result of the ternary GEMV.
//
// How (GB300, sm_103a).  Every operand is a small integer that fp16 holds
// exactly (weights -1, 0, 1; activations -127..127) and |dot| <= 127 * k <
// 2^24 for k <= 2^17, so tcgen05.mma kind::f16 with an f32 accumulator
// computes dot exactly over the whole k: unlike the Q4_0 product there are
// no per-block scales, so the tile's accumulator stays in TMEM until the end
// and the CUDA cores only run the epilogue.
//
// A persistent CTA (one per SM) walks output tiles of 128 weight rows x BN
// tokens (t = blockIdx.x, + gridDim.x, ...).  Roles:
//   warp 0      TMA producer: per stage of 64 k-elements the 128 x 16 B code
//               tile and the BN x 64 fp16 activation tile (128-byte swizzle).
//   warp 1      allocates TMEM; lane 0 issues the four K=16 MMAs of a stage
//               into the tile's accumulator (two in TMEM, so one tile's
//               epilogue overlaps the next tile's MMAs).
//   warps 2-5   converters: all four convert every stage together, 32 rows
//               each, turning the codes into the 128-byte-swizzled K-major
//               fp16 A tile (value code - 1); the stage is ready when all
//               four have arrived.
//   warps 6-21  epilogue: thread (warp % 4, lane) owns a weight row (a TMEM
//               lane quarter is readable only from the sub-partition with the
//               same index) and BN / 4 columns of the tile.
// Every mbarrier wait is bounded; on expiry the kernel records
// QMM_ERR_TIMEOUT in its device error word, waits (bounded) for its copies
// and MMAs in flight, frees TMEM and returns.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>

#include "qmm_internal.h"
#include "tcgen05.cuh"

namespace qmm {
namespace {

constexpr int kBM = 128;        // weight rows per tile (MMA M)
constexpr int kBK = 64;         // k-elements per stage
constexpr int kBN = 256;        // tokens per tile (MMA N)
constexpr int kStages = 4;
constexpr int kConvWarps = 4;   // each converts 32 rows of every stage
constexpr int kConvWarp0 = 2;
constexpr int kEpiWarp0 = kConvWarp0 + kConvWarps;
constexpr int kEpiWarps = 16;   // 4 lane quarters x 4 column groups
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kAccBufs = 2;     // TMEM accumulators (2 x 256 columns)

constexpr int kA = kBM * kBK * 2;      // fp16 weights, 16 KB
constexpr int kB = kBN * kBK * 2;      // fp16 activations, 32 KB
constexpr int kCodes = kBM * kBK / 4;  // 2-bit codes, 2 KB
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kA;
constexpr int kOffCodes = kOffB + kStages * kB;
constexpr int kOffBar = kOffCodes + kStages * kCodes;
constexpr int kNumBars = 3 * kStages + 2 * kAccBufs + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // slack for the 1024-byte round-up
static_assert(kOffB % 1024 == 0 && kB % 1024 == 0, "swizzled tiles are 1024-byte aligned");
static_assert(kBM == 32 * kConvWarps, "one row per converter lane and stage");

__device__ unsigned int g_bitnet_gemm_error = 0;

__device__ __forceinline__ bool wait_bounded(uint64_t *bar, uint32_t parity, uint32_t limit,
                                             volatile int *abort_flag) {
    return wait_bounded_err(bar, parity, limit, abort_flag, &g_bitnet_gemm_error);
}
__device__ __forceinline__ bool wait_bounded_warp(uint64_t *bar, uint32_t parity, uint32_t limit,
                                                  volatile int *abort_flag) {
    return wait_bounded_warp_err(bar, parity, limit, abort_flag, &g_bitnet_gemm_error);
}

// 16 codes of one word (element i at bits 2i) -> 16 fp16 values code - 1, in
// element order.  The fp16 bit pattern 0x6400 | c is the value 1024 + c, so
// (0x6400 | c) - 1025 = c - 1, exactly.
__device__ __forceinline__ void codes_to_f16(uint32_t w, uint32_t (&out)[8]) {
    const __half2 off = __halves2half2(__ushort_as_half(0x6401), __ushort_as_half(0x6401));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t t = w >> (4 * i);  // codes 2i (bits 0-1) and 2i+1 (bits 2-3)
        const uint32_t pair = (t & 3u) | ((t << 14) & 0x30000u) | 0x64006400u;
        __half2 h;
        memcpy(&h, &pair, 4);
        h = __hsub2(h, off);
        memcpy(&out[i], &h, 4);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
bitnet_gemm_kernel(const __grid_constant__ CUtensorMap tm_codes,
                   const __grid_constant__ CUtensorMap tm_act, float absmean,
                   const float *__restrict__ act_scale, float *__restrict__ y, int m, int n,
                   int k, uint32_t wait_limit) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *bar_load = bar;                   // TMA landed
    uint64_t *bar_conv = bar + kStages;         // A tile written
    uint64_t *bar_empty = bar + 2 * kStages;    // the stage's MMAs completed
    uint64_t *bar_accf = bar + 3 * kStages;     // accumulator holds a finished tile
    uint64_t *bar_acce = bar_accf + kAccBufs;   // epilogue done with the accumulator
    uint64_t *bar_drain = bar_acce + kAccBufs;  // final MMA completion
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int m_tiles = (m + kBN - 1) / kBN;
    const int tiles = m_tiles * ((n + kBM - 1) / kBM);
    const int ksteps = (k + kBK - 1) / kBK;
    constexpr uint32_t kTmemCols = kAccBufs * kBN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bar_load[s], 1);
            mbar_init(&bar_conv[s], kConvWarps);
            mbar_init(&bar_empty[s], 1);
        }
        for (int b = 0; b < kAccBufs; ++b) {
            mbar_init(&bar_accf[b], 1);
            mbar_init(&bar_acce[b], kEpiWarps);
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tmap_prefetch(&tm_codes);
        tmap_prefetch(&tm_act);
    }
    if (warp == 1) tmem_alloc(tmem_holder, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    // tile -> (first weight row, first token); consecutive tiles share rows
    auto tile_coords = [&](int tile, int &n0, int &t0) {
        n0 = (tile / m_tiles) * kBM;
        t0 = (tile % m_tiles) * kBN;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        uint32_t st = 0;  // stages issued
        bool ok = true;
        for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
            int n0, t0;
            tile_coords(tile, n0, t0);
            for (int ks = 0; ks < ksteps; ++ks, ++st) {
                const int s = (int)(st % kStages);
                const uint32_t ph = (st / kStages) & 1u;
                if (!wait_bounded_warp(&bar_empty[s], ph ^ 1u, wait_limit, abort_flag)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bar_load[s], (uint32_t)(kCodes + kB));
                    tma_load_2d(smem + kOffCodes + s * kCodes, &tm_codes, &bar_load[s], ks * 4, n0);
                    tma_load_2d(smem + kOffB + s * kB, &tm_act, &bar_load[s], ks * kBK, t0);
                }
                __syncwarp();
            }
        }
        // never leave a copy in flight
        for (uint32_t j = st > (uint32_t)kStages ? st - kStages : 0; j < st; ++j) {
            volatile int no_abort = 0;
            wait_bounded_warp(&bar_load[j % kStages], (j / kStages) & 1u, kDrainLimit, &no_abort);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(kBM, kBN);
            const uint64_t a_desc0 = smem_desc_sw128(smem_u32(smem + kOffA));
            const uint64_t b_desc0 = smem_desc_sw128(smem_u32(smem + kOffB));
            uint32_t st = 0;
            int issued_any = 0, tcount = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x, ++tcount) {
                const int ab = tcount % kAccBufs;
                const uint32_t aph = (uint32_t)(tcount / kAccBufs) & 1u;
                if (!wait_bounded(&bar_acce[ab], aph ^ 1u, wait_limit, abort_flag)) break;
                const uint32_t d = tmem_base + (uint32_t)(ab * kBN);
                for (int ks = 0; ks < ksteps; ++ks, ++st) {
                    const int s = (int)(st % kStages);
                    const uint32_t ph = (st / kStages) & 1u;
                    if (!wait_bounded(&bar_conv[s], ph, wait_limit, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a_desc = a_desc0 + (uint64_t)(s * (kA >> 4));
                    const uint64_t b_desc = b_desc0 + (uint64_t)(s * (kB >> 4));
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_f16(d, a_desc + 2 * kk, b_desc + 2 * kk, idesc,
                                (ks > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&bar_empty[s]);
                    issued_any = 1;
                }
                if (ok) mma_commit(&bar_accf[ab]);
            }
            if (issued_any) {
                mma_commit(bar_drain);
                volatile int no_abort = 0;
                wait_bounded(bar_drain, 0, kDrainLimit, &no_abort);
            }
        }
        __syncwarp();
    } else if (warp >= kConvWarp0 && warp < kConvWarp0 + kConvWarps) {
        // ------------------------------------------------------------ converters
        // Every converter takes every stage of the CTA's stage sequence, in
        // order: converter c, lane l converts row 32c + l, one 16-byte read
        // (64 codes) and eight swizzled 16-byte stores.
        const int cw = warp - kConvWarp0;
        const int row = 32 * cw + lane;
        const int per_cta = ((tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x) * ksteps;
        for (int stg = 0; stg < per_cta; ++stg) {
            const int s = stg % kStages;
            const uint32_t ph = (uint32_t)(stg / kStages) & 1u;
            if (!wait_bounded_warp(&bar_load[s], ph, wait_limit, abort_flag)) break;
            const uint8_t *codes = smem + kOffCodes + s * kCodes;
            uint8_t *a_tile = smem + kOffA + s * kA;
            const uint4 w4 = *reinterpret_cast<const uint4 *>(codes + row * 16);
            const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {  // word q: elements 16q .. 16q+15 (chunks 2q, 2q+1)
                uint32_t h[8];
                codes_to_f16(w[q], h);
                *reinterpret_cast<uint4 *>(a_tile + row * 128 + (((2 * q) ^ (row & 7)) * 16)) =
                    make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4 *>(a_tile + row * 128 + (((2 * q + 1) ^ (row & 7)) * 16)) =
                    make_uint4(h[4], h[5], h[6], h[7]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_conv[s]);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - kEpiWarp0;
        const int q = warp & 3;             // TMEM lane quarter = sub-partition
        const int grp = ew >> 2;            // column group 0..3
        constexpr int kCols = kBN / 4;      // 64 columns per thread
        int tcount = 0;
        for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++tcount) {
            int n0, t0;
            tile_coords(tile, n0, t0);
            const int ab = tcount % kAccBufs;
            if (!wait_bounded_warp(&bar_accf[ab], (uint32_t)(tcount / kAccBufs) & 1u, wait_limit,
                                   abort_flag))
                break;
            tc_fence_after();
            const int row = n0 + 32 * q + lane;
            const uint32_t col0 = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(ab * kBN + grp * kCols);
#pragma unroll 1
            for (int g = 0; g < kCols / 16; ++g) {
                uint32_t v[16];
                tmem_ld16(col0 + 16 * g, v);
                tmem_wait_ld();
                if (row < n) {
                    // the chunk's 16 activation scales: four 16-byte loads
                    // where the whole chunk exists and is aligned
                    const int tc = t0 + grp * kCols + 16 * g;
                    float sc[16];
                    if (tc + 16 <= m && (reinterpret_cast<uintptr_t>(act_scale + tc) & 15) == 0) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float4 f = __ldg(reinterpret_cast<const float4 *>(act_scale + tc) + i);
                            sc[4 * i] = f.x;
                            sc[4 * i + 1] = f.y;
                            sc[4 * i + 2] = f.z;
                            sc[4 * i + 3] = f.w;
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 16; ++c) sc[c] = tc + c < m ? __ldg(act_scale + tc + c) : 0.0f;
                    }
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const int t = tc + c;
                        if (t < m) {
                            const float s = sc[c];
                            // dot is the exact integer the accumulator holds; a
                            // zero dot gives the integer's +0, whatever sign the
                            // accumulator's zero carries
                            const float dot = __uint_as_float(v[c]);
                            const float out = (s == 0.0f || dot == 0.0f)
                                                  ? 0.0f
                                                  : __fdiv_rn(__fmul_rn(dot, absmean), s);
                            y[(int64_t)t * n + row] = out;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_acce[ab]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// int8 activations -> fp16 (exact), 16 per thread and turn.
__global__ void bitnet_gemm_prep_kernel(const int8_t *__restrict__ aq, __half *__restrict__ a16,
                                        int64_t count16) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < count16; g += stride) {
        const int4 v = reinterpret_cast<const int4 *>(aq)[g];
        const int w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int lo = (int)(int8_t)((w[i] >> (16 * j)) & 0xff);
                const int hi = (int)(int8_t)((w[i] >> (16 * j + 8)) & 0xff);
                __half2 hv = __halves2half2(__int2half_rn(lo), __int2half_rn(hi));
                memcpy(&o[2 * i + j], &hv, 4);
            }
        }
        uint4 *dst = reinterpret_cast<uint4 *>(a16) + 2 * g;
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

uint32_t g_wait_limit = kDefaultWaitLimit;
std::atomic<uint64_t> g_opted_in;  // bit per device
std::atomic<int> g_sm_count[64];

}  // namespace

size_t bitnet_gemm_workspace_bytes(int64_t m, int64_t k) {
    return ((size_t)m * (size_t)k * 2 + 255) / 256 * 256;
}

cudaError_t launch_bitnet_gemm(const uint32_t *w, float absmean, const int8_t *aq,
                               const float *act_scale, float *y, int64_t m, int64_t n, int64_t k,
                               void *workspace, cudaStream_t s) {
    __half *a16 = static_cast<__half *>(workspace);
    {
        const int threads = 256;
        const int64_t count16 = m * k / 16;
        const int64_t blocks = std::min<int64_t>((count16 + threads - 1) / threads, 152 * 8);
        bitnet_gemm_prep_kernel<<<(unsigned)std::max<int64_t>(blocks, 1), threads, 0, s>>>(
            aq, a16, count16);
        cudaError_t e = cudaPeekAtLastError();
        if (e != cudaSuccess) return e;
    }
    CUtensorMap tm_codes, tm_act;
    // codes: u32 [n rows, k/16 words], box 4 words x 128 rows
    if (!make_map_2d(&tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT32, w, (uint64_t)(k / 16), (uint64_t)n,
                     (uint64_t)(k / 16) * 4, kBK / 16, kBM, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    // activations: fp16 [m rows, k], box 64 x 256, 128-byte swizzle
    if (!make_map_2d(&tm_act, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a16, (uint64_t)k, (uint64_t)m,
                     (uint64_t)k * 2, kBK, kBN, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int sms = g_sm_count[dev].load(std::memory_order_relaxed);
    if (sms == 0) {
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_sm_count[dev].store(sms, std::memory_order_relaxed);
    }
    if (!(g_opted_in.load(std::memory_order_acquire) >> dev & 1)) {
        e = cudaFuncSetAttribute(bitnet_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes);
        if (e != cudaSuccess) return e;
        g_opted_in.fetch_or(uint64_t(1) << dev, std::memory_order_acq_rel);
    }
    const int64_t tiles = ((m + kBN - 1) / kBN) * ((n + kBM - 1) / kBM);
    const int64_t grid = tiles < sms ? tiles : sms;
    bitnet_gemm_kernel<<<(unsigned)grid, kThreads, kSmemBytes, s>>>(
        tm_codes, tm_act, absmean, act_scale, y, (int)m, (int)n, (int)k, g_wait_limit);
    return cudaPeekAtLastError();
}

void bitnet_gemm_set_wait_limit(uint32_t iterations) {
    g_wait_limit = iterations ? iterations : kDefaultWaitLimit;
}

cudaError_t bitnet_gemm_read_and_clear_error(unsigned int *word, cudaStream_t s) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_bitnet_gemm_error, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    if (*word) {
        e = cudaMemcpyToSymbolAsync(g_bitnet_gemm_error, &zero, sizeof(unsigned int), 0,
                                    cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

}  // namespace qmm
