// Streaming decode GEMV: the Q4_0 x Q8_0 product of the decode GEMV (llama.cpp
// visual guide, lesson 31 "The CPU backend", section "How the quantized dot
// product works") with the weight stream staged through shared memory by the
// bulk-copy engine instead of registers.
//
// A persistent CTA (one per SM) runs one producer warp and kConsumerWarps
// consumer warps over a ring of shared-memory stages.  A stage holds
// one tile: kTileRows consecutive weight rows x kChunkBlocks blocks (their
// nibbles and fp16 scales).  The producer fills a stage with two tensor
// copies (cp.async.bulk.tensor; the nibbles viewed as a 2-D uint64 tensor
// [n, k/16] with a 256 x 16 box, the scales as uint16 [n, k/32] with a
// 128 x 16 box; completion counted in bytes on the stage's "full" mbarrier,
// boxes past the matrix edge filled with zeros that no consumer reads);
// consumers wait on "full", copy their rows to registers, release the stage
// on its "empty" mbarrier and compute.  Up to kMaxStages * 36 KiB per SM are
// in flight whatever the register budget, so the HBM stream does not stall on
// CTA turnover.  The consumers first stage every problem's quantized
// activations in shared memory (codes, f32 scales and per-block code sums):
// with the HBM queues full, any load that reaches memory waits microseconds,
// so nothing on the consumers' path after that reads global memory.
//
// Work order: the CTA takes row groups (of kTileRows rows) i = blockIdx.x,
// +gridDim.x, ... over all problems of the table, and every row group's k
// chunks in order.  Consumer warp w owns rows 2w, 2w+1 of the tile; lane l
// takes the blocks l, l+32, l+64, l+96 of each chunk, i.e. the blocks l + 32j
// of the row in ascending order, exactly as the register GEMV does, and the
// lane partials are summed by the same xor-shuffle tree, so the two kernels
// give identical bits.
//
// With programmatic dependent launch the producer starts streaming weights
// (model parameters) at once; consumers wait for the previous kernel on the
// stream (griddepcontrol.wait) before they read the activations.
//
// Every mbarrier wait is bounded: after the poll limit the waiting role sets
// an abort flag and the library's error word (QMM_ERR_TIMEOUT through
// qmm_check_device_error), every role stops, and the CTA waits (again with a
// limit) for the copies it issued before it exits.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (kConsumerWarps + 1);  // + the producer warp
constexpr int kRowsPerWarp = 2;
constexpr int kTileRows = kConsumerWarps * kRowsPerWarp;  // 16
constexpr int kChunkBlocks = 128;                          // blocks per row in one stage
constexpr int kRowWBytes = kChunkBlocks * 16;              // nibble bytes per tile row
constexpr int kRowSBytes = kChunkBlocks * 2;               // scale bytes per tile row
constexpr int kStageBytes = kTileRows * (kRowWBytes + kRowSBytes);  // 36 KiB
constexpr int kMaxStages = 6;
constexpr int kMinStages = 2;
constexpr int kStreamMinM = 8;  // smallest m this kernel serves
constexpr int kSmemLimit = 227 * 1024;  // dynamic shared memory of one CTA
// full[kMaxStages], empty[kMaxStages], the activation barrier, the abort flag
constexpr int kBarBytes = 2 * kMaxStages * 8 + 8 + 8;

// What the work loops need of each problem, copied to shared memory at entry:
// the hot loops then never read the (large) parameter table, whose constant-
// cache misses would cost a trip to L2 each while HBM queues are full.
struct Meta {
    int64_t group_end;  // cumulative row groups up to and including this problem
    int64_t n;
    float *y;
    int k;
    uint32_t act_off;
};
constexpr int kMetaBytes = kGroupMax * (int)sizeof(Meta);

constexpr uint32_t kErrTimeout = 1u;
constexpr uint32_t kSuspendHintNs = 20000;
constexpr uint32_t kDefaultWaitLimit = 1u << 17;

__device__ unsigned int g_stream_error = 0;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}
// true when the phase completed; false after `limit` polls or once another
// role raised the abort flag (which this call then also raises)
__device__ __forceinline__ bool wait_bounded(uint64_t *bar, uint32_t parity, uint32_t limit,
                                             volatile int *abort_flag) {
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag || it >= limit) {
            *abort_flag = 1;
            atomicOr(&g_stream_error, kErrTimeout);
            return false;
        }
    }
}
__device__ __forceinline__ bool wait_bounded_warp(uint64_t *bar, uint32_t parity, uint32_t limit,
                                                  volatile int *abort_flag) {
    return __all_sync(0xffffffffu, wait_bounded(bar, parity, limit, abort_flag));
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// The problem table plus, per problem, the tensor maps of its nibbles and
// scales and the shared-memory offset of its staged activations; a kernel
// parameter read in place.
struct StreamTable {
    CUtensorMap wmap[kGroupMax];
    CUtensorMap smap[kGroupMax];
    LinearGroup g;
    uint32_t act_off[kGroupMax];  // from the start of the activation region
    uint32_t act_base;            // = stages * kStageBytes
    uint32_t bar_off;
    int stages;
};

// Staged activations of one problem (m rows of k), in shared memory:
//   codes int8 [m][k]      the Q8_0 codes, as in global memory
//   ad    fp16 [m][k/32]   the Q8_0 scales, as in global memory
//   asum  int  [m][k/32]   sum of each block's codes (for the -8 offset)
// codes and ad arrive by two bulk copies; asum is computed in place.
__host__ __device__ constexpr uint32_t act_bytes(int m, int64_t k) {
    return (uint32_t)(m * k + 6 * m * (k / kQK));
}
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ int dp4a_us(unsigned a, int b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ float h2f(unsigned short h) {
    return __half2float(__ushort_as_half(h));
}

// problem of row group i
__device__ __forceinline__ int problem_of(const Meta *meta, int count, int64_t i) {
    int p = 0;
    while (p + 1 < count && i >= meta[p].group_end) ++p;
    return p;
}

__device__ __forceinline__ void tmap_prefetch(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

template <int MT, bool PDL>
__global__ void __launch_bounds__(kThreads, 1)
gemv_stream_kernel(const __grid_constant__ StreamTable st_tab, uint32_t wait_limit, int withhold) {
    const LinearGroup &tab = st_tab.g;
    extern __shared__ __align__(128) unsigned char smem[];
    const int stages = st_tab.stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + st_tab.bar_off);
    uint64_t *empty = full + stages;
    uint64_t *act_bar = empty + stages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(act_bar + 1);
    unsigned char *act = smem + st_tab.act_base;
    Meta *meta = reinterpret_cast<Meta *>(smem + st_tab.bar_off + kBarBytes);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int count = tab.count;
    const int64_t groups = tab.cta_end[count - 1];
    if (threadIdx.x < count) {
        const int p = threadIdx.x;
        meta[p] = {tab.cta_end[p], tab.p[p].n, tab.p[p].y, (int)tab.p[p].k, st_tab.act_off[p]};
    } else if (warp == kConsumerWarps && lane >= 16 && lane - 16 < count) {
        tmap_prefetch(&st_tab.wmap[lane - 16]);
        tmap_prefetch(&st_tab.smap[lane - 16]);
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_init(act_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (PDL) pdl_launch_dependents();

    if (warp == kConsumerWarps) {
        // ---------------- producer: weights and scales into the ring
        uint32_t st = 0;  // stages armed so far
        bool ok = true;
        for (int64_t i = blockIdx.x; ok && i < groups; i += gridDim.x) {
            const int p = problem_of(meta, count, i);
            const int64_t row0 = (i - (p ? meta[p - 1].group_end : 0)) * kTileRows;
            const int kb = meta[p].k / kQK;
            for (int c0 = 0; c0 < kb; c0 += kChunkBlocks) {
                const int s = (int)(st % stages);
                const uint32_t ph = (st / stages) & 1u;
                if (!wait_bounded_warp(&empty[s], ph ^ 1u, wait_limit, abort_flag)) {
                    ok = false;
                    break;
                }
                if (withhold) {  // test hook: arm nothing, so the consumers' waits run out
                    ++st;
                    continue;
                }
                if (lane == 0) {
                    unsigned char *stage = smem + s * kStageBytes;
                    // whole boxes land, including their zero-filled parts
                    mbar_arrive_expect_tx(&full[s], (uint32_t)kStageBytes);
                    tma_load_2d(stage, &st_tab.wmap[p], &full[s], c0 * 2, (int)row0);
                    tma_load_2d(stage + kTileRows * kRowWBytes, &st_tab.smap[p], &full[s], c0,
                                (int)row0);
                }
                __syncwarp();
                ++st;
            }
        }
        // No CTA may exit while copies it issued are still landing: wait (with
        // the limit) until the last armed stages completed.  In a normal run
        // the consumers have waited for them already.
        if (lane == 0 && !withhold) {
            const uint32_t first = st > (uint32_t)stages ? st - stages : 0;
            for (uint32_t j = first; j < st; ++j)
                for (uint32_t it = 0;
                     it < wait_limit && !mbar_try_wait(&full[j % stages], (j / stages) & 1u);
                     ++it) {
                }
        }
        return;
    }

    // ---------------- consumers
    if (PDL) pdl_wait();  // the activations may come from the previous kernel
    const int m = tab.m;
    // stage every problem's activations once: two bulk copies per problem
    // (one round trip for all of them), then the block sums in place
    if (threadIdx.x == 0) {
        uint32_t bytes = 0;
        for (int p = 0; p < count; ++p) {
            const int64_t kb = tab.p[p].k / kQK;
            bytes += (uint32_t)(m * tab.p[p].k + 2 * m * kb);
        }
        mbar_arrive_expect_tx(act_bar, bytes);
        for (int p = 0; p < count; ++p) {
            const LinearProblem &P = tab.p[p];
            unsigned char *a = act + st_tab.act_off[p];
            bulk_load(a, P.aq, (uint32_t)(m * P.k), act_bar);
            bulk_load(a + m * P.k, P.ad, (uint32_t)(2 * m * (P.k / kQK)), act_bar);
        }
    }
    if (!wait_bounded(act_bar, 0, wait_limit, abort_flag)) return;
    for (int p = 0; p < count; ++p) {
        const int k = meta[p].k, kb = k / kQK;
        const unsigned char *a = act + meta[p].act_off;
        int *asum = reinterpret_cast<int *>(const_cast<unsigned char *>(a) + m * k + 2 * m * kb);
        for (int it = threadIdx.x; it < m * kb; it += 32 * kConsumerWarps) {
            const int4 *q = reinterpret_cast<const int4 *>(a + it * kQK);  // row t, block b
            const int4 a0 = q[0], a1 = q[1];
            int sum = dp4a_us(0x01010101u, a0.x, 0);
            sum = dp4a_us(0x01010101u, a0.y, sum);
            sum = dp4a_us(0x01010101u, a0.z, sum);
            sum = dp4a_us(0x01010101u, a0.w, sum);
            sum = dp4a_us(0x01010101u, a1.x, sum);
            sum = dp4a_us(0x01010101u, a1.y, sum);
            sum = dp4a_us(0x01010101u, a1.z, sum);
            sum = dp4a_us(0x01010101u, a1.w, sum);
            asum[it] = sum;
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumerWarps) : "memory");

    uint32_t st = 0;
    const int r0 = warp * kRowsPerWarp;
    for (int64_t i = blockIdx.x; i < groups; i += gridDim.x) {
        const int p = problem_of(meta, count, i);
        const Meta mp = meta[p];
        const int64_t row0 = (i - (p ? meta[p - 1].group_end : 0)) * kTileRows;
        const int kb = mp.k / kQK;
        const int k = mp.k;
        const int8_t *codes = reinterpret_cast<const int8_t *>(act + mp.act_off);
        const unsigned short *ads = reinterpret_cast<const unsigned short *>(codes + m * k);
        const int *asums = reinterpret_cast<const int *>(codes + m * k + 2 * m * kb);
        float acc[kRowsPerWarp][MT];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
            for (int t = 0; t < MT; ++t) acc[r][t] = 0.0f;
        for (int c0 = 0; c0 < kb; c0 += kChunkBlocks, ++st) {
            const int s = (int)(st % stages);
            const uint32_t ph = (st / stages) & 1u;
            if (!wait_bounded_warp(&full[s], ph, wait_limit, abort_flag)) return;
            const int cb = kb - c0 < kChunkBlocks ? kb - c0 : kChunkBlocks;
            const unsigned char *wst = smem + s * kStageBytes;
            const unsigned short *sst =
                reinterpret_cast<const unsigned short *>(wst + kTileRows * kRowWBytes);
            uint4 wv[4][kRowsPerWarp];
            unsigned short dwv[4][kRowsPerWarp];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int b = lane + 32 * u;
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; ++r) {
                    if (b < cb && row0 + r0 + r < mp.n) {
                        wv[u][r] = *reinterpret_cast<const uint4 *>(wst + (r0 + r) * kRowWBytes +
                                                                    b * 16);
                        dwv[u][r] = sst[(r0 + r) * kChunkBlocks + b];
                    } else {
                        wv[u][r] = make_uint4(0x88888888u, 0x88888888u, 0x88888888u,
                                              0x88888888u);
                        dwv[u][r] = 0;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);  // the stage is in registers now
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int b = lane + 32 * u;
                if (b >= cb) break;
                const int gb = c0 + b;
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    if (t >= m) break;
                    const int4 a0 = *reinterpret_cast<const int4 *>(codes + t * k + gb * kQK);
                    const int4 a1 = *reinterpret_cast<const int4 *>(codes + t * k + gb * kQK + 16);
                    const float da = h2f(ads[t * kb + gb]);
                    const int asum = asums[t * kb + gb];
#pragma unroll
                    for (int r = 0; r < kRowsPerWarp; ++r) {
                        const uint4 w = wv[u][r];
                        int sm = -8 * asum;
                        sm = dp4a_us(w.x & 0x0F0F0F0Fu, a0.x, sm);
                        sm = dp4a_us(w.y & 0x0F0F0F0Fu, a0.y, sm);
                        sm = dp4a_us(w.z & 0x0F0F0F0Fu, a0.z, sm);
                        sm = dp4a_us(w.w & 0x0F0F0F0Fu, a0.w, sm);
                        sm = dp4a_us((w.x >> 4) & 0x0F0F0F0Fu, a1.x, sm);
                        sm = dp4a_us((w.y >> 4) & 0x0F0F0F0Fu, a1.y, sm);
                        sm = dp4a_us((w.z >> 4) & 0x0F0F0F0Fu, a1.z, sm);
                        sm = dp4a_us((w.w >> 4) & 0x0F0F0F0Fu, a1.w, sm);
                        const float sc = __fmul_rn(h2f(dwv[u][r]), da);
                        acc[r][t] = fmaf((float)sm, sc, acc[r][t]);
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                float v = acc[r][t];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                acc[r][t] = v;
            }
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                const int64_t row = row0 + r0 + r;
                if (row >= mp.n) break;
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    if (t >= m) break;
                    mp.y[(int64_t)t * mp.n + row] = acc[r][t];
                }
            }
        }
    }
}

// Shared-memory plan: activations of every problem, then as many weight
// stages as fit (kMinStages at least), then the barriers.
bool plan_smem(const LinearGroup &g, StreamTable *tab, size_t *bytes) {
    uint32_t act = 0;
    for (int p = 0; p < g.count; ++p) {
        if (tab) tab->act_off[p] = act;
        act += (act_bytes(g.m, g.p[p].k) + 15u) & ~15u;
    }
    const int64_t room = (int64_t)kSmemLimit - kBarBytes - kMetaBytes - act;
    int stages = (int)(room / kStageBytes);
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < kMinStages) return false;
    if (tab) {
        tab->stages = stages;
        // stages first (tensor-copy destinations at 128-byte multiples)
        tab->act_base = (uint32_t)(stages * kStageBytes);
        tab->bar_off = tab->act_base + act;
    }
    if (bytes) *bytes = (size_t)stages * kStageBytes + act + kBarBytes + kMetaBytes;
    return true;
}

uint32_t g_wait_limit = kDefaultWaitLimit;
int g_withhold = 0;
std::atomic<uint64_t> g_opted_in[2][5];  // per PDL flag and MT: bit per device
std::atomic<int> g_sm_count[64];

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D row-major map over [outer, inner] elements with rows row_bytes apart
bool encode_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t inner,
               uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
    auto fn = get_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MT>
cudaError_t launch_mt(const LinearGroup &g, bool pdl, cudaStream_t s) {
    StreamTable tab;
    tab.g = g;
    size_t smem_bytes = 0;
    if (!plan_smem(g, &tab, &smem_bytes)) return cudaErrorInvalidValue;
    int64_t total = 0;
    for (int p = 0; p < g.count; ++p) {
        const LinearProblem &P = g.p[p];
        total += (P.n + kTileRows - 1) / kTileRows;
        tab.g.cta_end[p] = total;
        const uint64_t kb = (uint64_t)(P.k / kQK);
        if (!encode_2d(&tab.wmap[p], CU_TENSOR_MAP_DATA_TYPE_UINT64, P.wq, (uint64_t)P.k / 16,
                       (uint64_t)P.n, (uint64_t)P.k / 2, kRowWBytes / 8, kTileRows) ||
            !encode_2d(&tab.smap[p], CU_TENSOR_MAP_DATA_TYPE_UINT16, P.wd, kb, (uint64_t)P.n,
                       kb * 2, kChunkBlocks, kTileRows))
            return cudaErrorInvalidValue;
    }
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
    auto kernel = pdl ? gemv_stream_kernel<MT, true> : gemv_stream_kernel<MT, false>;
    constexpr int mt_index = MT == 1 ? 0 : MT == 2 ? 1 : MT == 4 ? 2 : MT == 8 ? 3 : 4;
    std::atomic<uint64_t> &mask = g_opted_in[pdl ? 1 : 0][mt_index];
    if (!(mask.load(std::memory_order_acquire) >> dev & 1)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        mask.fetch_or(uint64_t(1) << dev, std::memory_order_acq_rel);
    }
    const int64_t grid = total < sms ? total : sms;
    return launch_kernel(kernel, dim3((unsigned)grid), dim3(kThreads), smem_bytes, s, pdl,
                         tab, g_wait_limit, g_withhold);
}

}  // namespace

bool stream_gemv_supported(const LinearGroup &tab) {
    for (int p = 0; p < tab.count; ++p) {
        const LinearProblem &P = tab.p[p];
        // bulk copies need 16-byte aligned sources and sizes: every scale row
        // and chunk starts on a 16-byte boundary when k/32 is a multiple of 8
        if ((P.k / kQK) % 8 != 0) return false;
        if ((reinterpret_cast<uintptr_t>(P.wd) & 15) || (reinterpret_cast<uintptr_t>(P.wq) & 15) ||
            (reinterpret_cast<uintptr_t>(P.ad) & 15) || (reinterpret_cast<uintptr_t>(P.aq) & 15))
            return false;
    }
    // at m < 8 the register GEMV is faster: this kernel's start (shared
    // memory set-up, the first tile's round trip) costs more than it saves
    return tab.m >= kStreamMinM && tab.m <= 16 && plan_smem(tab, nullptr, nullptr);
}

cudaError_t launch_stream_gemv(const LinearGroup &tab, bool pdl, cudaStream_t s) {
    const int m = tab.m;
    if (m == 1) return launch_mt<1>(tab, pdl, s);
    if (m == 2) return launch_mt<2>(tab, pdl, s);
    if (m <= 4) return launch_mt<4>(tab, pdl, s);
    if (m <= 8) return launch_mt<8>(tab, pdl, s);
    return launch_mt<16>(tab, pdl, s);
}

void stream_set_wait_limit(uint32_t iterations) {
    g_wait_limit = iterations ? iterations : kDefaultWaitLimit;
}

void stream_set_withhold_loads(int enable) { g_withhold = enable ? 1 : 0; }

cudaError_t stream_read_and_clear_error(unsigned int *word, cudaStream_t s) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_stream_error, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    if (*word) {
        e = cudaMemcpyToSymbolAsync(g_stream_error, &zero, sizeof(unsigned int), 0,
                                    cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

}  // namespace qmm
