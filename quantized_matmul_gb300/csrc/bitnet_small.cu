// BitNet ternary product for a few tokens (m <= 32) on the warp-level
// tensor-core MMA: the decode-batch shape, where the tcgen05 product's
// 128-row tiles leave most SMs idle (6912 rows are 54 tiles) and the dp4a
// GEMV's work grows with every token.
//
// What it computes is the BitNet kernel's definition (Loom docs, "Plan 9 SIMD
// Forward", section "BitNet ternary MAD kernel"): dot[t, r] = sum over the k
// elements of (code[r, e] - 1) * aq[t, e], exact in int32 (equal to the
// identity sum(code * q) - sum(q)), then y[t, r] = ((float)dot * absmean) /
// act_scale[t] in IEEE f32, left to right (0 where act_scale is 0): bit for
// bit what the ternary GEMV and the tcgen05 product give.
//
// Operands.  One mma.sync m16n8k16 (f16 operands, f32 accumulators) covers
// 16 weight rows (A) by 8 tokens (B) over one packed word: 16 codes of a
// row, code of element e at bits 2e, 2e+1.  Lane (g = lane / 4, c = lane % 4)
// holds A at rows g and g + 8, k-slots 2c, 2c+1, 2c+8, 2c+9; the slots are
// mapped to the word's elements 2c, 2c+8, 2c+1, 2c+9, so that after one
// shift by 4c the lane's pairs sit 16 bits apart: (t & 0x00030003) | 0x6400
// 6400 is the fp16 pair (1024 + code(2c), 1024 + code(2c+8)), and the same on
// t >> 2 gives elements 2c+1, 2c+9.  A prepass writes the activations as fp16
// in the matching B order, and per token and 64-element group the exact
// correction cor = -1025 * (sum of the group's 64 activations): (1024 + code) * a
// - 1025 * a = (code - 1) * a.
//
// Exactness.  A group's four MMAs are chained from C = cor.  After any subset
// S of the group's elements has been added, in whatever order the tensor
// core adds them, the value is sum over S of (code - 1) a - 1025 * (sum of
// the other elements' a), at most 1025 * 64 * 127 < 2^23.1 in magnitude: an
// integer, held exactly in f32.  The chain ends at the group's dot (at most
// 64 * 127), which is added to the running dot, an integer of magnitude at
// most 127 k < 2^24 for k <= 131072: exact too, so (float)dot is the integer
// itself.  Chains of different groups do not depend on one another, so the
// scheduler can overlap them.
//
// Layout and roles, as in the few-token Q4_0 product: a producer warp fills a
// ring of stages, each 64 weight rows x 512 elements (128 bytes of codes per
// row: one tensor copy with 128-byte swizzle, so the 16-byte chunk q of row
// r sits at chunk q ^ (r % 8) and the 8 rows a lane group reads fall in 8
// bank groups) plus the stage's activation fragments and corrections (bulk
// copies).  Sixteen consumer warps in four quartets: warp w of quartet h
// owns rows 16 w .. 16 w + 15 and groups 2 h, 2 h + 1 of every stage, and
// keeps its partial dots in registers across k; at the end of a set
// quartets 1-3 hand their partials to quartet 0 through shared memory, which
// adds them (exact: integers below 2^24) and writes y.  Four warps per
// sub-partition instead of one hide the MMA chains' and shared-memory loads'
// latency, and each warp's work per stage is a quarter.  CTAs (one per SM) are persistent
// over 64-row sets: the first is the block index, further ones come from a
// counter in the workspace (zeroed by the prepass).  A last stage with row
// set -1 and no copies ends the consumers.  The product is a programmatic
// dependent launch after the prepass; every mbarrier wait is bounded.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "qmm_internal.h"
#include "tcgen05.cuh"

namespace qmm {
namespace {

constexpr int kBsRows = 64;         // weight rows per set (4 warps x one 16-row unit)
constexpr int kBsQuartets = 4;      // consumer quartets, each on a quarter of a stage's groups
constexpr int kBsWarps = 4 * kBsQuartets;  // consumer warps
constexpr int kBsThreads = 32 * (kBsWarps + 1);
constexpr int kBsGroups = 8;        // 64-element groups (16-byte chunks) per stage
constexpr int kBsQGroups = kBsGroups / kBsQuartets;  // groups per quartet and stage
constexpr int kBsStageElems = kBsGroups * 64;  // 512 elements, 128 bytes of codes per row

__device__ unsigned int g_bitnet_small_error = 0;

// MT: 16-token tiles; NT: 8-token tiles used per 16-token tile (1 for m <= 8)
template <int MT, int NT>
struct BsPlan {
    static constexpr int kStages = MT == 1 ? 4 : 2;
    static constexpr int kW = kBsRows * 128;                  // codes, 128-byte swizzle
    static constexpr int kA = kBsGroups * MT * NT * 1024;     // activation fragments
    static constexpr int kCor = kBsGroups * MT * 64;          // f32 corrections, 16 tokens
    static constexpr int kPart = (kBsQuartets - 1) * 4 * MT * NT * 4 * 32 * 4;  // partial dots
    static constexpr int kOffW = 0;
    static constexpr int kOffA = kOffW + kStages * kW;
    static constexpr int kOffCor = kOffA + kStages * kA;
    static constexpr int kOffPart = kOffCor + kStages * kCor;
    static constexpr int kOffBar = kOffPart + kPart;
    static constexpr int kOffMisc = kOffBar + (2 * kStages + 8) * 8;
    static constexpr int kBytes = kOffMisc + 16 + 4 * kStages;  // abort flag, stage row sets
    static constexpr int kAlloc = kBytes + 1024;                 // slack for the 1024-byte round-up
    static_assert(kW % 1024 == 0 && kA % 1024 == 0, "swizzled tiles stay 1024-byte aligned");
    static_assert(kAlloc + 1024 <= 227 * 1024, "one CTA fits one SM");
};

__device__ __forceinline__ bool bs_wait(uint64_t *bar, uint32_t parity, uint32_t limit,
                                        volatile int *abort_flag) {
    return wait_bounded_warp_err(bar, parity, limit, abort_flag, &g_bitnet_small_error, 8);
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint4 &a, uint32_t b0, uint32_t b1,
                                          const float (&c)[4]) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
          "f"(c[2]), "f"(c[3]));
}

// The lane's A registers for one packed word of rows g (w0) and g + 8 (w1):
// slots (2c, 2c+1) = elements (2c, 2c+8), slots (2c+8, 2c+9) = (2c+1, 2c+9),
// each code as the fp16 value 1024 + code.
__device__ __forceinline__ uint4 decode_word_pair(uint32_t w0, uint32_t w1, int c) {
    const uint32_t t0 = w0 >> (4 * c), t1 = w1 >> (4 * c);
    return make_uint4((t0 & 0x00030003u) | 0x64006400u, (t1 & 0x00030003u) | 0x64006400u,
                      ((t0 >> 2) & 0x00030003u) | 0x64006400u,
                      ((t1 >> 2) & 0x00030003u) | 0x64006400u);
}

template <int MT, int NT>
__global__ void __launch_bounds__(kBsThreads, 1)
bitnet_small_m_kernel(const __grid_constant__ CUtensorMap tm_w, const uint8_t *__restrict__ afrag,
                      const uint8_t *__restrict__ corrs, const float *__restrict__ act_scale,
                      float absmean, float *__restrict__ y, unsigned int *set_counter, int m, int n,
                      int nst, uint32_t wait_limit, int withhold_loads) {
    using P = BsPlan<MT, NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar_full = reinterpret_cast<uint64_t *>(smem + P::kOffBar);
    uint64_t *bar_empty = bar_full + P::kStages;
    uint64_t *bar_part = bar_empty + P::kStages;  // quartets 1.. have written a set's partials
    uint64_t *bar_pfree = bar_part + 4;           // quartet 0 has read them
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + P::kOffMisc);
    int *stage_set = reinterpret_cast<int *>(smem + P::kOffMisc + 16);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nsets = (n + kBsRows - 1) / kBsRows;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P::kStages; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_empty[s], kBsWarps);
        }
        for (int w = 0; w < 4; ++w) {
            mbar_init(&bar_part[w], kBsQuartets - 1);
            mbar_init(&bar_pfree[w], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
        tmap_prefetch(&tm_w);
    }
    __syncthreads();

    if (warp == kBsWarps) {
        // ---------------------------------------------------------------- producer
        constexpr uint32_t kTx = (uint32_t)(P::kW + P::kA + P::kCor);
        auto issue_weights = [&](int s, int rs, int j) {
            tma_load_2d(smem + P::kOffW + s * P::kW, &tm_w, &bar_full[s], j * 128, rs * kBsRows);
        };
        auto issue_acts = [&](int s, int j) {
            bulk_load(smem + P::kOffA + s * P::kA, afrag + (size_t)j * P::kA, P::kA, &bar_full[s]);
            bulk_load(smem + P::kOffCor + s * P::kCor, corrs + (size_t)j * P::kCor, P::kCor,
                      &bar_full[s]);
        };
        // first set: the block index; then sets from the counter.  The first
        // stage's codes are copied before the wait for the prepass (the codes
        // are model weights), its activations after.  withhold_loads (a test
        // hook) issues nothing.
        int rs = withhold_loads ? nsets : (int)blockIdx.x;
        const int pre = rs < nsets ? 1 : 0;
        if (lane == 0 && pre) {
            stage_set[0] = rs;
            mbar_arrive_expect_tx(&bar_full[0], kTx);
            issue_weights(0, rs, 0);
        }
        pdl_wait();
        __syncwarp();
        int it = 0;
        bool ok = true;
        while (ok && rs < nsets) {
            for (int j = 0; j < nst; ++j, ++it) {
                const int s = it % P::kStages;
                if (it >= pre) {
                    if (!bs_wait(&bar_empty[s], ((uint32_t)(it / P::kStages) & 1u) ^ 1u, wait_limit,
                                 abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        stage_set[s] = rs;
                        mbar_arrive_expect_tx(&bar_full[s], kTx);
                        issue_weights(s, rs, j);
                    }
                }
                if (lane == 0) issue_acts(s, j);
                __syncwarp();
            }
            int next = 0;
            if (lane == 0) next = (int)gridDim.x + (int)atomicAdd(set_counter, 1u);
            rs = __shfl_sync(0xffffffffu, next, 0);
        }
        // no further set: one more stage, with no copies, says so
        bool sent = false;
        if (ok && !withhold_loads) {
            const int s = it % P::kStages;
            if (bs_wait(&bar_empty[s], ((uint32_t)(it / P::kStages) & 1u) ^ 1u, wait_limit, abort_flag)) {
                if (lane == 0) {
                    stage_set[s] = -1;
                    mbar_arrive(&bar_full[s]);
                }
                sent = true;
            }
            __syncwarp();
        }
        // never leave a copy in flight (the end stage's slot, reused, is skipped)
        const int first_pending = (it > P::kStages ? it - P::kStages : 0) + (sent && it >= P::kStages ? 1 : 0);
        for (int i = first_pending; i < it; ++i) {
            volatile int no_abort = 0;
            bs_wait(&bar_full[i % P::kStages], (uint32_t)(i / P::kStages) & 1u, kDrainLimit, &no_abort);
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    // Warp w of quartet h owns rows 16 w .. 16 w + 15 of every set (one MMA
    // unit) and groups 2 h, 2 h + 1 of every stage; lane (g, c) reads rows g
    // and g + 8, whose swizzle rows are both g.
    const int g = lane >> 2, c = lane & 3;
    const int quartet = warp >> 2, wq = warp & 3;
    // partials of quartet h > 0 and warp w: MT * NT * 4 floats per lane, lane-contiguous
    float *part = reinterpret_cast<float *>(smem + P::kOffPart) + wq * (MT * NT * 4 * 32) + lane;
    constexpr int kPartStride = 4 * MT * NT * 4 * 32;  // floats per quartet
    float acc[MT][NT][4];
    int it = 0, sets = 0;
    bool ok = true;
    for (;;) {
        if (!bs_wait(&bar_full[it % P::kStages], (uint32_t)(it / P::kStages) & 1u, wait_limit,
                     abort_flag)) {
            ok = false;
            break;
        }
        const int rs = stage_set[it % P::kStages];
        if (rs < 0) break;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.0f;
        for (int j = 0; j < nst; ++j, ++it) {
            const int s = it % P::kStages;
            const uint32_t ph = (uint32_t)(it / P::kStages) & 1u;
            if (j > 0 && !bs_wait(&bar_full[s], ph, wait_limit, abort_flag)) {
                ok = false;
                break;
            }
            const uint8_t *wt = smem + P::kOffW + s * P::kW + (16 * wq + g) * 128;
            const uint8_t *at = smem + P::kOffA + s * P::kA;
            const float2 *cor = reinterpret_cast<const float2 *>(smem + P::kOffCor + s * P::kCor);
#pragma unroll
            for (int qq = 0; qq < kBsQGroups; ++qq) {
                const int q = quartet * kBsQGroups + qq;
                // 4 packed words (64 elements) of rows g and g + 8
                const uint4 w0 = *reinterpret_cast<const uint4 *>(wt + 16 * (q ^ g));
                const uint4 w1 = *reinterpret_cast<const uint4 *>(wt + 8 * 128 + 16 * (q ^ g));
                uint4 a[4];
                a[0] = decode_word_pair(w0.x, w1.x, c);
                a[1] = decode_word_pair(w0.y, w1.y, c);
                a[2] = decode_word_pair(w0.z, w1.z, c);
                a[3] = decode_word_pair(w0.w, w1.w, c);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        // B fragments of the group's 4 words for this 8-token
                        // tile: words 0-1 for all lanes, then words 2-3
                        // (lane-contiguous 16 bytes, conflict-free)
                        const uint4 *bf = reinterpret_cast<const uint4 *>(
                            at + ((q * MT + mt) * NT + nt) * 1024);
                        const uint4 b01 = bf[lane], b23 = bf[32 + lane];
                        const float2 cp = cor[(q * MT + mt) * 8 + nt * 4 + c];
                        // the group's dots, from its corrections; groups are
                        // independent chains, added to the running dots after
                        float d[4] = {cp.x, cp.y, cp.x, cp.y};
                        mma_16816(d, a[0], b01.x, b01.y, d);
                        mma_16816(d, a[1], b01.z, b01.w, d);
                        mma_16816(d, a[2], b23.x, b23.y, d);
                        mma_16816(d, a[3], b23.z, b23.w, d);
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[mt][nt][i] += d[i];
                    }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_empty[s]);
        }
        if (!ok) break;
        // quartets 1.. hand their partial dots to the warp of quartet 0 with
        // the same rows (once that warp has read the previous set's), which
        // adds them in quartet order and writes y
        if (quartet > 0) {
            if (sets > 0 && !bs_wait(&bar_pfree[wq], (uint32_t)(sets - 1) & 1u, wait_limit, abort_flag))
                break;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        part[(quartet - 1) * kPartStride + ((mt * NT + nt) * 4 + i) * 32] = acc[mt][nt][i];
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_part[wq]);
            ++sets;
            continue;
        }
        if (!bs_wait(&bar_part[wq], (uint32_t)sets & 1u, wait_limit, abort_flag)) break;
#pragma unroll
        for (int h = 1; h < kBsQuartets; ++h)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        acc[mt][nt][i] += part[(h - 1) * kPartStride + ((mt * NT + nt) * 4 + i) * 32];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_pfree[wq]);
        ++sets;
        // y = ((float)dot * absmean) / scale, the ternary GEMV's rule
        const int r0 = rs * kBsRows + 16 * wq + g;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int t = mt * 16 + nt * 8 + 2 * c + (i & 1);
                    const int r = r0 + 8 * (i >> 1);
                    if (t < m && r < n) {
                        const float st = act_scale[t];
                        y[(int64_t)t * n + r] =
                            st != 0.0f ? __fdiv_rn(__fmul_rn(acc[mt][nt][i], absmean), st) : 0.0f;
                    }
                }
    }
}

// Activation prepass, in the B-fragment order of the kernel above.  Unit u =
// ((group * mt_count + mt) * nt_count + nt) * 32 + lane covers token t = mt *
// 16 + nt * 8 + g and group q (elements 64 q ..): for each of the group's 4
// words j, the lane's registers (a[16j+2c], a[16j+2c+8]) and (a[16j+2c+1],
// a[16j+2c+9]) as fp16 (exact: -127..127): words 0-1 as 16 bytes at lane *
// 16 of the unit's 1 KB, words 2-3 at 512 + lane * 16.  The four lanes of a
// token hold all 64 of its group's activations, so their sum comes from two
// shuffle steps; lane c = 0 writes cor = -1025 * sum as float (group *
// mt_count + mt) * 16 + nt * 8 + g, so that the kernel reads tokens 2c, 2c+1
// of tile nt as one float2.  Elements past k and tokens past m are zeros.
__global__ void bitnet_small_prep_kernel(const int8_t *__restrict__ aq, uint4 *__restrict__ afrag,
                                         float *__restrict__ corrs, unsigned int *set_counter,
                                         int64_t m, int64_t k, int64_t groups, int mt_count,
                                         int nt_count) {
    pdl_launch_dependents();  // the product may start its first code copies now
    if (blockIdx.x == 0 && threadIdx.x == 0) *set_counter = 0;
    const int64_t units = groups * mt_count * nt_count * 32;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += stride) {
        const int lane = (int)(u & 31);
        const int64_t rest = u >> 5;
        const int nt = (int)(rest % nt_count);
        const int64_t qm = rest / nt_count;      // group * mt_count + mt
        const int mt = (int)(qm % mt_count);
        const int64_t q = qm / mt_count;
        const int g = lane >> 2, c = lane & 3;
        const int64_t t = mt * 16 + nt * 8 + g;
        uint32_t reg[8];
        int sum = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t e = 64 * q + 16 * j + 2 * c;  // elements e, e+1, e+8, e+9
            int v[4] = {0, 0, 0, 0};
            if (t < m) {
                const int64_t idx[4] = {e, e + 8, e + 1, e + 9};
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (idx[i] < k) v[i] = aq[t * k + idx[i]];
            }
            sum += v[0] + v[1] + v[2] + v[3];
            const __half2 lo = __halves2half2(__int2half_rn(v[0]), __int2half_rn(v[1]));
            const __half2 hi = __halves2half2(__int2half_rn(v[2]), __int2half_rn(v[3]));
            reg[2 * j] = *reinterpret_cast<const uint32_t *>(&lo);
            reg[2 * j + 1] = *reinterpret_cast<const uint32_t *>(&hi);
        }
        afrag[(u >> 5) * 64 + lane] = make_uint4(reg[0], reg[1], reg[2], reg[3]);
        afrag[(u >> 5) * 64 + 32 + lane] = make_uint4(reg[4], reg[5], reg[6], reg[7]);
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        if (c == 0) corrs[qm * 16 + nt * 8 + g] = (float)(-1025 * sum);
    }
}

uint32_t g_bs_wait_limit = kDefaultWaitLimit;
int g_bs_withhold = 0;

template <int MT, int NT>
cudaError_t launch_bs_tile(const CUtensorMap &tw, const uint8_t *afrag, const uint8_t *corrs,
                           const float *scale, float absmean, float *y, unsigned int *counter,
                           int64_t m, int64_t n, int nst, cudaStream_t s) {
    using P = BsPlan<MT, NT>;
    auto kern = bitnet_small_m_kernel<MT, NT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P::kAlloc);
    if (e != cudaSuccess) return e;
    // as many CTAs as fit at once (the first set of each is its index)
    static std::atomic<int> per_sm_cache{0};  // the same for every GB300
    int per_sm = per_sm_cache.load(std::memory_order_relaxed);
    if (per_sm == 0) {
        int v = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, kBsThreads, P::kAlloc);
        if (e != cudaSuccess) return e;
        per_sm = std::max(v, 1);
        per_sm_cache.store(per_sm, std::memory_order_relaxed);
    }
    const int64_t nsets = (n + kBsRows - 1) / kBsRows;
    const int grid = (int)std::min<int64_t>(nsets, (int64_t)per_sm * device_sm_count());
    return launch_kernel(kern, dim3(grid), dim3(kBsThreads), P::kAlloc, s, true, tw, afrag, corrs,
                         scale, absmean, y, counter, (int)m, (int)n, nst, g_bs_wait_limit,
                         g_bs_withhold);
}

struct BsWs {
    size_t frag, cor, total;
};

BsWs bs_plan(int64_t m, int64_t k) {
    const int64_t mt = (m + 15) / 16, nt = m <= 8 ? 1 : 2;
    const int64_t groups = (k + kBsStageElems - 1) / kBsStageElems * kBsGroups;
    BsWs p;
    p.frag = (size_t)(groups * mt * nt * 1024);
    p.cor = (size_t)(groups * mt * 64);
    p.total = (p.frag + 255) / 256 * 256 + (p.cor + 255) / 256 * 256 + 256;
    return p;
}

}  // namespace

bool bitnet_small_m_supported(int64_t m, int64_t n, int64_t k) {
    return m >= 1 && m <= 32 && n >= 1 && k % 64 == 0 && k <= 131072;
}

size_t bitnet_small_m_workspace_bytes(int64_t m, int64_t k) { return bs_plan(m, k).total; }

void bitnet_small_set_wait_limit(uint32_t iterations) {
    g_bs_wait_limit = iterations ? iterations : kDefaultWaitLimit;
}

void bitnet_small_set_withhold_loads(int enable) { g_bs_withhold = enable ? 1 : 0; }

cudaError_t bitnet_small_read_and_clear_error(unsigned int *word, cudaStream_t s) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_bitnet_small_error, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    if (*word) {
        e = cudaMemcpyToSymbolAsync(g_bitnet_small_error, &zero, sizeof(unsigned int), 0,
                                    cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

cudaError_t launch_bitnet_small_m(const uint32_t *w, float absmean, const int8_t *aq,
                                  const float *act_scale, float *y, int64_t m, int64_t n,
                                  int64_t k, void *workspace, cudaStream_t s) {
    const BsWs p = bs_plan(m, k);
    const int mt = (int)((m + 15) / 16), nt = m <= 8 ? 1 : 2;
    const int64_t groups = (k + kBsStageElems - 1) / kBsStageElems * kBsGroups;
    const int nst = (int)(groups / kBsGroups);
    auto *ws = static_cast<uint8_t *>(workspace);
    uint8_t *afrag = ws;
    uint8_t *corrs = ws + (p.frag + 255) / 256 * 256;
    auto *counter = reinterpret_cast<unsigned int *>(corrs + (p.cor + 255) / 256 * 256);
    {
        const int threads = 256;
        const int64_t units = groups * mt * nt * 32;
        const int64_t blocks = std::min<int64_t>((units + threads - 1) / threads, 152 * 8);
        bitnet_small_prep_kernel<<<(unsigned)blocks, threads, 0, s>>>(
            aq, reinterpret_cast<uint4 *>(afrag), reinterpret_cast<float *>(corrs), counter, m, k,
            groups, mt, nt);
        cudaError_t e = cudaPeekAtLastError();
        if (e != cudaSuccess) return e;
    }
    // codes: u8 [n rows, k/4 bytes], box 128 bytes x 64 rows, 128-byte
    // swizzle; a last stage past k reads zeros (code 0), which meet zero
    // activations
    CUtensorMap tw;
    const uint64_t row_bytes = (uint64_t)(k / 4);
    if (!make_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, row_bytes, (uint64_t)n, row_bytes, 128,
                     kBsRows, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (m <= 8)
        return launch_bs_tile<1, 1>(tw, afrag, corrs, act_scale, absmean, y, counter, m, n, nst, s);
    if (mt == 1)
        return launch_bs_tile<1, 2>(tw, afrag, corrs, act_scale, absmean, y, counter, m, n, nst, s);
    return launch_bs_tile<2, 2>(tw, afrag, corrs, act_scale, absmean, y, counter, m, n, nst, s);
}

}  // namespace qmm
