// Q4_0 x Q8_0 and Q8_0 x Q8_0 products for a few tokens (m <= 64 with Q4_0
// weights, m <= 32 with Q8_0): the decode-batch and small-prefill shape,
// where the weights stream once and the product should run at the speed of
// the weight read.
//
// What it computes is the GEMM's definition (llama.cpp visual guide, lesson
// 31 "The CPU backend", section "How the quantized dot product works"): for
// every output y[t, n] = sum over blocks b, in ascending order, of
// fma(sumi[t, n, b], dw[n, b] * da[t, b], acc), where sumi is the exact
// integer dot of the 32 weight values (nibbles minus 8, or int8 codes) with
// the 32 int8 activations of block b.  y is bit for bit the serial
// definition.
//
// Why not the tcgen05 GEMM here.  With 16 tokens a tcgen05 tile is
// 128 rows x 16 columns per block, and each block needs its own TMEM
// accumulator round trip (MMA, commit, drain, release): that chain, not the
// weight read, sets the time.  The warp-level tensor-core MMA
// (mma.sync m16n8k16, f16 operands, f32 accumulators) keeps the accumulators
// in registers, so a block's sums are scaled and added the moment the two
// MMAs return, with no hand-off at all.  Its rate (1024 MAC/clk/SM on
// GB300) covers a 16-token product at the weight-streaming speed.
//
// Exactness: weights (as 1024 + nibble or 1152 + code, see the decodes) and
// activations (-127..127, or that over 16) are exact in fp16, and every
// partial sum of a block's two MMAs is an integer of magnitude below 2^23
// (at most 32 x 1279 x 127 = 5.2e6), so the f32 accumulators hold it
// exactly; adding the integer correction that takes the 1024 / 1152 offsets
// out is exact too (tests compare the block sums bit for bit).  The scale
// product dw * da of two fp16 values is exact in f32.
//
// Layout.  One MMA covers 16 weight rows (A, row-major) by 8 tokens (B) over
// 16 k-slots.  Lane (g = lane / 4, c = lane % 4) holds A at rows g and g + 8,
// k-slots 2c, 2c+1, 2c+8, 2c+9.  The k-slots of a block's first MMA are
// mapped to its elements so that a row's four values are the low nibbles of
// the lane's own four nibble bytes 4c..4c+3 of that row (elements 4c..4c+3),
// and the same slots of the second MMA to their high nibbles (elements
// 16+4c..16+4c+3).  With Q8_0 weights the lane's 8 code bytes 8c..8c+7 of a
// row fill the same slots (8c, 8c+2, 8c+1, 8c+3 in the first MMA, the next
// four in the second).  The sum over a block does not depend on the order
// of its elements, so this only fixes how the activations are arranged: a
// prepass writes them as fp16 in exactly the B-fragment order of that
// mapping (16 bytes per lane, block and 8-token tile), together with the
// per-token block corrections and activation scales as f32.  With the
// weights as the 16-row operand, each activation fragment a warp loads from
// shared memory serves 16 weight rows.  Shared memory delivers 128 bytes
// per cycle to the lanes whatever the sharing, so every register a lane
// loads per block counts; the layouts keep that to one (Q4_0) or two (Q8_0)
// words of weights per row, four words of activations per 8-token tile, and
// one 16-byte load each of corrections and scales per 16-token tile.
//
// Roles: warp 4 is the producer; per stage of 8 blocks it copies a tile of
// 128 weight rows x 128 nibble bytes (two such tiles of code bytes for
// Q8_0; tensor copies with 128-byte swizzle, so the 8 rows a lane group
// reads fall in 8 different bank groups; a 3-D copy that lands the tile as
// [block][row][16 bytes] moved 16-byte pieces and streamed a third slower),
// the 128 x 8 dw scales (tensor copy), and the stage's activation
// fragments, corrections and scales (bulk copies).  Warps 0..3
// each own 32 weight rows for every token tile and keep their accumulators in
// registers across the whole reduction; two or three CTAs share an SM.
// CTAs are persistent over 128-row sets (sets of 128 rows keep the last
// round of a large product short: 1002 sets over 152 SMs is 6.6 per SM);
// after its first set (its block index) a CTA takes the next free one from a
// counter, so the sets spread evenly over the SMs however the CTAs were
// placed (a fixed stride put two 4-set CTAs on some SMs: 8 sets there against
// 6.6 on average).  The product is a programmatic dependent launch after the
// prepass: its first weight copies overlap the prepass.  Every mbarrier wait
// is bounded, as in the other kernels.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "qmm_internal.h"
#include "tcgen05.cuh"

namespace qmm {
namespace {

constexpr int kSmRows = 128;    // weight rows per row set (one stage's tile)
constexpr int kSmBlocks = 8;    // blocks per stage (256 k-elements)
constexpr int kSmWarps = 4;     // consumer warps, 32 weight rows (two 16-row units) each
// CTAs per SM and stages of each CTA's ring, per shape (WB: weight bytes per
// row and block, 16 for Q4_0 nibbles, 32 for Q8_0 codes; MT, NT as for the
// kernel).  Q4_0 with two 8-token tiles per 16-token tile up to 32 tokens
// runs three CTAs of two stages (vocabulary shape: 95.9 -> 92.4 us at 16
// tokens, 145.5 -> 138.5 us at 32, registers capped at 128); with one
// 8-token tile three CTAs gain nothing, and Q8_0's stages, and those of 33..64
// tokens, are too large for three: those run two CTAs, each within half the
// SM's shared memory.
template <int WB, int MT, int NT>
constexpr int sm_ctas() { return WB == 16 && NT == 2 && MT <= 2 ? 3 : 2; }
template <int WB, int MT, int NT>
constexpr int sm_stages() {
    return WB == 32 ? 2 : NT == 2 ? 2 : 4;
}
constexpr int kSmThreads = 32 * (kSmWarps + 1);

__device__ unsigned int g_small_error = 0;

template <int WB, int MT, int NT>
struct SmPlan {
    static constexpr int kW = kSmRows * kSmBlocks * WB;  // weight tile(s), 128-byte swizzle
    static constexpr int kDw = kSmRows * 16;           // dw tile: 8 fp16 per row
    static constexpr int kA = kSmBlocks * MT * 1024;   // activation fragments
    static constexpr int kDa = kSmBlocks * MT * 128;   // block corrections and scales (f32)
    static constexpr int kStages = sm_stages<WB, MT, NT>();
    static constexpr int kOffW = 0;                    // 1024-aligned swizzled tiles
    static constexpr int kOffDw = kOffW + kStages * kW;
    static constexpr int kOffA = kOffDw + kStages * kDw;
    static constexpr int kOffDa = kOffA + kStages * kA;
    static constexpr int kOffBar = kOffDa + kStages * kDa;
    static constexpr int kOffMisc = kOffBar + 2 * kStages * 8;
    static constexpr int kBytes = kOffMisc + 16 + 4 * kStages;  // abort flag, stage row sets
    static constexpr int kAlloc = kBytes + 1024;       // slack for the 1024-byte round-up
    static_assert(kW % 1024 == 0, "swizzled tiles stay 1024-byte aligned");
    // the SM's 228 KB hold the CTAs' allocations and 1 KB reserved per CTA
    static_assert(sm_ctas<WB, MT, NT>() * (kAlloc + 1024) <= 228 * 1024, "the CTAs fit one SM");
};

__device__ __forceinline__ bool sm_wait(uint64_t *bar, uint32_t parity, uint32_t limit,
                                        volatile int *abort_flag) {
    return wait_bounded_warp_err(bar, parity, limit, abort_flag, &g_small_error, 8);
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint4 &a, uint32_t b0, uint32_t b1,
                                          const float (&c)[4]) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
          "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) {
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
}

// The lane's 4 nibble bytes 4c..4c+3 of one block of one row (little-endian
// in w) -> the row's A values of the block's two MMAs, as fp16 pairs.  A
// nibble v becomes the fp16 pattern 0x6400 | v = 1024 + v (one mask-or, no
// arithmetic); the 1024 + 8 offset is taken out exactly by the block's
// correction (see the kernel).  Low nibbles (first MMA):
//   lo_a = elements (4c, 4c+2)   (bytes 0 and 2: bits 0-3 and 16-19)
//   lo_b = elements (4c+1, 4c+3) (bytes 1 and 3, after one 8-bit shift)
// High nibbles (second MMA), left at bits 4-7 of their 16-bit half, i.e.
// 1024 + 16 v: hi_a = elements (16+4c, 16+4c+2), hi_b = (16+4c+1, 16+4c+3).
__device__ __forceinline__ void decode_lane_bytes(uint32_t w, uint32_t &lo_a, uint32_t &lo_b,
                                                  uint32_t &hi_a, uint32_t &hi_b) {
    const uint32_t w8 = w >> 8;
    lo_a = (w & 0x000F000Fu) | 0x64006400u;
    lo_b = (w8 & 0x000F000Fu) | 0x64006400u;
    hi_a = (w & 0x00F000F0u) | 0x64006400u;
    hi_b = (w8 & 0x00F000F0u) | 0x64006400u;
}

// The lane's 8 Q8_0 code bytes 8c..8c+7 of one block of one row (lo: bytes
// 0-3, hi: bytes 4-7) -> the row's A values of the block's two MMAs.  A
// signed byte b becomes the fp16 pattern 0x6400 | (b ^ 0x80) = 1152 + b (one
// logic instruction); the 1152 offset is taken out exactly by the block's
// correction.  First MMA: lo_a = elements (8c, 8c+2),
// lo_b = (8c+1, 8c+3); second: hi_a = (8c+4, 8c+6), hi_b = (8c+5, 8c+7).
__device__ __forceinline__ uint32_t q8_pair(uint32_t w) {
    return ((w ^ 0x00800080u) & 0x00FF00FFu) | 0x64006400u;
}

__device__ __forceinline__ void decode_lane_codes(uint2 w, uint32_t &lo_a, uint32_t &lo_b,
                                                  uint32_t &hi_a, uint32_t &hi_b) {
    lo_a = q8_pair(w.x);
    lo_b = q8_pair(w.x >> 8);
    hi_a = q8_pair(w.y);
    hi_b = q8_pair(w.y >> 8);
}

// WB: weight bytes per row and block (16: Q4_0, 32: Q8_0);
// MT: 16-token tiles (m <= 16 MT); NT: 8-token tiles used per 16-token tile
// (1 when m <= 8: the second would hold only padding); EMIT: write the block
// sums instead of y.
template <int WB, int MT, int NT, bool EMIT>
__global__ void __launch_bounds__(kSmThreads, sm_ctas<WB, MT, NT>())
gemm_small_m_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_dw,
                    const uint8_t *__restrict__ afrag, const uint8_t *__restrict__ dafrag,
                    float *__restrict__ y, int32_t *__restrict__ sumi, unsigned int *set_counter, int m,
                    int n, int kb_total, uint32_t wait_limit, int withhold_loads) {
    using P = SmPlan<WB, MT, NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar_full = reinterpret_cast<uint64_t *>(smem + P::kOffBar);
    uint64_t *bar_empty = bar_full + P::kStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + P::kOffMisc);
    // the row set each stage of the ring holds (-1: no further set), written
    // by the producer before it arms the stage
    int *stage_set = reinterpret_cast<int *>(smem + P::kOffMisc + 16);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nst = kb_total / kSmBlocks;                 // stages per row set
    const int nsets = (n + kSmRows - 1) / kSmRows;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P::kStages; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_empty[s], kSmWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
        tmap_prefetch(&tm_w);
        if (!EMIT) tmap_prefetch(&tm_dw);
    }
    __syncthreads();

    if (warp == kSmWarps) {
        // ---------------------------------------------------------------- producer
        constexpr uint32_t kTx = (uint32_t)(P::kW + P::kA + P::kDa + (EMIT ? 0 : P::kDw));
        auto issue_weights = [&](int s, int rs, int j) {  // stage s <- weights, dw of (rs, j)
#pragma unroll
            for (int h = 0; h < WB / 16; ++h)  // one 128-byte box per 128 bytes of row
                tma_load_2d(smem + P::kOffW + s * P::kW + h * kSmRows * 128, &tm_w, &bar_full[s],
                            (j * (WB / 16) + h) * 128, rs * kSmRows);
            if (!EMIT)
                tma_load_2d(smem + P::kOffDw + s * P::kDw, &tm_dw, &bar_full[s], j * kSmBlocks,
                            rs * kSmRows);
        };
        auto issue_acts = [&](int s, int j) {  // stage s <- activation fragments, records of j
            bulk_load(smem + P::kOffA + s * P::kA, afrag + (size_t)j * P::kA, P::kA, &bar_full[s]);
            bulk_load(smem + P::kOffDa + s * P::kDa, dafrag + (size_t)j * P::kDa, P::kDa, &bar_full[s]);
        };
        // Row sets: the first is blockIdx.x, each further one the next free
        // set from a counter in the workspace (zeroed by the prepass), so the
        // sets spread over the SMs as they finish, wherever the CTAs were
        // placed.  withhold_loads (a test hook) issues nothing, so every
        // consumer wait can only run out its limit.
        int rs = withhold_loads ? nsets : (int)blockIdx.x;
        // The weights do not depend on the previous kernel on the stream (the
        // prepass): the first stage gets its weight copies before the wait
        // for it (programmatic dependent launch), its activation copies after.
        // A stage is armed once, for all its bytes.  (More stages ahead of the
        // wait put more weight traffic in front of the first activation
        // copies: 0.1-1 us slower per launch at the vocabulary shape.)
        const int pre = rs < nsets ? 1 : 0;
        if (lane == 0)
            for (int i = 0; i < pre; ++i) {
                stage_set[i] = rs;
                mbar_arrive_expect_tx(&bar_full[i], kTx);
                issue_weights(i, rs, i);
            }
        pdl_wait();
        __syncwarp();
        int it = 0;
        bool ok = true;
        while (ok && rs < nsets) {
            for (int j = 0; j < nst; ++j, ++it) {
                const int s = it % P::kStages;
                if (it >= pre) {
                    if (!sm_wait(&bar_empty[s], ((uint32_t)(it / P::kStages) & 1u) ^ 1u, wait_limit,
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
        // no further set: one more stage, with no copies, says so (once the
        // consumers released stage it - kStages, whose copies have landed)
        bool sent = false;
        if (ok && !withhold_loads) {
            const int s = it % P::kStages;
            if (sm_wait(&bar_empty[s], ((uint32_t)(it / P::kStages) & 1u) ^ 1u, wait_limit, abort_flag)) {
                if (lane == 0) {
                    stage_set[s] = -1;
                    mbar_arrive(&bar_full[s]);
                }
                sent = true;
            }
            __syncwarp();
        }
        // Never leave a copy in flight: wait for the last stages issued (an
        // abort can only come at it >= pre, so every stage armed before the
        // wait got its activation copies too).  Stage it - kStages is skipped
        // once the end stage went out on its slot: its copies landed, and its
        // barrier has moved on by two phases.
        const int first_pending = (it > P::kStages ? it - P::kStages : 0) + (sent && it >= P::kStages ? 1 : 0);
        for (int i = first_pending; i < it; ++i) {
            volatile int no_abort = 0;
            sm_wait(&bar_full[i % P::kStages], (uint32_t)(i / P::kStages) & 1u, kDrainLimit, &no_abort);
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    // Warp w owns weight rows 32 w .. 32 w + 31 of every row set, as two
    // units of 16 rows (u = 0, 1).  A unit is the MMA's A operand (16 rows),
    // with the tokens as B in tiles of 8 (two per 16-token tile); both units
    // use the same activation fragments, loaded once per block.  Lane (g, c)
    // holds A at rows g and g + 8 of a unit and B at token g of the 8-token
    // tile; its accumulators are rows g, g + 8 x tokens 2c, 2c + 1.
    const int g = lane >> 2, c = lane & 3;
    uint64_t acc[2][MT][NT][2];  // [unit][tile][8-token tile][row g | row g + 8], token pairs
    int it = 0;
    bool ok = true;
    for (;;) {
        // the next set: its first stage says which (or that there is none)
        if (!sm_wait(&bar_full[it % P::kStages], (uint32_t)(it / P::kStages) & 1u, wait_limit,
                     abort_flag)) {
            ok = false;
            break;
        }
        const int rs = stage_set[it % P::kStages];
        if (rs < 0) break;
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) acc[u][mt][nt][0] = acc[u][mt][nt][1] = 0ull;
        for (int j = 0; j < nst; ++j, ++it) {
            const int s = it % P::kStages;
            const uint32_t ph = (uint32_t)(it / P::kStages) & 1u;
            if (j > 0 && !sm_wait(&bar_full[s], ph, wait_limit, abort_flag)) {
                ok = false;
                break;
            }
            // weight tile(s): 128 rows of 128 bytes each under the 128-byte
            // swizzle, 16-byte chunk q of row r at chunk q ^ (r % 8).  This
            // lane's rows all have r % 8 = g, and its offsets have bits 4..6
            // clear before the chunk is set, so one XOR per row and block
            // places each read:
            //   Q4_0: 4 bytes of block b (chunk b) at (r*128 + 4c + 16g) ^ 16b;
            //   Q8_0: 8 bytes of block b (chunk 2(b%4) + c/2 of tile b/4) at
            //         16384 (b/4) + ((r*128 + 8(c%2) + 16(c/2 ^ g)) ^ 32(b%4)).
            const uint8_t *wt = smem + P::kOffW + s * P::kW;
            const uint32_t wl = WB == 16 ? (32 * warp + g) * 128 + 4 * c + 16 * g
                                         : (32 * warp + g) * 128 + 8 * (c & 1) + 16 * ((c >> 1) ^ g);
            const uint8_t *at = smem + P::kOffA + s * P::kA;
            const float4 *rec = reinterpret_cast<const float4 *>(smem + P::kOffDa + s * P::kDa);
            // dw of rows g and g + 8 of both units, the stage's 8 blocks (fp16 pairs)
            uint4 dwr[2][2];
            if (!EMIT) {
                const uint8_t *dt = smem + P::kOffDw + s * P::kDw + (32 * warp + g) * 16;
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        dwr[u][h] = *reinterpret_cast<const uint4 *>(dt + (16 * u + 8 * h) * 16);
            }
#pragma unroll
            for (int b = 0; b < kSmBlocks; ++b) {
                uint4 a_lo[2], a_hi[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    uint32_t la0, lb0, ha0, hb0, la1, lb1, ha1, hb1;
                    if constexpr (WB == 16) {
                        const uint32_t w0 = *reinterpret_cast<const uint32_t *>(wt + ((wl + (16 * u) * 128) ^ (16u * b)));
                        const uint32_t w1 = *reinterpret_cast<const uint32_t *>(wt + ((wl + (16 * u + 8) * 128) ^ (16u * b)));
                        decode_lane_bytes(w0, la0, lb0, ha0, hb0);
                        decode_lane_bytes(w1, la1, lb1, ha1, hb1);
                    } else {
                        const uint8_t *wb = wt + (b >> 2) * (kSmRows * 128);
                        const uint2 w0 = *reinterpret_cast<const uint2 *>(wb + ((wl + (16 * u) * 128) ^ (32u * (b & 3))));
                        const uint2 w1 = *reinterpret_cast<const uint2 *>(wb + ((wl + (16 * u + 8) * 128) ^ (32u * (b & 3))));
                        decode_lane_codes(w0, la0, lb0, ha0, hb0);
                        decode_lane_codes(w1, la1, lb1, ha1, hb1);
                    }
                    // A registers: (row g, slots 2c..), (row g+8, 2c..), (row g,
                    // 2c+8..), (row g+8, 2c+8..); slots 2c, 2c+1, 2c+8, 2c+9 of
                    // the first MMA hold elements 4c, 4c+2, 4c+1, 4c+3, of the
                    // second 16 more (Q4_0), or 8c, 8c+2, 8c+1, 8c+3 and 4 more
                    // (Q8_0)
                    a_lo[u] = make_uint4(la0, la1, lb0, lb1);
                    a_hi[u] = make_uint4(ha0, ha1, hb0, hb1);
                }
                // dw of the units' rows g, g + 8 for block b, as f32 pairs (dw, dw)
                uint64_t dwp[2][2];
                if (!EMIT) {
#pragma unroll
                    for (int u = 0; u < 2; ++u)
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t wv = (&dwr[u][h].x)[b >> 1];
                            const float f = __half2float(__ushort_as_half(
                                (unsigned short)((b & 1) ? (wv >> 16) : (wv & 0xFFFFu))));
                            dwp[u][h] = f2_pack(f, f);
                        }
                }
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    // activation fragments of (block b, tile mt): two 512-byte
                    // pieces (tokens 0..7, 8..15), lane-contiguous 16 bytes
                    const uint4 *af = reinterpret_cast<const uint4 *>(at + (b * MT + mt) * 1024);
                    // corrections and scales of tokens 2c, 2c+1 of both 8-token tiles
                    const float4 cor = rec[(b * MT + mt) * 8 + c];
                    const float4 da = EMIT ? make_float4(0.f, 0.f, 0.f, 0.f) : rec[(b * MT + mt) * 8 + 4 + c];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const uint4 bf = af[32 * nt + lane];
                        const uint64_t corp = nt ? f2_pack(cor.z, cor.w) : f2_pack(cor.x, cor.y);
                        const uint64_t dap = nt ? f2_pack(da.z, da.w) : f2_pack(da.x, da.y);
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const float zero[4] = {0.f, 0.f, 0.f, 0.f};
                            float d[4];
                            mma_16816(d, a_lo[u], bf.x, bf.y, zero);
                            mma_16816(d, a_hi[u], bf.z, bf.w, d);
                            // the block sums: add the tokens' corrections (exact, integers)
                            const uint64_t s0 = f2_add(f2_pack(d[0], d[1]), corp);  // row g
                            const uint64_t s1 = f2_add(f2_pack(d[2], d[3]), corp);  // row g + 8
                            if constexpr (EMIT) {
                                const int kbi = j * kSmBlocks + b;
                                const int t0 = mt * 16 + nt * 8 + 2 * c;
                                const int n0 = rs * kSmRows + 32 * warp + 16 * u + g;
                                float v[4];
                                f2_unpack(s0, v[0], v[1]);
                                f2_unpack(s1, v[2], v[3]);
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const int t = t0 + (i & 1);
                                    const int nn = n0 + 8 * (i >> 1);
                                    if (t < m && nn < n)
                                        sumi[((int64_t)t * n + nn) * kb_total + kbi] = __float2int_rn(v[i]);
                                }
                            } else {
                                // S = dw * da (exact); acc = fma(sumi, S, acc), two
                                // outputs per instruction
                                acc[u][mt][nt][0] = f2_fma(s0, f2_mul(dwp[u][0], dap), acc[u][mt][nt][0]);
                                acc[u][mt][nt][1] = f2_fma(s1, f2_mul(dwp[u][1], dap), acc[u][mt][nt][1]);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_empty[s]);
        }
        if (!ok) break;
        if (!EMIT) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int n0 = rs * kSmRows + 32 * warp + 16 * u + g;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            float v[2];
                            f2_unpack(acc[u][mt][nt][r], v[0], v[1]);
                            const int nn = n0 + 8 * r;
#pragma unroll
                            for (int i = 0; i < 2; ++i) {
                                const int t = mt * 16 + nt * 8 + 2 * c + i;
                                if (t < m && nn < n) y[(int64_t)t * n + nn] = v[i];
                            }
                        }
            }
        }
    }
}

// Activation prepass, in the B-fragment order of the kernel above.  Per
// block b and 16-token tile mt, 1 KB in two 512-byte pieces, one per 8-token
// tile nt; lane l = 4 g + c owns 16 bytes of piece nt at l * 16, for token
// t = mt * 16 + nt * 8 + g: the first MMA's registers (a[4c], a[4c+2]) and
// (a[4c+1], a[4c+3]), then the second's (a[16+4c] / 16, a[16+4c+2] / 16) and
// (a[16+4c+1] / 16, a[16+4c+3] / 16), all exact in fp16 (a = the int8 code
// of element e of block b).  The first MMA sees the weights as 1024 + v and
// the second as 1024 + 16 v against activations scaled by 1/16, i.e. 64 + v,
// so a block's two MMAs sum (v - 8) a exactly once the correction
//   cor[t] = -1032 * (a[0] + .. + a[15]) - 72 * (a[16] + .. + a[31])
// is added (every partial sum is an integer below 2^24 in magnitude).  Then
// a 128-byte record per (b, mt): for c = 0..3 the f32 corrections of tokens
// (nt0: 2c, 2c+1, nt1: 2c, 2c+1), then for c = 0..3 their scales da as f32.
// Tokens past m are zeros.  The four lanes of a token hold all its codes of
// the block, so its sums come from two shuffle steps.
//
// With Q8_0 weights (q8) the element order follows that kernel's Q8_0
// mapping: registers (a[8c], a[8c+2]), (a[8c+1], a[8c+3]), then
// (a[8c+4], a[8c+6]), (a[8c+5], a[8c+7]), nothing scaled, and the weights
// seen as 1152 + code, so cor[t] = -1152 * (a[0] + .. + a[31]).
__global__ void gemm_small_prep_kernel(const int8_t *__restrict__ aq, const unsigned short *__restrict__ ad,
                                       uint4 *__restrict__ afrag, uint8_t *__restrict__ rec,
                                       unsigned int *set_counter, int64_t m, int64_t k, int mt_count,
                                       int q8) {
    // the product (launched with programmatic dependent launch) may start its
    // weight copies now; it reads what this kernel writes only after its wait
    pdl_launch_dependents();
    if (blockIdx.x == 0 && threadIdx.x == 0) *set_counter = 0;  // the product's row-set counter
    const int64_t kb = k / kQK;
    const int64_t units = kb * mt_count * 64;  // (block, tile, piece, lane)
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const __half sixteenth = __float2half_rn(0.0625f);
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += stride) {
        const int lane = (int)(u & 31);
        const int nt = (int)((u >> 5) & 1);
        const int64_t bm = u >> 6;                 // b * mt_count + mt
        const int mt = (int)(bm % mt_count);
        const int64_t b = bm / mt_count;
        const int g = lane >> 2, c = lane & 3;
        const int64_t t = mt * 16 + nt * 8 + g;
        uint32_t reg[4];
        int part[2] = {0, 0};  // sums of the two groups of four codes
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            // four int8 codes of token t: elements 16 half + 4c .. (Q4_0) or
            // 8c + 4 half .. (Q8_0)
            const int64_t e = q8 ? 8 * c + 4 * half : 16 * half + 4 * c;
            uint32_t q = 0;
            if (t < m) q = *reinterpret_cast<const uint32_t *>(aq + t * k + b * kQK + e);
            __half h[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int v = (int)(int8_t)((q >> (8 * i)) & 0xff);
                part[half] += v;
                h[i] = __int2half_rn(v);
                if (half && !q8) h[i] = __hmul(h[i], sixteenth);  // exact: a power of two
            }
            reg[2 * half] = h2_bits(__halves2half2(h[0], h[2]));
            reg[2 * half + 1] = h2_bits(__halves2half2(h[1], h[3]));
        }
        afrag[u] = make_uint4(reg[0], reg[1], reg[2], reg[3]);
        // the four lanes of token t hold all 32 of its codes in the block:
        // lo = a[0] + .. + a[15], hi = a[16] + .. + a[31] for Q4_0 (for Q8_0
        // only their total is used)
        int lo = part[0], hi = part[1];
        lo += __shfl_xor_sync(0xffffffffu, lo, 1);
        hi += __shfl_xor_sync(0xffffffffu, hi, 1);
        lo += __shfl_xor_sync(0xffffffffu, lo, 2);
        hi += __shfl_xor_sync(0xffffffffu, hi, 2);
        // token g of 8-token tile nt sits at float 4 (g / 2) + 2 nt + g % 2 of
        // the record's correction half (and 16 floats on, its scale)
        float *r = reinterpret_cast<float *>(rec + bm * 128) + 4 * (g >> 1) + 2 * nt + (g & 1);
        if (c == 0) r[0] = q8 ? (float)(-1152 * (lo + hi)) : (float)(-1032 * lo - 72 * hi);
        if (c == 1) r[16] = ad && t < m ? __half2float(__ushort_as_half(ad[t * kb + b])) : 0.0f;
    }
}

uint32_t g_small_wait_limit = kDefaultWaitLimit;
int g_small_withhold = 0;

template <int WB, int MT, int NT, bool EMIT>
cudaError_t launch_small_tile(const CUtensorMap &tw, const CUtensorMap &tdw, const uint8_t *afrag,
                              const uint8_t *dafrag, float *y, int32_t *sumi, unsigned int *counter,
                              int64_t m, int64_t n, int64_t k, cudaStream_t s) {
    using P = SmPlan<WB, MT, NT>;
    auto kern = gemm_small_m_kernel<WB, MT, NT, EMIT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P::kAlloc);
    if (e != cudaSuccess) return e;
    const int64_t nsets = (n + kSmRows - 1) / kSmRows;
    const int grid = (int)std::min<int64_t>(nsets, sm_ctas<WB, MT, NT>() * device_sm_count());
    // programmatic dependent launch: the CTAs start their weight copies
    // while the prepass before them still runs
    return launch_kernel(kern, dim3(grid), dim3(kSmThreads), P::kAlloc, s, true, tw, tdw, afrag,
                         dafrag, y, sumi, counter, (int)m, (int)n, (int)(k / kQK), g_small_wait_limit,
                         g_small_withhold);
}

}  // namespace

bool gemm_small_m_supported(int64_t m, int64_t /*n*/, int64_t k) {
    return m >= 1 && m <= 32 && k % (kQK * kSmBlocks) == 0;
}

bool gemm_small_m_supported_q4(int64_t m, int64_t n, int64_t k) {
    return gemm_small_m_supported(std::min<int64_t>(m, 32), n, k) && m <= 64;
}

// activation fragments, then the records, then the row-set counter, each
// 256-byte aligned
size_t gemm_small_m_workspace_bytes(int64_t m, int64_t k) {
    const int64_t mt = (m + 15) / 16;
    const int64_t kb = k / kQK;
    const size_t a = (size_t)(kb * mt * 1024), r = (size_t)(kb * mt * 128);
    return (a + 255) / 256 * 256 + (r + 255) / 256 * 256 + 256;
}

void gemm_small_set_wait_limit(uint32_t iterations) {
    g_small_wait_limit = iterations ? iterations : kDefaultWaitLimit;
}

void gemm_small_set_withhold_loads(int enable) { g_small_withhold = enable ? 1 : 0; }

cudaError_t gemm_small_read_and_clear_error(unsigned int *word, cudaStream_t s) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_small_error, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    if (*word) {
        e = cudaMemcpyToSymbolAsync(g_small_error, &zero, sizeof(unsigned int), 0,
                                    cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

namespace {

// WB = 16: Q4_0 nibbles [n, k/2]; WB = 32: Q8_0 codes [n, k].
template <int WB>
cudaError_t launch_small(const void *w, const uint16_t *wd, const int8_t *aq, const uint16_t *ad,
                         float *y, int32_t *sumi, int64_t m, int64_t n, int64_t k, void *workspace,
                         cudaStream_t s) {
    const int mt = (int)((m + 15) / 16);
    const int64_t kb = k / kQK;
    auto *ws = static_cast<uint8_t *>(workspace);
    const size_t a_bytes = (size_t)(kb * mt * 1024), r_bytes = (size_t)(kb * mt * 128);
    uint8_t *afrag = ws;
    uint8_t *dafrag = ws + (a_bytes + 255) / 256 * 256;
    auto *counter = reinterpret_cast<unsigned int *>(dafrag + (r_bytes + 255) / 256 * 256);
    {
        const int threads = 256;
        const int64_t units = kb * mt * 64;
        const int64_t blocks = std::min<int64_t>((units + threads - 1) / threads, 152 * 8);
        gemm_small_prep_kernel<<<(unsigned)blocks, threads, 0, s>>>(
            aq, reinterpret_cast<const unsigned short *>(sumi ? nullptr : ad),
            reinterpret_cast<uint4 *>(afrag), dafrag, counter, m, k, mt, WB == 32 ? 1 : 0);
        cudaError_t e = cudaPeekAtLastError();
        if (e != cudaSuccess) return e;
    }
    CUtensorMap tw, tdw;
    // weights: u8 [n rows, k WB / 32 bytes], box 128 bytes x 128 rows,
    // 128-byte swizzle (a Q8_0 stage takes two boxes)
    const uint64_t row_bytes = (uint64_t)(kb * WB);
    if (!make_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, row_bytes, (uint64_t)n, row_bytes, 128,
                     kSmRows, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    // dw: fp16 [n rows, k/32], box 8 x 128 (the block-sum variant reads none
    // and maps the weights again as a placeholder)
    if (sumi) {
        tdw = tw;
    } else if (!make_map_2d(&tdw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, wd, (uint64_t)kb, (uint64_t)n,
                            (uint64_t)kb * 2, kSmBlocks, kSmRows, CU_TENSOR_MAP_SWIZZLE_NONE)) {
        return cudaErrorInvalidValue;
    }
    // m <= 8 runs one 8-token tile per block (measured 74 against 94 us at
    // the vocabulary shape with Q4_0 weights)
    if (m <= 8)
        return sumi ? launch_small_tile<WB, 1, 1, true>(tw, tdw, afrag, dafrag, y, sumi, counter, m, n, k, s)
                    : launch_small_tile<WB, 1, 1, false>(tw, tdw, afrag, dafrag, y, sumi, counter, m, n, k, s);
    if (mt == 1)
        return sumi ? launch_small_tile<WB, 1, 2, true>(tw, tdw, afrag, dafrag, y, sumi, counter, m, n, k, s)
                    : launch_small_tile<WB, 1, 2, false>(tw, tdw, afrag, dafrag, y, sumi, counter, m, n, k, s);
    if constexpr (WB == 16) {
        // 33..64 tokens, Q4_0 only (Q8_0 stages of that width would not fit
        // two CTAs per SM)
        if (mt == 3)
            return sumi ? launch_small_tile<WB, 3, 2, true>(tw, tdw, afrag, dafrag, y, sumi, counter, m, n, k, s)
                        : launch_small_tile<WB, 3, 2, false>(tw, tdw, afrag, dafrag, y, sumi, counter, m, n, k, s);
        if (mt == 4)
            return sumi ? launch_small_tile<WB, 4, 2, true>(tw, tdw, afrag, dafrag, y, sumi, counter, m, n, k, s)
                        : launch_small_tile<WB, 4, 2, false>(tw, tdw, afrag, dafrag, y, sumi, counter, m, n, k, s);
    }
    return sumi ? launch_small_tile<WB, 2, 2, true>(tw, tdw, afrag, dafrag, y, sumi, counter, m, n, k, s)
                : launch_small_tile<WB, 2, 2, false>(tw, tdw, afrag, dafrag, y, sumi, counter, m, n, k, s);
}

}  // namespace

// wd / ad may be null (block-sum variant, sumi != null).
cudaError_t launch_gemm_small_m(const uint8_t *wq, const uint16_t *wd, const int8_t *aq,
                                const uint16_t *ad, float *y, int32_t *sumi, int64_t m, int64_t n,
                                int64_t k, void *workspace, cudaStream_t s) {
    return launch_small<16>(wq, wd, aq, ad, y, sumi, m, n, k, workspace, s);
}

cudaError_t launch_gemm_small_m_q8(const int8_t *w8, const uint16_t *wd, const int8_t *aq,
                                   const uint16_t *ad, float *y, int32_t *sumi, int64_t m, int64_t n,
                                   int64_t k, void *workspace, cudaStream_t s) {
    return launch_small<32>(w8, wd, aq, ad, y, sumi, m, n, k, workspace, s);
}

}  // namespace qmm
