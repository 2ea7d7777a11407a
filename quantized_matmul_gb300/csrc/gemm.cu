// Prefill-shaped Q4_0 x Q8_0 and Q8_0 x Q8_0 products on the 5th-generation
// tensor cores.
//
// What it computes (llama.cpp visual guide, lesson 31 "The CPU backend",
// section "How the quantized dot product works"): for every output
// y[t, n] = sum over blocks b of sumi[t, n, b] * (dw[n, b] * da[t, b]) where
// sumi is the exact integer dot of the 32 nibbles (minus 8) with the 32 int8
// activations of the block, accumulated block by block in ascending order.
// With Q8_0 weights (the Fucina reference, section 9, uses the Q8_0 block as
// a weight format too) the weight values are the 32 int8 codes of the block
// (|sumi| <= 32 * 127 * 127 < 2^24); only the weight tile and its converter
// differ (template parameter WB, the weight bytes per row and stage).
// Q4_0 weights repacked at load time into the tile order (template flag RP;
// Fucina reference, section 9.7, packs weights once into the kernel's
// interleaved layout) arrive as one contiguous 4 KB bulk copy per stage, and
// the converter decodes each word with one shift and masks.  (A tile is 16
// rows of 256 bytes in the copy's 2-D view.)
//
// How (GB300, sm_103a).  There is no int8 MMA on sm_103a, but every operand
// value is a small integer that fp16 holds exactly (weights -8..7,
// activations -127..127) and every partial sum of one block is an integer of
// magnitude <= 32 * 8 * 127 < 2^24, so tcgen05.mma kind::f16 with an f32
// accumulator produces each block sum exactly.  The scale product dw * da of
// two fp16 values is exact in f32 too, so the tensor core computes it as
// well: one more MMA per block whose A tile holds dw[n, b] in column 0 and
// zeros elsewhere and whose B tile holds da[t, b] in column 0 writes the
// matrix S[n, t] = dw * da, exactly, next to the block sums.  The CUDA cores
// then do one fused multiply-add per output and block,
// acc = fma(sumi, S, acc): the same operations, in the same order, as the
// serial definition, so y is reproducible bit for bit.
//
// One CTA computes a tile of 128 weight rows (the MMA's M, TMEM lanes) by BN
// tokens (the MMA's N, TMEM columns).  Roles:
//   warp 0      TMA producer: per stage of two blocks (64 k-elements) the
//               128 x 32 B nibble tile (128 x 64 B of codes for Q8_0), the BN x 64 fp16 activation tile
//               (128-byte swizzle) and the two BN x 16 B scale rows (da in
//               the first fp16 of each row, written by the prepass).
//   warps 1, 2  warp 1 allocates TMEM; lane 0 of warp 1 (even blocks) and of
//               warp 2 (odd blocks) issues, per block, the two K=16
//               block-sum MMAs and the scale MMA into accumulator slot
//               b % NACC (2 * BN columns: sums, then S) and commits.
//   warps 3..6  converters: all four convert every stage together, each a
//               quarter of its 256 (row, block) units, turning the weights
//               into the 128-byte-swizzled K-major fp16 A tile and writing
//               the 128 rows x 16 B dw tile of each block.
//   then        drains: thread (warp % 4, lane) owns weight row n (a TMEM
//               lane quarter is readable only from the sub-partition with the
//               same index) and BN / groups columns; per block it loads the
//               sums and S from TMEM and applies the multiply-adds.
// The roles meet only at mbarriers; each slot's S and sums are drained while
// the tensor core fills the next slot.  The scale tiles use the no-swizzle
// K-major layout: 16-byte rows (8 fp16, the value and seven zeros), 8-row
// groups 128 bytes apart, and the second K core matrix of every group read
// from one shared block of zeros through the descriptor's leading offset.
// An activation prepass (same stream) writes the fp16 copy of the int8
// activations and the scale rows into the workspace.
//
// Every mbarrier wait is bounded.  On expiry a kernel raises a CTA-wide abort
// flag, records QMM_ERR_TIMEOUT in a device error word, waits (bounded) for
// its own TMA copies and MMAs still in flight, releases TMEM and returns.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "qmm_internal.h"
#include "tcgen05.cuh"

namespace qmm {
namespace {

constexpr int kBM = 128;       // weight rows per tile (MMA M)
constexpr int kBK = 64;        // k-elements per pipeline stage (two blocks)
constexpr int kMmaWarps = 2;   // warps 1 and 2 issue the MMAs of even and odd blocks
constexpr int kConvWarp0 = 1 + kMmaWarps;  // converters follow the producer and MMA warps
constexpr int kSmemBudget = 200 * 1024;  // per SM
constexpr int kZeroBytes = 2048;         // zeros behind every scale tile's second K half

// drain warps per TMEM lane quarter, each taking BN / groups columns
template <int BN>
__host__ __device__ constexpr int drain_groups() { return BN >= 64 ? BN / 32 : 1; }
template <int BN>
__host__ __device__ constexpr int ctas_per_sm() { return BN <= 32 ? 2 : 1; }
// WB: weight bytes per row and stage (two blocks): 32 for Q4_0 nibbles, 64
// for Q8_0 codes.
// bytes of one pipeline stage: A tile, B tile, weight tile, dw tile, da tile
template <int BN, int WB>
__host__ __device__ constexpr int stage_bytes() {
    return kBM * kBK * 2 + BN * kBK * 2 + kBM * WB + 2 * kBM * 16 + 2 * BN * 16;
}
template <int BN, int WB>
__host__ __device__ constexpr int stages_fit() {
    return ((kSmemBudget / ctas_per_sm<BN>()) - kZeroBytes - 1024) / stage_bytes<BN, WB>() < 8
               ? ((kSmemBudget / ctas_per_sm<BN>()) - kZeroBytes - 1024) / stage_bytes<BN, WB>()
               : 8;
}
// Converter warps: four (their number divides the 8 units per lane of a
// stage).  Every converter visits every stage in order, so no waiter can run
// a phase ahead of a barrier.
template <int BN, int WB>
__host__ __device__ constexpr int conv_warps() { return 4; }
template <int BN, int WB>
__host__ __device__ constexpr int stages_for() {
    return stages_fit<BN, WB>();
}
template <int BN, int WB>
__host__ __device__ constexpr int epi_warp0() { return kConvWarp0 + conv_warps<BN, WB>(); }
template <int BN, int WB>
__host__ __device__ constexpr int threads_for() { return 32 * (epi_warp0<BN, WB>() + 4 * drain_groups<BN>()); }
// TMEM accumulator slots, one per block in flight (2 * BN columns each)
template <int BN>
constexpr int nacc_for() {
    return (512 / ctas_per_sm<BN>()) / (2 * BN) < 8 ? (512 / ctas_per_sm<BN>()) / (2 * BN) : 8;
}
__device__ unsigned int g_gemm_error = 0;

// Polls of a phase before a waiter asks to be suspended.  A CTA that has the
// SM to itself (BN >= 64) polls for a while: a suspended warp resumes later
// than a polling one sees the phase complete (4% at the prefill shape).  Two
// CTAs per SM share the issue slots, and there polling costs more than it
// saves (8% at m = 16), so their waiters suspend at once.
template <int BN>
__host__ __device__ constexpr int spin_polls() { return ctas_per_sm<BN>() == 1 ? 200 : 1; }

// the shared bounded waits, reporting into this kernel's error word
template <int BN>
__device__ __forceinline__ bool wait_bounded(uint64_t *bar, uint32_t parity, uint32_t limit,
                                             volatile int *abort_flag) {
    return wait_bounded_err(bar, parity, limit, abort_flag, &g_gemm_error, spin_polls<BN>());
}
template <int BN>
__device__ __forceinline__ bool wait_bounded_warp(uint64_t *bar, uint32_t parity, uint32_t limit,
                                                  volatile int *abort_flag) {
    return wait_bounded_warp_err(bar, parity, limit, abort_flag, &g_gemm_error, spin_polls<BN>());
}


// Pairs of f32 in one 64-bit register: the paired FP32 instructions give two
// independent IEEE round-to-nearest results per instruction.
__device__ __forceinline__ uint64_t pack_u32x2(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}

__device__ __forceinline__ void unpack_f32x2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) {
    __half2 h;
    memcpy(&h, &u, 4);
    return h;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) {
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
}

// 16 nibble bytes of one block -> 32 fp16 values (nibble - 8) in element
// order: element j is the low nibble of byte j, element j+16 the high one.
// Exact: fp16 holds every integer in [-8, 7].  The fp16 bit pattern
// 0x6400 | v is the value 1024 + v (v < 1024), so a low nibble becomes
// (0x6400 | v) - 1032 and a high nibble, left at bits 4..7, becomes
// (0x6400 | 16 v) / 16 - 72; every step is exact.
__device__ __forceinline__ void unpack_block_f16(uint4 v, uint4 (&out)[4]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const __half2 off = u32_as_h2(0x64086408u);        // (1032, 1032)
    const __half2 sixteenth = u32_as_h2(0x2C002C00u);  // (1/16, 1/16)
    const __half2 m72 = u32_as_h2(0xD480D480u);        // (-72, -72)
    uint32_t lo[8], hi[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // bytes (b0, b1) and (b2, b3) of word i spread to the two 16-bit halves
        const uint32_t p0 = __byte_perm(w[i], 0, 0x4140);
        const uint32_t p1 = __byte_perm(w[i], 0, 0x4342);
        lo[2 * i] = h2_as_u32(__hsub2(u32_as_h2((p0 & 0x000F000Fu) | 0x64006400u), off));
        lo[2 * i + 1] = h2_as_u32(__hsub2(u32_as_h2((p1 & 0x000F000Fu) | 0x64006400u), off));
        hi[2 * i] = h2_as_u32(__hfma2(u32_as_h2((p0 & 0x00F000F0u) | 0x64006400u), sixteenth, m72));
        hi[2 * i + 1] = h2_as_u32(__hfma2(u32_as_h2((p1 & 0x00F000F0u) | 0x64006400u), sixteenth, m72));
    }
    out[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);  // elements 0..7
    out[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);  // elements 8..15
    out[2] = make_uint4(hi[0], hi[1], hi[2], hi[3]);  // elements 16..23
    out[3] = make_uint4(hi[4], hi[5], hi[6], hi[7]);  // elements 24..31
}

// One repacked Q4_0 block (16 bytes, word c carrying elements 8c..8c+7 with
// element 8c + 2i + h at bits 4i + 16h) -> 32 fp16 values (nibble - 8).  The
// pairs at bits 0-3/16-19 and 8-11/24-27 (after one 8-bit shift) become
// (0x6400 | v) - 1032; the pairs at bits 4-7/20-23 and 12-15/28-31 become
// (0x6400 | 16 v) / 16 - 72, with no shift: nine operations per word, all
// exact.
__device__ __forceinline__ void unpack_repacked_f16(uint4 v, uint4 (&out)[4]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const __half2 off = u32_as_h2(0x64086408u);        // (1032, 1032)
    const __half2 sixteenth = u32_as_h2(0x2C002C00u);  // (1/16, 1/16)
    const __half2 m72 = u32_as_h2(0xD480D480u);        // (-72, -72)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t w8 = w[c] >> 8;
        out[c] = make_uint4(
            h2_as_u32(__hsub2(u32_as_h2((w[c] & 0x000F000Fu) | 0x64006400u), off)),
            h2_as_u32(__hfma2(u32_as_h2((w[c] & 0x00F000F0u) | 0x64006400u), sixteenth, m72)),
            h2_as_u32(__hsub2(u32_as_h2((w8 & 0x000F000Fu) | 0x64006400u), off)),
            h2_as_u32(__hfma2(u32_as_h2((w8 & 0x00F000F0u) | 0x64006400u), sixteenth, m72)));
    }
}

// 32 int8 codes of one Q8_0 block (two 16-byte words, elements in order) ->
// 32 fp16 values.  Exact: the fp16 pattern 0x6400 | u is 1024 + u for
// u < 1024, and u = b ^ 0x80 = b + 128 for a signed byte b, so subtracting
// 1152 leaves b.
__device__ __forceinline__ void unpack_block_q8_f16(uint4 v0, uint4 v1, uint4 (&out)[4]) {
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    const __half2 off = u32_as_h2(0x64806480u);  // (1152, 1152)
    uint32_t h[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t p0 = __byte_perm(w[i], 0, 0x4140);  // bytes 0, 1 -> halves
        const uint32_t p1 = __byte_perm(w[i], 0, 0x4342);  // bytes 2, 3 -> halves
        h[2 * i] = h2_as_u32(__hsub2(u32_as_h2((p0 ^ 0x00800080u) | 0x64006400u), off));
        h[2 * i + 1] = h2_as_u32(__hsub2(u32_as_h2((p1 ^ 0x00800080u) | 0x64006400u), off));
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) out[c] = make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
}


// Shared-memory descriptor for the scale tiles: K-major, no swizzle, 16-byte
// rows, 8-row groups 128 bytes apart (stride offset), the second K core
// matrix `lead` bytes after the first (the block of zeros).
__device__ __forceinline__ uint64_t smem_desc_scale(uint32_t saddr, uint32_t lead) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lead >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)(128u >> 4) << 32;
    d |= 1ull << 46;  // swizzle mode 0 (none) at bits 61-63
    return d;
}

// ---------------------------------------------------------------------------
// Shared memory plan (dynamic; the base is rounded up to 1024 bytes)

template <int BN, int WB>
struct Smem {
    static constexpr int kStages = stages_for<BN, WB>();
    static constexpr int kNacc = nacc_for<BN>();
    static constexpr int kEpiWarps = 4 * drain_groups<BN>();
    static constexpr int kA = kBM * kBK * 2;   // fp16 weights, 16 KB
    static constexpr int kB = BN * kBK * 2;    // fp16 activations
    static constexpr int kNib = kBM * WB;      // weight bytes (nibbles or int8 codes)
    static constexpr int kAs = 2 * kBM * 16;   // dw tiles of the two blocks
    static constexpr int kBs = 2 * BN * 16;    // da tiles of the two blocks
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kA;
    static constexpr int kOffNib = kOffB + kStages * kB;
    static constexpr int kOffAs = kOffNib + kStages * kNib;
    static constexpr int kOffBs = kOffAs + kStages * kAs;
    static constexpr int kOffZ = kOffBs + kStages * kBs;
    static constexpr int kOffBar = kOffZ + kZeroBytes;
    static constexpr int kNumBars = 3 * kStages + 2 * kNacc + kMmaWarps;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kBytes = kOffMisc + 16;
    static constexpr int kAlloc = kBytes + 1024;  // slack for the 1024-byte round-up
    static constexpr uint32_t kTx = kNib + kB + kBs;
    static_assert(kOffB % 1024 == 0 && kB % 1024 == 0, "swizzled tiles are 1024-byte aligned");
};

template <int BN, bool EMIT, int WB, bool RP>
__global__ void __launch_bounds__(threads_for<BN, WB>(), ctas_per_sm<BN>())
gemm_blocks_kernel(const __grid_constant__ CUtensorMap tm_nib,
                      const __grid_constant__ CUtensorMap tm_act,
                      const __grid_constant__ CUtensorMap tm_bs,
                      const unsigned short *__restrict__ wd, float *__restrict__ y,
                      int32_t *__restrict__ sumi, int m, int n, int kb_total, int m4,
                      uint32_t wait_limit, int withhold_loads, const uint8_t *__restrict__ wr) {
    static_assert(!RP || WB == 32, "the repacked layout holds Q4_0 nibbles");
    using S = Smem<BN, WB>;
    constexpr int kStages = S::kStages;
    constexpr int kNacc = S::kNacc;
    constexpr int kEpiWarps = S::kEpiWarps;
    constexpr int kConvWarps = conv_warps<BN, WB>();
    constexpr int kEpiWarp0 = epi_warp0<BN, WB>();
    static_assert(8 % kConvWarps == 0, "every converter takes a whole number of units per lane");
    static_assert(kNacc % kMmaWarps == 0, "block b's slot b % NACC belongs to issuer b % 2");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::kOffBar);
    uint64_t *bar_load = bar;                  // TMA landed (tx) + producer arrive
    uint64_t *bar_conv = bar + kStages;        // A and dw tiles written (one converter)
    uint64_t *bar_empty = bar + 2 * kStages;   // the stage's MMAs completed (both issuers)
    uint64_t *bar_accf = bar + 3 * kStages;    // accumulator slot full (one block)
    uint64_t *bar_acce = bar_accf + kNacc;     // accumulator slot drained
    uint64_t *bar_drain = bar_acce + kNacc;    // final MMA completion, one per issuer
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + S::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * BN;   // first token of the tile
    const int n0 = blockIdx.y * kBM;  // first weight row of the tile
    const int num_stages = (kb_total + 1) / 2;
    constexpr uint32_t kTmemCols = (uint32_t)(2 * kNacc * BN) < 32 ? 32 : (uint32_t)(2 * kNacc * BN);

    // the block of zeros the scale tiles' second K halves read
    for (int i = threadIdx.x; i < kZeroBytes / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(smem + S::kOffZ)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bar_load[s], 1);
            mbar_init(&bar_conv[s], kConvWarps);
            mbar_init(&bar_empty[s], kMmaWarps);
        }
        for (int b = 0; b < kNacc; ++b) {
            mbar_init(&bar_accf[b], 1);
            mbar_init(&bar_acce[b], kEpiWarps);
        }
        for (int w = 0; w < kMmaWarps; ++w) mbar_init(&bar_drain[w], 1);
        *abort_flag = 0;
        fence_mbar_init();
        tmap_prefetch(&tm_nib);
        tmap_prefetch(&tm_act);
        tmap_prefetch(&tm_bs);
    }
    fence_proxy_async_smem();  // the zeros are read by the tensor core
    if (warp == 1) tmem_alloc(tmem_holder, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int issued = 0;
        // withhold_loads (test hook): issue nothing, so every consumer wait
        // can only run out its poll limit
        for (int it = 0; it < (withhold_loads ? 0 : num_stages); ++it) {
            const int s = it % kStages;
            const uint32_t ph = (uint32_t)(it / kStages) & 1u;
            if (!wait_bounded_warp<BN>(&bar_empty[s], ph ^ 1u, wait_limit, abort_flag)) break;
            if (lane == 0) {
                const bool two = 2 * it + 1 < kb_total;
                mbar_arrive_expect_tx(&bar_load[s], S::kTx - (two ? 0u : (uint32_t)(BN * 16)));
                if constexpr (RP)  // tile (row group, stage): 4096 contiguous bytes = 16 map rows
                    tma_load_2d(smem + S::kOffNib + s * S::kNib, &tm_nib, &bar_load[s], 0,
                                (int)(((int64_t)blockIdx.y * num_stages + it) * 16));
                else
                    tma_load_2d(smem + S::kOffNib + s * S::kNib, &tm_nib, &bar_load[s], it * WB, n0);
                tma_load_2d(smem + S::kOffB + s * S::kB, &tm_act, &bar_load[s], it * kBK, t0);
                uint8_t *bs = smem + S::kOffBs + s * S::kBs;
                tma_load_2d(bs, &tm_bs, &bar_load[s], 0, (2 * it) * m4 + t0);
                if (two) tma_load_2d(bs + BN * 16, &tm_bs, &bar_load[s], 0, (2 * it + 1) * m4 + t0);
            }
            __syncwarp();
            issued = it + 1;
        }
        // Never leave a copy in flight: wait for every stage still pending.
        for (int it = issued > kStages ? issued - kStages : 0; it < issued; ++it) {
            volatile int no_abort = 0;
            wait_bounded_warp<BN>(&bar_load[it % kStages], (uint32_t)(it / kStages) & 1u, kDrainLimit,
                              &no_abort);
        }
    } else if (warp >= 1 && warp < 1 + kMmaWarps) {
        // ------------------------------------------------------------ MMA issuers
        // Lane 0 of warp 1 issues the even blocks, lane 0 of warp 2 the odd
        // ones: one thread's tcgen05 instructions issue one after another, so
        // two issuers keep the tensor core fed.  NACC is even, so block b's
        // slot b % NACC always belongs to the same issuer.  Per block: two
        // K=16 block-sum MMAs and the scale MMA, then a commit for the slot;
        // per stage each issuer commits to the stage's "empty" barrier.
        const int h = warp - 1;  // block parity
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(kBM, BN);
            const uint64_t a_desc0 = smem_desc_sw128(smem_u32(smem + S::kOffA));
            const uint64_t b_desc0 = smem_desc_sw128(smem_u32(smem + S::kOffB));
            const uint32_t zaddr = smem_u32(smem + S::kOffZ);
            int issued_any = 0;
            for (int it = 0; it < num_stages; ++it) {
                const int s = it % kStages;
                const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                const int kbi = 2 * it + h;
                const int slot = kbi % kNacc;
                const uint32_t sph = (uint32_t)(kbi / kNacc) & 1u;
                // operands first, so the MMAs issue back to back after the waits
                const uint64_t a_desc = a_desc0 + (uint64_t)(s * (S::kA >> 4)) + 4 * h;
                const uint64_t b_desc = b_desc0 + (uint64_t)(s * (S::kB >> 4)) + 4 * h;
                const uint32_t d = tmem_base + (uint32_t)(slot * 2 * BN);
                const uint32_t as = smem_u32(smem + S::kOffAs + s * S::kAs + h * kBM * 16);
                const uint32_t bs = smem_u32(smem + S::kOffBs + s * S::kBs + h * BN * 16);
                const uint64_t as_desc = smem_desc_scale(as, zaddr - as);
                const uint64_t bs_desc = smem_desc_scale(bs, zaddr - bs);
                if (!wait_bounded<BN>(&bar_conv[s], ph, wait_limit, abort_flag)) break;
                if (kbi < kb_total) {
                    if (!wait_bounded<BN>(&bar_acce[slot], sph ^ 1u, wait_limit, abort_flag)) break;
                    tc_fence_after();
                    mma_f16(d, a_desc, b_desc, idesc, 0u);
                    mma_f16(d, a_desc + 2, b_desc + 2, idesc, 1u);
                    if (!EMIT) mma_f16(d + BN, as_desc, bs_desc, idesc, 0u);
                    mma_commit(&bar_accf[slot]);
                    issued_any = 1;
                }
                // the stage's tiles are free once both issuers' MMAs completed
                mma_commit(&bar_empty[s]);
            }
            // Wait until every MMA issued here has finished.
            if (issued_any) {
                mma_commit(&bar_drain[h]);
                volatile int no_abort = 0;
                wait_bounded<BN>(&bar_drain[h], 0, kDrainLimit, &no_abort);
            }
        }
        __syncwarp();
    } else if (warp >= kConvWarp0 && warp < kConvWarp0 + kConvWarps) {
        // ------------------------------------------------------------ converters
        // Every converter takes every stage, in order, and converts its share
        // of the stage's 256 (row, block) units, kUpl per lane: unit
        // u = 32 (kUpl c + i) + lane is row u / 2, block u % 2.  A stage is
        // ready when all converters have arrived, so its conversion latency
        // is a fraction of one warp's pass.  Contiguous 16-byte reads; the
        // swizzled 16-byte stores of 8 consecutive lanes hit 8 different bank
        // groups.
        const int cw = warp - kConvWarp0;
        constexpr int kUpl = 8 / kConvWarps;
        for (int j = 0; j < num_stages; ++j) {
            const int s = j % kStages;
            const uint32_t ph = (uint32_t)(j / kStages) & 1u;
            // the stage's weight scales (global, L2) are requested before the
            // wait so their latency overlaps it
            unsigned short dwv[kUpl];
#pragma unroll
            for (int i = 0; i < kUpl; ++i) {
                const int u = 32 * (kUpl * cw + i) + lane;
                const int row = n0 + (u >> 1), kbi = 2 * j + (u & 1);
                dwv[i] = (!EMIT && row < n && kbi < kb_total) ? __ldg(wd + (int64_t)row * kb_total + kbi)
                                                               : (unsigned short)0;
            }
            if (!wait_bounded_warp<BN>(&bar_load[s], ph, wait_limit, abort_flag)) break;
            const uint8_t *nib = smem + S::kOffNib + s * S::kNib;
            uint8_t *a_tile = smem + S::kOffA + s * S::kA;
            uint8_t *as_tile = smem + S::kOffAs + s * S::kAs;
            // units in flight per batch: up to four nibble blocks, or two
            // blocks of codes (the same bytes in registers)
            constexpr int kBatch = (WB == 32 ? 4 : 2) < kUpl ? (WB == 32 ? 4 : 2) : kUpl;
#pragma unroll
            for (int g = 0; g < kUpl / kBatch; ++g) {
                uint4 v[kBatch][WB / 32];
#pragma unroll
                for (int i = 0; i < kBatch; ++i)
#pragma unroll
                    for (int jj = 0; jj < WB / 32; ++jj)
                        v[i][jj] = *reinterpret_cast<const uint4 *>(
                            nib + (32 * (kUpl * cw + kBatch * g + i) + lane) * (WB / 2) + 16 * jj);
#pragma unroll
                for (int i = 0; i < kBatch; ++i) {
                    const int u = 32 * (kUpl * cw + kBatch * g + i) + lane;
                    const int row = u >> 1, blk = u & 1;
                    uint4 out[4];
                    if constexpr (RP)
                        unpack_repacked_f16(v[i][0], out);
                    else if constexpr (WB == 32)
                        unpack_block_f16(v[i][0], out);
                    else
                        unpack_block_q8_f16(v[i][0], v[i][WB / 32 - 1], out);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4 *>(a_tile + row * 128 +
                                                   (((blk * 4 + c) ^ (row & 7)) * 16)) = out[c];
                    if (!EMIT)
                        *reinterpret_cast<uint4 *>(as_tile + blk * kBM * 16 + row * 16) =
                            make_uint4((uint32_t)dwv[kBatch * g + i], 0u, 0u, 0u);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_conv[s]);
        }
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + kEpiWarps) {
        // ------------------------------------------------------------ drains
        constexpr int kCols = BN / drain_groups<BN>();  // columns per thread (16 or 32)
        const int ew = warp - kEpiWarp0;
        const int q = warp & 3;                  // TMEM lane quarter = sub-partition
        const int grp = ew >> 2;                 // column group
        const int row = n0 + 32 * q + lane;      // weight row owned by this thread
        const int c0 = grp * kCols;              // first column (token) in the tile
        const bool row_ok = row < n;
        const uint32_t lane_base = tmem_base + ((uint32_t)(32 * q) << 16);
        uint64_t acc[kCols / 2];  // f32 pairs
#pragma unroll
        for (int c = 0; c < kCols / 2; ++c) acc[c] = 0ull;
        bool ok = true;
        for (int kbi = 0; kbi < kb_total; ++kbi) {
            const int slot = kbi % kNacc;
            if (!wait_bounded_warp<BN>(&bar_accf[slot], (uint32_t)(kbi / kNacc) & 1u, wait_limit,
                                   abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t col = lane_base + (uint32_t)(slot * 2 * BN + c0);
#pragma unroll
            for (int g = 0; g < kCols / 16; ++g) {
                uint32_t sv[16], scv[16];
                tmem_ld16(col + 16 * g, sv);
                if constexpr (!EMIT) tmem_ld16(col + BN + 16 * g, scv);
                tmem_wait_ld();
                if constexpr (EMIT) {
                    if (row_ok) {
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const int t = t0 + c0 + 16 * g + c;
                            if (t < m)
                                sumi[((int64_t)t * n + row) * kb_total + kbi] =
                                    __float2int_rn(__uint_as_float(sv[c]));
                        }
                    }
                } else {
                    // acc += sumi * S, two columns per instruction
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        acc[8 * g + c] = fma_f32x2(pack_u32x2(sv[2 * c], sv[2 * c + 1]),
                                                   pack_u32x2(scv[2 * c], scv[2 * c + 1]),
                                                   acc[8 * g + c]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_acce[slot]);
        }
        if (!EMIT && ok && !*abort_flag && row_ok) {
#pragma unroll
            for (int c = 0; c < kCols / 2; ++c) {
                float lo, hi;
                unpack_f32x2(acc[c], lo, hi);
                const int t = t0 + c0 + 2 * c;
                if (t < m) y[(int64_t)t * n + row] = lo;
                if (t + 1 < m) y[(int64_t)(t + 1) * n + row] = hi;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// Activation prepass: int8 -> fp16 (exact), and per block b and token t one
// 16-byte scale row {da[t, b], 0 x 7} (fp16) at row b * m4 + t (zero rows for
// t >= m, and all zeros when no scales are given: the block-sum variant).
__global__ void gemm_prep_kernel(const int8_t *__restrict__ aq, const unsigned short *__restrict__ ad,
                                 __half *__restrict__ a16, uint4 *__restrict__ bs, int64_t m,
                                 int64_t k, int64_t m4) {
    const int64_t kb = k / kQK;
    const int64_t n16 = m * k / 16;  // 16-element groups
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < n16; g += stride) {
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
                o[2 * i + j] = *reinterpret_cast<uint32_t *>(&hv);
            }
        }
        uint4 *dst = reinterpret_cast<uint4 *>(a16) + 2 * g;
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
    const int64_t nrows = kb * m4;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < nrows; g += stride) {
        const int64_t b = g / m4, t = g - b * m4;
        const uint32_t d = (t < m && ad != nullptr) ? (uint32_t)ad[t * kb + b] : 0u;
        bs[g] = make_uint4(d, 0u, 0u, 0u);
    }
}

// ---------------------------------------------------------------------------
// Host side

int choose_bn(int64_t m) {
    if (m <= 16) return 16;
    if (m <= 32) return 32;
    if (m <= 64) return 64;
    return 128;
}

struct WsPlan {
    size_t a16_off, a16_bytes, bs_off, bs_bytes, total;
    int64_t m4;
};

WsPlan plan_ws(int64_t m, int64_t k) {
    WsPlan p;
    p.m4 = (m + 3) / 4 * 4;
    p.a16_off = 0;
    p.a16_bytes = (size_t)m * (size_t)k * 2;
    p.bs_off = (p.a16_bytes + 255) / 256 * 256;
    p.bs_bytes = (size_t)(k / kQK) * (size_t)p.m4 * 16;
    p.total = p.bs_off + (p.bs_bytes + 255) / 256 * 256;
    return p;
}

uint32_t g_wait_limit = kDefaultWaitLimit;
int g_withhold_loads = 0;

template <int BN, int WB, bool RP>
cudaError_t launch_tile(const CUtensorMap &nib, const CUtensorMap &act, const CUtensorMap &bs,
                        const uint16_t *wd, float *y, int32_t *sumi, int64_t m, int64_t n,
                        int64_t k, int64_t m4, const uint8_t *wr, cudaStream_t s) {
    using S = Smem<BN, WB>;
    const int kb = (int)(k / kQK);
    dim3 grid((unsigned)((m + BN - 1) / BN), (unsigned)((n + kBM - 1) / kBM));
    const auto *wdp = reinterpret_cast<const unsigned short *>(wd);
    if (sumi) {
        auto kern = gemm_blocks_kernel<BN, true, WB, RP>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kAlloc);
        kern<<<grid, threads_for<BN, WB>(), S::kAlloc, s>>>(nib, act, bs, wdp, y, sumi, (int)m, (int)n, kb,
                                                        (int)m4, g_wait_limit, g_withhold_loads, wr);
    } else {
        auto kern = gemm_blocks_kernel<BN, false, WB, RP>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kAlloc);
        kern<<<grid, threads_for<BN, WB>(), S::kAlloc, s>>>(nib, act, bs, wdp, y, sumi, (int)m, (int)n, kb,
                                                        (int)m4, g_wait_limit, g_withhold_loads, wr);
    }
    return cudaPeekAtLastError();
}

}  // namespace

// Covers both products a GEMM call may launch (the few-token kernel of
// gemm_small.cu for m <= 64 with Q4_0 weights, m <= 32 with Q8_0, the
// tcgen05 kernel otherwise), either weight format.
size_t gemm_workspace_bytes(int64_t m, int64_t n, int64_t k) {
    const size_t t = plan_ws(m, k).total;
    return gemm_small_m_supported_q4(m, n, k) ? std::max(t, gemm_small_m_workspace_bytes(m, k)) : t;
}

void gemm_set_wait_limit(uint32_t iterations) { g_wait_limit = iterations ? iterations : kDefaultWaitLimit; }

void gemm_set_withhold_loads(int enable) {
    g_withhold_loads = enable ? 1 : 0;
    gemm_small_set_withhold_loads(enable);
}

cudaError_t gemm_read_and_clear_error(unsigned int *word, cudaStream_t s) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_gemm_error, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    if (*word) {
        e = cudaMemcpyToSymbolAsync(g_gemm_error, &zero, sizeof(unsigned int), 0,
                                    cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

namespace {

// Shared host path of both weight formats: prepass, tensor maps, launch.
// WB = weight bytes per row and stage (32: Q4_0 nibbles [n, k/2]; 64: Q8_0
// codes [n, k]).
template <int WB, bool RP>
cudaError_t launch_gemm(const void *w, const uint16_t *wd, const int8_t *aq, const uint16_t *ad,
                        float *y, int32_t *sumi, int64_t m, int64_t n, int64_t k, void *workspace,
                        cudaStream_t s) {
    const WsPlan p = plan_ws(m, k);
    auto *ws = static_cast<uint8_t *>(workspace);
    __half *a16 = reinterpret_cast<__half *>(ws + p.a16_off);
    uint4 *bs = reinterpret_cast<uint4 *>(ws + p.bs_off);
    {
        const int threads = 256;
        const int64_t work = std::max<int64_t>(m * k / 16, (k / kQK) * p.m4);  // groups, scale rows
        const int64_t blocks = std::min<int64_t>((work + threads - 1) / threads, 152 * 8);
        gemm_prep_kernel<<<(unsigned)blocks, threads, 0, s>>>(
            aq, reinterpret_cast<const unsigned short *>(ad), a16, bs, m, k, p.m4);
        cudaError_t e = cudaPeekAtLastError();
        if (e != cudaSuccess) return e;
    }
    const int bn = choose_bn(m);
    const uint64_t row_bytes = (uint64_t)(k * WB / kBK);  // k/2 (Q4_0) or k (Q8_0)
    CUtensorMap tm_nib, tm_act, tm_bs;
    // weights: u8 [n rows, row_bytes], box WB bytes x 128 rows; the repacked
    // tiles as u8 [tiles * 16 rows, 256 bytes], box 256 x 16 (one tile)
    if (RP) {
        const uint64_t map_rows = (uint64_t)((n + kBM - 1) / kBM) * (uint64_t)((k / kQK + 1) / 2) * 16;
        if (!make_map_2d(&tm_nib, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, 256, map_rows, 256, 256, 16,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else if (!make_map_2d(&tm_nib, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, row_bytes, (uint64_t)n,
                            row_bytes, WB, kBM, CU_TENSOR_MAP_SWIZZLE_NONE)) {
        return cudaErrorInvalidValue;
    }
    const uint8_t *wr = RP ? static_cast<const uint8_t *>(w) : nullptr;
    // activations: fp16 [m rows, k], box 64 x BN, 128-byte swizzle
    if (!make_map_2d(&tm_act, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a16, (uint64_t)k, (uint64_t)m,
                     (uint64_t)k * 2, kBK, (uint32_t)bn, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    // activation scale rows: fp16 [k/32 * m4 rows, 8], box 8 x BN
    if (!make_map_2d(&tm_bs, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, bs, 8, (uint64_t)(k / kQK) * p.m4, 16,
                     8, (uint32_t)bn, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    switch (bn) {
        case 16: return launch_tile<16, WB, RP>(tm_nib, tm_act, tm_bs, wd, y, sumi, m, n, k, p.m4, wr, s);
        case 32: return launch_tile<32, WB, RP>(tm_nib, tm_act, tm_bs, wd, y, sumi, m, n, k, p.m4, wr, s);
        case 64: return launch_tile<64, WB, RP>(tm_nib, tm_act, tm_bs, wd, y, sumi, m, n, k, p.m4, wr, s);
        default: return launch_tile<128, WB, RP>(tm_nib, tm_act, tm_bs, wd, y, sumi, m, n, k, p.m4, wr, s);
    }
}

}  // namespace

cudaError_t launch_gemm_q4_0_q8_0(const uint8_t *wq, const uint16_t *wd, const int8_t *aq,
                                  const uint16_t *ad, float *y, int32_t *sumi, int64_t m,
                                  int64_t n, int64_t k, void *workspace, cudaStream_t s) {
    // the few-token kernel copies dw with a tensor map, whose base must be
    // 16-byte aligned (the entry point only asks for 2)
    if (gemm_small_m_supported_q4(m, n, k) && (reinterpret_cast<uintptr_t>(wd) & 15) == 0)
        return launch_gemm_small_m(wq, wd, aq, ad, y, sumi, m, n, k, workspace, s);
    return launch_gemm<32, false>(wq, wd, aq, ad, y, sumi, m, n, k, workspace, s);
}

cudaError_t launch_gemm_q8_0_q8_0(const int8_t *w8, const uint16_t *wd, const int8_t *aq,
                                  const uint16_t *ad, float *y, int32_t *sumi, int64_t m,
                                  int64_t n, int64_t k, void *workspace, cudaStream_t s) {
    if (gemm_small_m_supported(m, n, k) && (reinterpret_cast<uintptr_t>(wd) & 15) == 0)
        return launch_gemm_small_m_q8(w8, wd, aq, ad, y, sumi, m, n, k, workspace, s);
    return launch_gemm<64, false>(w8, wd, aq, ad, y, sumi, m, n, k, workspace, s);
}

size_t repack_q4_0_gemm_bytes(int64_t n, int64_t k) {
    return (size_t)((n + kBM - 1) / kBM) * (size_t)((k / kQK + 1) / 2) * (size_t)(kBM * 32);
}

cudaError_t launch_gemm_q4_0_q8_0_repacked(const uint8_t *wr, const uint16_t *wd, const int8_t *aq,
                                           const uint16_t *ad, float *y, int32_t *sumi, int64_t m,
                                           int64_t n, int64_t k, void *workspace, cudaStream_t s) {
    return launch_gemm<32, true>(wr, wd, aq, ad, y, sumi, m, n, k, workspace, s);
}

// Load-time repack: thread t writes 16-byte unit t of the tiles (row group g,
// stage j, unit u = 2 * row + block), from block b = 2j + u % 2 of row
// r = 128 g + u / 2: word c carries elements 8c..8c+7 (low nibbles of bytes
// 8c.. for c < 2, high nibbles of bytes 8(c-2).. for c >= 2), element
// 8c + 2i + h at bits 4i + 16h.  Rows past n and blocks past k/32: nibble 8.
__global__ void repack_q4_0_gemm_kernel(const uint8_t *__restrict__ wq, int64_t n, int64_t k,
                                        uint4 *__restrict__ wr, int64_t units, int64_t tiles_k) {
    const int64_t kb = k / kQK;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < units;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tile = t / 256;
        const int u = (int)(t % 256);
        const int64_t g = tile / tiles_k, j = tile % tiles_k;
        const int64_t r = g * kBM + u / 2, b = 2 * j + u % 2;
        uint4 out = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
        if (r < n && b < kb) {
            const uint4 src = *reinterpret_cast<const uint4 *>(wq + r * (k / 2) + b * 16);
            const uint32_t bw[4] = {src.x, src.y, src.z, src.w};
            uint32_t word[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t acc = 0;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int byte = 8 * (c & 1) + e;
                    const uint32_t v = (bw[byte >> 2] >> (8 * (byte & 3) + (c >= 2 ? 4 : 0))) & 0xFu;
                    acc |= v << (4 * (e >> 1) + 16 * (e & 1));
                }
                word[c] = acc;
            }
            out = make_uint4(word[0], word[1], word[2], word[3]);
        }
        wr[t] = out;
    }
}

cudaError_t launch_repack_q4_0_gemm(const uint8_t *wq, int64_t n, int64_t k, uint8_t *wr,
                                    cudaStream_t s) {
    const int64_t tiles_k = (k / kQK + 1) / 2;
    const int64_t units = ((n + kBM - 1) / kBM) * tiles_k * 256;
    const int threads = 256;
    const int64_t blocks = std::min<int64_t>((units + threads - 1) / threads, 152 * 16);
    repack_q4_0_gemm_kernel<<<(unsigned)blocks, threads, 0, s>>>(wq, n, k, reinterpret_cast<uint4 *>(wr),
                                                                 units, tiles_k);
    return cudaPeekAtLastError();
}

}  // namespace qmm
