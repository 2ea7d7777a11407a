/*
 * qmm.h -- C ABI of libqmm.so: quantized weight-by-activation matmul on GB300
 * (sm_103a).
 *
 * The operation (llama.cpp visual guide, lesson 31 "The CPU backend", section
 * "How the quantized dot product works"): weights are Q4_0 blocks of 32
 * four-bit values with one fp16 scale each (value = (nibble - 8) * dw),
 * activations are Q8_0 blocks of 32 int8 values with one fp16 scale each
 * (value = q * da).  For every output the kernels form the exact integer dot
 * of each block pair, sumi = sum_j (nibble_j - 8) * q_j, and accumulate
 * sumi * (dw * da) in f32.  The ternary variant (Loom docs, "Plan 9 SIMD
 * Forward", section "BitNet ternary MAD kernel") packs weights in {-1,0,+1}
 * as 2-bit codes 16 per uint32 and computes dot = sum(code*q) - sum(q),
 * then y = dot * weight_absmean / activation_scale.
 *
 * Conventions shared by every entry point
 *  - Every data pointer is a DEVICE pointer owned by the caller (allocated
 *    through any CUDA allocator); the library never allocates, frees or
 *    keeps a pointer after the call returns.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Work is enqueued asynchronously on it; the library never
 *    synchronizes the host.  Outputs are valid once the stream reaches the
 *    point after the call.
 *  - All argument checks run on the host before anything is launched.  A
 *    failed check returns a non-zero qmm_status and launches nothing.  The
 *    kernels themselves check nothing (the caller-validated contract of the
 *    Fucina course, chapter 06, section 6.3).
 *  - Sizes are int64_t element counts.  m = activation rows (tokens),
 *    n = output columns (weight rows), k = reduction length.
 *  - Layouts are row-major and dense:
 *      x   f32  [m, k] (row stride ldx where given)
 *      aq  int8 [m, k]          ad  fp16 (raw bits) [m, k/32]
 *      wq  u8   [n, k/2]        wd  fp16 (raw bits) [n, k/32]
 *      y   f32  [m, n]
 *    wq/wd are the two planes of an array of block_q4_0: byte j of a block
 *    holds element j in its low nibble and element j+16 in its high nibble;
 *    the 16 bytes of block b of row r start at wq + r*k/2 + 16*b.
 *  - Rounding: quantizers divide in IEEE f32 and round half away from zero;
 *    stored scales are fp16 round-to-nearest-even of the f32 scale.
 *  - Requires a device of compute capability 10.3 (GB300); any other device
 *    gives QMM_ERR_UNSUPPORTED_DEVICE.
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum qmm_status {
    QMM_OK = 0,
    QMM_ERR_NULL = 1,               /* a required pointer is NULL */
    QMM_ERR_SHAPE = 2,              /* a size is <= 0, too large, or not a block multiple */
    QMM_ERR_ALIGN = 3,              /* a pointer lacks the alignment stated for it */
    QMM_ERR_WORKSPACE = 4,          /* workspace NULL or smaller than qmm_workspace_bytes() */
    QMM_ERR_UNSUPPORTED_DEVICE = 5, /* the current device is not compute capability 10.3 */
    QMM_ERR_CUDA = 6,               /* a CUDA runtime call or a kernel launch failed */
    QMM_ERR_TIMEOUT = 7,            /* a bounded device-side wait gave up (see qmm_check_device_error) */
    QMM_ERR_ARG = 8                 /* another invalid argument (split_k, op id, path id) */
} qmm_status;

/* Workspace-taking operations, for qmm_workspace_bytes(). */
enum {
    QMM_OP_GEMV_Q4_0_Q8_0 = 1,
    QMM_OP_GEMM_Q4_0_Q8_0 = 2,
    QMM_OP_BITNET_GEMM = 3,
    QMM_OP_GEMV_Q8_0_Q8_0 = 4,
    QMM_OP_GEMM_Q8_0_Q8_0 = 5
};

/* Largest m accepted by the GEMV entry points (decode and small batches). */
#define QMM_GEMV_MAX_M 16

/* ---------------------------------------------------------------------- */
/* Activation quantization to Q8_0 (lesson 31, "How the quantized dot product
 * works": activations are Q8_0 int8 blocks with an fp16 scale).  For every
 * row i and block b: amax = max |x|, d = amax / 127 (f32), q = 0 if d == 0
 * else clamp(round(x / d), -127, 127); ad = fp16(d).
 *   x    f32 [m, ldx] (only the first k columns are read); 4-byte aligned
 *   aq   int8 [m, k] output;  ad  fp16 bits [m, k/32] output, 2-byte aligned
 *   k % 32 == 0, ldx >= k.  Inputs must be finite. */
qmm_status qmm_quantize_act_q8_0(const float *x, int64_t m, int64_t k, int64_t ldx,
                                 int8_t *aq, uint16_t *ad, void *stream);

/* Weight quantization to Q4_0 (load-time, not on the per-token path).  For
 * every row and block: the element of largest |w| (first one on ties) keeps
 * its sign as `max`; d = max / -8; q = 8 if d == 0 else
 * clamp(round(w / d) + 8, 0, 15); packed as described above; wd = fp16(d).
 *   w   f32 [n, k], 4-byte aligned;  wq u8 [n, k/2];  wd fp16 bits [n, k/32]
 *   k % 32 == 0.  Inputs must be finite. */
qmm_status qmm_quantize_weight_q4_0(const float *w, int64_t n, int64_t k,
                                    uint8_t *wq, uint16_t *wd, void *stream);

/* ---------------------------------------------------------------------- */
/* Q4_0 x Q8_0 matrix-vector product for decode (1 <= m <= QMM_GEMV_MAX_M):
 *   y[i, r] = sum over blocks b of sumi[i, r, b] * (dw[r, b] * da[i, b]),
 * sumi exact in int32, the scaled terms accumulated in f32 (the order differs
 * from a serial loop; results agree to f32 rounding).  Weights stream once
 * from HBM for all m rows.
 *   wq 16-byte aligned; aq 16-byte aligned; wd, ad 2-byte aligned; y 4-byte.
 *   k % 32 == 0.
 *   split_k: 1 = no split; S > 1 = the k range is cut into S slices whose f32
 *   partials go to the workspace and are summed in slice order by a second
 *   kernel on the same stream (deterministic); 0 = the library picks S from
 *   the shape.  S may not exceed k/32.  workspace: device memory of at least
 *   qmm_workspace_bytes(QMM_OP_GEMV_Q4_0_Q8_0, m, n, k, split_k) bytes,
 *   16-byte aligned (NULL allowed when that size is 0).
 * With split_k = 0, 3 <= m, k % 256 == 0, wd 16-byte aligned and a 256-byte
 * aligned workspace of at least the queried size (the query for split_k = 0
 * covers it), the call runs the few-token product described at
 * qmm_gemm_q4_0_q8_0 instead, which is faster from three tokens on; its y is
 * the serial definition bit for bit, within this entry's tolerance.  A
 * smaller or absent workspace keeps the GEMV kernels.  Explicit split_k >= 1
 * always runs the GEMV kernels.
 * With one slice and 8 <= m, when k/32 is a multiple of 8, wq, wd, aq and
 * ad are 16-byte aligned and the quantized activations fit in shared memory,
 * a persistent kernel streams the weights through shared memory with tensor
 * copies; otherwise each warp streams them through registers.  At m = 1 with
 * at most 1024 blocks per slice (k <= 32768 unsplit) each CTA first reads
 * the activation slice once into shared memory for all its warps.  All of
 * these give the same bits. */
qmm_status qmm_gemv_q4_0_q8_0(const uint8_t *wq, const uint16_t *wd,
                              const int8_t *aq, const uint16_t *ad, float *y,
                              int64_t m, int64_t n, int64_t k, int split_k,
                              void *workspace, size_t workspace_bytes, void *stream);

/* The GEMV above for callers that cannot allocate device memory where they
 * run it -- for instance a latency-critical decode loop that must not enter
 * the CUDA allocator (its locks and possible implicit synchronization), or a
 * component that only receives device pointers and owns no allocator.  The
 * pages this library follows have no counterpart: this is a deployment
 * convenience.  Same arguments, result and rules as qmm_gemv_q4_0_q8_0
 * except that there is no workspace: the split-K partials go to a device
 * array owned by the library, QMM_NOALLOC_SCRATCH_FLOATS floats (4 MiB)
 * reserved on every GPU that loads the library and held until the process
 * exits.  The call itself allocates nothing.  It always runs the GEMV
 * kernels, never the few-token product (whose activation layout would need
 * a workspace), so at m >= 3 with split_k = 0 its bits can differ from
 * those of qmm_gemv_q4_0_q8_0 given a workspace; both meet the same
 * tolerance.
 *   - A split_k > 1 with split_k * m * n > QMM_NOALLOC_SCRATCH_FLOATS
 *     returns QMM_ERR_WORKSPACE and launches nothing.  The automatic split
 *     (split_k = 0) always fits: it exceeds 1 only for short grids (n below
 *     ~1200 rows) and never passes 32.
 *   - The first call on a device looks up the array's device address with
 *     that device current and keeps it for the life of the process; make
 *     that first call before any stream capture.  Calls after
 *     cudaDeviceReset (or any teardown of the device's primary context) are
 *     not supported: the kept address would no longer be valid.
 *   - Every call on a device shares the one array (it keeps the last call's
 *     partials; each call overwrites all it reads, so nothing needs
 *     clearing): calls whose executions overlap on the GPU, e.g. on two
 *     streams, race and give wrong results.  Order them on one stream. */
#define QMM_NOALLOC_SCRATCH_FLOATS (1 << 20)
qmm_status qmm_gemv_q4_0_q8_0_noalloc(const uint8_t *wq, const uint16_t *wd,
                                      const int8_t *aq, const uint16_t *ad, float *y,
                                      int64_t m, int64_t n, int64_t k, int split_k,
                                      void *stream);

/* Decode linear layer y = x W^T with Q8_0 activations (1 <= m <=
 * QMM_GEMV_MAX_M): qmm_quantize_act_q8_0 of x into aq/ad, then
 * qmm_gemv_q4_0_q8_0 with split_k = 1, enqueued as one call; y, aq and ad
 * are bit for bit those of the two calls.
 *   x f32 [m, ldx] (first k columns), 4-byte aligned; aq int8 [m, k] 16-byte
 *   aligned; ad fp16 bits [m, k/32] 2-byte aligned; wq, wd, y as for
 *   qmm_gemv_q4_0_q8_0.
 *   flags: 0, or QMM_LINEAR_PDL: launch both kernels with programmatic
 *   dependent launch.  Each may then start while its predecessor on the
 *   stream is still running: the quantizer reads x, and the GEMV reads aq/ad
 *   and writes y, only after the predecessor completed, while the GEMV loads
 *   its first weight blocks (wq, wd) before that.  So layer i+1's first
 *   weight traffic overlaps layer i's tail and the launch gaps close.  Only
 *   valid when wq and wd are not written by work still running on the
 *   stream when the call is enqueued (true for model weights).  A chain of
 *   such calls on one stream stays ordered: every kernel reads its inputs
 *   after the kernel before it completed, which completed after the one
 *   before that, and so on. */
#define QMM_LINEAR_PDL 1
#define QMM_LINEAR_HOST_DIRECT 2  /* qmm_linear_q4_0_grouped_host only */
qmm_status qmm_linear_q4_0(const uint8_t *wq, const uint16_t *wd, const float *x, int64_t ldx,
                           int8_t *aq, uint16_t *ad, float *y, int64_t m, int64_t n, int64_t k,
                           int flags, void *stream);

/* One problem of qmm_linear_q4_0_grouped: the arguments of qmm_linear_q4_0
 * for one weight matrix (same meaning, layout and alignment rules). */
typedef struct qmm_linear_problem {
    const uint8_t *wq;   /* Q4_0 nibbles [n, k/2] */
    const uint16_t *wd;  /* Q4_0 scales, fp16 bits [n, k/32] */
    const float *x;      /* activations f32 [m, ldx] */
    int64_t ldx;
    int8_t *aq;          /* receives the Q8_0 codes [m, k] */
    uint16_t *ad;        /* receives the Q8_0 scales, fp16 bits [m, k/32] */
    float *y;            /* receives y f32 [m, n] */
    int64_t n;
    int64_t k;
} qmm_linear_problem;

/* Up to QMM_GROUP_MAX independent decode linear layers with the same m in
 * two launches in all: one quantizer launch over every problem's x, then
 * one GEMV launch whose CTAs cover every problem's rows (the way a model's
 * Q/K/V or gate/up projections, or the experts of a mixture, are batched).
 * Each problem's y, aq and ad are bit for bit those of qmm_linear_q4_0 on
 * it alone.  `problems` is a host array read during the call.  The problems
 * must be independent: no problem's aq, ad or y may overlap any buffer of
 * another problem.  flags as for qmm_linear_q4_0. */
#define QMM_GROUP_MAX 16
qmm_status qmm_linear_q4_0_grouped(const qmm_linear_problem *problems, int count, int64_t m,
                                   int flags, void *stream);

/* qmm_linear_q4_0_grouped with its input coming from, and its output going
 * to, host memory, in one call: a copy of x_bytes from x_host (host) to
 * x_dev (device), the grouped layers, then a copy of y_bytes from y_dev
 * (device) to y_host (host).  All three are enqueued on `stream` in that
 * order (cudaMemcpyAsync).  With page-locked host buffers the call returns
 * before they run, so the caller must keep x_host and y_host alive and
 * unchanged until the stream has passed the copies; pageable host memory
 * makes the copies synchronous.  The problems' x must lie in
 * [x_dev, x_dev + x_bytes) and their y in [y_dev, y_dev + y_bytes) for the
 * copies to carry them; without QMM_LINEAR_HOST_DIRECT the library does
 * not check this.  A size of 0 skips that copy (its pointers may then be
 * NULL).
 *   flags: QMM_LINEAR_PDL as for qmm_linear_q4_0, and QMM_LINEAR_HOST_DIRECT:
 *   where the runtime reports a device address for both host buffers
 *   (page-locked memory on a system with unified addressing, as over
 *   NVLink-C2C on GB300), the kernels read x from x_host and write y to
 *   y_host themselves and x_dev and y_dev are not touched.  The problems' x
 *   and y must then lie in the device buffers (checked, QMM_ERR_ARG
 *   otherwise), and each is redirected to the same offset in the host
 *   buffer.  Where the runtime reports none, the call copies as without the
 *   flag.
 * The same checks as qmm_linear_q4_0_grouped run first, and a failure
 * enqueues nothing; a failed copy or launch returns QMM_ERR_CUDA, possibly
 * after the earlier steps were enqueued. */
qmm_status qmm_linear_q4_0_grouped_host(const qmm_linear_problem *problems, int count, int64_t m,
                                        int flags, const void *x_host, void *x_dev, size_t x_bytes,
                                        const void *y_dev, void *y_host, size_t y_bytes,
                                        void *stream);

/* 1 when the current device can address the host memory at `host` itself
 * (the condition QMM_LINEAR_HOST_DIRECT acts on), else 0.  Asks the runtime
 * for the pointer's attributes; dereferences nothing. */
int qmm_host_addressable(const void *host);

/* Q4_0 x Q8_0 matrix product for prefill (m >= 1, any n, k % 32 == 0), same
 * result definition as the GEMV.  The block sums run on the tensor cores
 * (tcgen05.mma kind::f16 with f32 accumulators in TMEM): the int4 and int8
 * values are exact in fp16 and every partial sum is an integer below 2^24,
 * so each block sum is exact; each f32 output then accumulates
 * fma(sumi, dw*da, acc) over blocks in ascending order; the exact products
 * dw*da come from the tensor core too.  The workspace holds an fp16 copy of
 * the activations and one 16-byte activation-scale row per (block, token).
 * For a few tokens (m <= 64, k % 256 == 0, wd 16-byte aligned) the call runs
 * a product on the warp-level tensor-core MMA instead (mma.sync, f16
 * operands, f32 accumulators in registers), with the same block sums and the
 * same bits of y; its workspace holds the activations as fp16 in the MMA's
 * fragment order (1 KB per block and 16-token tile) and, per block and tile,
 * a 128-byte record of per-token block corrections and scales (f32).  The workspace query covers whichever
 * product the shape can take.
 *   wq 16-byte aligned; aq 16-byte aligned; wd, ad 2-byte aligned; y 4-byte;
 *   workspace 256-byte aligned, at least
 *   qmm_workspace_bytes(QMM_OP_GEMM_Q4_0_Q8_0, m, n, k, 0) bytes.
 *   Not reentrant on one workspace: calls that share a workspace must be
 *   ordered on one stream. */
qmm_status qmm_gemm_q4_0_q8_0(const uint8_t *wq, const uint16_t *wd,
                              const int8_t *aq, const uint16_t *ad, float *y,
                              int64_t m, int64_t n, int64_t k,
                              void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* Load-time repack of Q4_0 weights for the prefill GEMM (Fucina reference,
 * section 9.7: weights are packed once, at load time, into the layout the
 * kernel reads).  A pure permutation of the nibble plane wq [n, k/2]:
 * ceil(n/128) * ceil(k/64) tiles of 4096 bytes, tile (g, j) for rows
 * 128g..128g+127 and blocks 2j, 2j+1, at byte (g * ceil(k/64) + j) * 4096.
 * Inside a tile, 16-byte unit u = 2 * row + block holds one block as four
 * 32-bit words; word c carries elements 8c..8c+7, element 8c + 2i + h at
 * bits 4i + 16h, so (word >> 4i) & 0x000F000F yields a pair of elements in
 * the two 16-bit halves.  Rows past n and the block past an odd k/32 hold
 * nibble 8 (value 0).  The scales wd are not repacked.
 *   qmm_repack_q4_0_gemm_bytes: size of wr (SIZE_MAX for a bad shape).
 *   wq, wr 16-byte aligned; k % 32 == 0. */
size_t qmm_repack_q4_0_gemm_bytes(int64_t n, int64_t k);
qmm_status qmm_repack_q4_0_gemm(const uint8_t *wq, int64_t n, int64_t k, uint8_t *wr,
                                size_t wr_bytes, void *stream);

/* qmm_gemm_q4_0_q8_0 on repacked weights: identical results, bit for bit.
 * Each pipeline stage's weight tile then arrives as one contiguous bulk copy
 * and unpacks with shifts and masks only.  wr of at least
 * qmm_repack_q4_0_gemm_bytes(n, k) bytes, 16-byte aligned; other arguments
 * as for qmm_gemm_q4_0_q8_0. */
qmm_status qmm_gemm_q4_0_q8_0_repacked(const uint8_t *wr, size_t wr_bytes, const uint16_t *wd,
                                       const int8_t *aq, const uint16_t *ad, float *y,
                                       int64_t m, int64_t n, int64_t k,
                                       void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* Q8_0 weights x Q8_0 activations.  The Q8_0 block (lesson 31: 32 int8 codes
 * and one fp16 scale) also serves as a weight format (Fucina reference,
 * section 9: the Q8_0 right-hand side of 9.2 and 9.7, Q8_0 decode and
 * prefill in 9.9.2).  Weights are quantized with the activation recipe:
 * qmm_quantize_act_q8_0 on the f32 weight rows gives the two planes, codes
 * w8 int8 [n, k] and scales wd fp16 bits [n, k/32].  The block dot is
 * sumi = sum_j q_w * q_a (no offset), exact in int32 (|sumi| <= 516,128),
 * and y follows the same rule as the Q4_0 products.
 *
 * The decode GEMV (1 <= m <= QMM_GEMV_MAX_M): arguments, split_k and
 * workspace as for qmm_gemv_q4_0_q8_0 (workspace size from
 * qmm_workspace_bytes(QMM_OP_GEMV_Q8_0_Q8_0, ...)); w8 16-byte aligned.
 * Each warp streams its rows through registers, two 16-byte loads per
 * block.  With split_k = 0 and the conditions stated at qmm_gemv_q4_0_q8_0
 * the call runs the few-token product of qmm_gemm_q8_0_q8_0 instead. */
qmm_status qmm_gemv_q8_0_q8_0(const int8_t *w8, const uint16_t *wd,
                              const int8_t *aq, const uint16_t *ad, float *y,
                              int64_t m, int64_t n, int64_t k, int split_k,
                              void *workspace, size_t workspace_bytes, void *stream);

/* The prefill product (any m >= 1) on the tensor cores, as
 * qmm_gemm_q4_0_q8_0: the int8 codes are exact in fp16, the block sums exact
 * in the f32 TMEM accumulators, and each f32 output accumulates
 * fma(sumi, dw*da, acc) over blocks in ascending order, bit for bit the
 * serial definition.  For a few tokens (m <= 32, k % 256 == 0, wd 16-byte
 * aligned) the call runs the warp-level product described at
 * qmm_gemm_q4_0_q8_0, reading each int8 code as the fp16 value 1152 + code
 * (one logic instruction) and taking 1152 times the activations' block sum
 * out exactly; same block sums, same bits of y.  Workspace:
 * qmm_workspace_bytes(QMM_OP_GEMM_Q8_0_Q8_0, m, n, k, 0) bytes (it covers
 * either product), 256-byte aligned; w8 16-byte aligned; the rest as for
 * qmm_gemm_q4_0_q8_0. */
qmm_status qmm_gemm_q8_0_q8_0(const int8_t *w8, const uint16_t *wd,
                              const int8_t *aq, const uint16_t *ad, float *y,
                              int64_t m, int64_t n, int64_t k,
                              void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* BitNet activation quantization (Loom, "BitNet ternary MAD kernel"): per row
 * s = 127 / max|x| (s = 0 for an all-zero row), q = clamp(round(x * s),
 * -127, 127), act_sum = sum q.
 *   x f32 [m, k] 4-byte aligned; aq int8 [m, k]; act_scale f32 [m];
 *   act_sum int32 [m].  k % 16 == 0.  Inputs must be finite. */
qmm_status qmm_quantize_act_bitnet(const float *x, int64_t m, int64_t k,
                                   int8_t *aq, float *act_scale, int32_t *act_sum,
                                   void *stream);

/* Pack ternary weights t in {-1, 0, +1} (int8 [n, k]) as code = t + 1,
 * 16 codes per uint32, element i of each word at bits [2i, 2i+1] (load-time).
 * Values outside {-1, 0, 1} give unspecified codes.  k % 16 == 0;
 * w uint32 [n, k/16], 4-byte aligned. */
qmm_status qmm_pack_ternary(const int8_t *t, int64_t n, int64_t k, uint32_t *w,
                            void *stream);

/* BitNet ternary matrix-vector product (1 <= m <= QMM_GEMV_MAX_M):
 *   dot[i, r] = sum_j code[r, j] * aq[i, j] - act_sum[i]   (exact int32)
 *   y[i, r]   = act_scale[i] == 0 ? 0 : ((float)dot * weight_absmean) / act_scale[i]
 * (two IEEE f32 operations, left to right, so y is reproducible bit for bit).
 *   w uint32 [n, k/16] 16-byte aligned; aq 16-byte aligned; k % 16 == 0,
 *   k <= 2^21 (so |dot| fits int32). */
qmm_status qmm_bitnet_gemv(const uint32_t *w, float weight_absmean,
                           const int8_t *aq, const float *act_scale, const int32_t *act_sum,
                           float *y, int64_t m, int64_t n, int64_t k, void *stream);

/* BitNet decode linear layer (Loom, "BitNet ternary MAD kernel"): the
 * activation quantization of qmm_quantize_act_bitnet on x, then
 * qmm_bitnet_gemv, enqueued as one call; aq, act_scale, act_sum and y are bit
 * for bit those of the two calls.  1 <= m <= QMM_GEMV_MAX_M.  For m = 1 with
 * k % 64 == 0, k <= 32768 and x, aq 16-byte aligned this is one kernel in
 * which every CTA quantizes the row itself (the same operations) and CTA 0
 * writes aq, act_scale and act_sum; otherwise two kernels.
 *   x f32 [m, ldx] (first k columns, ldx >= k), 4-byte aligned; aq int8
 *   [m, k] 16-byte aligned; act_scale f32 [m], act_sum int32 [m] 4-byte
 *   aligned; w, y and the limits on k as for qmm_bitnet_gemv.  Inputs must
 *   be finite.
 *   flags: 0, or QMM_LINEAR_PDL: both kernels launch with programmatic
 *   dependent launch, with the same rules as qmm_linear_q4_0 (the GEMV loads
 *   its first weight words before the quantizer has finished, so w must not
 *   be written by work still running on the stream; a chain of such calls
 *   on one stream stays ordered).
 * Errors as for the two calls; QMM_ERR_ARG for unknown flags. */
qmm_status qmm_linear_bitnet(const uint32_t *w, float weight_absmean, const float *x, int64_t ldx,
                             int8_t *aq, float *act_scale, int32_t *act_sum, float *y,
                             int64_t m, int64_t n, int64_t k, int flags, void *stream);

/* BitNet ternary matrix product for prefill (any m >= 1), on the tensor
 * cores.  Same result as qmm_bitnet_gemv, bit for bit:
 *   dot[i, r] = sum_j (code[r, j] - 1) * aq[i, j]    (exact; equal to the
 *               identity sum(code * q) - sum(q), so no act_sum is needed)
 *   y[i, r]   = act_scale[i] == 0 ? 0 : ((float)dot * weight_absmean) / act_scale[i]
 * Every operand is exact in fp16 and |dot| < 2^24, so the tensor core's f32
 * accumulation over all of k is exact.  For a few tokens (m <= 32) the call
 * runs a product on the warp-level tensor-core MMA instead
 * (mma.sync, codes as the fp16 values 1024 + code, exact per-group
 * corrections, accumulators in registers, 64-row sets over the SMs): the
 * same dots and the same bits of y; the workspace query covers its layout
 * (activations in the MMA's fragment order, the corrections, a counter).
 *   w uint32 [n, k/16] 16-byte aligned; aq int8 [m, k] 16-byte aligned;
 *   act_scale f32 [m]; y f32 [m, n]; k % 64 == 0 and k <= 131072.
 *   workspace 256-byte aligned, at least
 *   qmm_workspace_bytes(QMM_OP_BITNET_GEMM, m, n, k, 0) bytes (an fp16 copy
 *   of the activations).  Not reentrant on one workspace. */
qmm_status qmm_bitnet_gemm(const uint32_t *w, float weight_absmean, const int8_t *aq,
                           const float *act_scale, float *y, int64_t m, int64_t n, int64_t k,
                           void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* Workspace size in bytes for `op` (QMM_OP_*) at this shape; 0 when none is
 * needed; SIZE_MAX for an invalid op or shape.  For the GEMV ops with
 * split_k = 0 it covers both products the call may choose (the GEMV's
 * split-K partials, the few-token product's activation layout). */
size_t qmm_workspace_bytes(int op, int64_t m, int64_t n, int64_t k, int split_k);

/* The split-K factor qmm_gemv_q4_0_q8_0 uses for split_k = 0 at this shape. */
int qmm_gemv_auto_split(int64_t m, int64_t n, int64_t k);

/* Reads and clears the library's device error word after synchronizing
 * `stream`.  QMM_OK if no kernel reported an error since the last call;
 * QMM_ERR_TIMEOUT if a bounded wait inside a kernel gave up (the kernel then
 * stopped early and its outputs are unspecified); QMM_ERR_CUDA if the
 * synchronization itself failed.  This is the only entry point that blocks
 * the host. */
qmm_status qmm_check_device_error(void *stream);

/* A static, human-readable name for a status code. */
const char *qmm_status_string(qmm_status status);

/* Library version as 10000*major + 100*minor + patch. */
int qmm_version(void);

/* ---------------------------------------------------------------------- */
/* Test entry points.  They run the same kernels as the product entry points
 * compiled to also emit their intermediate integers, so tests can compare
 * them bit for bit with a reference.  Not for production use. */

/* Test and measurement entry: runs a tensor-pipe throughput loop on every SM
 * (one CTA of 512 threads per SM, each warp issuing independent warp-level
 * MMAs back to back) so the caller can time it and obtain the peak rate of
 * that instruction.  kind 0: mma.sync m16n8k32 s8 x s8 -> s32, the only int8
 * tensor-core instruction sm_103a accepts (the assembler rejects
 * tcgen05.mma kind::i8 for this target); kind 1: mma.sync m16n8k16 f16 x f16
 * -> f32.  *macs receives the multiply-accumulates of the launch.  The pages
 * have no counterpart; it only supplies the int8 peak that products are
 * reported against.
 *   out int32 device buffer of at least (SM count) * 512 * 4 bytes (written
 *   with values of no meaning); iters > 0.
 *   QMM_ERR_ARG for another kind or iters <= 0; QMM_ERR_WORKSPACE when out is
 *   too small. */
qmm_status qmm_debug_mma_probe(int kind, int iters, int *out, size_t out_bytes, int64_t *macs,
                               void *stream);

/* Per-block sums sumi int32 [m, n, k/32] = sum_j (nibble_j - 8) * q_j.
 * path 0: the decode GEMV kernel (m <= QMM_GEMV_MAX_M); path 1: the GEMM
 * call (the few-token product for m <= 64 and k % 256 == 0, else the tensor-
 * core GEMM kernel; needs the GEMM workspace); path 2: the GEMM on repacked
 * weights (wq then points at the repacked tiles, see qmm_repack_q4_0_gemm).  Same alignment rules as the
 * product entry points; sumi 4-byte aligned. */
qmm_status qmm_debug_block_sums_q4_0_q8_0(int path, const uint8_t *wq, const int8_t *aq,
                                          int32_t *sumi, int64_t m, int64_t n, int64_t k,
                                          void *workspace, size_t workspace_bytes,
                                          void *stream);

/* Per-block sums sumi int32 [m, n, k/32] = sum_j q_w * q_a of the Q8_0-weight
 * kernels: path 0 the decode GEMV, path 1 the GEMM call (the few-token
 * product for m <= 32 and k % 256 == 0, else the tcgen05 kernel; needs its
 * workspace).  Rules as for qmm_debug_block_sums_q4_0_q8_0. */
qmm_status qmm_debug_block_sums_q8_0_q8_0(int path, const int8_t *w8, const int8_t *aq,
                                          int32_t *sumi, int64_t m, int64_t n, int64_t k,
                                          void *workspace, size_t workspace_bytes,
                                          void *stream);

/* BitNet integer dots dot int32 [m, n] from the ternary GEMV kernel. */
qmm_status qmm_debug_bitnet_dot(const uint32_t *w, const int8_t *aq, const int32_t *act_sum,
                                int32_t *dot, int64_t m, int64_t n, int64_t k, void *stream);

/* Upper bound on the polling iterations of every bounded wait inside the
 * GEMM and the streaming GEMV kernels (default 1 << 17; 0 restores the
 * default).  Each poll
 * suspends the waiting warp for at most 20 microseconds (it resumes as soon
 * as the awaited phase completes).  Affects kernels launched after the
 * call. */
void qmm_debug_set_wait_limit(uint32_t iterations);

/* Test hook: while enabled, the load stages of the GEMM kernel, of the
 * few-token products (Q4_0, Q8_0 and BitNet) issue no copies, so their
 * pipeline waits can only run out their poll limit.  Tests use it
 * with a small limit to check that the kernel then records QMM_ERR_TIMEOUT
 * (read by qmm_check_device_error), releases its resources and returns, and
 * that the device stays usable.  Outputs of such a call are unspecified. */
void qmm_debug_withhold_gemm_loads(int enable);

/* The same hook for the shared-memory streaming decode GEMV (see
 * qmm_gemv_q4_0_q8_0): while enabled its producer arms no stage, so the
 * consumers' waits run out their limit. */
void qmm_debug_withhold_gemv_loads(int enable);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */
