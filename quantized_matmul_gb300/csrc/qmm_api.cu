// C ABI of libqmm.so (declared in include/qmm.h).
//
// Every entry point validates its arguments on the host and launches nothing
// when a check fails; the kernels behind it check nothing (the split of the
// Fucina course, chapter 06, section 6.3: validation happens once, above
// small unchecked kernels, and output buffers come from the caller).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>

#include "../../include/qmm.h"
#include "qmm_internal.h"

namespace {

using qmm::kQK;
static_assert(qmm::kGemvNoAllocScratchFloats == QMM_NOALLOC_SCRATCH_FLOATS,
              "the header and the library must agree on the built-in scratch size");
static_assert(qmm::kGroupMax == QMM_GROUP_MAX, "the header and the library must agree");

constexpr int kMaxDevices = 64;
std::atomic<int> g_dev_ok[kMaxDevices];  // 0 unknown, 1 supported, 2 not supported

qmm_status check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return QMM_ERR_UNSUPPORTED_DEVICE;
    int state = g_dev_ok[dev].load(std::memory_order_relaxed);
    if (state == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return QMM_ERR_CUDA;
        state = (major == 10 && minor == 3) ? 1 : 2;
        g_dev_ok[dev].store(state, std::memory_order_relaxed);
    }
    return state == 1 ? QMM_OK : QMM_ERR_UNSUPPORTED_DEVICE;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

qmm_status launch_status(cudaError_t e) { return e == cudaSuccess ? QMM_OK : QMM_ERR_CUDA; }

cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

// Grid dimension limits of the launchers: counts that end up in a 32-bit
// grid.x stay well below 2^31.
constexpr int64_t kMaxElems = int64_t(1) << 40;

qmm_status check_q4_common(const uint8_t *wq, const uint16_t *wd, const int8_t *aq,
                           const uint16_t *ad, const void *y, int64_t m, int64_t n, int64_t k) {
    if (!wq || !wd || !aq || !ad || !y) return QMM_ERR_NULL;
    if (m <= 0 || n <= 0 || k <= 0 || k % kQK != 0) return QMM_ERR_SHAPE;
    if (n >= (int64_t(1) << 31) || m >= (int64_t(1) << 31) || k >= (int64_t(1) << 31))
        return QMM_ERR_SHAPE;
    if (m * k > kMaxElems || n * k > kMaxElems || m * n > kMaxElems) return QMM_ERR_SHAPE;
    if (!aligned(wq, 16) || !aligned(aq, 16) || !aligned(wd, 2) || !aligned(ad, 2) ||
        !aligned(y, 4))
        return QMM_ERR_ALIGN;
    return QMM_OK;
}

qmm_status gemv_split(int split_k, int64_t m, int64_t n, int64_t k, int *out) {
    if (split_k < 0) return QMM_ERR_ARG;
    int s = split_k == 0 ? qmm::gemv_auto_split(m, n, k) : split_k;
    if (s > k / kQK || s > 65535) return QMM_ERR_ARG;
    *out = s;
    return QMM_OK;
}

// The decode GEMV entries with split_k = 0 (the library's choice) hand the
// call to the few-token product of gemm_small.cu where that is faster: from
// three tokens on (vocabulary shape, K=4096, N=128256: 70 against 117 us at
// m = 3, 88 against 323 us at m = 16; at m = 2 the GEMV kernel is faster, 57
// against 70), for k % 256 == 0, when the caller's workspace holds the
// product's activation layout (qmm_workspace_bytes reports that size for
// split_k = 0) and wd is 16-byte aligned (the product copies it with a
// tensor map).  The product's y is the serial definition, bit for bit,
// which is within the GEMV's tolerance.
constexpr int64_t kFewTokenMinM = 3;

bool few_token_shape(int64_t m, int64_t n, int64_t k, int split_k) {
    return split_k == 0 && m >= kFewTokenMinM && m <= QMM_GEMV_MAX_M &&
           qmm::gemm_small_m_supported(m, n, k);
}

bool few_token_route(int64_t m, int64_t n, int64_t k, int split_k, const void *wd,
                     const void *workspace, size_t workspace_bytes) {
    return few_token_shape(m, n, k, split_k) && aligned(wd, 16) && workspace &&
           aligned(workspace, 256) && workspace_bytes >= qmm::gemm_small_m_workspace_bytes(m, k);
}

// Workspace of qmm_bitnet_gemm: enough for either product it may run.
size_t bitnet_gemm_need(int64_t m, int64_t n, int64_t k) {
    const size_t t = qmm::bitnet_gemm_workspace_bytes(m, k);
    return qmm::bitnet_small_m_supported(m, n, k)
               ? std::max(t, qmm::bitnet_small_m_workspace_bytes(m, k))
               : t;
}

qmm_status check_linear(const uint8_t *wq, const uint16_t *wd, const float *x, int64_t ldx,
                        const int8_t *aq, const uint16_t *ad, const float *y, int64_t m,
                        int64_t n, int64_t k) {
    if (!x) return QMM_ERR_NULL;
    if (qmm_status st = check_q4_common(wq, wd, aq, ad, y, m, n, k)) return st;
    if (m > QMM_GEMV_MAX_M || ldx < k || m * ldx > kMaxElems) return QMM_ERR_SHAPE;
    if (!aligned(x, 4)) return QMM_ERR_ALIGN;
    return QMM_OK;
}

qmm_status gemm_shape_ok(int64_t m, int64_t n, int64_t k) {
    // The tensor maps use 32-bit dimensions and the tile grid uses 16-bit grid.y.
    if (k / 2 >= (int64_t(1) << 32) || (n + 127) / 128 > 65535) return QMM_ERR_SHAPE;
    return QMM_OK;
}

}  // namespace

extern "C" {

qmm_status qmm_quantize_act_q8_0(const float *x, int64_t m, int64_t k, int64_t ldx, int8_t *aq,
                                 uint16_t *ad, void *stream) {
    if (!x || !aq || !ad) return QMM_ERR_NULL;
    if (m <= 0 || k <= 0 || k % kQK != 0 || ldx < k) return QMM_ERR_SHAPE;
    if (m * k > kMaxElems || m * ldx > kMaxElems) return QMM_ERR_SHAPE;
    if (!aligned(x, 4) || !aligned(ad, 2)) return QMM_ERR_ALIGN;
    if (qmm_status st = check_device()) return st;
    return launch_status(qmm::launch_quantize_act_q8_0(x, m, k, ldx, aq, ad, as_stream(stream)));
}

qmm_status qmm_quantize_weight_q4_0(const float *w, int64_t n, int64_t k, uint8_t *wq,
                                    uint16_t *wd, void *stream) {
    if (!w || !wq || !wd) return QMM_ERR_NULL;
    if (n <= 0 || k <= 0 || k % kQK != 0 || n * k > kMaxElems) return QMM_ERR_SHAPE;
    if (!aligned(w, 4) || !aligned(wd, 2)) return QMM_ERR_ALIGN;
    if (qmm_status st = check_device()) return st;
    return launch_status(qmm::launch_quantize_weight_q4_0(w, n, k, wq, wd, as_stream(stream)));
}

qmm_status qmm_gemv_q4_0_q8_0(const uint8_t *wq, const uint16_t *wd, const int8_t *aq,
                              const uint16_t *ad, float *y, int64_t m, int64_t n, int64_t k,
                              int split_k, void *workspace, size_t workspace_bytes, void *stream) {
    if (qmm_status st = check_q4_common(wq, wd, aq, ad, y, m, n, k)) return st;
    if (m > QMM_GEMV_MAX_M) return QMM_ERR_SHAPE;
    if (few_token_route(m, n, k, split_k, wd, workspace, workspace_bytes)) {
        if (qmm_status st = check_device()) return st;
        return launch_status(qmm::launch_gemm_small_m(wq, wd, aq, ad, y, nullptr, m, n, k, workspace,
                                                      as_stream(stream)));
    }
    int split = 1;
    if (qmm_status st = gemv_split(split_k, m, n, k, &split)) return st;
    const size_t need = qmm::gemv_workspace_bytes(m, n, k, split);
    if (need > 0 && (!workspace || workspace_bytes < need)) return QMM_ERR_WORKSPACE;
    if (need > 0 && !aligned(workspace, 16)) return QMM_ERR_ALIGN;
    if (qmm_status st = check_device()) return st;
    return launch_status(qmm::launch_gemv_q4_0_q8_0(wq, wd, aq, ad, y, nullptr, m, n, k, split,
                                                    static_cast<float *>(workspace),
                                                    as_stream(stream)));
}

qmm_status qmm_gemv_q4_0_q8_0_noalloc(const uint8_t *wq, const uint16_t *wd, const int8_t *aq,
                                      const uint16_t *ad, float *y, int64_t m, int64_t n,
                                      int64_t k, int split_k, void *stream) {
    if (qmm_status st = check_q4_common(wq, wd, aq, ad, y, m, n, k)) return st;
    if (m > QMM_GEMV_MAX_M) return QMM_ERR_SHAPE;
    int split = 1;
    if (qmm_status st = gemv_split(split_k, m, n, k, &split)) return st;
    // The automatic split only exceeds 1 when the grid is short of two CTAs
    // per SM, i.e. for n below ~1200 rows, and it never passes 32: its
    // partials stay below 20 Ki floats for every m <= QMM_GEMV_MAX_M (a CPU
    // test sweeps the bound).  Only an explicit split_k can overflow the
    // array, and the same check rejects both.
    if (split > 1 && (int64_t)split * m * n > qmm::kGemvNoAllocScratchFloats)
        return QMM_ERR_WORKSPACE;
    if (qmm_status st = check_device()) return st;
    return launch_status(qmm::launch_gemv_q4_0_q8_0_noalloc(wq, wd, aq, ad, y, m, n, k, split,
                                                            as_stream(stream)));
}

qmm_status qmm_linear_q4_0(const uint8_t *wq, const uint16_t *wd, const float *x, int64_t ldx,
                           int8_t *aq, uint16_t *ad, float *y, int64_t m, int64_t n, int64_t k,
                           int flags, void *stream) {
    if (qmm_status st = check_linear(wq, wd, x, ldx, aq, ad, y, m, n, k)) return st;
    if (flags & ~QMM_LINEAR_PDL) return QMM_ERR_ARG;
    if (qmm_status st = check_device()) return st;
    const bool pdl = (flags & QMM_LINEAR_PDL) != 0;
    const cudaStream_t s = as_stream(stream);
    cudaError_t e = qmm::launch_quantize_act_q8_0(x, m, k, ldx, aq, ad, s, pdl);
    if (e != cudaSuccess) return QMM_ERR_CUDA;
    return launch_status(qmm::launch_gemv_q4_0_q8_0(wq, wd, aq, ad, y, nullptr, m, n, k, 1,
                                                    nullptr, s, pdl));
}

namespace {

// Checks a grouped call's table and fills its launch table; launches nothing.
qmm_status build_group(const qmm_linear_problem *problems, int count, int64_t m,
                       qmm::LinearGroup &tab) {
    if (!problems) return QMM_ERR_NULL;
    if (count < 1 || count > QMM_GROUP_MAX) return QMM_ERR_ARG;
    tab = {};
    int64_t ctas = 0, blocks = 0;
    for (int p = 0; p < count; ++p) {
        const qmm_linear_problem &P = problems[p];
        if (qmm_status st = check_linear(P.wq, P.wd, P.x, P.ldx, P.aq, P.ad, P.y, m, P.n, P.k))
            return st;
        ctas += (P.n + 1) / 2;  // at least 2 rows per CTA of the grouped GEMV
        blocks += m * (P.k / kQK);
        tab.p[p] = {P.wq, P.wd, P.x, P.ldx, P.aq, P.ad, P.y, P.n, P.k};
    }
    if (ctas >= (int64_t(1) << 31) || blocks >= (int64_t(1) << 33)) return QMM_ERR_SHAPE;
    tab.count = count;
    tab.m = (int)m;
    return QMM_OK;
}

// The device address of page-locked host memory, or nullptr when the device
// cannot address it (the runtime's pointer attributes decide; nothing is
// dereferenced here).
const void *host_device_address(const void *host) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
        cudaGetLastError();  // an unknown pointer leaves a (non-sticky) error behind
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// [lo, hi) of bytes inside [base, base + bytes)?
bool within(const void *lo, size_t len, const void *base, size_t bytes) {
    const uintptr_t l = reinterpret_cast<uintptr_t>(lo), b = reinterpret_cast<uintptr_t>(base);
    return l >= b && len <= bytes && l - b <= bytes - len;
}

}  // namespace

qmm_status qmm_linear_q4_0_grouped(const qmm_linear_problem *problems, int count, int64_t m,
                                   int flags, void *stream) {
    if (flags & ~QMM_LINEAR_PDL) return QMM_ERR_ARG;
    qmm::LinearGroup tab;
    if (qmm_status st = build_group(problems, count, m, tab)) return st;
    if (qmm_status st = check_device()) return st;
    return launch_status(
        qmm::launch_linear_grouped(tab, (flags & QMM_LINEAR_PDL) != 0, as_stream(stream)));
}

qmm_status qmm_linear_q4_0_grouped_host(const qmm_linear_problem *problems, int count, int64_t m,
                                        int flags, const void *x_host, void *x_dev, size_t x_bytes,
                                        const void *y_dev, void *y_host, size_t y_bytes,
                                        void *stream) {
    if (flags & ~(QMM_LINEAR_PDL | QMM_LINEAR_HOST_DIRECT)) return QMM_ERR_ARG;
    qmm::LinearGroup tab;
    if (qmm_status st = build_group(problems, count, m, tab)) return st;
    if (x_bytes && (!x_host || !x_dev)) return QMM_ERR_NULL;
    if (y_bytes && (!y_dev || !y_host)) return QMM_ERR_NULL;
    const bool pdl = (flags & QMM_LINEAR_PDL) != 0;
    if (flags & QMM_LINEAR_HOST_DIRECT) {
        // every problem's x and y inside the device buffers the host buffers mirror
        for (int p = 0; p < count; ++p) {
            const qmm_linear_problem &P = problems[p];
            const size_t xlen = (size_t)(((m - 1) * P.ldx + P.k) * 4), ylen = (size_t)(m * P.n * 4);
            if (!within(P.x, xlen, x_dev, x_bytes) || !within(P.y, ylen, y_dev, y_bytes))
                return QMM_ERR_ARG;
        }
    }
    if (qmm_status st = check_device()) return st;
    cudaStream_t s = as_stream(stream);
    if (flags & QMM_LINEAR_HOST_DIRECT) {
        const auto *xh = static_cast<const uint8_t *>(host_device_address(x_host));
        auto *yh = static_cast<uint8_t *>(const_cast<void *>(host_device_address(y_host)));
        if (xh && yh) {
            // the kernels read x from, and write y to, host memory themselves
            qmm::LinearGroup direct = tab;
            bool ok = true;
            for (int p = 0; p < count && ok; ++p) {
                auto &D = direct.p[p];
                D.x = reinterpret_cast<const float *>(
                    xh + (reinterpret_cast<const uint8_t *>(problems[p].x) -
                          static_cast<const uint8_t *>(x_dev)));
                D.y = reinterpret_cast<float *>(
                    yh + (reinterpret_cast<const uint8_t *>(problems[p].y) -
                          static_cast<const uint8_t *>(y_dev)));
                ok = aligned(D.x, 4) && aligned(D.y, 4);
            }
            if (ok) return launch_status(qmm::launch_linear_grouped(direct, pdl, s));
        }
        // not addressable from the device: copy instead
    }
    if (x_bytes && cudaMemcpyAsync(x_dev, x_host, x_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return QMM_ERR_CUDA;
    if (qmm_status st = launch_status(qmm::launch_linear_grouped(tab, pdl, s))) return st;
    if (y_bytes && cudaMemcpyAsync(y_host, y_dev, y_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return QMM_ERR_CUDA;
    return QMM_OK;
}

int qmm_host_addressable(const void *host) { return host && host_device_address(host) ? 1 : 0; }

qmm_status qmm_gemm_q4_0_q8_0(const uint8_t *wq, const uint16_t *wd, const int8_t *aq,
                              const uint16_t *ad, float *y, int64_t m, int64_t n, int64_t k,
                              void *workspace, size_t workspace_bytes, void *stream) {
    if (qmm_status st = check_q4_common(wq, wd, aq, ad, y, m, n, k)) return st;
    if (qmm_status st = gemm_shape_ok(m, n, k)) return st;
    const size_t need = qmm::gemm_workspace_bytes(m, n, k);
    if (!workspace || workspace_bytes < need) return QMM_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return QMM_ERR_ALIGN;
    if (qmm_status st = check_device()) return st;
    return launch_status(qmm::launch_gemm_q4_0_q8_0(wq, wd, aq, ad, y, nullptr, m, n, k, workspace,
                                                    as_stream(stream)));
}

size_t qmm_repack_q4_0_gemm_bytes(int64_t n, int64_t k) {
    if (n <= 0 || k <= 0 || k % kQK != 0 || n * k > kMaxElems) return SIZE_MAX;
    return qmm::repack_q4_0_gemm_bytes(n, k);
}

qmm_status qmm_repack_q4_0_gemm(const uint8_t *wq, int64_t n, int64_t k, uint8_t *wr,
                                size_t wr_bytes, void *stream) {
    if (!wq || !wr) return QMM_ERR_NULL;
    if (n <= 0 || k <= 0 || k % kQK != 0 || n * k > kMaxElems) return QMM_ERR_SHAPE;
    if (!aligned(wq, 16) || !aligned(wr, 16)) return QMM_ERR_ALIGN;
    if (wr_bytes < qmm::repack_q4_0_gemm_bytes(n, k)) return QMM_ERR_WORKSPACE;
    if (qmm_status st = check_device()) return st;
    return launch_status(qmm::launch_repack_q4_0_gemm(wq, n, k, wr, as_stream(stream)));
}

qmm_status qmm_gemm_q4_0_q8_0_repacked(const uint8_t *wr, size_t wr_bytes, const uint16_t *wd,
                                       const int8_t *aq, const uint16_t *ad, float *y, int64_t m,
                                       int64_t n, int64_t k, void *workspace,
                                       size_t workspace_bytes, void *stream) {
    if (qmm_status st = check_q4_common(wr, wd, aq, ad, y, m, n, k)) return st;
    if (qmm_status st = gemm_shape_ok(m, n, k)) return st;
    if (wr_bytes < qmm::repack_q4_0_gemm_bytes(n, k)) return QMM_ERR_WORKSPACE;
    const size_t need = qmm::gemm_workspace_bytes(m, n, k);
    if (!workspace || workspace_bytes < need) return QMM_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return QMM_ERR_ALIGN;
    if (qmm_status st = check_device()) return st;
    return launch_status(qmm::launch_gemm_q4_0_q8_0_repacked(wr, wd, aq, ad, y, nullptr, m, n, k,
                                                             workspace, as_stream(stream)));
}

qmm_status qmm_gemv_q8_0_q8_0(const int8_t *w8, const uint16_t *wd, const int8_t *aq,
                              const uint16_t *ad, float *y, int64_t m, int64_t n, int64_t k,
                              int split_k, void *workspace, size_t workspace_bytes, void *stream) {
    const auto *wb = reinterpret_cast<const uint8_t *>(w8);
    if (qmm_status st = check_q4_common(wb, wd, aq, ad, y, m, n, k)) return st;
    if (m > QMM_GEMV_MAX_M) return QMM_ERR_SHAPE;
    if (few_token_route(m, n, k, split_k, wd, workspace, workspace_bytes)) {
        if (qmm_status st = check_device()) return st;
        return launch_status(qmm::launch_gemm_small_m_q8(w8, wd, aq, ad, y, nullptr, m, n, k,
                                                         workspace, as_stream(stream)));
    }
    int split = 1;
    if (qmm_status st = gemv_split(split_k, m, n, k, &split)) return st;
    const size_t need = qmm::gemv_workspace_bytes(m, n, k, split);
    if (need > 0 && (!workspace || workspace_bytes < need)) return QMM_ERR_WORKSPACE;
    if (need > 0 && !aligned(workspace, 16)) return QMM_ERR_ALIGN;
    if (qmm_status st = check_device()) return st;
    return launch_status(qmm::launch_gemv_q8_0_q8_0(w8, wd, aq, ad, y, nullptr, m, n, k, split,
                                                    static_cast<float *>(workspace),
                                                    as_stream(stream)));
}

qmm_status qmm_gemm_q8_0_q8_0(const int8_t *w8, const uint16_t *wd, const int8_t *aq,
                              const uint16_t *ad, float *y, int64_t m, int64_t n, int64_t k,
                              void *workspace, size_t workspace_bytes, void *stream) {
    const auto *wb = reinterpret_cast<const uint8_t *>(w8);
    if (qmm_status st = check_q4_common(wb, wd, aq, ad, y, m, n, k)) return st;
    if (qmm_status st = gemm_shape_ok(m, n, 2 * k)) return st;  // Q8_0 rows are k bytes
    const size_t need = qmm::gemm_workspace_bytes(m, n, k);
    if (!workspace || workspace_bytes < need) return QMM_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return QMM_ERR_ALIGN;
    if (qmm_status st = check_device()) return st;
    return launch_status(qmm::launch_gemm_q8_0_q8_0(w8, wd, aq, ad, y, nullptr, m, n, k, workspace,
                                                    as_stream(stream)));
}

qmm_status qmm_quantize_act_bitnet(const float *x, int64_t m, int64_t k, int8_t *aq,
                                   float *act_scale, int32_t *act_sum, void *stream) {
    if (!x || !aq || !act_scale || !act_sum) return QMM_ERR_NULL;
    if (m <= 0 || k <= 0 || k % 16 != 0 || m >= (int64_t(1) << 31) || m * k > kMaxElems ||
        k > (int64_t(1) << 21))
        return QMM_ERR_SHAPE;
    if (!aligned(x, 4) || !aligned(act_scale, 4) || !aligned(act_sum, 4)) return QMM_ERR_ALIGN;
    if (qmm_status st = check_device()) return st;
    return launch_status(
        qmm::launch_quantize_act_bitnet(x, m, k, k, aq, act_scale, act_sum, as_stream(stream)));
}

qmm_status qmm_pack_ternary(const int8_t *t, int64_t n, int64_t k, uint32_t *w, void *stream) {
    if (!t || !w) return QMM_ERR_NULL;
    if (n <= 0 || k <= 0 || k % 16 != 0 || n * k > kMaxElems) return QMM_ERR_SHAPE;
    if (!aligned(w, 4)) return QMM_ERR_ALIGN;
    if (qmm_status st = check_device()) return st;
    return launch_status(qmm::launch_pack_ternary(t, n, k, w, as_stream(stream)));
}

static qmm_status check_bitnet(const uint32_t *w, const int8_t *aq, const float *act_scale,
                               const int32_t *act_sum, const void *out, int64_t m, int64_t n,
                               int64_t k) {
    if (!w || !aq || !act_scale || !act_sum || !out) return QMM_ERR_NULL;
    if (m <= 0 || m > QMM_GEMV_MAX_M || n <= 0 || k <= 0 || k % 16 != 0 ||
        k > (int64_t(1) << 21) || n >= (int64_t(1) << 31) || n * k > kMaxElems)
        return QMM_ERR_SHAPE;
    if (!aligned(w, 16) || !aligned(aq, 16) || !aligned(act_scale, 4) || !aligned(act_sum, 4) ||
        !aligned(out, 4))
        return QMM_ERR_ALIGN;
    return QMM_OK;
}

qmm_status qmm_bitnet_gemv(const uint32_t *w, float weight_absmean, const int8_t *aq,
                           const float *act_scale, const int32_t *act_sum, float *y, int64_t m,
                           int64_t n, int64_t k, void *stream) {
    if (qmm_status st = check_bitnet(w, aq, act_scale, act_sum, y, m, n, k)) return st;
    if (qmm_status st = check_device()) return st;
    return launch_status(qmm::launch_bitnet_gemv(w, weight_absmean, aq, act_scale, act_sum, y,
                                                 nullptr, m, n, k, as_stream(stream)));
}

qmm_status qmm_linear_bitnet(const uint32_t *w, float weight_absmean, const float *x, int64_t ldx,
                             int8_t *aq, float *act_scale, int32_t *act_sum, float *y, int64_t m,
                             int64_t n, int64_t k, int flags, void *stream) {
    if (!x) return QMM_ERR_NULL;
    if (qmm_status st = check_bitnet(w, aq, act_scale, act_sum, y, m, n, k)) return st;
    if (ldx < k || m * ldx > kMaxElems) return QMM_ERR_SHAPE;
    if (!aligned(x, 4)) return QMM_ERR_ALIGN;
    if (flags & ~QMM_LINEAR_PDL) return QMM_ERR_ARG;
    if (qmm_status st = check_device()) return st;
    const bool pdl = (flags & QMM_LINEAR_PDL) != 0;
    const cudaStream_t s = as_stream(stream);
    if (qmm::bitnet_linear_fused_supported(m, k, ldx, x, aq))
        return launch_status(qmm::launch_bitnet_linear_fused(w, weight_absmean, x, aq, act_scale,
                                                             act_sum, y, n, k, s, pdl));
    cudaError_t e = qmm::launch_quantize_act_bitnet(x, m, k, ldx, aq, act_scale, act_sum, s, pdl);
    if (e != cudaSuccess) return QMM_ERR_CUDA;
    return launch_status(qmm::launch_bitnet_gemv(w, weight_absmean, aq, act_scale, act_sum, y, nullptr,
                                                 m, n, k, s, pdl));
}

qmm_status qmm_bitnet_gemm(const uint32_t *w, float weight_absmean, const int8_t *aq,
                           const float *act_scale, float *y, int64_t m, int64_t n, int64_t k,
                           void *workspace, size_t workspace_bytes, void *stream) {
    if (!w || !aq || !act_scale || !y) return QMM_ERR_NULL;
    if (m <= 0 || n <= 0 || k <= 0 || k % 64 != 0 || k > (int64_t(1) << 17)) return QMM_ERR_SHAPE;
    if (m >= (int64_t(1) << 31) || n >= (int64_t(1) << 31) || m * k > kMaxElems ||
        n * k > kMaxElems || m * n > kMaxElems)
        return QMM_ERR_SHAPE;
    if (!aligned(w, 16) || !aligned(aq, 16) || !aligned(act_scale, 4) || !aligned(y, 4))
        return QMM_ERR_ALIGN;
    const size_t need = bitnet_gemm_need(m, n, k);
    if (!workspace || workspace_bytes < need) return QMM_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return QMM_ERR_ALIGN;
    if (qmm_status st = check_device()) return st;
    // a few tokens: the warp-level MMA product (the tcgen05 tiles of 128 rows
    // would leave most SMs idle); the same bits
    if (qmm::bitnet_small_m_supported(m, n, k))
        return launch_status(qmm::launch_bitnet_small_m(w, weight_absmean, aq, act_scale, y, m, n,
                                                        k, workspace, as_stream(stream)));
    return launch_status(qmm::launch_bitnet_gemm(w, weight_absmean, aq, act_scale, y, m, n, k,
                                                 workspace, as_stream(stream)));
}

size_t qmm_workspace_bytes(int op, int64_t m, int64_t n, int64_t k, int split_k) {
    if (op == QMM_OP_BITNET_GEMM)
        return (m <= 0 || n <= 0 || k <= 0 || k % 64 != 0) ? SIZE_MAX : bitnet_gemm_need(m, n, k);
    if (m <= 0 || n <= 0 || k <= 0 || k % kQK != 0) return SIZE_MAX;
    switch (op) {
        case QMM_OP_GEMV_Q4_0_Q8_0:
        case QMM_OP_GEMV_Q8_0_Q8_0: {
            if (m > QMM_GEMV_MAX_M) return SIZE_MAX;
            int split = 1;
            if (gemv_split(split_k, m, n, k, &split) != QMM_OK) return SIZE_MAX;
            const size_t need = qmm::gemv_workspace_bytes(m, n, k, split);
            // enough for either product the call may run
            return few_token_shape(m, n, k, split_k)
                       ? std::max(need, qmm::gemm_small_m_workspace_bytes(m, k))
                       : need;
        }
        case QMM_OP_GEMM_Q4_0_Q8_0:
        case QMM_OP_GEMM_Q8_0_Q8_0:
            return qmm::gemm_workspace_bytes(m, n, k);
        default:
            return SIZE_MAX;
    }
}

int qmm_gemv_auto_split(int64_t m, int64_t n, int64_t k) {
    if (m <= 0 || n <= 0 || k <= 0 || k % kQK != 0) return 1;
    return qmm::gemv_auto_split(m, n, k);
}

qmm_status qmm_check_device_error(void *stream) {
    unsigned int word = 0, word2 = 0, word3 = 0, word4 = 0, word5 = 0;
    if (qmm::gemm_read_and_clear_error(&word, as_stream(stream)) != cudaSuccess) return QMM_ERR_CUDA;
    if (qmm::gemm_small_read_and_clear_error(&word4, as_stream(stream)) != cudaSuccess)
        return QMM_ERR_CUDA;
    if (qmm::stream_read_and_clear_error(&word2, as_stream(stream)) != cudaSuccess)
        return QMM_ERR_CUDA;
    if (qmm::bitnet_gemm_read_and_clear_error(&word3, as_stream(stream)) != cudaSuccess)
        return QMM_ERR_CUDA;
    if (qmm::bitnet_small_read_and_clear_error(&word5, as_stream(stream)) != cudaSuccess)
        return QMM_ERR_CUDA;
    return (word | word2 | word3 | word4 | word5) ? QMM_ERR_TIMEOUT : QMM_OK;
}

const char *qmm_status_string(qmm_status status) {
    switch (status) {
        case QMM_OK: return "ok";
        case QMM_ERR_NULL: return "null pointer";
        case QMM_ERR_SHAPE: return "invalid shape";
        case QMM_ERR_ALIGN: return "misaligned pointer";
        case QMM_ERR_WORKSPACE: return "workspace missing or too small";
        case QMM_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
        case QMM_ERR_CUDA: return "CUDA error";
        case QMM_ERR_TIMEOUT: return "device-side wait timed out";
        case QMM_ERR_ARG: return "invalid argument";
    }
    return "unknown status";
}

int qmm_version(void) { return 100; }

qmm_status qmm_debug_block_sums_q4_0_q8_0(int path, const uint8_t *wq, const int8_t *aq,
                                          int32_t *sumi, int64_t m, int64_t n, int64_t k,
                                          void *workspace, size_t workspace_bytes, void *stream) {
    // The scale planes are not read by the block-sum variants; pass aligned
    // dummies through the shared shape/alignment check.
    static const uint16_t dummy[8] = {0};
    if (!sumi) return QMM_ERR_NULL;
    if (qmm_status st = check_q4_common(wq, dummy, aq, dummy, sumi, m, n, k)) return st;
    if (path == 0) {
        if (m > QMM_GEMV_MAX_M) return QMM_ERR_SHAPE;
        if (qmm_status st = check_device()) return st;
        return launch_status(qmm::launch_gemv_q4_0_q8_0(wq, nullptr, aq, nullptr, nullptr, sumi, m,
                                                        n, k, 1, nullptr, as_stream(stream)));
    }
    if (path == 1) {
        if (qmm_status st = gemm_shape_ok(m, n, k)) return st;
        const size_t need = qmm::gemm_workspace_bytes(m, n, k);
        if (!workspace || workspace_bytes < need) return QMM_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return QMM_ERR_ALIGN;
        if (qmm_status st = check_device()) return st;
        // The block-sum variant reads no scale planes (passed as NULL).
        return launch_status(qmm::launch_gemm_q4_0_q8_0(wq, nullptr, aq, nullptr, nullptr, sumi, m,
                                                        n, k, workspace, as_stream(stream)));
    }
    if (path == 2) {  // wq: the repacked tiles
        if (qmm_status st = gemm_shape_ok(m, n, k)) return st;
        const size_t need = qmm::gemm_workspace_bytes(m, n, k);
        if (!workspace || workspace_bytes < need) return QMM_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return QMM_ERR_ALIGN;
        if (qmm_status st = check_device()) return st;
        return launch_status(qmm::launch_gemm_q4_0_q8_0_repacked(wq, nullptr, aq, nullptr, nullptr,
                                                                 sumi, m, n, k, workspace,
                                                                 as_stream(stream)));
    }
    return QMM_ERR_ARG;
}

qmm_status qmm_debug_block_sums_q8_0_q8_0(int path, const int8_t *w8, const int8_t *aq,
                                          int32_t *sumi, int64_t m, int64_t n, int64_t k,
                                          void *workspace, size_t workspace_bytes, void *stream) {
    static const uint16_t dummy[8] = {0};
    if (!sumi) return QMM_ERR_NULL;
    const auto *wb = reinterpret_cast<const uint8_t *>(w8);
    if (qmm_status st = check_q4_common(wb, dummy, aq, dummy, sumi, m, n, k)) return st;
    if (path == 0) {
        if (m > QMM_GEMV_MAX_M) return QMM_ERR_SHAPE;
        if (qmm_status st = check_device()) return st;
        return launch_status(qmm::launch_gemv_q8_0_q8_0(w8, nullptr, aq, nullptr, nullptr, sumi, m,
                                                        n, k, 1, nullptr, as_stream(stream)));
    }
    if (path == 1) {
        if (qmm_status st = gemm_shape_ok(m, n, 2 * k)) return st;  // Q8_0 rows are k bytes
        const size_t need = qmm::gemm_workspace_bytes(m, n, k);
        if (!workspace || workspace_bytes < need) return QMM_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return QMM_ERR_ALIGN;
        if (qmm_status st = check_device()) return st;
        return launch_status(qmm::launch_gemm_q8_0_q8_0(w8, nullptr, aq, nullptr, nullptr, sumi, m,
                                                        n, k, workspace, as_stream(stream)));
    }
    return QMM_ERR_ARG;
}

qmm_status qmm_debug_bitnet_dot(const uint32_t *w, const int8_t *aq, const int32_t *act_sum,
                                int32_t *dot, int64_t m, int64_t n, int64_t k, void *stream) {
    static const float dummy_scale[4] = {0};
    if (qmm_status st = check_bitnet(w, aq, dummy_scale, act_sum, dot, m, n, k)) return st;
    if (qmm_status st = check_device()) return st;
    return launch_status(qmm::launch_bitnet_gemv(w, 0.0f, aq, nullptr, act_sum, nullptr, dot, m, n,
                                                 k, as_stream(stream)));
}

qmm_status qmm_debug_mma_probe(int kind, int iters, int *out, size_t out_bytes, int64_t *macs,
                               void *stream) {
    if (!out || !macs) return QMM_ERR_NULL;
    if ((kind != 0 && kind != 1) || iters <= 0) return QMM_ERR_ARG;
    if (!aligned(out, 4)) return QMM_ERR_ALIGN;
    if (qmm_status st = check_device()) return st;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return QMM_ERR_CUDA;
    if (out_bytes < (size_t)sms * 512 * sizeof(int)) return QMM_ERR_WORKSPACE;
    *macs = qmm::mma_probe_macs_per_iter(kind, sms) * iters;
    return launch_status(qmm::launch_mma_probe(kind, iters, sms, out, as_stream(stream)));
}

void qmm_debug_set_wait_limit(uint32_t iterations) {
    qmm::gemm_set_wait_limit(iterations);
    qmm::gemm_small_set_wait_limit(iterations);
    qmm::stream_set_wait_limit(iterations);
    qmm::bitnet_gemm_set_wait_limit(iterations);
    qmm::bitnet_small_set_wait_limit(iterations);
}

void qmm_debug_withhold_gemm_loads(int enable) {
    qmm::gemm_set_withhold_loads(enable);
    qmm::bitnet_small_set_withhold_loads(enable);
}

void qmm_debug_withhold_gemv_loads(int enable) { qmm::stream_set_withhold_loads(enable); }

}  // extern "C"
