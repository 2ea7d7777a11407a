"""The C ABI without a GPU: the library builds and loads, it exports every
symbol include/qmm.h declares, and argument checks run on the host before
anything touches the device (so every call below returns without a launch)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qmm.h")

QMM_OK, QMM_ERR_NULL, QMM_ERR_SHAPE, QMM_ERR_ALIGN, QMM_ERR_WORKSPACE = 0, 1, 2, 3, 4
QMM_ERR_ARG = 8


@pytest.fixture(scope="module")
def lib():
    from quantized_matmul_gb300 import build
    build.build()
    import quantized_matmul_gb300 as q
    return q.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qmm_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ["qmm_quantize_act_q8_0", "qmm_gemv_q4_0_q8_0", "qmm_gemm_q4_0_q8_0",
                     "qmm_bitnet_gemv", "qmm_quantize_act_bitnet", "qmm_workspace_bytes",
                     "qmm_linear_q4_0", "qmm_linear_q4_0_grouped",
                     "qmm_check_device_error", "qmm_status_string"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_exports_are_unmangled_c_symbols():
    from quantized_matmul_gb300 import build
    build.build()
    out = os.popen(f"nm -D --defined-only {build.LIB}").read()
    exported = set(re.findall(r"\bT (qmm_[a-z0-9_]+)\b", out))
    assert set(declared_functions()) <= exported


def test_status_strings_and_version(lib):
    assert lib.qmm_status_string(0) == b"ok"
    assert lib.qmm_status_string(7) == b"device-side wait timed out"
    assert lib.qmm_status_string(99) == b"unknown status"
    assert lib.qmm_version() >= 100


def test_workspace_queries(lib):
    # no split: no workspace
    assert lib.qmm_workspace_bytes(1, 1, 4096, 4096, 1) == 0
    # explicit split of 4 at m=2, n=100: 4 * 2 * 100 floats
    assert lib.qmm_workspace_bytes(1, 2, 100, 4096, 4) == 4 * 2 * 100 * 4
    # GEMM: fp16 activations + one 16-byte scale row per (block, token),
    # tokens rounded up to 4, each part 256-byte rounded
    m, k = 512, 4096
    a16 = m * k * 2
    rows = (k // 32) * m * 16
    assert lib.qmm_workspace_bytes(2, m, 14336, k, 0) == a16 + rows
    m = 3
    a16 = (m * k * 2 + 255) // 256 * 256
    rows = ((k // 32) * 4 * 16 + 255) // 256 * 256
    # m <= 32 with k a multiple of 256 may run the few-token product: fp16
    # activation fragments (1 KB per block and 16-token tile) + a 128-byte
    # record of f32 block corrections and scales per block and tile + 256
    # bytes for its row-set counter, each part 256-byte rounded; the query
    # covers the larger layout
    frags = (k // 32) * 1024
    pairs = (k // 32) * 128
    assert lib.qmm_workspace_bytes(2, m, 14336, k, 0) == max(a16 + rows, frags + pairs + 256)
    assert lib.qmm_workspace_bytes(2, 32, 14336, k, 0) == max(32 * k * 2 + (k // 32) * 32 * 16,
                                                               2 * (frags + pairs) + 256)
    assert lib.qmm_workspace_bytes(5, 16, 14336, k, 0) == max(16 * k * 2 + (k // 32) * 16 * 16,
                                                              frags + pairs + 256)
    # the decode GEMV with split_k = 0 from three tokens on may run the
    # few-token product: the query covers its layout (and stays 0 for an
    # explicit unsplit call, which always runs the GEMV kernels)
    for op in (1, 4):
        assert lib.qmm_workspace_bytes(op, 3, 14336, k, 0) == frags + pairs + 256
        assert lib.qmm_workspace_bytes(op, 16, 14336, k, 0) == frags + pairs + 256
        assert lib.qmm_workspace_bytes(op, 3, 14336, k, 1) == 0
        assert lib.qmm_workspace_bytes(op, 2, 14336, k, 0) == 0
    # Q4_0 weights take the few-token product up to 64 tokens: the query
    # covers its layout there too (three and four 16-token tiles)
    for mm in (33, 48, 64):
        mt = (mm + 15) // 16
        small = (k // 32) * mt * 1024 + (k // 32) * mt * 128 + 256
        assert lib.qmm_workspace_bytes(2, mm, 14336, k, 0) >= small
    k = 4064  # not a multiple of 256: the tcgen05 product only
    assert lib.qmm_workspace_bytes(2, m, 14336, k, 0) == (
        (m * k * 2 + 255) // 256 * 256 + ((k // 32) * 4 * 16 + 255) // 256 * 256)
    bad = ctypes.c_size_t(-1).value
    assert lib.qmm_workspace_bytes(9, 1, 1, 32, 0) == bad        # unknown op
    assert lib.qmm_workspace_bytes(1, 1, 1, 33, 0) == bad        # k not a block multiple
    assert lib.qmm_workspace_bytes(1, 17, 1, 32, 0) == bad       # GEMV m > 16
    assert lib.qmm_workspace_bytes(1, 1, 1, 64, 3) == bad        # more slices than blocks


def test_q8_0_weight_entry_points(lib):
    A16 = _p(0x10000)  # never dereferenced: every call below fails its host checks
    A2 = _p(0x10002)
    # workspace queries: the Q4_0 formulas
    assert lib.qmm_workspace_bytes(4, 2, 100, 4096, 4) == lib.qmm_workspace_bytes(1, 2, 100, 4096, 4)
    assert lib.qmm_workspace_bytes(5, 512, 14336, 4096, 0) == lib.qmm_workspace_bytes(2, 512, 14336, 4096, 0)
    assert lib.qmm_workspace_bytes(4, 17, 1, 32, 0) == ctypes.c_size_t(-1).value
    # argument errors
    assert lib.qmm_gemv_q8_0_q8_0(None, A16, A16, A16, A16, 1, 1, 32, 1, None, 0, None) == QMM_ERR_NULL
    assert lib.qmm_gemv_q8_0_q8_0(A16, A16, A16, A16, A16, 17, 1, 32, 1, None, 0, None) == QMM_ERR_SHAPE
    assert lib.qmm_gemv_q8_0_q8_0(A16, A16, A16, A16, A16, 1, 1, 48, 1, None, 0, None) == QMM_ERR_SHAPE
    assert lib.qmm_gemv_q8_0_q8_0(A2, A16, A16, A16, A16, 1, 1, 32, 1, None, 0, None) == QMM_ERR_ALIGN
    assert lib.qmm_gemv_q8_0_q8_0(A16, A16, A16, A16, A16, 1, 4, 64, 2, None, 0, None) == QMM_ERR_WORKSPACE
    assert lib.qmm_gemv_q8_0_q8_0(A16, A16, A16, A16, A16, 1, 4, 64, 3, A16, 1 << 20, None) == QMM_ERR_ARG
    assert lib.qmm_gemm_q8_0_q8_0(A16, A16, A16, None, A16, 1, 1, 32, A16, 1 << 20, None) == QMM_ERR_NULL
    assert lib.qmm_gemm_q8_0_q8_0(A16, A16, A16, A16, A16, 1, 1, 40, A16, 1 << 20, None) == QMM_ERR_SHAPE
    assert lib.qmm_gemm_q8_0_q8_0(A16, A16, A2, A16, A16, 1, 1, 32, A16, 1 << 20, None) == QMM_ERR_ALIGN
    assert lib.qmm_gemm_q8_0_q8_0(A16, A16, A16, A16, A16, 4, 4, 32, A16, 16, None) == QMM_ERR_WORKSPACE
    assert lib.qmm_debug_block_sums_q8_0_q8_0(2, A16, A16, A16, 1, 1, 32, None, 0, None) == QMM_ERR_ARG
    assert lib.qmm_debug_block_sums_q8_0_q8_0(0, A16, A16, None, 1, 1, 32, None, 0, None) == QMM_ERR_NULL


def test_repack_entry_points(lib):
    A16 = _p(0x10000)
    A2 = _p(0x10002)
    bad = ctypes.c_size_t(-1).value
    lib.qmm_repack_q4_0_gemm_bytes.restype = ctypes.c_size_t
    lib.qmm_repack_q4_0_gemm_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
    # ceil(n/128) row groups x ceil(k/64) stages x 4096 bytes
    assert lib.qmm_repack_q4_0_gemm_bytes(14336, 4096) == 112 * 64 * 4096
    assert lib.qmm_repack_q4_0_gemm_bytes(129, 96) == 2 * 2 * 4096
    assert lib.qmm_repack_q4_0_gemm_bytes(1, 33) == bad
    assert lib.qmm_repack_q4_0_gemm(None, 1, 32, A16, 1 << 20, None) == QMM_ERR_NULL
    assert lib.qmm_repack_q4_0_gemm(A16, 1, 48, A16, 1 << 20, None) == QMM_ERR_SHAPE
    assert lib.qmm_repack_q4_0_gemm(A16, 1, 32, A2, 1 << 20, None) == QMM_ERR_ALIGN
    assert lib.qmm_repack_q4_0_gemm(A16, 1, 32, A16, 4095, None) == QMM_ERR_WORKSPACE
    gemm = lib.qmm_gemm_q4_0_q8_0_repacked
    assert gemm(A16, 1 << 20, A16, A16, A16, None, 1, 1, 32, A16, 1 << 20, None) == QMM_ERR_NULL
    assert gemm(A16, 4095, A16, A16, A16, A16, 1, 1, 32, A16, 1 << 20, None) == QMM_ERR_WORKSPACE
    assert gemm(A16, 1 << 20, A16, A16, A16, A16, 4, 4, 32, A16, 16, None) == QMM_ERR_WORKSPACE
    assert gemm(A2, 1 << 20, A16, A16, A16, A16, 1, 1, 32, A16, 1 << 20, None) == QMM_ERR_ALIGN


def test_linear_bitnet_argument_errors(lib):
    A16 = _p(0x10000)  # never dereferenced: every call below fails its host checks
    A2 = _p(0x10002)
    f = lib.qmm_linear_bitnet
    f.restype = ctypes.c_int
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    f.argtypes = [P, ctypes.c_float, P, I64, P, P, P, P, I64, I64, I64, I, P]
    assert f(A16, 1.0, None, 32, A16, A16, A16, A16, 1, 1, 32, 0, None) == QMM_ERR_NULL
    assert f(None, 1.0, A16, 32, A16, A16, A16, A16, 1, 1, 32, 0, None) == QMM_ERR_NULL
    assert f(A16, 1.0, A16, 32, A16, A16, A16, A16, 17, 1, 32, 0, None) == QMM_ERR_SHAPE
    assert f(A16, 1.0, A16, 32, A16, A16, A16, A16, 1, 1, 24, 0, None) == QMM_ERR_SHAPE
    assert f(A16, 1.0, A16, 16, A16, A16, A16, A16, 1, 1, 32, 0, None) == QMM_ERR_SHAPE  # ldx < k
    assert f(A2, 1.0, A16, 32, A16, A16, A16, A16, 1, 1, 32, 0, None) == QMM_ERR_ALIGN
    assert f(A16, 1.0, A2, 32, A16, A16, A16, A16, 1, 1, 32, 0, None) == QMM_ERR_ALIGN
    assert f(A16, 1.0, A16, 32, A16, A16, A16, A16, 1, 1, 32, 4, None) == QMM_ERR_ARG


def test_mma_probe_argument_errors(lib):
    A16 = _p(0x10000)  # never dereferenced: every call below fails its host checks
    f = lib.qmm_debug_mma_probe
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                  ctypes.c_void_p]
    macs = ctypes.c_int64(0)
    assert f(0, 10, None, 1 << 20, ctypes.byref(macs), None) == QMM_ERR_NULL
    assert f(0, 10, A16, 1 << 20, None, None) == QMM_ERR_NULL
    assert f(2, 10, A16, 1 << 20, ctypes.byref(macs), None) == QMM_ERR_ARG
    assert f(0, 0, A16, 1 << 20, ctypes.byref(macs), None) == QMM_ERR_ARG


def test_auto_split_policy(lib):
    # a narrow output with a long reduction is split, a wide one is not
    assert lib.qmm_gemv_auto_split(1, 256, 16384) > 1
    assert lib.qmm_gemv_auto_split(1, 128256, 4096) == 1
    assert lib.qmm_gemv_auto_split(1, 4096, 4096) >= 1


def test_auto_split_always_fits_the_noalloc_array(lib):
    # qmm_gemv_q4_0_q8_0_noalloc rejects any split whose partials exceed its
    # built-in array; the automatic split must never be rejected, at any
    # m <= 16, any n and any k
    cap = 1 << 20
    worst = 0
    for m in range(1, 17):
        for n in list(range(1, 1400)) + [2048, 4096, 11008, 128256]:
            for k in (32, 2048, 4096, 11008, 1 << 17):
                s = lib.qmm_gemv_auto_split(m, n, k)
                assert 1 <= s <= max(1, k // 32 // 64) or s == 1
                worst = max(worst, s * m * n if s > 1 else 0)
    assert 0 < worst <= cap // 32, worst


def _p(v):
    return ctypes.c_void_p(v)


def test_argument_errors_return_before_any_launch(lib):
    A16 = _p(0x10000)  # never dereferenced: every call below fails its host checks
    A2 = _p(0x10002)   # 2-byte aligned only
    # null pointers
    assert lib.qmm_quantize_act_q8_0(None, 1, 32, 32, A16, A16, None) == QMM_ERR_NULL
    assert lib.qmm_gemv_q4_0_q8_0(A16, A16, None, A16, A16, 1, 1, 32, 1, None, 0, None) == QMM_ERR_NULL
    assert lib.qmm_gemm_q4_0_q8_0(A16, A16, A16, A16, None, 1, 1, 32, A16, 1 << 20, None) == QMM_ERR_NULL
    assert lib.qmm_bitnet_gemv(None, 1.0, A16, A16, A16, A16, 1, 1, 16, None) == QMM_ERR_NULL
    # shapes
    assert lib.qmm_quantize_act_q8_0(A16, 1, 33, 33, A16, A16, None) == QMM_ERR_SHAPE
    assert lib.qmm_quantize_act_q8_0(A16, 1, 64, 32, A16, A16, None) == QMM_ERR_SHAPE  # ldx < k
    assert lib.qmm_quantize_act_q8_0(A16, 0, 32, 32, A16, A16, None) == QMM_ERR_SHAPE
    assert lib.qmm_gemv_q4_0_q8_0(A16, A16, A16, A16, A16, 17, 1, 32, 1, None, 0, None) == QMM_ERR_SHAPE
    assert lib.qmm_gemv_q4_0_q8_0(A16, A16, A16, A16, A16, 1, 0, 32, 1, None, 0, None) == QMM_ERR_SHAPE
    assert lib.qmm_gemm_q4_0_q8_0(A16, A16, A16, A16, A16, 1, 1, 48, A16, 1 << 20, None) == QMM_ERR_SHAPE
    assert lib.qmm_bitnet_gemv(A16, 1.0, A16, A16, A16, A16, 1, 1, 24, None) == QMM_ERR_SHAPE
    assert lib.qmm_bitnet_gemv(A16, 1.0, A16, A16, A16, A16, 17, 1, 16, None) == QMM_ERR_SHAPE
    assert lib.qmm_quantize_act_bitnet(A16, 1, 20, A16, A16, A16, None) == QMM_ERR_SHAPE
    assert lib.qmm_pack_ternary(A16, 1, 8, A16, None) == QMM_ERR_SHAPE
    # alignment
    assert lib.qmm_gemv_q4_0_q8_0(A2, A16, A16, A16, A16, 1, 1, 32, 1, None, 0, None) == QMM_ERR_ALIGN
    assert lib.qmm_gemv_q4_0_q8_0(A16, A16, A2, A16, A16, 1, 1, 32, 1, None, 0, None) == QMM_ERR_ALIGN
    assert lib.qmm_gemm_q4_0_q8_0(A16, A16, A16, A16, A2, 1, 1, 32, A16, 1 << 20, None) == QMM_ERR_ALIGN
    assert lib.qmm_bitnet_gemv(A2, 1.0, A16, A16, A16, A16, 1, 1, 16, None) == QMM_ERR_ALIGN
    # workspace
    assert lib.qmm_gemm_q4_0_q8_0(A16, A16, A16, A16, A16, 4, 4, 32, None, 0, None) == QMM_ERR_WORKSPACE
    assert lib.qmm_gemm_q4_0_q8_0(A16, A16, A16, A16, A16, 4, 4, 32, A16, 16, None) == QMM_ERR_WORKSPACE
    assert lib.qmm_gemv_q4_0_q8_0(A16, A16, A16, A16, A16, 1, 4, 64, 2, None, 0, None) == QMM_ERR_WORKSPACE
    assert lib.qmm_gemm_q4_0_q8_0(A16, A16, A16, A16, A16, 4, 4, 32, _p(0x10010), 1 << 20, None) == QMM_ERR_ALIGN
    # split_k out of range
    assert lib.qmm_gemv_q4_0_q8_0(A16, A16, A16, A16, A16, 1, 4, 64, 3, A16, 1 << 20, None) == QMM_ERR_ARG
    assert lib.qmm_gemv_q4_0_q8_0(A16, A16, A16, A16, A16, 1, 4, 64, -1, A16, 1 << 20, None) == QMM_ERR_ARG
    # decode linear: m above the GEMV limit, ldx below k, bad flags
    assert lib.qmm_linear_q4_0(A16, A16, A16, 32, A16, A16, A16, 17, 1, 32, 0, None) == QMM_ERR_SHAPE
    assert lib.qmm_linear_q4_0(A16, A16, A16, 16, A16, A16, A16, 1, 1, 32, 0, None) == QMM_ERR_SHAPE
    assert lib.qmm_linear_q4_0(A16, A16, A16, 32, A16, A16, A16, 1, 1, 32, 2, None) == QMM_ERR_ARG
    assert lib.qmm_linear_q4_0(A16, A16, None, 32, A16, A16, A16, 1, 1, 32, 0, None) == QMM_ERR_NULL
    assert lib.qmm_linear_q4_0(A16, A16, A2, 32, A16, A16, A16, 1, 1, 32, 0, None) == QMM_ERR_ALIGN
    # grouped: table checks
    import quantized_matmul_gb300 as q
    tab = (q.LinearProblem * 17)()
    for i in range(17):
        tab[i] = q.LinearProblem(0x10000, 0x10000, 0x10000, 32, 0x10000, 0x10000, 0x10000, 1, 32)
    assert lib.qmm_linear_q4_0_grouped(None, 1, 1, 0, None) == QMM_ERR_NULL
    assert lib.qmm_linear_q4_0_grouped(ctypes.addressof(tab), 0, 1, 0, None) == QMM_ERR_ARG
    assert lib.qmm_linear_q4_0_grouped(ctypes.addressof(tab), 17, 1, 0, None) == QMM_ERR_ARG
    tab[3].k = 48
    assert lib.qmm_linear_q4_0_grouped(ctypes.addressof(tab), 5, 1, 0, None) == QMM_ERR_SHAPE
    tab[3].k = 32
    tab[2].aq = 0x10004
    assert lib.qmm_linear_q4_0_grouped(ctypes.addressof(tab), 5, 1, 0, None) == QMM_ERR_ALIGN
    tab[2].aq = 0x10000
    # the host-buffer variant: the same table checks, then its copy arguments
    host = lib.qmm_linear_q4_0_grouped_host
    assert host(None, 1, 1, 0, 0x10000, 0x10000, 64, 0x10000, 0x10000, 64, None) == QMM_ERR_NULL
    assert host(ctypes.addressof(tab), 17, 1, 0, 0x10000, 0x10000, 64, 0x10000, 0x10000, 64,
                None) == QMM_ERR_ARG
    assert host(ctypes.addressof(tab), 5, 1, 2, 0x10000, 0x10000, 64, 0x10000, 0x10000, 64,
                None) == QMM_ERR_ARG
    assert host(ctypes.addressof(tab), 5, 1, 0, None, 0x10000, 64, 0x10000, 0x10000, 64,
                None) == QMM_ERR_NULL
    assert host(ctypes.addressof(tab), 5, 1, 0, 0x10000, 0x10000, 64, 0x10000, None, 64,
                None) == QMM_ERR_NULL
    # debug entry: unknown path
    assert lib.qmm_debug_block_sums_q4_0_q8_0(5, A16, A16, A16, 1, 1, 32, None, 0, None) == QMM_ERR_ARG


def test_python_binding_refuses_cpu_tensors():
    import torch
    import quantized_matmul_gb300 as q
    with pytest.raises(ValueError, match="CUDA"):
        q.quantize_act_q8_0(torch.zeros(1, 32))
