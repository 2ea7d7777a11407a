"""CPU oracle for the quantized matmul path -- TEST INFRASTRUCTURE ONLY.

Plain scalar C (``qmm_oracle.c``) behind a numpy/ctypes binding.  Only the
test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library in ``quantized_matmul_gb300/`` and neither side imports the other.

Sources: llama.cpp visual guide, lesson 31 "The CPU backend", section "How the
quantized dot product works" (Q4_0 x Q8_0; the Q8_0 block, which the Fucina
reference, section 9, also uses as a weight format: Q8_0 x Q8_0); Loom docs, "Plan 9 SIMD Forward",
section "BitNet ternary MAD kernel" (ternary path); Fucina course ch. 06,
section 6.4 (the scalar referee).  The readings taken where the pages are
silent are listed at the top of ``qmm_oracle.c``.

Every function here has at least one pin in ``tests/test_oracle_pins.py``
that does not go through the oracle's own formula: hand-worked blocks under
``tests/golden/``, brute-force double-precision dequantize-then-dot, an exact
integer-matmul reduction, the ternary identity against a direct signed sum,
and format invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

QK = 32  # elements per block

CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with gcc (no-op when it is newer than the source)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int64
            sig = {
                "orc_fp16_to_fp32": (ctypes.c_float, [ctypes.c_uint16]),
                "orc_fp32_to_fp16": (ctypes.c_uint16, [ctypes.c_float]),
                "orc_fp16_to_fp32_array": (None, [P, I, P]),
                "orc_fp32_to_fp16_array": (None, [P, I, P]),
                "orc_quantize_q8_0": (None, [P, I, I, I, P, P]),
                "orc_quantize_q4_0": (None, [P, I, I, P, P]),
                "orc_block_sums_q4_0_q8_0": (None, [P, P, I, I, I, P]),
                "orc_gemm_q4_0_q8_0": (None, [P, P, P, P, I, I, I, P]),
                "orc_gemm_q4_0_q8_0_f64": (None, [P, P, P, P, I, I, I, P]),
                "orc_gemm_q4_0_q8_0_absterms": (None, [P, P, P, P, I, I, I, P]),
                "orc_block_sums_q8_0_q8_0": (None, [P, P, I, I, I, P]),
                "orc_gemm_q8_0_q8_0": (None, [P, P, P, P, I, I, I, P]),
                "orc_gemm_q8_0_q8_0_f64": (None, [P, P, P, P, I, I, I, P, P]),
                "orc_repack_q4_0_gemm": (None, [P, I, I, P]),
                "orc_unrepack_q4_0_gemm": (None, [P, I, I, P]),
                "orc_q4_0_blocks_to_planes": (None, [P, I, I, P, P]),
                "orc_q4_0_planes_to_blocks": (None, [P, P, I, I, P]),
                "orc_quantize_act_bitnet": (None, [P, I, I, P, P, P]),
                "orc_pack_ternary": (None, [P, I, I, P]),
                "orc_bitnet_dot": (None, [P, P, P, I, I, I, P]),
                "orc_bitnet_gemv": (None, [P, ctypes.c_float, P, P, P, I, I, I, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# fp16 scalar conversions (IEEE-754 binary16, round to nearest even)

def fp32_to_fp16_bits(v: float) -> int:
    return int(_load().orc_fp32_to_fp16(float(v)))


def fp16_bits_to_fp32(h: int) -> float:
    return float(_load().orc_fp16_to_fp32(int(h)))


def fp32_to_fp16_bits_array(a) -> np.ndarray:
    """Element-wise fp32 -> fp16 bits through the oracle's own conversion."""
    a = _c(a, np.float32).ravel()
    out = np.empty(a.size, np.uint16)
    _load().orc_fp32_to_fp16_array(_p(a), a.size, _p(out))
    return out


def fp16_bits_to_fp32_array(h) -> np.ndarray:
    h = _c(h, np.uint16).ravel()
    out = np.empty(h.size, np.float32)
    _load().orc_fp16_to_fp32_array(_p(h), h.size, _p(out))
    return out


# --------------------------------------------------------------------------
# Q4_0 x Q8_0

def quantize_q8_0(x) -> tuple[np.ndarray, np.ndarray]:
    """f32 [m, k] -> (aq int8 [m, k], ad fp16-bits uint16 [m, k/32])."""
    x = _c(x, np.float32)
    if x.ndim == 1:
        x = x[None, :]
    m, k = x.shape
    assert k % QK == 0
    aq = np.empty((m, k), np.int8)
    ad = np.empty((m, k // QK), np.uint16)
    _load().orc_quantize_q8_0(_p(x), m, k, k, _p(aq), _p(ad))
    return aq, ad


def quantize_q8_0_strided(xbuf, k) -> tuple[np.ndarray, np.ndarray]:
    """The first k columns of f32 [m, ldx] rows (row stride ldx >= k)
    -> (aq int8 [m, k], ad fp16-bits uint16 [m, k/32])."""
    xbuf = _c(xbuf, np.float32)
    m, ldx = xbuf.shape
    assert k % QK == 0 and ldx >= k
    aq = np.empty((m, k), np.int8)
    ad = np.empty((m, k // QK), np.uint16)
    _load().orc_quantize_q8_0(_p(xbuf), m, k, ldx, _p(aq), _p(ad))
    return aq, ad


def quantize_q4_0(w) -> tuple[np.ndarray, np.ndarray]:
    """f32 [n, k] -> (wq uint8 [n, k/2], wd fp16-bits uint16 [n, k/32])."""
    w = _c(w, np.float32)
    n, k = w.shape
    assert k % QK == 0
    wq = np.empty((n, k // 2), np.uint8)
    wd = np.empty((n, k // QK), np.uint16)
    _load().orc_quantize_q4_0(_p(w), n, k, _p(wq), _p(wd))
    return wq, wd


def block_sums(wq, aq) -> np.ndarray:
    """int32 [m, n, k/32] per-block integer dots."""
    wq = _c(wq, np.uint8)
    aq = _c(aq, np.int8)
    n = wq.shape[0]
    m, k = aq.shape
    assert wq.shape[1] * 2 == k
    out = np.empty((m, n, k // QK), np.int32)
    _load().orc_block_sums_q4_0_q8_0(_p(wq), _p(aq), m, n, k, _p(out))
    return out


def _gemm_args(wq, wd, aq, ad):
    wq = _c(wq, np.uint8)
    wd = _c(wd, np.uint16)
    aq = _c(aq, np.int8)
    ad = _c(ad, np.uint16)
    n = wq.shape[0]
    m, k = aq.shape
    assert wq.shape == (n, k // 2) and wd.shape == (n, k // QK) and ad.shape == (m, k // QK)
    return wq, wd, aq, ad, m, n, k


def gemm_q4_0_q8_0(wq, wd, aq, ad) -> np.ndarray:
    """y f32 [m, n] = sum_b fma(sumi, dw*da, acc), blocks ascending."""
    wq, wd, aq, ad, m, n, k = _gemm_args(wq, wd, aq, ad)
    y = np.empty((m, n), np.float32)
    _load().orc_gemm_q4_0_q8_0(_p(wq), _p(wd), _p(aq), _p(ad), m, n, k, _p(y))
    return y


def gemm_q4_0_q8_0_f64(wq, wd, aq, ad) -> np.ndarray:
    wq, wd, aq, ad, m, n, k = _gemm_args(wq, wd, aq, ad)
    y = np.empty((m, n), np.float64)
    _load().orc_gemm_q4_0_q8_0_f64(_p(wq), _p(wd), _p(aq), _p(ad), m, n, k, _p(y))
    return y


def gemm_q4_0_q8_0_absterms(wq, wd, aq, ad) -> np.ndarray:
    wq, wd, aq, ad, m, n, k = _gemm_args(wq, wd, aq, ad)
    y = np.empty((m, n), np.float64)
    _load().orc_gemm_q4_0_q8_0_absterms(_p(wq), _p(wd), _p(aq), _p(ad), m, n, k, _p(y))
    return y


def q4_0_blocks_to_planes(blocks, n: int, k: int):
    blocks = _c(blocks, np.uint8)
    assert blocks.size == n * (k // QK) * 18
    wq = np.empty((n, k // 2), np.uint8)
    wd = np.empty((n, k // QK), np.uint16)
    _load().orc_q4_0_blocks_to_planes(_p(blocks), n, k, _p(wq), _p(wd))
    return wq, wd


def q4_0_planes_to_blocks(wq, wd) -> np.ndarray:
    wq = _c(wq, np.uint8)
    wd = _c(wd, np.uint16)
    n, k = wq.shape[0], wq.shape[1] * 2
    out = np.empty(n * (k // QK) * 18, np.uint8)
    _load().orc_q4_0_planes_to_blocks(_p(wq), _p(wd), n, k, _p(out))
    return out


def repack_q4_0_gemm_bytes(n: int, k: int) -> int:
    return ((n + 127) // 128) * ((k // QK + 1) // 2) * 4096


def repack_q4_0_gemm(wq) -> np.ndarray:
    """Q4_0 nibble plane [n, k/2] -> the GEMM tile order (uint8, flat)."""
    wq = _c(wq, np.uint8)
    n, k = wq.shape[0], wq.shape[1] * 2
    out = np.empty(repack_q4_0_gemm_bytes(n, k), np.uint8)
    _load().orc_repack_q4_0_gemm(_p(wq), n, k, _p(out))
    return out


def unrepack_q4_0_gemm(wr, n: int, k: int) -> np.ndarray:
    wr = _c(wr, np.uint8)
    assert wr.size == repack_q4_0_gemm_bytes(n, k)
    out = np.zeros((n, k // 2), np.uint8)
    _load().orc_unrepack_q4_0_gemm(_p(wr), n, k, _p(out))
    return out


# --------------------------------------------------------------------------
# Q8_0 weights x Q8_0 activations (weights quantized by quantize_q8_0)

def _q8w_args(w8, wd, aq, ad):
    w8 = _c(w8, np.int8)
    wd = _c(wd, np.uint16)
    aq = _c(aq, np.int8)
    ad = _c(ad, np.uint16)
    n = w8.shape[0]
    m, k = aq.shape
    assert w8.shape == (n, k) and wd.shape == (n, k // QK) and ad.shape == (m, k // QK)
    return w8, wd, aq, ad, m, n, k


def block_sums_q8_0(w8, aq) -> np.ndarray:
    """int32 [m, n, k/32]: sum_j q_w * q_a per block."""
    w8 = _c(w8, np.int8)
    aq = _c(aq, np.int8)
    n = w8.shape[0]
    m, k = aq.shape
    assert w8.shape[1] == k
    out = np.empty((m, n, k // QK), np.int32)
    _load().orc_block_sums_q8_0_q8_0(_p(w8), _p(aq), m, n, k, _p(out))
    return out


def gemm_q8_0_q8_0(w8, wd, aq, ad) -> np.ndarray:
    """y f32 [m, n] = sum_b fma(sumi, dw*da, acc), blocks ascending."""
    w8, wd, aq, ad, m, n, k = _q8w_args(w8, wd, aq, ad)
    y = np.empty((m, n), np.float32)
    _load().orc_gemm_q8_0_q8_0(_p(w8), _p(wd), _p(aq), _p(ad), m, n, k, _p(y))
    return y


def gemm_q8_0_q8_0_f64(w8, wd, aq, ad) -> tuple[np.ndarray, np.ndarray]:
    """(y in double, per-output sum of |sumi*dw*da|)."""
    w8, wd, aq, ad, m, n, k = _q8w_args(w8, wd, aq, ad)
    y = np.empty((m, n), np.float64)
    a = np.empty((m, n), np.float64)
    _load().orc_gemm_q8_0_q8_0_f64(_p(w8), _p(wd), _p(aq), _p(ad), m, n, k, _p(y), _p(a))
    return y, a


# --------------------------------------------------------------------------
# BitNet ternary

def quantize_act_bitnet(x):
    """f32 [m, k] -> (aq int8 [m, k], scale f32 [m], asum int32 [m])."""
    x = _c(x, np.float32)
    if x.ndim == 1:
        x = x[None, :]
    m, k = x.shape
    aq = np.empty((m, k), np.int8)
    s = np.empty(m, np.float32)
    asum = np.empty(m, np.int32)
    _load().orc_quantize_act_bitnet(_p(x), m, k, _p(aq), _p(s), _p(asum))
    return aq, s, asum


def pack_ternary(t) -> np.ndarray:
    """int8 {-1,0,1} [n, k] -> uint32 [n, k/16]."""
    t = _c(t, np.int8)
    n, k = t.shape
    assert k % 16 == 0
    out = np.empty((n, k // 16), np.uint32)
    _load().orc_pack_ternary(_p(t), n, k, _p(out))
    return out


def bitnet_dot(tw, aq, asum) -> np.ndarray:
    tw = _c(tw, np.uint32)
    aq = _c(aq, np.int8)
    asum = _c(asum, np.int32)
    n = tw.shape[0]
    m, k = aq.shape
    assert tw.shape[1] * 16 == k
    out = np.empty((m, n), np.int32)
    _load().orc_bitnet_dot(_p(tw), _p(aq), _p(asum), m, n, k, _p(out))
    return out


def bitnet_gemv(tw, absmean: float, aq, scale, asum) -> np.ndarray:
    tw = _c(tw, np.uint32)
    aq = _c(aq, np.int8)
    scale = _c(scale, np.float32)
    asum = _c(asum, np.int32)
    n = tw.shape[0]
    m, k = aq.shape
    assert tw.shape[1] * 16 == k
    y = np.empty((m, n), np.float32)
    _load().orc_bitnet_gemv(_p(tw), float(np.float32(absmean)), _p(aq), _p(scale), _p(asum),
                            m, n, k, _p(y))
    return y
