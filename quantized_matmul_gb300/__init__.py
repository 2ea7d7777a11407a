"""quantized_matmul_gb300 -- Q4_0 x Q8_0 and BitNet ternary matmul on GB300.

A thin ctypes binding over the C ABI of ``libqmm.so`` (declared in
``include/qmm.h``).  Every function marshals torch tensors (device memory,
dtype and shape checks) and the current CUDA stream into one C call; all
arithmetic runs in the library's CUDA kernels.  There is no CPU fallback:
if the library is missing or does not load, every call raises.

Tensor conventions (row-major, contiguous, on the current CUDA device):
  x   float32 [m, k]            activations
  aq  int8    [m, k]            Q8_0 codes;  ad float16 [m, k/32] scales
  wq  uint8   [n, k/2]          Q4_0 nibbles; wd float16 [n, k/32] scales
  y   float32 [m, n]
  tw  int32   [n, k/16]         packed ternary codes (uint32 bit patterns)
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libqmm.so")

QK = 32
GEMV_MAX_M = 16
OP_GEMV = 1
OP_GEMM = 2
OP_BITNET_GEMM = 3
OP_GEMV_Q8 = 4
OP_GEMM_Q8 = 5

STATUS_NAMES = {0: "ok", 1: "null pointer", 2: "invalid shape", 3: "misaligned pointer",
                4: "workspace missing or too small", 5: "unsupported device", 6: "CUDA error",
                7: "device-side wait timed out", 8: "invalid argument"}

_lock = threading.Lock()
_lib = None


class QmmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: qmm status {status} ({STATUS_NAMES.get(status, '?')})")


def load() -> ctypes.CDLL:
    """Load libqmm.so (built in-tree by ``quantized_matmul_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m quantized_matmul_gb300.build` (there is no fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        P, I64, I, U32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32
        F, SZ = ctypes.c_float, ctypes.c_size_t
        sigs = {
            "qmm_quantize_act_q8_0": (I, [P, I64, I64, I64, P, P, P]),
            "qmm_quantize_weight_q4_0": (I, [P, I64, I64, P, P, P]),
            "qmm_gemv_q4_0_q8_0": (I, [P, P, P, P, P, I64, I64, I64, I, P, SZ, P]),
            "qmm_gemm_q4_0_q8_0": (I, [P, P, P, P, P, I64, I64, I64, P, SZ, P]),
            "qmm_gemv_q4_0_q8_0_noalloc": (I, [P, P, P, P, P, I64, I64, I64, I, P]),
            "qmm_gemv_q8_0_q8_0": (I, [P, P, P, P, P, I64, I64, I64, I, P, SZ, P]),
            "qmm_repack_q4_0_gemm_bytes": (SZ, [I64, I64]),
            "qmm_repack_q4_0_gemm": (I, [P, I64, I64, P, SZ, P]),
            "qmm_gemm_q4_0_q8_0_repacked": (I, [P, SZ, P, P, P, P, I64, I64, I64, P, SZ, P]),
            "qmm_gemm_q8_0_q8_0": (I, [P, P, P, P, P, I64, I64, I64, P, SZ, P]),
            "qmm_linear_q4_0": (I, [P, P, P, I64, P, P, P, I64, I64, I64, I, P]),
            "qmm_linear_q4_0_grouped": (I, [P, I, I64, I, P]),
            "qmm_linear_q4_0_grouped_host": (I, [P, I, I64, I, P, P, SZ, P, P, SZ, P]),
            "qmm_host_addressable": (I, [P]),
            "qmm_quantize_act_bitnet": (I, [P, I64, I64, P, P, P, P]),
            "qmm_pack_ternary": (I, [P, I64, I64, P, P]),
            "qmm_bitnet_gemv": (I, [P, F, P, P, P, P, I64, I64, I64, P]),
            "qmm_bitnet_gemm": (I, [P, F, P, P, P, I64, I64, I64, P, SZ, P]),
            "qmm_linear_bitnet": (I, [P, F, P, I64, P, P, P, P, I64, I64, I64, I, P]),
            "qmm_workspace_bytes": (SZ, [I, I64, I64, I64, I]),
            "qmm_gemv_auto_split": (I, [I64, I64, I64]),
            "qmm_check_device_error": (I, [P]),
            "qmm_status_string": (ctypes.c_char_p, [I]),
            "qmm_version": (I, []),
            "qmm_debug_block_sums_q4_0_q8_0": (I, [I, P, P, P, I64, I64, I64, P, SZ, P]),
            "qmm_debug_block_sums_q8_0_q8_0": (I, [I, P, P, P, I64, I64, I64, P, SZ, P]),
            "qmm_debug_bitnet_dot": (I, [P, P, P, P, I64, I64, I64, P]),
            "qmm_debug_mma_probe": (I, [I, I, P, SZ, P, P]),
            "qmm_debug_set_wait_limit": (None, [U32]),
            "qmm_debug_withhold_gemm_loads": (None, [I]),
            "qmm_debug_withhold_gemv_loads": (None, [I]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(status: int, where: str) -> None:
    if status != 0:
        raise QmmError(status, where)


def _torch():
    import torch
    return torch


def _stream() -> int:
    """The current CUDA stream of the current device, as a raw handle.  The
    raw accessor costs ~0.3 us a call against ~2.9 us for building a
    torch.cuda.Stream object (measured on the GB300 host), a fifth of a
    decode step's host time; the public call is the fallback."""
    torch = _torch()
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _dev(t, dtype, name: str, shape=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _empty(shape, dtype, like):
    return _torch().empty(shape, dtype=dtype, device=like.device)


# ---------------------------------------------------------------------------
# Q4_0 x Q8_0

def quantize_act_q8_0(x, aq=None, ad=None):
    """f32 [m, k] -> (aq int8 [m, k], ad fp16 [m, k/32])."""
    torch = _torch()
    if x.dim() == 1:
        x = x.unsqueeze(0)
    m, k = x.shape
    aq = _empty((m, k), torch.int8, x) if aq is None else aq
    ad = _empty((m, k // QK), torch.float16, x) if ad is None else ad
    st = load().qmm_quantize_act_q8_0(_dev(x, torch.float32, "x"), m, k, k,
                                      _dev(aq, torch.int8, "aq", (m, k)),
                                      _dev(ad, torch.float16, "ad", (m, k // QK)), _stream())
    _check(st, "qmm_quantize_act_q8_0")
    return aq, ad


def quantize_weight_q4_0(w, wq=None, wd=None):
    """f32 [n, k] -> (wq uint8 [n, k/2], wd fp16 [n, k/32])."""
    torch = _torch()
    n, k = w.shape
    wq = _empty((n, k // 2), torch.uint8, w) if wq is None else wq
    wd = _empty((n, k // QK), torch.float16, w) if wd is None else wd
    st = load().qmm_quantize_weight_q4_0(_dev(w, torch.float32, "w"), n, k,
                                         _dev(wq, torch.uint8, "wq", (n, k // 2)),
                                         _dev(wd, torch.float16, "wd", (n, k // QK)), _stream())
    _check(st, "qmm_quantize_weight_q4_0")
    return wq, wd


def workspace_bytes(op: int, m: int, n: int, k: int, split_k: int = 0) -> int:
    v = load().qmm_workspace_bytes(op, m, n, k, split_k)
    if v == ctypes.c_size_t(-1).value:
        raise ValueError(f"invalid workspace query op={op} m={m} n={n} k={k} split_k={split_k}")
    return int(v)


def gemv_auto_split(m: int, n: int, k: int) -> int:
    return int(load().qmm_gemv_auto_split(m, n, k))


def _workspace(ws, need, like):
    torch = _torch()
    if need == 0:
        return None, 0
    if ws is None:
        ws = _empty((need,), torch.uint8, like)
    if ws.numel() < need:
        raise ValueError(f"workspace has {ws.numel()} bytes, needs {need}")
    return ws, ws.numel()


def _q4_shapes(wq, wd, aq, ad):
    torch = _torch()
    n = wq.shape[0]
    m, k = aq.shape
    _dev(wq, torch.uint8, "wq", (n, k // 2))
    _dev(wd, torch.float16, "wd", (n, k // QK))
    _dev(aq, torch.int8, "aq", (m, k))
    _dev(ad, torch.float16, "ad", (m, k // QK))
    return m, n, k


def gemv_q4_0_q8_0(wq, wd, aq, ad, y=None, split_k: int = 0, workspace=None):
    """Decode GEMV (m <= 16): y f32 [m, n]."""
    torch = _torch()
    m, n, k = _q4_shapes(wq, wd, aq, ad)
    y = _empty((m, n), torch.float32, aq) if y is None else y
    ws, ws_bytes = _workspace(workspace, workspace_bytes(OP_GEMV, m, n, k, split_k)
                              if m <= GEMV_MAX_M else 0, aq)
    st = load().qmm_gemv_q4_0_q8_0(wq.data_ptr(), wd.data_ptr(), aq.data_ptr(), ad.data_ptr(),
                                   _dev(y, torch.float32, "y", (m, n)), m, n, k, split_k,
                                   ws.data_ptr() if ws is not None else None, ws_bytes, _stream())
    _check(st, "qmm_gemv_q4_0_q8_0")
    return y


def gemv_q4_0_q8_0_noalloc(wq, wd, aq, ad, y=None, split_k: int = 0):
    """The decode GEMV for callers that cannot allocate device memory where
    they run it: the split-K partials use a 4 MiB array the library reserves
    on each GPU, so no workspace is passed.  Calls that overlap on the GPU
    share that array and race; order them on one stream."""
    torch = _torch()
    m, n, k = _q4_shapes(wq, wd, aq, ad)
    y = _empty((m, n), torch.float32, aq) if y is None else y
    st = load().qmm_gemv_q4_0_q8_0_noalloc(wq.data_ptr(), wd.data_ptr(), aq.data_ptr(),
                                           ad.data_ptr(), _dev(y, torch.float32, "y", (m, n)),
                                           m, n, k, split_k, _stream())
    _check(st, "qmm_gemv_q4_0_q8_0_noalloc")
    return y


def gemm_q4_0_q8_0(wq, wd, aq, ad, y=None, workspace=None):
    """Prefill GEMM on the tensor cores: y f32 [m, n]."""
    torch = _torch()
    m, n, k = _q4_shapes(wq, wd, aq, ad)
    y = _empty((m, n), torch.float32, aq) if y is None else y
    ws, ws_bytes = _workspace(workspace, workspace_bytes(OP_GEMM, m, n, k), aq)
    st = load().qmm_gemm_q4_0_q8_0(wq.data_ptr(), wd.data_ptr(), aq.data_ptr(), ad.data_ptr(),
                                   _dev(y, torch.float32, "y", (m, n)), m, n, k,
                                   ws.data_ptr() if ws is not None else None, ws_bytes, _stream())
    _check(st, "qmm_gemm_q4_0_q8_0")
    return y


def quantize_weight_q8_0(w):
    """Q8_0 weights: the activation recipe on the f32 weight rows, giving
    (w8 int8 [n, k], wd fp16 [n, k/32])."""
    return quantize_act_q8_0(w)


def _q8_shapes(w8, wd, aq, ad):
    torch = _torch()
    n = w8.shape[0]
    m, k = aq.shape
    _dev(w8, torch.int8, "w8", (n, k))
    _dev(wd, torch.float16, "wd", (n, k // QK))
    _dev(aq, torch.int8, "aq", (m, k))
    _dev(ad, torch.float16, "ad", (m, k // QK))
    return m, n, k


def gemv_q8_0_q8_0(w8, wd, aq, ad, y=None, split_k: int = 0, workspace=None):
    """Decode GEMV with Q8_0 weights (m <= 16): y f32 [m, n]."""
    torch = _torch()
    m, n, k = _q8_shapes(w8, wd, aq, ad)
    y = _empty((m, n), torch.float32, aq) if y is None else y
    ws, ws_bytes = _workspace(workspace, workspace_bytes(OP_GEMV_Q8, m, n, k, split_k)
                              if m <= GEMV_MAX_M else 0, aq)
    st = load().qmm_gemv_q8_0_q8_0(w8.data_ptr(), wd.data_ptr(), aq.data_ptr(), ad.data_ptr(),
                                   _dev(y, torch.float32, "y", (m, n)), m, n, k, split_k,
                                   ws.data_ptr() if ws is not None else None, ws_bytes, _stream())
    _check(st, "qmm_gemv_q8_0_q8_0")
    return y


def gemm_q8_0_q8_0(w8, wd, aq, ad, y=None, workspace=None):
    """Prefill GEMM with Q8_0 weights on the tensor cores: y f32 [m, n]."""
    torch = _torch()
    m, n, k = _q8_shapes(w8, wd, aq, ad)
    y = _empty((m, n), torch.float32, aq) if y is None else y
    ws, ws_bytes = _workspace(workspace, workspace_bytes(OP_GEMM_Q8, m, n, k), aq)
    st = load().qmm_gemm_q8_0_q8_0(w8.data_ptr(), wd.data_ptr(), aq.data_ptr(), ad.data_ptr(),
                                   _dev(y, torch.float32, "y", (m, n)), m, n, k,
                                   ws.data_ptr() if ws is not None else None, ws_bytes, _stream())
    _check(st, "qmm_gemm_q8_0_q8_0")
    return y


def repack_q4_0_gemm(wq):
    """Load-time repack of the Q4_0 nibble plane [n, k/2] into the GEMM's tile
    order (uint8, flat; see qmm_repack_q4_0_gemm in include/qmm.h)."""
    torch = _torch()
    n, k = wq.shape[0], wq.shape[1] * 2
    nbytes = load().qmm_repack_q4_0_gemm_bytes(n, k)
    if nbytes == ctypes.c_size_t(-1).value:
        raise ValueError(f"invalid shape n={n} k={k}")
    wr = _empty((nbytes,), torch.uint8, wq)
    st = load().qmm_repack_q4_0_gemm(_dev(wq, torch.uint8, "wq"), n, k, wr.data_ptr(), nbytes,
                                     _stream())
    _check(st, "qmm_repack_q4_0_gemm")
    return wr


def gemm_q4_0_q8_0_repacked(wr, wd, aq, ad, y=None, workspace=None):
    """The prefill GEMM on repacked weights (bit for bit gemm_q4_0_q8_0)."""
    torch = _torch()
    n = wd.shape[0]
    m, k = aq.shape
    _dev(wd, torch.float16, "wd", (n, k // QK))
    _dev(aq, torch.int8, "aq", (m, k))
    _dev(ad, torch.float16, "ad", (m, k // QK))
    y = _empty((m, n), torch.float32, aq) if y is None else y
    ws, ws_bytes = _workspace(workspace, workspace_bytes(OP_GEMM, m, n, k), aq)
    st = load().qmm_gemm_q4_0_q8_0_repacked(_dev(wr, torch.uint8, "wr"), wr.numel(), wd.data_ptr(),
                                            aq.data_ptr(), ad.data_ptr(),
                                            _dev(y, torch.float32, "y", (m, n)), m, n, k,
                                            ws.data_ptr() if ws is not None else None, ws_bytes,
                                            _stream())
    _check(st, "qmm_gemm_q4_0_q8_0_repacked")
    return y


LINEAR_PDL = 1
LINEAR_HOST_DIRECT = 2
GROUP_MAX = 16


class LinearProblem(ctypes.Structure):
    """qmm_linear_problem: one weight matrix of qmm_linear_q4_0_grouped."""
    _fields_ = [("wq", ctypes.c_void_p), ("wd", ctypes.c_void_p), ("x", ctypes.c_void_p),
                ("ldx", ctypes.c_int64), ("aq", ctypes.c_void_p), ("ad", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("n", ctypes.c_int64), ("k", ctypes.c_int64)]


def linear_q4_0(x, wq, wd, y=None, pdl: bool = False, aq=None, ad=None, workspace=None,
                codes: bool = False):
    """y = x @ dequant(W)^T with Q8_0 activations, one library call.

    m <= 16: qmm_linear_q4_0, the quantizer then the decode GEMV; pdl=True
    launches both with programmatic dependent launch,
    so in a chain of layers on one stream each layer's weights stream while
    the previous layer finishes (the weights must not be written by work
    still running on the stream).  m > 16: quantizer + tensor-core GEMM
    (workspace used there).  aq/ad are optional preallocated code and scale
    buffers; codes=True also returns (aq, ad)."""
    torch = _torch()
    if x.dim() == 1:
        x = x.unsqueeze(0)
    m, k = x.shape
    n = wq.shape[0]
    if m <= GEMV_MAX_M:
        _dev(wq, torch.uint8, "wq", (n, k // 2))
        _dev(wd, torch.float16, "wd", (n, k // QK))
        aq = _empty((m, k), torch.int8, x) if aq is None else aq
        ad = _empty((m, k // QK), torch.float16, x) if ad is None else ad
        y = _empty((m, n), torch.float32, x) if y is None else y
        st = load().qmm_linear_q4_0(wq.data_ptr(), wd.data_ptr(), _dev(x, torch.float32, "x"), k,
                                    _dev(aq, torch.int8, "aq", (m, k)),
                                    _dev(ad, torch.float16, "ad", (m, k // QK)),
                                    _dev(y, torch.float32, "y", (m, n)), m, n, k,
                                    LINEAR_PDL if pdl else 0, _stream())
        _check(st, "qmm_linear_q4_0")
        return (y, aq, ad) if codes else y
    aq, ad = quantize_act_q8_0(x, aq=aq, ad=ad)
    y = gemm_q4_0_q8_0(wq, wd, aq, ad, y=y, workspace=workspace)
    return (y, aq, ad) if codes else y


def linear_q4_0_grouped(problems, pdl: bool = False):
    """Independent decode linear layers with the same m in two launches.

    problems: a list of (x, wq, wd) or (x, wq, wd, y, aq, ad) tuples (missing
    outputs are allocated).  Returns the list of (y, aq, ad).  Each result is
    bit for bit that of linear_q4_0 on the problem alone."""
    table, m, outs = _grouped_table(problems)
    st = load().qmm_linear_q4_0_grouped(ctypes.addressof(table), len(problems), m,
                                        LINEAR_PDL if pdl else 0, _stream())
    _check(st, "qmm_linear_q4_0_grouped")
    return outs


def host_addressable(t) -> bool:
    """Whether the current GPU can read and write the host tensor t's memory
    itself (page-locked memory with a device mapping), as host_direct needs."""
    if t.is_cuda:
        raise ValueError("a host (CPU) tensor is expected")
    return bool(load().qmm_host_addressable(t.data_ptr()))


class GroupedLinear:
    """A prepared linear_q4_0_grouped call for a decode loop.

    The problem table is built and checked once, here; each call then only
    enqueues the two launches on the current stream with one ctypes call.
    The tensors given (and the outputs allocated here) are used in place on
    every call: keep them alive and write new activations into the same x
    tensors between calls.  `outputs` is the list of (y, aq, ad).

    host_io=(x_host, x_dev, y_dev, y_host) makes every call carry its input
    from and its output to host memory as well (qmm_linear_q4_0_grouped_host):
    x_host (CPU) is copied into x_dev (CUDA) before the layers, and y_dev
    (CUDA) into y_host (CPU) after them, all on the current stream.  Every
    problem's x must be a view of x_dev and its y a view of y_dev.  Use
    page-locked host tensors (pin_memory()) to keep the call asynchronous;
    the host tensors must then stay unchanged until the stream has passed
    the copies.  host_direct=True lets the kernels read x_host and write
    y_host themselves where the device can address them (page-locked memory
    over NVLink-C2C), with no copy engine transfer; elsewhere it copies.

    graph=True suits a loop that waits for every call's outputs before the
    next: the first call runs the layers and captures the same C call into a
    CUDA graph, and every later call replays that graph on the current stream
    (one launch instead of one per kernel: measured 29.5 against 36.1 us per
    layer-set step with the outputs awaited each time).  Calls issued back to
    back are faster without it, since consecutive graph launches do not
    overlap the way dependent launches do.  The graph keeps the pointers of
    the first call, which GroupedLinear fixes anyway; with host_io the host
    tensors must be page-locked (a copy from pageable memory cannot be
    captured)."""

    def __init__(self, problems, pdl: bool = False, host_io=None, host_direct: bool = False,
                 graph: bool = False):
        self._table, self._m, self.outputs = _grouped_table(problems)
        self._keep = [tuple(p) for p in problems]  # the tensors the table points at
        self._count = len(problems)
        self._flags = LINEAR_PDL if pdl else 0
        self._fn = load().qmm_linear_q4_0_grouped
        self._addr = ctypes.addressof(self._table)
        self._host = None
        if host_direct and host_io is None:
            raise ValueError("host_direct needs host_io")
        if host_io is not None:
            x_host, x_dev, y_dev, y_host = host_io
            for name, t, cuda in (("x_host", x_host, False), ("x_dev", x_dev, True),
                                  ("y_dev", y_dev, True), ("y_host", y_host, False)):
                if t.is_cuda != cuda or not t.is_contiguous():
                    raise ValueError(f"{name}: a contiguous {'CUDA' if cuda else 'CPU'} tensor")
            xb = x_dev.numel() * x_dev.element_size()
            yb = y_dev.numel() * y_dev.element_size()
            if x_host.numel() * x_host.element_size() != xb or \
                    y_host.numel() * y_host.element_size() != yb:
                raise ValueError("host and device tensors of host_io differ in size")
            self._keep.append(tuple(host_io))
            self._host = (x_host.data_ptr(), x_dev.data_ptr(), xb,
                          y_dev.data_ptr(), y_host.data_ptr(), yb)
            self._fn_host = load().qmm_linear_q4_0_grouped_host
            self._host_flags = self._flags | (LINEAR_HOST_DIRECT if host_direct else 0)
            if graph and not (host_io[0].is_pinned() and host_io[3].is_pinned()):
                raise ValueError("graph=True with host_io needs page-locked host tensors")
        self._use_graph = graph
        self._graph = None

    def __call__(self):
        if not self._use_graph:
            return self._run()
        if self._graph is None:
            torch = _torch()
            self._run()  # this call's results; also any one-time set-up
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._run()
            self._graph = g
            return self.outputs
        self._graph.replay()
        return self.outputs

    def _run(self):
        if self._host is not None:
            st = self._fn_host(self._addr, self._count, self._m, self._host_flags, *self._host,
                               _stream())
            if st != 0:
                raise QmmError(st, "qmm_linear_q4_0_grouped_host")
            return self.outputs
        st = self._fn(self._addr, self._count, self._m, self._flags, _stream())
        if st != 0:
            raise QmmError(st, "qmm_linear_q4_0_grouped")
        return self.outputs


def _grouped_table(problems):
    """The qmm_linear_problem table for a list of problems (checked), the
    common m, and the (y, aq, ad) of every problem (allocated when missing)."""
    torch = _torch()
    if not 1 <= len(problems) <= GROUP_MAX:
        raise ValueError(f"1..{GROUP_MAX} problems, got {len(problems)}")
    table = (LinearProblem * len(problems))()
    outs = []
    m = None
    for p, prob in enumerate(problems):
        x, wq, wd = prob[:3]
        if x.dim() == 1:
            x = x.unsqueeze(0)
        mp, k = x.shape
        if m is None:
            m = mp
        if mp != m:
            raise ValueError("every problem of a group has the same m")
        n = wq.shape[0]
        y, aq, ad = (tuple(prob[3:6]) + (None, None, None))[:3]
        y = _empty((m, n), torch.float32, x) if y is None else y
        aq = _empty((m, k), torch.int8, x) if aq is None else aq
        ad = _empty((m, k // QK), torch.float16, x) if ad is None else ad
        table[p] = LinearProblem(_dev(wq, torch.uint8, "wq", (n, k // 2)),
                                 _dev(wd, torch.float16, "wd", (n, k // QK)),
                                 _dev(x, torch.float32, "x"), k,
                                 _dev(aq, torch.int8, "aq", (m, k)),
                                 _dev(ad, torch.float16, "ad", (m, k // QK)),
                                 _dev(y, torch.float32, "y", (m, n)), n, k)
        outs.append((y, aq, ad))
    return table, m, outs


# ---------------------------------------------------------------------------
# BitNet ternary

def quantize_act_bitnet(x):
    """f32 [m, k] -> (aq int8 [m, k], act_scale f32 [m], act_sum int32 [m])."""
    torch = _torch()
    if x.dim() == 1:
        x = x.unsqueeze(0)
    m, k = x.shape
    aq = _empty((m, k), torch.int8, x)
    s = _empty((m,), torch.float32, x)
    asum = _empty((m,), torch.int32, x)
    st = load().qmm_quantize_act_bitnet(_dev(x, torch.float32, "x"), m, k, aq.data_ptr(),
                                        s.data_ptr(), asum.data_ptr(), _stream())
    _check(st, "qmm_quantize_act_bitnet")
    return aq, s, asum


def pack_ternary(t):
    """int8 {-1,0,1} [n, k] -> int32 [n, k/16] (uint32 bit patterns)."""
    torch = _torch()
    n, k = t.shape
    w = _empty((n, k // 16), torch.int32, t)
    st = load().qmm_pack_ternary(_dev(t, torch.int8, "t"), n, k, w.data_ptr(), _stream())
    _check(st, "qmm_pack_ternary")
    return w


def linear_bitnet(x, tw, weight_absmean: float, y=None, pdl: bool = False, aq=None,
                  act_scale=None, act_sum=None, codes: bool = False):
    """BitNet decode layer in one library call (qmm_linear_bitnet): the
    per-row activation quantizer then the ternary GEMV, m <= 16.  pdl=True
    launches both with programmatic dependent launch (see linear_q4_0).
    codes=True also returns (aq, act_scale, act_sum)."""
    torch = _torch()
    if x.dim() == 1:
        x = x.unsqueeze(0)
    m, k = x.shape
    n = tw.shape[0]
    _dev(tw, torch.int32, "tw", (n, k // 16))
    aq = _empty((m, k), torch.int8, x) if aq is None else aq
    act_scale = _empty((m,), torch.float32, x) if act_scale is None else act_scale
    act_sum = _empty((m,), torch.int32, x) if act_sum is None else act_sum
    y = _empty((m, n), torch.float32, x) if y is None else y
    st = load().qmm_linear_bitnet(tw.data_ptr(), float(weight_absmean), _dev(x, torch.float32, "x"), k,
                                  _dev(aq, torch.int8, "aq", (m, k)),
                                  _dev(act_scale, torch.float32, "act_scale", (m,)),
                                  _dev(act_sum, torch.int32, "act_sum", (m,)),
                                  _dev(y, torch.float32, "y", (m, n)), m, n, k,
                                  LINEAR_PDL if pdl else 0, _stream())
    _check(st, "qmm_linear_bitnet")
    return (y, aq, act_scale, act_sum) if codes else y


def mma_probe_tops(kind: int = 0, iters: int = 4096, repeats: int = 3) -> float:
    """Measured warp-level tensor-core rate, in tera multiply-accumulates x 2
    per second (TOPS for kind 0, int8; TFLOPS for kind 1, f16): the best of
    `repeats` timed launches of qmm_debug_mma_probe after one untimed one."""
    torch = _torch()
    dev = torch.cuda.current_device()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = torch.empty((sms * 512,), dtype=torch.int32, device="cuda")
    macs = ctypes.c_int64(0)
    best = 0.0
    for r in range(repeats + 1):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record()
        st = load().qmm_debug_mma_probe(kind, iters, out.data_ptr(), out.numel() * 4,
                                        ctypes.byref(macs), _stream())
        end.record()
        _check(st, "qmm_debug_mma_probe")
        end.synchronize()
        if r:
            best = max(best, 2.0 * macs.value / (start.elapsed_time(end) * 1e-3) / 1e12)
    return best


def bitnet_gemv(tw, weight_absmean: float, aq, act_scale, act_sum, y=None):
    torch = _torch()
    n = tw.shape[0]
    m, k = aq.shape
    _dev(tw, torch.int32, "tw", (n, k // 16))
    _dev(aq, torch.int8, "aq", (m, k))
    _dev(act_scale, torch.float32, "act_scale", (m,))
    _dev(act_sum, torch.int32, "act_sum", (m,))
    y = _empty((m, n), torch.float32, aq) if y is None else y
    st = load().qmm_bitnet_gemv(tw.data_ptr(), float(weight_absmean), aq.data_ptr(),
                                act_scale.data_ptr(), act_sum.data_ptr(),
                                _dev(y, torch.float32, "y", (m, n)), m, n, k, _stream())
    _check(st, "qmm_bitnet_gemv")
    return y


def bitnet_gemm(tw, weight_absmean: float, aq, act_scale, y=None, workspace=None):
    """BitNet prefill on the tensor cores (any m, k % 64 == 0): y f32 [m, n],
    bit for bit what bitnet_gemv gives."""
    torch = _torch()
    n = tw.shape[0]
    m, k = aq.shape
    _dev(tw, torch.int32, "tw", (n, k // 16))
    _dev(aq, torch.int8, "aq", (m, k))
    _dev(act_scale, torch.float32, "act_scale", (m,))
    y = _empty((m, n), torch.float32, aq) if y is None else y
    ws, ws_bytes = _workspace(workspace, workspace_bytes(OP_BITNET_GEMM, m, n, k), aq)
    st = load().qmm_bitnet_gemm(tw.data_ptr(), float(weight_absmean), aq.data_ptr(),
                                act_scale.data_ptr(), _dev(y, torch.float32, "y", (m, n)), m, n, k,
                                ws.data_ptr() if ws is not None else None, ws_bytes, _stream())
    _check(st, "qmm_bitnet_gemm")
    return y


# ---------------------------------------------------------------------------
# errors and test hooks

def check_device_error() -> int:
    """Synchronizes the current stream and returns (and clears) the device
    error status: 0 ok, 7 a bounded wait gave up."""
    return int(load().qmm_check_device_error(_stream()))


def debug_block_sums(path: int, wq, aq, workspace=None, n=None):
    """int32 [m, n, k/32] block sums from the GEMV (path 0) or GEMM (path 1)
    kernel, or the GEMM on repacked weights (path 2: wq is the repacked
    tile array and n must be given)."""
    torch = _torch()
    m, k = aq.shape
    if path == 2:
        _dev(wq, torch.uint8, "wr")
    else:
        n = wq.shape[0]
        _dev(wq, torch.uint8, "wq", (n, k // 2))
    _dev(aq, torch.int8, "aq", (m, k))
    sumi = _empty((m, n, k // QK), torch.int32, aq)
    ws, ws_bytes = (None, 0)
    if path in (1, 2):
        ws, ws_bytes = _workspace(workspace, workspace_bytes(OP_GEMM, m, n, k), aq)
    st = load().qmm_debug_block_sums_q4_0_q8_0(path, wq.data_ptr(), aq.data_ptr(), sumi.data_ptr(),
                                               m, n, k, ws.data_ptr() if ws is not None else None,
                                               ws_bytes, _stream())
    _check(st, "qmm_debug_block_sums_q4_0_q8_0")
    return sumi


def debug_block_sums_q8(path: int, w8, aq, workspace=None):
    """int32 [m, n, k/32] block sums of the Q8_0-weight GEMV (path 0) or GEMM
    (path 1) kernel."""
    torch = _torch()
    n = w8.shape[0]
    m, k = aq.shape
    _dev(w8, torch.int8, "w8", (n, k))
    _dev(aq, torch.int8, "aq", (m, k))
    sumi = _empty((m, n, k // QK), torch.int32, aq)
    ws, ws_bytes = (None, 0)
    if path == 1:
        ws, ws_bytes = _workspace(workspace, workspace_bytes(OP_GEMM_Q8, m, n, k), aq)
    st = load().qmm_debug_block_sums_q8_0_q8_0(path, w8.data_ptr(), aq.data_ptr(), sumi.data_ptr(),
                                               m, n, k, ws.data_ptr() if ws is not None else None,
                                               ws_bytes, _stream())
    _check(st, "qmm_debug_block_sums_q8_0_q8_0")
    return sumi


def debug_bitnet_dot(tw, aq, act_sum):
    torch = _torch()
    n = tw.shape[0]
    m, k = aq.shape
    dot = _empty((m, n), torch.int32, aq)
    st = load().qmm_debug_bitnet_dot(tw.data_ptr(), aq.data_ptr(), act_sum.data_ptr(),
                                     dot.data_ptr(), m, n, k, _stream())
    _check(st, "qmm_debug_bitnet_dot")
    return dot


def set_wait_limit(iterations: int) -> None:
    load().qmm_debug_set_wait_limit(int(iterations))


def withhold_gemm_loads(enable: bool) -> None:
    load().qmm_debug_withhold_gemm_loads(1 if enable else 0)


def withhold_gemv_loads(enable: bool) -> None:
    """Test hook: the streaming GEMV arms no stage while enabled."""
    load().qmm_debug_withhold_gemv_loads(1 if enable else 0)
