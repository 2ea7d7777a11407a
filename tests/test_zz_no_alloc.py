"""The allocation-free decode GEMV, qmm_gemv_q4_0_q8_0_noalloc.

It serves callers that cannot allocate device memory where they run the
product (a latency-critical loop that must stay out of the CUDA allocator,
or a component handed device pointers but no allocator): its split-K
partials live in a 4 MiB array the library reserves on each GPU.  This file
sorts last so that a run stopping at the first failure has already run every
other test; it also passes when run alone in a fresh process.

The entry point is called through the C ABI (ctypes on libqmm.so) twice in a
row, on two different problems that both split the reduction, so both go
through the shared array.  Each result must equal, bit for bit, the
workspace-taking qmm_gemv_q4_0_q8_0 with the same split (the same kernels in
the same order), and must pass the CPU oracle under the f32 gate of the other
GPU tests."""
import ctypes

import numpy as np
import pytest

from conftest import rel_gate
from quantized_matmul_gb300 import synthetic

pytestmark = pytest.mark.gpu

QMM_ERR_WORKSPACE = 4


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _entry(qmm):
    fn = qmm.load().qmm_gemv_q4_0_q8_0_noalloc
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.restype = I
    fn.argtypes = [P, P, P, P, P, I64, I64, I64, I, P]
    return fn


def _case(orc, seed, m, n, k):
    w, x = synthetic.q4_0_case(seed, n, k, m)
    wq, wd = orc.quantize_q4_0(w)
    aq, ad = orc.quantize_q8_0(x)
    return wq, wd, aq, ad


def test_noalloc_gemv_matches_workspace_gemv_on_two_calls(qmm, orc):
    import torch
    fn = _entry(qmm)
    stream = torch.cuda.current_stream().cuda_stream
    # two different problems back to back, both split (so both use the
    # shared array), the second smaller than the first: it must read only
    # the partials it wrote, not what the first call left behind
    for seed, (m, n, k, split) in [(901, (1, 300, 4096, 4)), (902, (3, 129, 2048, 3))]:
        wq, wd, aq, ad = _case(orc, seed, m, n, k)
        d = (_dev(wq), _dev(wd.view(np.float16)), _dev(aq), _dev(ad.view(np.float16)))
        y = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
        st = fn(d[0].data_ptr(), d[1].data_ptr(), d[2].data_ptr(), d[3].data_ptr(), y.data_ptr(),
                m, n, k, split, stream)
        assert st == 0
        y_ws = qmm.gemv_q4_0_q8_0(*d, split_k=split)
        torch.cuda.synchronize()
        assert qmm.check_device_error() == 0
        got, ref = y.cpu().numpy(), y_ws.cpu().numpy()
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
        absterms = orc.gemm_q4_0_q8_0_absterms(wq, wd, aq, ad)
        ok, worst, maxrel = rel_gate(got, orc.gemm_q4_0_q8_0(wq, wd, aq, ad), absterms)
        assert ok, (worst, maxrel)


def test_noalloc_gemv_rejects_partials_larger_than_its_array(qmm):
    fn = _entry(qmm)
    a16 = ctypes.c_void_p(0x10000)  # never dereferenced: the host check fails first
    # 64 slices x 16 rows x 4096 outputs = 4 Mi floats > the 1 Mi-float array
    assert fn(a16, a16, a16, a16, a16, 16, 4096, 4096, 64, None) == QMM_ERR_WORKSPACE
