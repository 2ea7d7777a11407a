"""GPU parity at the benchmark workloads' full sizes, in the calls bench.py times.

Each workload is drawn with its seed and recipe (synthetic.py), quantized by
the oracle on the CPU (except where the timed call quantizes the activations
itself, and the codes are then compared bit for bit first), run through the
same entry point and launch configuration as the benchmark, and compared with
the oracle: on every output where the oracle finishes in a second or two,
else on sampled output rows, which the oracle computes alone (its results do
not depend on the other rows).  Integer parts and the tensor-core products are
compared bit for bit, decode f32 outputs with the gate of conftest.rel_gate.
"""
import numpy as np
import pytest

from conftest import rel_gate
from quantized_matmul_gb300 import synthetic

pytestmark = pytest.mark.gpu

QK = 32


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_np(t):
    return t.cpu().numpy()


def f16(a):
    return to_dev(np.ascontiguousarray(a).view(np.float16))


def f16_bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _check_decode(y, orc, wq, wd, aq, ad):
    y_ref = orc.gemm_q4_0_q8_0(wq, wd, aq, ad)
    absterms = orc.gemm_q4_0_q8_0_absterms(wq, wd, aq, ad)
    ok, worst, maxrel = rel_gate(y, y_ref, absterms)
    assert ok, (worst, maxrel)


def test_gemv_4096x4096_full(qmm, orc):
    """GEMV m=1, K=4096, N=4096, seed 0: every output, split_k=1 as timed."""
    w, x = synthetic.q4_0_case(0, 4096, 4096, 1)
    wq, wd = orc.quantize_q4_0(w)
    aq, ad = orc.quantize_q8_0(x)
    y = to_np(qmm.gemv_q4_0_q8_0(to_dev(wq), f16(wd), to_dev(aq), f16(ad), split_k=1))
    _check_decode(y, orc, wq, wd, aq, ad)
    sumi = to_np(qmm.debug_block_sums(0, to_dev(wq), to_dev(aq)))
    assert np.array_equal(sumi, orc.block_sums(wq, aq))


def test_layer_set_grouped_full(qmm, orc):
    """The 7-matrix layer set (seeds 1..7) through one grouped call with PDL,
    the headline step: every Q8_0 code and scale bit-exact, every output
    within the gate."""
    import torch
    table, refs = [], []
    for j, (n, k) in enumerate(synthetic.LAYER_SET_7B):
        w, x = synthetic.q4_0_case(j + 1, n, k, 1)
        wq, wd = orc.quantize_q4_0(w)
        aq_ref, ad_ref = orc.quantize_q8_0(x)
        xd = to_dev(x)
        aq = torch.empty((1, k), dtype=torch.int8, device="cuda")
        ad = torch.empty((1, k // QK), dtype=torch.float16, device="cuda")
        y = torch.empty((1, n), dtype=torch.float32, device="cuda")
        table.append((xd, to_dev(wq), f16(wd), y, aq, ad))
        refs.append((wq, wd, aq_ref, ad_ref))
    qmm.linear_q4_0_grouped(table, pdl=True)
    torch.cuda.synchronize()
    for (xd, _, _, y, aq, ad), (wq, wd, aq_ref, ad_ref) in zip(table, refs):
        assert np.array_equal(to_np(aq), aq_ref)
        assert np.array_equal(f16_bits(ad), ad_ref)
        _check_decode(to_np(y), orc, wq, wd, aq_ref, ad_ref)


def test_bitnet_6912x2560_full(qmm, orc):
    """BitNet GEMV m=1, K=2560, N=6912, seed 3: every output bit for bit."""
    n, k = 6912, 2560
    t, x, absmean = synthetic.bitnet_case(3, n, k, 1)
    tw = orc.pack_ternary(t)
    aq, scale, asum = orc.quantize_act_bitnet(x)
    y = to_np(qmm.bitnet_gemv(to_dev(tw.view(np.int32)), absmean, to_dev(aq), to_dev(scale),
                              to_dev(asum)))
    ref = orc.bitnet_gemv(tw, absmean, aq, scale, asum)
    assert np.array_equal(y.view(np.uint32), ref.view(np.uint32))


def test_bitnet_decode_step_6912x2560_full(qmm, orc):
    """The BitNet decode step as the benchmark times it (qmm_linear_bitnet with
    PDL, one kernel at m = 1), seed 3: codes, scale and sum, and every output,
    bit for bit."""
    n, k = 6912, 2560
    t, x, absmean = synthetic.bitnet_case(3, n, k, 1)
    tw = orc.pack_ternary(t)
    aq_ref, s_ref, asum_ref = orc.quantize_act_bitnet(x)
    y, aq, s, asum = qmm.linear_bitnet(to_dev(x), to_dev(tw.view(np.int32)), absmean, pdl=True,
                                       codes=True)
    assert np.array_equal(to_np(aq), aq_ref)
    assert np.array_equal(to_np(s).view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(to_np(asum), asum_ref)
    ref = orc.bitnet_gemv(tw, absmean, aq_ref, s_ref, asum_ref)
    assert np.array_equal(to_np(y).view(np.uint32), ref.view(np.uint32))


# token rows of the prefill outputs the oracle recomputes (first, tile edges, last)
PREFILL_ROWS = np.r_[0, 1, 127, 128, 255, 300, 383, 384, 510, 511]


def test_prefill_512x14336x4096_sampled_rows(qmm, orc):
    """Prefill GEMM m=512, K=4096, N=14336, seed 11, 1% outliers x20: the full
    product on the tensor cores; ten token rows (every weight row) compared
    bit for bit with the serial definition."""
    m, n, k = 512, 14336, 4096
    w, x = synthetic.q4_0_case(11, n, k, m, outlier_p=0.01)
    wq, wd = orc.quantize_q4_0(w)
    aq, ad = orc.quantize_q8_0(x)
    y = to_np(qmm.gemm_q4_0_q8_0(to_dev(wq), f16(wd), to_dev(aq), f16(ad)))
    r = PREFILL_ROWS
    ref = orc.gemm_q4_0_q8_0(wq, wd, np.ascontiguousarray(aq[r]), np.ascontiguousarray(ad[r]))
    assert np.array_equal(y[r].view(np.uint32), ref.view(np.uint32))


def test_prefill_repacked_weights_sampled_rows(qmm, orc):
    """The prefill shape on weights repacked at load time on the GPU: the
    repacked tiles equal the oracle's, and the sampled rows the serial
    definition, bit for bit."""
    m, n, k = 512, 14336, 4096
    w, x = synthetic.q4_0_case(11, n, k, m, outlier_p=0.01)
    wq, wd = orc.quantize_q4_0(w)
    aq, ad = orc.quantize_q8_0(x)
    wr = qmm.repack_q4_0_gemm(to_dev(wq))
    assert np.array_equal(to_np(wr), orc.repack_q4_0_gemm(wq))
    y = to_np(qmm.gemm_q4_0_q8_0_repacked(wr, f16(wd), to_dev(aq), f16(ad)))
    r = PREFILL_ROWS
    ref = orc.gemm_q4_0_q8_0(wq, wd, np.ascontiguousarray(aq[r]), np.ascontiguousarray(ad[r]))
    assert np.array_equal(y[r].view(np.uint32), ref.view(np.uint32))


def test_prefill_q8_0_weights_sampled_rows(qmm, orc):
    """The prefill shape with Q8_0 weights (the widened row), as timed."""
    m, n, k = 512, 14336, 4096
    w, x = synthetic.q4_0_case(11, n, k, m, outlier_p=0.01)
    w8, wd = orc.quantize_q8_0(w)
    aq, ad = orc.quantize_q8_0(x)
    y = to_np(qmm.gemm_q8_0_q8_0(to_dev(w8), f16(wd), to_dev(aq), f16(ad)))
    r = PREFILL_ROWS
    ref = orc.gemm_q8_0_q8_0(w8, wd, np.ascontiguousarray(aq[r]), np.ascontiguousarray(ad[r]))
    assert np.array_equal(y[r].view(np.uint32), ref.view(np.uint32))


def test_vocab_128256x4096(qmm, orc):
    """Vocabulary projection K=4096, N=128256, seed 13, for m = 1, 8, 16, 32,
    64, 128 as the benchmark runs them: the m=1 GEMV on every output; for m=8
    and 16 the GEMV and the GEMM (the few-token product), for m=32 and 64 the
    few-token product and for m=128 the tcgen05 GEMM, on sampled weight rows
    (ends of the range and of 128-row tiles)."""
    n, k = 128256, 4096
    w, x = synthetic.q4_0_case(13, n, k, 128)
    wq, wd = orc.quantize_q4_0(w)
    del w
    aq, ad = orc.quantize_q8_0(x)
    dwq, dwd = to_dev(wq), f16(wd)
    # m = 1: every output
    y1 = to_np(qmm.gemv_q4_0_q8_0(dwq, dwd, to_dev(aq[:1]), f16(ad[:1]), split_k=1))
    _check_decode(y1, orc, wq, wd, np.ascontiguousarray(aq[:1]), np.ascontiguousarray(ad[:1]))
    cols = np.r_[0:130, 64000:64130, n - 130:n]
    wqs, wds = np.ascontiguousarray(wq[cols]), np.ascontiguousarray(wd[cols])
    for m in (8, 16, 32, 64, 128):
        a, d = np.ascontiguousarray(aq[:m]), np.ascontiguousarray(ad[:m])
        ref = orc.gemm_q4_0_q8_0(wqs, wds, a, d)
        y_gemm = to_np(qmm.gemm_q4_0_q8_0(dwq, dwd, to_dev(a), f16(d)))
        assert np.array_equal(y_gemm[:, cols].view(np.uint32), ref.view(np.uint32))
        if m <= 16:
            y_gemv = to_np(qmm.gemv_q4_0_q8_0(dwq, dwd, to_dev(a), f16(d), split_k=1))
            absterms = orc.gemm_q4_0_q8_0_absterms(wqs, wds, a, d)
            ok, worst, maxrel = rel_gate(y_gemv[:, cols], ref, absterms)
            assert ok, (m, worst, maxrel)


def test_vocab_q8_0_weights_few_tokens(qmm, orc):
    """The vocabulary projection with Q8_0 weights (K=4096, N=128256, seed
    13) for m = 8 and 16, the few-token product as timed, on sampled weight
    rows (ends of the range and of 128-row sets), bit for bit."""
    n, k = 128256, 4096
    w, x = synthetic.q4_0_case(13, n, k, 16)
    w8, wd = orc.quantize_q8_0(w)
    del w
    aq, ad = orc.quantize_q8_0(x)
    dw8, dwd = to_dev(w8), f16(wd)
    cols = np.r_[0:130, 64000:64130, n - 130:n]
    w8s, wds = np.ascontiguousarray(w8[cols]), np.ascontiguousarray(wd[cols])
    for m in (8, 16):
        a, d = np.ascontiguousarray(aq[:m]), np.ascontiguousarray(ad[:m])
        y = to_np(qmm.gemm_q8_0_q8_0(dw8, dwd, to_dev(a), f16(d)))
        ref = orc.gemm_q8_0_q8_0(w8s, wds, a, d)
        assert np.array_equal(y[:, cols].view(np.uint32), ref.view(np.uint32))
