"""GPU parity: the CUDA library against the CPU oracle, element by element.

Integer results (quantized codes, fp16 scale bits, per-block sums, ternary
words, BitNet dots and BitNet outputs) must match bit for bit.  Q4_0 x Q8_0
f32 outputs must pass the gate of conftest.rel_gate: each output within
1e-5 * sum_b |sumi * dw * da| of the oracle, and max|diff| / max|y| <= 1e-5.
Shapes straddle the kernels' tiles (32-block lanes, 16-row CTAs, 128-row and
16..128-token tensor-core tiles) with ragged tails, plus the degenerate cases
(one row, one block, all-zero blocks, large outliers)."""
import ctypes

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


def f16_bits(t):
    """fp16 device tensor -> uint16 bit patterns on the host."""
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def adversarial_x(seed, m, k):
    w, x = synthetic.q4_0_case(seed, 1, k, m, outlier_p=0.02)
    x = x.copy()
    if m > 1:
        x[1, :QK] = 0.0                      # an all-zero block
    if m > 2:
        x[2, 5] = 1e4                        # an outlier
    if k > QK:
        x[0, QK:2 * QK] = np.float32(1e-30)  # scale far below fp16 range
    return x


def q4_case(orc, seed, m, n, k):
    """Oracle-quantized operands (weights and activations) for a parity case."""
    w, x = synthetic.q4_0_case(seed, n, k, m)
    wq, wd = orc.quantize_q4_0(w)
    aq, ad = orc.quantize_q8_0(x)
    return wq, wd, aq, ad


# ---------------------------------------------------------------------------
# quantizers

@pytest.mark.parametrize("m,k", [(1, 32), (3, 64), (17, 4064), (2, 4096), (1, 11008)])
def test_quantize_act_q8_0_bit_exact(qmm, orc, m, k):
    x = adversarial_x(10 + m, m, k)
    aq_ref, ad_ref = orc.quantize_q8_0(x)
    aq, ad = qmm.quantize_act_q8_0(to_dev(x))
    assert np.array_equal(to_np(aq), aq_ref)
    assert np.array_equal(f16_bits(ad), ad_ref)


@pytest.mark.parametrize("n,k", [(1, 32), (7, 96), (129, 4096)])
def test_quantize_weight_q4_0_bit_exact(qmm, orc, n, k):
    w, _ = synthetic.q4_0_case(20 + n, n, k, 1)
    w = w.copy()
    w[0, :QK] = 0.0                    # zero block: d = -0, all nibbles 8
    if n > 1:
        w[1, 3], w[1, 9] = 0.5, -0.5   # tie on |w|: the first index wins
    wq_ref, wd_ref = orc.quantize_q4_0(w)
    wq, wd = qmm.quantize_weight_q4_0(to_dev(w))
    assert np.array_equal(to_np(wq), wq_ref)
    assert np.array_equal(f16_bits(wd), wd_ref)


# ---------------------------------------------------------------------------
# GEMV

GEMV_SHAPES = [(1, 1, 32), (1, 31, 64), (1, 33, 4064), (1, 129, 4096), (2, 127, 4096),
               (3, 32, 96), (4, 128, 4096), (7, 65, 1024), (8, 17, 4096), (15, 33, 512),
               (16, 129, 4096), (1, 4097, 256),
               # one token: the staged form with 8-row CTAs (many rows, ragged
               # last CTA), the largest staged slice (k = 32768), and past it
               # the per-warp form unless the reduction is split
               (1, 16384 + 5, 256), (1, 9, 32768), (1, 40, 32768 + 64)]


@pytest.mark.parametrize("m,n,k", GEMV_SHAPES)
def test_gemv_block_sums_bit_exact(qmm, orc, m, n, k):
    wq, wd, aq, ad = q4_case(orc, 1000 + m * 7 + n, m, n, k)
    ref = orc.block_sums(wq, aq)
    got = qmm.debug_block_sums(0, to_dev(wq), to_dev(aq))
    assert np.array_equal(to_np(got), ref)


@pytest.mark.parametrize("m,n,k", GEMV_SHAPES)
@pytest.mark.parametrize("split", [1, 0, 3])
def test_gemv_matches_oracle(qmm, orc, m, n, k, split):
    if split > k // QK:
        pytest.skip("more slices than blocks")
    wq, wd, aq, ad = q4_case(orc, 2000 + m * 7 + n, m, n, k)
    y_ref = orc.gemm_q4_0_q8_0(wq, wd, aq, ad)
    absterms = orc.gemm_q4_0_q8_0_absterms(wq, wd, aq, ad)
    y = qmm.gemv_q4_0_q8_0(to_dev(wq), to_dev(wd.view(np.float16)), to_dev(aq),
                           to_dev(ad.view(np.float16)), split_k=split)
    ok, worst, maxrel = rel_gate(to_np(y), y_ref, absterms)
    assert ok, (worst, maxrel)


# ---------------------------------------------------------------------------
# tensor-core GEMM

GEMM_SHAPES = [(1, 1, 32), (1, 128, 64), (16, 129, 96), (17, 127, 4096), (33, 300, 256),
               (64, 128, 4064), (128, 256, 4096), (129, 130, 512), (200, 520, 1024),
               (512, 384, 4096)]


@pytest.mark.parametrize("m,n,k", GEMM_SHAPES)
def test_gemm_block_sums_bit_exact(qmm, orc, m, n, k):
    wq, wd, aq, ad = q4_case(orc, 3000 + m + n, m, n, k)
    ref = orc.block_sums(wq, aq)
    got = qmm.debug_block_sums(1, to_dev(wq), to_dev(aq))
    assert np.array_equal(to_np(got), ref)


@pytest.mark.parametrize("m,n,k", GEMM_SHAPES)
def test_gemm_matches_oracle(qmm, orc, m, n, k):
    wq, wd, aq, ad = q4_case(orc, 4000 + m + n, m, n, k)
    y_ref = orc.gemm_q4_0_q8_0(wq, wd, aq, ad)
    absterms = orc.gemm_q4_0_q8_0_absterms(wq, wd, aq, ad)
    y = to_np(qmm.gemm_q4_0_q8_0(to_dev(wq), to_dev(wd.view(np.float16)), to_dev(aq),
                                 to_dev(ad.view(np.float16))))
    ok, worst, maxrel = rel_gate(y, y_ref, absterms)
    assert ok, (worst, maxrel)


@pytest.mark.parametrize("m,n,k", [(5, 130, 4096), (129, 257, 1024)])
def test_gemm_is_bit_identical_to_serial_order(qmm, orc, m, n, k):
    """Each GEMM output accumulates fma(sumi, dw*da, acc) over blocks in
    ascending order, the oracle's order, so the f32 bits agree exactly."""
    wq, wd, aq, ad = q4_case(orc, 5000 + m, m, n, k)
    y_ref = orc.gemm_q4_0_q8_0(wq, wd, aq, ad)
    y = to_np(qmm.gemm_q4_0_q8_0(to_dev(wq), to_dev(wd.view(np.float16)), to_dev(aq),
                                 to_dev(ad.view(np.float16))))
    assert np.array_equal(y.view(np.uint32), y_ref.view(np.uint32))


# More tiles than CTAs fit on the GPU at once (152 SMs; one CTA per SM at
# BN >= 64, two at BN <= 32), odd block counts, ragged row and token tiles.
@pytest.mark.parametrize("m,n,k", [(40, 128 * 310 + 5, 32 * 33), (16, 128 * 330 + 77, 32 * 5),
                                   (130, 128 * 80 + 3, 32 * 9)])
def test_gemm_more_tiles_than_resident_ctas(qmm, orc, m, n, k):
    """y on sampled weight rows (tile edges and the last rows) and, where
    small enough, every block sum, bit for bit."""
    wq, wd, aq, ad = q4_case(orc, 5600 + m, m, n, k)
    dwq, dwd = to_dev(wq), to_dev(wd.view(np.float16))
    y = to_np(qmm.gemm_q4_0_q8_0(dwq, dwd, to_dev(aq), to_dev(ad.view(np.float16))))
    rows = np.unique(np.r_[0:3, 125:131, 128 * 152 - 2:128 * 152 + 2, 128 * 305:128 * 305 + 3,
                           n - 4:n].clip(0, n - 1))
    ref = orc.gemm_q4_0_q8_0(np.ascontiguousarray(wq[rows]), np.ascontiguousarray(wd[rows]), aq, ad)
    assert np.array_equal(y[:, rows].view(np.uint32), ref.view(np.uint32))
    if m * n * (k // 32) <= 64 * 1024 * 1024:
        sumi = to_np(qmm.debug_block_sums(1, dwq, to_dev(aq)))
        assert np.array_equal(sumi, orc.block_sums(wq, aq))


# The few-token product (m <= 32, k a multiple of 256: warp-level MMAs with
# register accumulators, persistent CTAs over 128-row sets): one and two
# 16-token tiles, ragged row sets, more row sets than SMs, long reductions,
# and more row sets than resident CTAs (two or three per SM), so that CTAs
# take further sets from the counter, with one stage per set (k = 256).
GEMM_SMALL_SHAPES = [(1, 1, 256), (8, 129, 512), (16, 128, 4096), (16, 257, 2048),
                     (17, 300, 768), (31, 1000, 1024), (32, 128 * 152 * 2 + 77, 256),
                     (20, 65, 11008), (8, 128 * 700 + 3, 256), (16, 128 * 1000 + 5, 512),
                     (29, 128 * 600 + 127, 256),
                     # three and four 16-token tiles (Q4_0 weights; Q8_0 takes the
                     # tcgen05 product from 33 tokens on)
                     (33, 300, 1024), (48, 1000, 512), (64, 257, 4096), (40, 129, 11008),
                     (64, 128 * 600 + 5, 256)]


@pytest.mark.parametrize("m,n,k", GEMM_SMALL_SHAPES)
def test_gemm_small_m_block_sums_and_y_bit_exact(qmm, orc, m, n, k):
    wq, wd, aq, ad = q4_case(orc, 8100 + m + n, m, n, k)
    dwq, daq = to_dev(wq), to_dev(aq)
    sumi = to_np(qmm.debug_block_sums(1, dwq, daq))
    assert np.array_equal(sumi, orc.block_sums(wq, aq))
    y = to_np(qmm.gemm_q4_0_q8_0(dwq, to_dev(wd.view(np.float16)), daq, to_dev(ad.view(np.float16))))
    assert np.array_equal(y.view(np.uint32), orc.gemm_q4_0_q8_0(wq, wd, aq, ad).view(np.uint32))


def test_gemm_small_m_adversarial_activations_bit_exact(qmm, orc):
    m, n, k = 16, 200, 1024
    wq, wd, _, _ = q4_case(orc, 8200, m, n, k)
    x = adversarial_x(8201, m, k)
    aq, ad = orc.quantize_q8_0(x)
    y = to_np(qmm.gemm_q4_0_q8_0(to_dev(wq), to_dev(wd.view(np.float16)), to_dev(aq),
                                 to_dev(ad.view(np.float16))))
    assert np.array_equal(y.view(np.uint32), orc.gemm_q4_0_q8_0(wq, wd, aq, ad).view(np.uint32))


def test_gemm_small_m_wait_timeout_reports_and_device_stays_usable(qmm, orc):
    """The few-token product with its stages never armed: every bounded wait
    runs out, QMM_ERR_TIMEOUT is recorded, and the next call is exact."""
    import torch
    wq, wd, aq, ad = q4_case(orc, 8300, 16, 300, 1024)
    args = (to_dev(wq), to_dev(wd.view(np.float16)), to_dev(aq), to_dev(ad.view(np.float16)))
    assert qmm.check_device_error() == 0
    try:
        qmm.set_wait_limit(2000)
        qmm.withhold_gemm_loads(True)
        qmm.gemm_q4_0_q8_0(*args)
        torch.cuda.synchronize()
        status = qmm.check_device_error()
    finally:
        qmm.withhold_gemm_loads(False)
        qmm.set_wait_limit(0)
    assert status == 7
    y = to_np(qmm.gemm_q4_0_q8_0(*args))
    torch.cuda.synchronize()
    assert qmm.check_device_error() == 0
    assert np.array_equal(y.view(np.uint32), orc.gemm_q4_0_q8_0(wq, wd, aq, ad).view(np.uint32))


@pytest.mark.parametrize("fmt", ["q4", "q8"])
def test_gemv_auto_runs_the_few_token_product_from_three_tokens(qmm, orc, fmt):
    """split_k = 0 with m >= 3 and k % 256 == 0 hands the GEMV call to the
    few-token product (the serial definition, bit for bit); m = 2, an
    explicit split_k = 1, or no workspace keep the GEMV kernels (within the
    f32 gate)."""
    import torch
    n, k = 300, 1024
    for m in (2, 3, 8, 16):
        if fmt == "q4":
            w, wd, aq, ad = q4_case(orc, 8700 + m, m, n, k)
            ref = orc.gemm_q4_0_q8_0(w, wd, aq, ad)
            absterms = orc.gemm_q4_0_q8_0_absterms(w, wd, aq, ad)
            gemv, entry = qmm.gemv_q4_0_q8_0, "qmm_gemv_q4_0_q8_0"
        else:
            w, wd, aq, ad = q8_case(orc, 8700 + m, m, n, k)
            ref = orc.gemm_q8_0_q8_0(w, wd, aq, ad)
            _, absterms = orc.gemm_q8_0_q8_0_f64(w, wd, aq, ad)
            gemv, entry = qmm.gemv_q8_0_q8_0, "qmm_gemv_q8_0_q8_0"
        args = (to_dev(w), to_dev(wd.view(np.float16)), to_dev(aq), to_dev(ad.view(np.float16)))
        y_auto = to_np(gemv(*args))
        if m >= 3:
            assert np.array_equal(y_auto.view(np.uint32), ref.view(np.uint32)), m
        else:
            ok, worst, maxrel = rel_gate(y_auto, ref, absterms)
            assert ok, (m, worst, maxrel)
        ok, worst, maxrel = rel_gate(to_np(gemv(*args, split_k=1)), ref, absterms)
        assert ok, (m, worst, maxrel)
        # no workspace at all: the GEMV kernels (this shape needs no split)
        y = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
        fn = getattr(qmm.load(), entry)
        st = fn(args[0].data_ptr(), args[1].data_ptr(), args[2].data_ptr(), args[3].data_ptr(),
                y.data_ptr(), m, n, k, 0, None, 0, torch.cuda.current_stream().cuda_stream)
        assert st == 0
        ok, worst, maxrel = rel_gate(to_np(y), ref, absterms)
        assert ok, (m, worst, maxrel)


def test_gemm_and_gemv_agree_with_adversarial_activations(qmm, orc):
    m, n, k = 9, 200, 4096
    w, _ = synthetic.q4_0_case(61, n, k, 1)
    x = adversarial_x(62, m, k)
    wq, wd = orc.quantize_q4_0(w)
    aq, ad = orc.quantize_q8_0(x)
    y_ref = orc.gemm_q4_0_q8_0(wq, wd, aq, ad)
    absterms = orc.gemm_q4_0_q8_0_absterms(wq, wd, aq, ad)
    args = (to_dev(wq), to_dev(wd.view(np.float16)), to_dev(aq), to_dev(ad.view(np.float16)))
    for y in (qmm.gemv_q4_0_q8_0(*args), qmm.gemm_q4_0_q8_0(*args)):
        ok, worst, maxrel = rel_gate(to_np(y), y_ref, absterms)
        assert ok, (worst, maxrel)


# ---------------------------------------------------------------------------
# BitNet ternary

BITNET_SHAPES = [(1, 1, 16), (1, 33, 48), (1, 6912, 2560), (2, 129, 2560), (3, 65, 160),
                 (5, 100, 4096), (16, 31, 1024), (1, 40, 2576),
                 # one token with k % 64 == 0 and k <= 32768: the activation row
                 # staged once per CTA (a ragged last CTA of 8 rows, the
                 # largest k); past 32768 the per-warp form
                 (1, 7, 64), (1, 300, 11008), (1, 1000, 32768), (1, 9, 32832)]


@pytest.mark.parametrize("m,n,k", BITNET_SHAPES)
def test_bitnet_path_bit_exact(qmm, orc, m, n, k):
    t, x, absmean = synthetic.bitnet_case(70 + m + n, n, k, m)
    x = x.copy()
    if m > 1:
        x[1] = 0.0  # zero row: scale 0, y 0
    tw_ref = orc.pack_ternary(t)
    aq_ref, s_ref, asum_ref = orc.quantize_act_bitnet(x)
    tw = qmm.pack_ternary(to_dev(t))
    assert np.array_equal(to_np(tw).view(np.uint32), tw_ref)
    aq, s, asum = qmm.quantize_act_bitnet(to_dev(x))
    assert np.array_equal(to_np(aq), aq_ref)
    assert np.array_equal(to_np(s).view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(to_np(asum), asum_ref)
    dot = qmm.debug_bitnet_dot(tw, aq, asum)
    assert np.array_equal(to_np(dot), orc.bitnet_dot(tw_ref, aq_ref, asum_ref))
    y = qmm.bitnet_gemv(tw, absmean, aq, s, asum)
    y_ref = orc.bitnet_gemv(tw_ref, absmean, aq_ref, s_ref, asum_ref)
    assert np.array_equal(to_np(y).view(np.uint32), y_ref.view(np.uint32))


@pytest.mark.parametrize("m,n,k", [(1, 6912, 2560), (1, 33, 48), (3, 65, 160), (16, 31, 1024),
                                   (2, 129, 2576)])
@pytest.mark.parametrize("pdl", [False, True])
def test_linear_bitnet_bit_exact(qmm, orc, m, n, k, pdl):
    """The decode step in one call: codes, scale, sum and y bit for bit the
    oracle's, with and without programmatic dependent launch, on rows read
    with a row stride larger than k."""
    import torch
    t, x, absmean = synthetic.bitnet_case(170 + m + n, n, k, m)
    x = x.copy()
    if m > 1:
        x[1] = 0.0  # zero row: scale 0, y 0
    tw_ref = orc.pack_ternary(t)
    aq_ref, s_ref, asum_ref = orc.quantize_act_bitnet(x)
    tw = to_dev(tw_ref.view(np.int32))
    xbuf = torch.full((m, k + 48), 3.0e3, dtype=torch.float32, device="cuda")
    xbuf[:, :k] = to_dev(x)
    aq = torch.empty((m, k), dtype=torch.int8, device="cuda")
    sc = torch.empty((m,), dtype=torch.float32, device="cuda")
    asum = torch.empty((m,), dtype=torch.int32, device="cuda")
    y = torch.empty((m, n), dtype=torch.float32, device="cuda")
    st = qmm.load().qmm_linear_bitnet(tw.data_ptr(), float(absmean), xbuf.data_ptr(), k + 48,
                                      aq.data_ptr(), sc.data_ptr(), asum.data_ptr(), y.data_ptr(),
                                      m, n, k, 1 if pdl else 0,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert np.array_equal(to_np(aq), aq_ref)
    assert np.array_equal(to_np(sc).view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(to_np(asum), asum_ref)
    y_ref = orc.bitnet_gemv(tw_ref, absmean, aq_ref, s_ref, asum_ref)
    assert np.array_equal(to_np(y).view(np.uint32), y_ref.view(np.uint32))


@pytest.mark.parametrize("pdl", [False, True])
def test_linear_bitnet_one_token_unaligned_row_bit_exact(qmm, orc, pdl):
    """One token whose f32 row is not 16-byte aligned: the step runs as the
    quantizer and then the one-token GEMV (with programmatic dependent
    launch when asked), still bit for bit the oracle's."""
    import torch
    n, k = 1000, 2560
    t, x, absmean = synthetic.bitnet_case(175, n, k, 1)
    tw_ref = orc.pack_ternary(t)
    aq_ref, s_ref, asum_ref = orc.quantize_act_bitnet(x)
    tw = to_dev(tw_ref.view(np.int32))
    xbuf = torch.full((k + 4,), 3.0e3, dtype=torch.float32, device="cuda")
    xbuf[1:k + 1] = to_dev(x[0])
    aq = torch.empty((1, k), dtype=torch.int8, device="cuda")
    sc = torch.empty((1,), dtype=torch.float32, device="cuda")
    asum = torch.empty((1,), dtype=torch.int32, device="cuda")
    y = torch.full((1, n), float("nan"), dtype=torch.float32, device="cuda")
    st = qmm.load().qmm_linear_bitnet(tw.data_ptr(), float(absmean), xbuf.data_ptr() + 4, k,
                                      aq.data_ptr(), sc.data_ptr(), asum.data_ptr(), y.data_ptr(),
                                      1, n, k, 1 if pdl else 0,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert np.array_equal(to_np(aq), aq_ref)
    y_ref = orc.bitnet_gemv(tw_ref, absmean, aq_ref, s_ref, asum_ref)
    assert np.array_equal(to_np(y).view(np.uint32), y_ref.view(np.uint32))


@pytest.mark.parametrize("m", [1, 4])
def test_linear_bitnet_pdl_chain_reads_the_previous_layer_output(qmm, orc, m):
    """BitNet layers chained on one stream, each consuming the previous
    layer's y and sharing one code buffer: with programmatic dependent
    launch every kernel still reads its inputs after its predecessor, so the
    chain gives the same bits as without, and each layer's output is the
    oracle's on that layer's actual input."""
    import torch
    dims = [2560, 6912, 2560, 2560]
    layers = []
    for j in range(len(dims) - 1):
        t, _, absmean = synthetic.bitnet_case(6400 + j, dims[j + 1], dims[j], 1)
        tw_ref = orc.pack_ternary(t)
        layers.append((tw_ref, absmean, to_dev(tw_ref.view(np.int32))))
    _, x0, _ = synthetic.bitnet_case(6499, 1, dims[0], m)
    aq_flat = torch.empty(m * max(dims), dtype=torch.int8, device="cuda")
    outs = {}
    for pdl in (False, True):
        hs = [to_dev(x0)]
        for j, (_, absmean, tw_d) in enumerate(layers):
            aq_j = aq_flat[: m * dims[j]].view(m, dims[j])
            hs.append(qmm.linear_bitnet(hs[-1], tw_d, absmean, pdl=pdl, aq=aq_j))
        torch.cuda.synchronize()
        outs[pdl] = [to_np(h) for h in hs]
    for a, b in zip(outs[False], outs[True]):
        assert np.isfinite(a).all()
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    for j, (tw_ref, absmean, _) in enumerate(layers):
        aq_r, s_r, asum_r = orc.quantize_act_bitnet(outs[True][j])
        y_ref = orc.bitnet_gemv(tw_ref, absmean, aq_r, s_r, asum_r)
        assert np.array_equal(outs[True][j + 1].view(np.uint32), y_ref.view(np.uint32)), j


# ---------------------------------------------------------------------------
# BitNet prefill on the tensor cores

# ---------------------------------------------------------------------------
# load-time repack for the GEMM

@pytest.mark.parametrize("n,k", [(1, 32), (3, 96), (130, 64), (257, 4096), (1000, 11008)])
def test_repack_q4_0_gemm_bit_exact(qmm, orc, n, k):
    rng = np.random.default_rng(n + k)
    wq = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    assert np.array_equal(to_np(qmm.repack_q4_0_gemm(to_dev(wq))), orc.repack_q4_0_gemm(wq))


@pytest.mark.parametrize("m,n,k", GEMM_SHAPES)
def test_gemm_on_repacked_weights_is_identical(qmm, orc, m, n, k):
    """The repacked tiles give the planes' GEMM bit for bit, and its block
    sums match the oracle's."""
    wq, wd, aq, ad = q4_case(orc, 8500 + m + n, m, n, k)
    wr = to_dev(orc.repack_q4_0_gemm(wq))
    args = (to_dev(wd.view(np.float16)), to_dev(aq), to_dev(ad.view(np.float16)))
    y_planes = to_np(qmm.gemm_q4_0_q8_0(to_dev(wq), *args))
    y_rep = to_np(qmm.gemm_q4_0_q8_0_repacked(wr, *args))
    assert np.array_equal(y_rep.view(np.uint32), y_planes.view(np.uint32))
    sumi = to_np(qmm.debug_block_sums(2, wr, to_dev(aq), n=n))
    assert np.array_equal(sumi, orc.block_sums(wq, aq))


# ---------------------------------------------------------------------------
# Q8_0 weights x Q8_0 activations (GEMV and tensor-core GEMM)

def q8_case(orc, seed, m, n, k):
    """Oracle-quantized Q8_0 weights (the activation recipe) and activations."""
    w, x = synthetic.q4_0_case(seed, n, k, m)
    w = w.copy()
    w[0, :QK] = 0.0  # an all-zero weight block: d = 0, codes 0
    w8, wd = orc.quantize_q8_0(w)
    aq, ad = orc.quantize_q8_0(x)
    return w8, wd, aq, ad


def test_quantize_weight_q8_0_is_the_activation_recipe(qmm, orc):
    w, _ = synthetic.q4_0_case(31, 37, 4096, 1)
    w8_ref, wd_ref = orc.quantize_q8_0(w)
    w8, wd = qmm.quantize_weight_q8_0(to_dev(w))
    assert np.array_equal(to_np(w8), w8_ref)
    assert np.array_equal(f16_bits(wd), wd_ref)


@pytest.mark.parametrize("m,n,k", GEMV_SHAPES)
def test_gemv_q8_0_block_sums_bit_exact(qmm, orc, m, n, k):
    w8, wd, aq, ad = q8_case(orc, 6000 + m * 7 + n, m, n, k)
    ref = orc.block_sums_q8_0(w8, aq)
    got = qmm.debug_block_sums_q8(0, to_dev(w8), to_dev(aq))
    assert np.array_equal(to_np(got), ref)


@pytest.mark.parametrize("m,n,k", GEMV_SHAPES)
@pytest.mark.parametrize("split", [1, 0, 3])
def test_gemv_q8_0_matches_oracle(qmm, orc, m, n, k, split):
    if split > k // QK:
        pytest.skip("more slices than blocks")
    w8, wd, aq, ad = q8_case(orc, 6500 + m * 7 + n, m, n, k)
    y_ref = orc.gemm_q8_0_q8_0(w8, wd, aq, ad)
    _, absterms = orc.gemm_q8_0_q8_0_f64(w8, wd, aq, ad)
    y = qmm.gemv_q8_0_q8_0(to_dev(w8), to_dev(wd.view(np.float16)), to_dev(aq),
                           to_dev(ad.view(np.float16)), split_k=split)
    ok, worst, maxrel = rel_gate(to_np(y), y_ref, absterms)
    assert ok, (worst, maxrel)


@pytest.mark.parametrize("m,n,k", GEMM_SHAPES)
def test_gemm_q8_0_block_sums_bit_exact(qmm, orc, m, n, k):
    w8, wd, aq, ad = q8_case(orc, 7000 + m + n, m, n, k)
    ref = orc.block_sums_q8_0(w8, aq)
    got = qmm.debug_block_sums_q8(1, to_dev(w8), to_dev(aq))
    assert np.array_equal(to_np(got), ref)


@pytest.mark.parametrize("m,n,k", GEMM_SHAPES)
def test_gemm_q8_0_is_bit_identical_to_serial_order(qmm, orc, m, n, k):
    """The Q8_0-weight GEMM accumulates fma(sumi, dw*da, acc) over blocks in
    ascending order, the oracle's order: identical f32 bits (so the 1e-5
    gate holds a fortiori)."""
    w8, wd, aq, ad = q8_case(orc, 7500 + m + n, m, n, k)
    y_ref = orc.gemm_q8_0_q8_0(w8, wd, aq, ad)
    y = to_np(qmm.gemm_q8_0_q8_0(to_dev(w8), to_dev(wd.view(np.float16)), to_dev(aq),
                                 to_dev(ad.view(np.float16))))
    assert np.array_equal(y.view(np.uint32), y_ref.view(np.uint32))


# The few-token product with Q8_0 weights (m <= 32, k % 256 == 0): each code
# read as the fp16 value 1152 + code, two 128-byte swizzled boxes per stage.
@pytest.mark.parametrize("m,n,k", GEMM_SMALL_SHAPES)
def test_gemm_small_m_q8_0_block_sums_and_y_bit_exact(qmm, orc, m, n, k):
    w8, wd, aq, ad = q8_case(orc, 8400 + m + n, m, n, k)
    dw8, daq = to_dev(w8), to_dev(aq)
    sumi = to_np(qmm.debug_block_sums_q8(1, dw8, daq))
    assert np.array_equal(sumi, orc.block_sums_q8_0(w8, aq))
    y = to_np(qmm.gemm_q8_0_q8_0(dw8, to_dev(wd.view(np.float16)), daq, to_dev(ad.view(np.float16))))
    assert np.array_equal(y.view(np.uint32), orc.gemm_q8_0_q8_0(w8, wd, aq, ad).view(np.uint32))


def test_gemm_small_m_q8_0_extreme_codes_bit_exact(qmm, orc):
    """Codes at the ends of the int8 range, whole blocks of them, so that a
    block's MMA partial sums reach their largest magnitude (32 x (1152 + 127)
    x 127 = 5.2e6, still an integer an f32 holds): block sums and y bit for
    bit."""
    m, n, k = 16, 136, 2048
    rng = np.random.default_rng(8500)
    w8 = rng.choice(np.array([-128, -127, 127], dtype=np.int8), size=(n, k))
    aq = rng.choice(np.array([-127, 127], dtype=np.int8), size=(m, k))
    w8[:8, :] = 127                   # whole rows of the largest code ...
    aq[:4, :] = 127                   # ... against whole tokens of +127
    w8[8:16, :] = -128                # and of the smallest code
    aq[4:8, :] = -127
    wd = (rng.random((n, k // QK)) * 0.01).astype(np.float16).view(np.uint16)
    ad = (rng.random((m, k // QK)) * 0.05).astype(np.float16).view(np.uint16)
    dw8, daq = to_dev(w8), to_dev(aq)
    sumi = to_np(qmm.debug_block_sums_q8(1, dw8, daq))
    ref = orc.block_sums_q8_0(w8, aq)
    assert ref.max() == 32 * 128 * 127 and ref.min() == -32 * 128 * 127
    assert np.array_equal(sumi, ref)
    y = to_np(qmm.gemm_q8_0_q8_0(dw8, to_dev(wd.view(np.float16)), daq, to_dev(ad.view(np.float16))))
    assert np.array_equal(y.view(np.uint32), orc.gemm_q8_0_q8_0(w8, wd, aq, ad).view(np.uint32))


def test_gemm_small_m_q8_0_wait_timeout_reports_and_device_stays_usable(qmm, orc):
    import torch
    w8, wd, aq, ad = q8_case(orc, 8600, 16, 300, 1024)
    args = (to_dev(w8), to_dev(wd.view(np.float16)), to_dev(aq), to_dev(ad.view(np.float16)))
    assert qmm.check_device_error() == 0
    try:
        qmm.set_wait_limit(2000)
        qmm.withhold_gemm_loads(True)
        qmm.gemm_q8_0_q8_0(*args)
        torch.cuda.synchronize()
        status = qmm.check_device_error()
    finally:
        qmm.withhold_gemm_loads(False)
        qmm.set_wait_limit(0)
    assert status == 7
    y = to_np(qmm.gemm_q8_0_q8_0(*args))
    torch.cuda.synchronize()
    assert qmm.check_device_error() == 0
    assert np.array_equal(y.view(np.uint32), orc.gemm_q8_0_q8_0(w8, wd, aq, ad).view(np.uint32))


def test_gemm_and_gemv_q8_0_agree_with_adversarial_activations(qmm, orc):
    m, n, k = 9, 200, 4096
    w, _ = synthetic.q4_0_case(63, n, k, 1)
    x = adversarial_x(64, m, k)
    w8, wd = orc.quantize_q8_0(w)
    aq, ad = orc.quantize_q8_0(x)
    y_ref = orc.gemm_q8_0_q8_0(w8, wd, aq, ad)
    _, absterms = orc.gemm_q8_0_q8_0_f64(w8, wd, aq, ad)
    args = (to_dev(w8), to_dev(wd.view(np.float16)), to_dev(aq), to_dev(ad.view(np.float16)))
    y_gemm = to_np(qmm.gemm_q8_0_q8_0(*args))
    assert np.array_equal(y_gemm.view(np.uint32), y_ref.view(np.uint32))
    ok, worst, maxrel = rel_gate(to_np(qmm.gemv_q8_0_q8_0(*args)), y_ref, absterms)
    assert ok, (worst, maxrel)


BITNET_GEMM_SHAPES = [(1, 1, 64), (17, 130, 256), (100, 300, 2560), (256, 128, 512),
                      (300, 257, 1024), (600, 1000, 128)]


def _bitnet_operands(orc, seed, m, n, k):
    t, x, absmean = synthetic.bitnet_case(seed, n, k, m)
    x = x.copy()
    if m > 1:
        x[1] = 0.0  # zero row: scale 0, y 0
    tw = orc.pack_ternary(t)
    aq, scale, asum = orc.quantize_act_bitnet(x)
    return tw, absmean, aq, scale, asum


@pytest.mark.parametrize("m,n,k", BITNET_GEMM_SHAPES)
def test_bitnet_gemm_bit_exact(qmm, orc, m, n, k):
    """The tensor-core product gives the oracle's y bit for bit (and the
    GEMV's, where m allows it)."""
    tw, absmean, aq, scale, asum = _bitnet_operands(orc, 8000 + m + n, m, n, k)
    y = to_np(qmm.bitnet_gemm(to_dev(tw.view(np.int32)), absmean, to_dev(aq), to_dev(scale)))
    ref = orc.bitnet_gemv(tw, absmean, aq, scale, asum)
    assert np.array_equal(y.view(np.uint32), ref.view(np.uint32))
    if m <= 16:
        y2 = to_np(qmm.bitnet_gemv(to_dev(tw.view(np.int32)), absmean, to_dev(aq), to_dev(scale),
                                   to_dev(asum)))
        assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


def test_bitnet_gemm_scales_at_any_alignment(qmm, orc):
    """act_scale 4-byte but not 16-byte aligned (a view one element into a
    buffer): the epilogue then reads the scales one by one; same bits."""
    import torch
    m, n, k = 48, 130, 128
    tw, absmean, aq, scale, asum = _bitnet_operands(orc, 8300, m, n, k)
    buf = torch.zeros(m + 1, dtype=torch.float32, device="cuda")
    buf[1:] = to_dev(scale)
    y = to_np(qmm.bitnet_gemm(to_dev(tw.view(np.int32)), absmean, to_dev(aq), buf[1:]))
    ref = orc.bitnet_gemv(tw, absmean, aq, scale, asum)
    assert np.array_equal(y.view(np.uint32), ref.view(np.uint32))


def test_bitnet_gemm_division_over_wide_scales(qmm, orc):
    """The epilogue's scaling against the oracle's IEEE operations, bit for
    bit: activation rows scaled across 40 decades (act_scale from ~1e-19 to
    ~1e22), a zero row (scale 0), a zero weight row against an all-negative
    activation row (products of -0, which the accumulator sums to -0, while
    the integer dot is +0), and absmean of 2^40 and 2^-40 besides the drawn
    one."""
    m, n, k = 1024, 256, 64
    t, x, absmean = synthetic.bitnet_case(8200, n, k, m)
    rng = np.random.default_rng(8201)
    x = (x * (10.0 ** rng.uniform(-20.0, 20.0, size=(m, 1)))).astype(np.float32)
    x[3] = 0.0
    x[5] = -np.abs(x[5]) - 1.0
    t = t.copy()
    t[7] = 0  # weight value 0: code 1
    tw = orc.pack_ternary(t)
    aq, scale, asum = orc.quantize_act_bitnet(x)
    assert scale[scale > 0].min() < 1e-18 and scale.max() > 1e21
    for am in (absmean, np.float32(2.0 ** 40), np.float32(2.0 ** -40)):
        y = to_np(qmm.bitnet_gemm(to_dev(tw.view(np.int32)), float(am), to_dev(aq), to_dev(scale)))
        ref = orc.bitnet_gemv(tw, float(am), aq, scale, asum)
        assert np.array_equal(y.view(np.uint32), ref.view(np.uint32)), float(am)


def test_bitnet_gemm_prefill_size_sampled_rows(qmm, orc):
    """The benchmark shape (m=2048, N=6912, K=2560), checked against the
    oracle on a sample of weight rows."""
    m, n, k = 2048, 6912, 2560
    tw, absmean, aq, scale, asum = _bitnet_operands(orc, 8100, m, n, k)
    y = to_np(qmm.bitnet_gemm(to_dev(tw.view(np.int32)), absmean, to_dev(aq), to_dev(scale)))
    rows = np.r_[0:3, 127:130, 3400:3403, n - 3:n]
    ref = orc.bitnet_gemv(np.ascontiguousarray(tw[rows]), absmean, aq, scale, asum)
    assert np.array_equal(y[:, rows].view(np.uint32), ref.view(np.uint32))


# ---------------------------------------------------------------------------
# the two decode GEMV kernels (shared-memory streaming and register streaming)

def _misaligned_copy(t):
    """The same values at a 2-byte offset from a 16-byte boundary: the library
    then takes the register-streaming kernel."""
    import torch
    flat = torch.empty(t.numel() + 8, dtype=t.dtype, device=t.device)
    v = flat[1:1 + t.numel()].view(t.shape)
    v.copy_(t)
    assert v.data_ptr() % 16 == 2
    return v


@pytest.mark.parametrize("m,n,k", [(8, 300, 4096), (16, 129, 11008), (12, 77, 8192),
                                   (16, 40, 2048), (9, 16, 256), (8, 1, 4096),
                                   (10, 4099, 4096)])
def test_streaming_and_register_gemv_agree_bitwise(qmm, orc, m, n, k):
    wq, wd, aq, ad = q4_case(orc, 7000 + m + n, m, n, k)
    wq_d, wd_d = to_dev(wq), to_dev(wd.view(np.float16))
    aq_d, ad_d = to_dev(aq), to_dev(ad.view(np.float16))
    y_stream = to_np(qmm.gemv_q4_0_q8_0(wq_d, wd_d, aq_d, ad_d, split_k=1))
    y_reg = to_np(qmm.gemv_q4_0_q8_0(wq_d, _misaligned_copy(wd_d), aq_d, ad_d, split_k=1))
    assert np.array_equal(y_stream.view(np.uint32), y_reg.view(np.uint32))
    ok, worst, maxrel = rel_gate(y_stream, orc.gemm_q4_0_q8_0(wq, wd, aq, ad),
                                 orc.gemm_q4_0_q8_0_absterms(wq, wd, aq, ad))
    assert ok, (worst, maxrel)


def test_streaming_gemv_wait_timeout_reports_and_device_stays_usable(qmm, orc):
    """With the streaming GEMV's stages never armed, the consumers' bounded
    waits must run out, the kernel must record QMM_ERR_TIMEOUT and return;
    afterwards a normal call on the same context gives the usual result."""
    import torch
    wq, wd, aq, ad = q4_case(orc, 7100, 8, 256, 4096)
    args = (to_dev(wq), to_dev(wd.view(np.float16)), to_dev(aq), to_dev(ad.view(np.float16)))
    assert qmm.check_device_error() == 0
    try:
        qmm.set_wait_limit(200)
        qmm.withhold_gemv_loads(True)
        qmm.gemv_q4_0_q8_0(*args, split_k=1)
        torch.cuda.synchronize()
        status = qmm.check_device_error()
    finally:
        qmm.withhold_gemv_loads(False)
        qmm.set_wait_limit(0)
    assert status == 7
    y = to_np(qmm.gemv_q4_0_q8_0(*args, split_k=1))
    torch.cuda.synchronize()
    assert qmm.check_device_error() == 0
    ok, worst, maxrel = rel_gate(y, orc.gemm_q4_0_q8_0(wq, wd, aq, ad),
                                 orc.gemm_q4_0_q8_0_absterms(wq, wd, aq, ad))
    assert ok, (worst, maxrel)


# ---------------------------------------------------------------------------
# bounded waits

def test_gemm_wait_timeout_reports_and_device_stays_usable(qmm, orc):
    """With the GEMM's loads withheld no pipeline barrier can complete: every
    bounded wait must run out, the kernel must record QMM_ERR_TIMEOUT in the
    device error word, release TMEM and return; afterwards a normal call on
    the same context gives the exact result."""
    import torch
    wq, wd, aq, ad = q4_case(orc, 77, 40, 256, 2048)
    args = (to_dev(wq), to_dev(wd.view(np.float16)), to_dev(aq), to_dev(ad.view(np.float16)))
    assert qmm.check_device_error() == 0
    try:
        qmm.set_wait_limit(2000)
        qmm.withhold_gemm_loads(True)
        qmm.gemm_q4_0_q8_0(*args)
        torch.cuda.synchronize()
        status = qmm.check_device_error()
    finally:
        qmm.withhold_gemm_loads(False)
        qmm.set_wait_limit(0)
    assert status == 7
    y = to_np(qmm.gemm_q4_0_q8_0(*args))
    torch.cuda.synchronize()
    assert qmm.check_device_error() == 0
    y_ref = orc.gemm_q4_0_q8_0(wq, wd, aq, ad)
    assert np.array_equal(y.view(np.uint32), y_ref.view(np.uint32))


# ---------------------------------------------------------------------------
# decode linear layer: quantizer + GEMV in one call, optionally chained with
# programmatic dependent launch

LINEAR_SHAPES = [(1, 1, 32), (1, 129, 4096), (2, 300, 11008), (3, 65, 4064), (4, 33, 1024),
                 (5, 33, 1024), (8, 257, 4096), (16, 70, 2048), (1, 4096, 11008),
                 (1, 11008, 4096), (2, 17, 96), (4, 40, 16384), (3, 9, 19680)]


@pytest.mark.parametrize("m,n,k", LINEAR_SHAPES)
@pytest.mark.parametrize("pdl", [False, True])
def test_linear_matches_separate_calls_and_oracle(qmm, orc, m, n, k, pdl):
    """qmm_linear_q4_0 gives the oracle's codes bit for bit and the separate
    calls' y."""
    w, _ = synthetic.q4_0_case(6000 + m + n, n, k, 1)
    x = adversarial_x(6100 + m, m, k)
    wq, wd = orc.quantize_q4_0(w)
    aq_ref, ad_ref = orc.quantize_q8_0(x)
    wq_d, wd_d = to_dev(wq), to_dev(wd.view(np.float16))
    y, aq, ad = qmm.linear_q4_0(to_dev(x), wq_d, wd_d, pdl=pdl, codes=True)
    assert np.array_equal(to_np(aq), aq_ref)
    assert np.array_equal(f16_bits(ad), ad_ref)
    aq2, ad2 = qmm.quantize_act_q8_0(to_dev(x))
    y2 = qmm.gemv_q4_0_q8_0(wq_d, wd_d, aq2, ad2, split_k=1)
    assert np.array_equal(to_np(y).view(np.uint32), to_np(y2).view(np.uint32))
    ok, worst, maxrel = rel_gate(to_np(y), orc.gemm_q4_0_q8_0(wq, wd, aq_ref, ad_ref),
                                 orc.gemm_q4_0_q8_0_absterms(wq, wd, aq_ref, ad_ref))
    assert ok, (worst, maxrel)


# at m >= 8 the first set streams through shared memory; the second (k/32
# not a multiple of 8 in some problems) always streams through registers; at
# m = 1 the third (a row longer than 32768) takes the per-warp form, the
# others stage each CTA's activation row in shared memory
GROUP_SHAPE_SETS = {
    "streaming": [(129, 1024), (300, 2048), (1, 256), (4096, 1024), (40, 2048),
                  (1100, 512), (17, 512)],
    "register": [(129, 4096), (300, 11008), (65, 4064), (1, 32), (4096, 4096), (40, 96),
                 (11008, 4096)],
    "long": [(40, 32768 + 64), (300, 4096), (7, 32768)],
}


@pytest.mark.parametrize("shapes", sorted(GROUP_SHAPE_SETS))
@pytest.mark.parametrize("m", [1, 3, 8, 16])
@pytest.mark.parametrize("pdl", [False, True])
def test_linear_grouped_matches_single_calls_and_oracle(qmm, orc, m, pdl, shapes):
    """Every problem of a group gets the bits qmm_linear_q4_0 gives it alone,
    and the oracle's codes."""
    probs, refs = [], []
    for j, (n, k) in enumerate(GROUP_SHAPE_SETS[shapes]):
        w, _ = synthetic.q4_0_case(6500 + j, n, k, 1)
        x = adversarial_x(6600 + j + m, m, k)
        wq, wd = orc.quantize_q4_0(w)
        wq_d, wd_d = to_dev(wq), to_dev(wd.view(np.float16))
        probs.append((to_dev(x), wq_d, wd_d))
        refs.append((x, wq, wd))
    outs = qmm.linear_q4_0_grouped(probs, pdl=pdl)
    for (x_d, wq_d, wd_d), (x, wq, wd), (y, aq, ad) in zip(probs, refs, outs):
        y1, aq1, ad1 = qmm.linear_q4_0(x_d, wq_d, wd_d, codes=True)
        assert np.array_equal(to_np(aq), to_np(aq1))
        assert np.array_equal(f16_bits(ad), f16_bits(ad1))
        assert np.array_equal(to_np(y).view(np.uint32), to_np(y1).view(np.uint32))
        aq_ref, ad_ref = orc.quantize_q8_0(x)
        assert np.array_equal(to_np(aq), aq_ref)
        assert np.array_equal(f16_bits(ad), ad_ref)
        ok, worst, maxrel = rel_gate(to_np(y), orc.gemm_q4_0_q8_0(wq, wd, aq_ref, ad_ref),
                                     orc.gemm_q4_0_q8_0_absterms(wq, wd, aq_ref, ad_ref))
        assert ok, (worst, maxrel)


def test_prepared_grouped_linear_matches_the_one_shot_call(qmm, orc):
    """GroupedLinear builds the table once; every call then gives the bits of
    linear_q4_0_grouped, and reads the x tensors' current contents."""
    import torch
    shapes = [(300, 4096), (77, 1024), (129, 11008)]
    probs, refs = [], []
    for j, (n, k) in enumerate(shapes):
        w, x = synthetic.q4_0_case(900 + j, n, k, 1)
        wq, wd = orc.quantize_q4_0(w)
        probs.append((to_dev(x), to_dev(wq), to_dev(wd.view(np.float16))))
    once = qmm.linear_q4_0_grouped(probs, pdl=True)
    call = qmm.GroupedLinear(probs, pdl=True)
    for (y1, aq1, ad1), (y2, aq2, ad2) in zip(once, call()):
        assert torch.equal(y1, y2) and torch.equal(aq1, aq2) and torch.equal(ad1, ad2)
    # new activations written in place are picked up by the next call
    for j, (x, _, _) in enumerate(probs):
        x.mul_(-0.5)
    again = qmm.linear_q4_0_grouped([(x, wq, wd) for x, wq, wd in probs], pdl=False)
    for (y1, _, _), (y2, _, _) in zip(again, call()):
        assert torch.equal(y1, y2)


def test_grouped_linear_with_host_buffers(qmm, orc):
    """GroupedLinear(host_io=...): one call copies the activations in from
    page-locked host memory, runs the layers and copies the outputs back.
    The host outputs equal, bit for bit, the device outputs of the plain
    call, and a new host input is picked up by the next call."""
    import torch
    shapes = [(300, 4096), (77, 1024), (129, 11008)]
    xs, mats = [], []
    for j, (n, k) in enumerate(shapes):
        w, x = synthetic.q4_0_case(950 + j, n, k, 1)
        wq, wd = orc.quantize_q4_0(w)
        xs.append(x.ravel())
        mats.append((n, k, to_dev(wq), to_dev(wd.view(np.float16))))
    k_off = np.cumsum([0] + [k for _, k in shapes])
    n_off = np.cumsum([0] + [n for n, _ in shapes])
    x_host = torch.from_numpy(np.concatenate(xs)).pin_memory()
    y_host = torch.full((int(n_off[-1]),), np.nan, dtype=torch.float32).pin_memory()
    x_dev = torch.zeros_like(x_host, device="cuda")
    y_dev = torch.zeros((int(n_off[-1]),), dtype=torch.float32, device="cuda")
    probs = [(x_dev[k_off[j]:k_off[j + 1]].view(1, -1), wq, wd,
              y_dev[n_off[j]:n_off[j + 1]].view(1, -1))
             for j, (_, _, wq, wd) in enumerate(mats)]
    assert qmm.host_addressable(x_host) and qmm.host_addressable(y_host)
    # graph=True: the first call runs and captures, later calls replay the
    # graph; each must pick up the new host input like the eager form
    for direct, graph in ((False, False), (True, False), (False, True), (True, True)):
        call = qmm.GroupedLinear(probs, pdl=True, host_io=(x_host, x_dev, y_dev, y_host),
                                 host_direct=direct, graph=graph)
        for scale in (1.0, -0.5, 3.0):
            if scale != 1.0:
                x_host.mul_(scale)
            y_host.fill_(np.nan)
            call()
            torch.cuda.synchronize()
            plain = qmm.linear_q4_0_grouped(
                [(x_host[k_off[j]:k_off[j + 1]].view(1, -1).cuda(), wq, wd)
                 for j, (_, _, wq, wd) in enumerate(mats)])
            for j, (y, _, _) in enumerate(plain):
                assert torch.equal(y.cpu().ravel(), y_host[n_off[j]:n_off[j + 1]]), (direct, graph, j)
    # a graph cannot capture copies from pageable memory: refused up front
    with pytest.raises(ValueError):
        qmm.GroupedLinear(probs, host_io=(x_host.clone(), x_dev, y_dev, y_host.clone()), graph=True)
    # direct mode checks that every x and y lies in the mirrored device buffers
    lib = qmm.load()
    outside = torch.zeros((1, shapes[0][1]), dtype=torch.float32, device="cuda")
    tab, m, _ = qmm._grouped_table(probs + [(outside, *mats[0][2:])])
    st = lib.qmm_linear_q4_0_grouped_host(
        ctypes.addressof(tab), len(probs) + 1, m, qmm.LINEAR_HOST_DIRECT, x_host.data_ptr(),
        x_dev.data_ptr(), x_dev.numel() * 4, y_dev.data_ptr(), y_host.data_ptr(),
        y_dev.numel() * 4, None)
    assert st == 8  # QMM_ERR_ARG
    with pytest.raises(ValueError, match="differ in size"):
        qmm.GroupedLinear(probs, host_io=(x_host[:-1], x_dev, y_dev, y_host))


def test_linear_grouped_full_table(qmm, orc):
    """A table of QMM_GROUP_MAX problems, all of one tiny shape."""
    probs, refs = [], []
    for j in range(qmm.GROUP_MAX):
        w, x = synthetic.q4_0_case(6700 + j, 24 + j, 64, 2)
        wq, wd = orc.quantize_q4_0(w)
        probs.append((to_dev(x), to_dev(wq), to_dev(wd.view(np.float16))))
        refs.append((x, wq, wd))
    outs = qmm.linear_q4_0_grouped(probs)
    for (x, wq, wd), (y, aq, ad) in zip(refs, outs):
        aq_ref, ad_ref = orc.quantize_q8_0(x)
        assert np.array_equal(to_np(aq), aq_ref)
        ok, worst, maxrel = rel_gate(to_np(y), orc.gemm_q4_0_q8_0(wq, wd, aq_ref, ad_ref),
                                     orc.gemm_q4_0_q8_0_absterms(wq, wd, aq_ref, ad_ref))
        assert ok, (worst, maxrel)


def test_linear_reads_strided_rows(qmm, orc):
    """x rows with a leading dimension above k (a column slice of a wider
    buffer) quantize exactly like a packed copy."""
    import torch
    m, n, k = 3, 50, 2048
    w, _ = synthetic.q4_0_case(6400, n, k, 1)
    x = adversarial_x(6401, m, k + 96)
    wq, wd = orc.quantize_q4_0(w)
    xd = to_dev(x)[:, :k]
    aq_ref, ad_ref = orc.quantize_q8_0(np.ascontiguousarray(x[:, :k]))
    wq_d, wd_d = to_dev(wq), to_dev(wd.view(np.float16))
    aq = torch.empty(m, k, dtype=torch.int8, device="cuda")
    ad = torch.empty(m, k // 32, dtype=torch.float16, device="cuda")
    y = torch.empty(m, n, dtype=torch.float32, device="cuda")
    lib = qmm.load()
    st = lib.qmm_linear_q4_0(wq_d.data_ptr(), wd_d.data_ptr(), xd.data_ptr(), k + 96,
                             aq.data_ptr(), ad.data_ptr(), y.data_ptr(), m, n, k, 0,
                             torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert np.array_equal(to_np(aq), aq_ref)
    assert np.array_equal(f16_bits(ad), ad_ref)
    ok, worst, maxrel = rel_gate(to_np(y), orc.gemm_q4_0_q8_0(wq, wd, aq_ref, ad_ref),
                                 orc.gemm_q4_0_q8_0_absterms(wq, wd, aq_ref, ad_ref))
    assert ok, (worst, maxrel)


@pytest.mark.parametrize("m", [1, 4])
def test_linear_pdl_chain_reads_the_previous_layer_output(qmm, orc, m):
    """Layer i+1 consumes layer i's output and shares its aq buffer; with
    programmatic dependent launch every kernel must still wait for its
    predecessor before it reads them, so the chain gives the same bits with
    and without PDL, and each layer's output matches the oracle applied to
    that layer's actual input.  The 11008 -> 4096 layer is split over k
    (three kernels in that layer)."""
    import torch
    dims = [4096, 11008, 4096, 4096]
    layers = []
    for j in range(len(dims) - 1):
        w, _ = synthetic.q4_0_case(6200 + j, dims[j + 1], dims[j], 1)
        wq, wd = orc.quantize_q4_0(w)
        layers.append((wq, wd, to_dev(wq), to_dev(wd.view(np.float16))))
    _, x0 = synthetic.q4_0_case(6299, 1, dims[0], m)
    aq_flat = torch.empty(m * max(dims), dtype=torch.int8, device="cuda")
    outs = {}
    for pdl in (False, True):
        hs = [to_dev(x0)]
        for j, (_, _, wq_d, wd_d) in enumerate(layers):
            aq_j = aq_flat[: m * dims[j]].view(m, dims[j])
            hs.append(qmm.linear_q4_0(hs[-1], wq_d, wd_d, pdl=pdl, aq=aq_j))
        torch.cuda.synchronize()
        outs[pdl] = [to_np(h) for h in hs]
    for a, b in zip(outs[False], outs[True]):
        assert np.isfinite(a).all()
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    for j, (wq, wd, _, _) in enumerate(layers):
        aq_r, ad_r = orc.quantize_q8_0(outs[True][j])
        ok, worst, maxrel = rel_gate(outs[True][j + 1], orc.gemm_q4_0_q8_0(wq, wd, aq_r, ad_r),
                                     orc.gemm_q4_0_q8_0_absterms(wq, wd, aq_r, ad_r))
        assert ok, (j, worst, maxrel)


@pytest.mark.parametrize("fmt", ["q4", "q8"])
def test_gemm_few_token_shape_with_unaligned_scales_takes_the_tcgen05_product(qmm, orc, fmt):
    """The few-token product copies dw with a tensor map (16-byte aligned
    base); with dw 2 bytes off a 16-byte boundary the GEMM call runs the
    tcgen05 product instead.  Both are the serial definition, bit for bit."""
    m, n, k = 16, 300, 1024
    if fmt == "q4":
        w, wd, aq, ad = q4_case(orc, 8800, m, n, k)
        ref, gemm = orc.gemm_q4_0_q8_0(w, wd, aq, ad), qmm.gemm_q4_0_q8_0
    else:
        w, wd, aq, ad = q8_case(orc, 8801, m, n, k)
        ref, gemm = orc.gemm_q8_0_q8_0(w, wd, aq, ad), qmm.gemm_q8_0_q8_0
    w_d, wd_d = to_dev(w), to_dev(wd.view(np.float16))
    aq_d, ad_d = to_dev(aq), to_dev(ad.view(np.float16))
    for scales in (wd_d, _misaligned_copy(wd_d)):
        y = to_np(gemm(w_d, scales, aq_d, ad_d))
        assert np.array_equal(y.view(np.uint32), ref.view(np.uint32))


def test_few_token_product_random_shapes_bit_exact(qmm, orc):
    """Seeded random shapes for the few-token product (1 <= m <= 32, any n,
    k a multiple of 256), both weight formats: y bit for bit the serial
    definition, through the GEMM entries and, for 3 <= m <= 16, the GEMV
    entries with split_k = 0."""
    rng = np.random.default_rng(9100)
    for case in range(12):
        m = int(rng.integers(1, 33))
        n = int(rng.integers(1, 3000))
        k = 256 * int(rng.integers(1, 13))
        fmt = "q4" if case % 2 == 0 else "q8"
        if fmt == "q4":
            w, wd, aq, ad = q4_case(orc, 9100 + case, m, n, k)
            ref = orc.gemm_q4_0_q8_0(w, wd, aq, ad)
            gemm, gemv = qmm.gemm_q4_0_q8_0, qmm.gemv_q4_0_q8_0
        else:
            w, wd, aq, ad = q8_case(orc, 9100 + case, m, n, k)
            ref = orc.gemm_q8_0_q8_0(w, wd, aq, ad)
            gemm, gemv = qmm.gemm_q8_0_q8_0, qmm.gemv_q8_0_q8_0
        args = (to_dev(w), to_dev(wd.view(np.float16)), to_dev(aq), to_dev(ad.view(np.float16)))
        y = to_np(gemm(*args))
        assert np.array_equal(y.view(np.uint32), ref.view(np.uint32)), (fmt, m, n, k)
        if 3 <= m <= 16:
            y = to_np(gemv(*args))
            assert np.array_equal(y.view(np.uint32), ref.view(np.uint32)), (fmt, m, n, k, "gemv")


# The BitNet product for a few tokens (qmm_bitnet_gemm with m <= 32:
# warp-level MMAs over 64-row sets): one and two 8-token tiles, two 16-token
# tiles, a ragged last stage (k not a multiple of 512), more row sets than
# resident CTAs, the longest rows the entry takes (k = 131072).
BITNET_SMALL_SHAPES = [(1, 1, 64), (2, 65, 576), (5, 6912, 2560), (8, 129, 1024),
                       (9, 300, 4096), (16, 1000, 2560), (17, 64 * 152 * 2 + 7, 512),
                       (32, 6912, 6912), (31, 100, 131072)]


@pytest.mark.parametrize("m,n,k", BITNET_SMALL_SHAPES)
def test_bitnet_small_m_bit_exact(qmm, orc, m, n, k):
    tw, absmean, aq, scale, asum = _bitnet_operands(orc, 9300 + m + n, m, n, k)
    y = to_np(qmm.bitnet_gemm(to_dev(tw.view(np.int32)), absmean, to_dev(aq), to_dev(scale)))
    ref = orc.bitnet_gemv(tw, absmean, aq, scale, asum)
    assert np.array_equal(y.view(np.uint32), ref.view(np.uint32))


def test_bitnet_small_m_extreme_activations_bit_exact(qmm, orc):
    """Whole rows of the largest codes (+1) and of -1 against activations of
    +127 and -127: the chained corrections at their largest magnitude, and
    at the longest rows the entry takes the dots reach 127 k = 16,646,144,
    just below 2^24."""
    m, n, k = 8, 96, 131072
    rng = np.random.default_rng(9400)
    t = rng.integers(-1, 2, size=(n, k)).astype(np.int8)
    t[:16] = 1
    t[16:32] = -1
    aq = rng.choice(np.array([-127, 127], dtype=np.int8), size=(m, k))
    aq[:2] = 127
    aq[2:4] = -127
    scale = np.full(m, 0.25, dtype=np.float32)
    asum = aq.astype(np.int64).sum(axis=1).astype(np.int32)
    tw = orc.pack_ternary(t)
    y = to_np(qmm.bitnet_gemm(to_dev(tw.view(np.int32)), 0.5, to_dev(aq), to_dev(scale)))
    ref = orc.bitnet_gemv(tw, 0.5, aq, scale, asum)
    assert np.array_equal(y.view(np.uint32), ref.view(np.uint32))


def test_bitnet_small_m_wait_timeout_reports_and_device_stays_usable(qmm, orc):
    import torch
    tw, absmean, aq, scale, asum = _bitnet_operands(orc, 9500, 16, 300, 1024)
    args = (to_dev(tw.view(np.int32)), absmean, to_dev(aq), to_dev(scale))
    assert qmm.check_device_error() == 0
    try:
        qmm.set_wait_limit(2000)
        qmm.withhold_gemm_loads(True)
        qmm.bitnet_gemm(*args)
        torch.cuda.synchronize()
        status = qmm.check_device_error()
    finally:
        qmm.withhold_gemm_loads(False)
        qmm.set_wait_limit(0)
    assert status == 7
    y = to_np(qmm.bitnet_gemm(*args))
    torch.cuda.synchronize()
    assert qmm.check_device_error() == 0
    ref = orc.bitnet_gemv(tw, absmean, aq, scale, asum)
    assert np.array_equal(y.view(np.uint32), ref.view(np.uint32))
