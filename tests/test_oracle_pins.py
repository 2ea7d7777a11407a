"""Pins for the CPU oracle that do not go through its own formulas.

Each test checks the oracle against something fixed independently of it: the
hand-worked blocks in tests/golden/ (worked from the definitions on the
llama.cpp visual guide, lesson 31 "How the quantized dot product works", and
Loom "Plan 9 SIMD Forward", "BitNet ternary MAD kernel"), numpy's IEEE binary16
conversion, brute-force dequantize-then-dot in double precision, an exact
integer-matmul reduction, the ternary identity against a direct signed sum,
and invariants of the block formats.  tests/test_oracle_mutants.py re-runs
these pins against deliberately broken copies of the oracle and requires each
copy to fail at least one of them.
"""
import numpy as np
import pytest

from conftest import load_golden
from quantized_matmul_gb300 import synthetic

QK = 32


# ---------------------------------------------------------------------------
# helpers written from the block layout only (no quantizer arithmetic)

def unpack_q4_0(wq: np.ndarray) -> np.ndarray:
    """uint8 [n, k/2] -> int64 [n, k] nibble values 0..15; byte j of a block
    holds element j (low nibble) and element j+16 (high nibble)."""
    n, half = wq.shape
    blocks = wq.reshape(n, half // 16, 16).astype(np.int64)
    out = np.concatenate([blocks & 0x0F, blocks >> 4], axis=2)
    return out.reshape(n, half * 2)


def fp16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def unpack_ternary(tw: np.ndarray) -> np.ndarray:
    """uint32 [n, k/16] -> int64 codes [n, k], element i of a word at bits 2i."""
    shifts = (2 * np.arange(16, dtype=np.uint64))
    codes = (tw.astype(np.uint64)[:, :, None] >> shifts) & np.uint64(3)
    return codes.reshape(tw.shape[0], -1).astype(np.int64)


def ints(vals):
    return np.array([int(v, 0) for v in vals], np.int64)


def floats(vals):
    return np.array([float(v) for v in vals], np.float64)


# ---------------------------------------------------------------------------
# IEEE binary16 conversions vs numpy

def test_fp16_to_fp32_exhaustive(orc):
    h = np.arange(65536, dtype=np.uint16)
    got = orc.fp16_bits_to_fp32_array(h)
    ref = h.view(np.float16).astype(np.float32)
    same = (got.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_fp32_to_fp16_vs_numpy(orc):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    # every binary16 value, the midpoints between neighbours, and +-1 ulp (f32) around them
    h = np.arange(0, 0x7C00, dtype=np.uint16)
    v = h.view(np.float16).astype(np.float64)
    mids = ((v[:-1] + v[1:]) / 2).astype(np.float32)
    edge = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)),
                           np.nextafter(mids, np.float32(0)), v.astype(np.float32),
                           np.array([65504, 65519.99, 65520, 65536, 1e30, 2**-25, 2**-24, 2**-26],
                                    np.float32)])
    f = np.concatenate([bits.view(np.float32), edge, -edge])
    f = f[~np.isnan(f)]
    got = orc.fp32_to_fp16_bits_array(f)
    with np.errstate(over="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------------------
# hand-worked blocks

def test_q8_0_hand_block(orc):
    g = load_golden("q4_0_q8_0_hand_block.txt")
    aq, ad = orc.quantize_q8_0(floats(g["x"]).astype(np.float32)[None])
    assert np.array_equal(aq[0].astype(np.int64), ints(g["aq"]))
    assert int(ad[0, 0]) == int(g["ad_bits"][0], 0)


def test_q4_0_hand_block(orc):
    g = load_golden("q4_0_q8_0_hand_block.txt")
    wq, wd = orc.quantize_q4_0(floats(g["w"]).astype(np.float32)[None])
    assert [int(b) for b in wq[0]] == [int(v, 16) for v in g["wq_hex"]]
    assert int(wd[0, 0]) == int(g["wd_bits"][0], 0)


def test_block_dot_hand(orc):
    g = load_golden("q4_0_q8_0_hand_block.txt")
    wq = np.array([[int(v, 16) for v in g["wq_hex"]]], np.uint8)
    wd = np.array([[int(g["wd_bits"][0], 0)]], np.uint16)
    aq = ints(g["aq"]).astype(np.int8)[None]
    ad = np.array([[int(g["ad_bits"][0], 0)]], np.uint16)
    assert int(orc.block_sums(wq, aq)[0, 0, 0]) == int(g["sumi"][0])
    y = orc.gemm_q4_0_q8_0(wq, wd, aq, ad)
    assert float(y[0, 0]) == float(g["y"][0])
    assert float(orc.gemm_q4_0_q8_0_f64(wq, wd, aq, ad)[0, 0]) == float(g["y"][0])


def test_aos_block_layout_hand(orc):
    g = load_golden("q4_0_q8_0_hand_block.txt")
    blk = np.array([int(v, 16) for v in g["block_aos_hex"]], np.uint8)
    wq, wd = orc.q4_0_blocks_to_planes(blk, 1, 32)
    assert [int(b) for b in wq[0]] == [int(v, 16) for v in g["wq_hex"]]
    assert int(wd[0, 0]) == int(g["wd_bits"][0], 0)
    assert np.array_equal(orc.q4_0_planes_to_blocks(wq, wd), blk)


def test_bitnet_hand_word(orc):
    g = load_golden("bitnet_hand_word.txt")
    tw = orc.pack_ternary(ints(g["t"]).astype(np.int8)[None])
    assert int(tw[0, 0]) == int(g["word_hex"][0], 16)
    aq, s, asum = orc.quantize_act_bitnet(floats(g["x"]).astype(np.float32)[None])
    assert np.array_equal(aq[0].astype(np.int64), ints(g["aq"]))
    assert float(s[0]) == float(g["act_scale"][0])
    assert int(asum[0]) == int(g["act_sum"][0])
    assert int(orc.bitnet_dot(tw, aq, asum)[0, 0]) == int(g["dot"][0])
    y = orc.bitnet_gemv(tw, float(g["absmean"][0]), aq, s, asum)
    assert float(y[0, 0]) == float(g["y"][0])


# ---------------------------------------------------------------------------
# brute force on small inputs

SMALL_SHAPES = [(m, n, k) for k in (32, 64, 96) for n in (1, 3, 7, 17) for m in (1, 2, 3, 5)]


def _small_case(seed, m, n, k):
    w, x = synthetic.q4_0_case(seed, n, k, m)
    return w, x


def test_block_sums_vs_integer_einsum(orc):
    for i, (m, n, k) in enumerate(SMALL_SHAPES):
        w, x = _small_case(100 + i, m, n, k)
        wq, _ = orc.quantize_q4_0(w)
        aq, _ = orc.quantize_q8_0(x)
        wv = (unpack_q4_0(wq) - 8).reshape(n, k // QK, QK)
        av = aq.astype(np.int64).reshape(m, k // QK, QK)
        ref = np.einsum("nbj,mbj->mnb", wv, av)
        assert np.array_equal(orc.block_sums(wq, aq), ref), (m, n, k)


def test_brute_force_dequantize_then_dot(orc):
    for i, (m, n, k) in enumerate(SMALL_SHAPES):
        w, x = _small_case(200 + i, m, n, k)
        wq, wd = orc.quantize_q4_0(w)
        aq, ad = orc.quantize_q8_0(x)
        # dequantize each side in double with numpy's binary16, then a plain dot
        wf = (unpack_q4_0(wq) - 8).astype(np.float64) * np.repeat(fp16_bits_to_f64(wd), QK, axis=1)
        af = aq.astype(np.float64) * np.repeat(fp16_bits_to_f64(ad), QK, axis=1)
        y_bf = af @ wf.T
        y64 = orc.gemm_q4_0_q8_0_f64(wq, wd, aq, ad)
        np.testing.assert_allclose(y64, y_bf, rtol=1e-12, atol=1e-12 * np.abs(y_bf).max())
        y32 = orc.gemm_q4_0_q8_0(wq, wd, aq, ad).astype(np.float64)
        absterms = np.abs(af) @ np.abs(wf).T  # >= the per-block |terms| sum
        assert (np.abs(y32 - y_bf) <= 1e-6 * absterms + 1e-30).all(), (m, n, k)
        at = orc.gemm_q4_0_q8_0_absterms(wq, wd, aq, ad)
        assert (at <= absterms * (1 + 1e-12)).all() and (at >= np.abs(y_bf) * (1 - 1e-12)).all()


def test_integer_matmul_reduction(orc):
    """With every scale fp16(1.0) the product is the plain integer matmul."""
    rng = np.random.default_rng(3)
    for (m, n, k) in [(1, 5, 64), (3, 17, 96), (7, 33, 256)]:
        wq = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
        aq = rng.integers(-127, 128, size=(m, k), dtype=np.int64).astype(np.int8)
        one = np.uint16(0x3C00)
        wd = np.full((n, k // QK), one, np.uint16)
        ad = np.full((m, k // QK), one, np.uint16)
        ref = aq.astype(np.int64) @ (unpack_q4_0(wq) - 8).T
        y = orc.gemm_q4_0_q8_0(wq, wd, aq, ad)
        assert np.array_equal(y.astype(np.int64), ref)
        assert np.array_equal(orc.block_sums(wq, aq).sum(axis=2), ref)


def test_row_independence(orc):
    w, x = _small_case(5, 6, 23, 128)
    wq, wd = orc.quantize_q4_0(w)
    aq, ad = orc.quantize_q8_0(x)
    y = orc.gemm_q4_0_q8_0(wq, wd, aq, ad)
    rows, cols = [1, 4], [0, 5, 22]
    ys = orc.gemm_q4_0_q8_0(wq[cols], wd[cols], aq[rows], ad[rows])
    assert np.array_equal(ys.view(np.uint32), y[np.ix_(rows, cols)].view(np.uint32))
    # quantizers are row/block local too
    aq2, ad2 = orc.quantize_q8_0(x[rows])
    assert np.array_equal(aq2, aq[rows]) and np.array_equal(ad2, ad[rows])
    wq2, wd2 = orc.quantize_q4_0(w[cols])
    assert np.array_equal(wq2, wq[cols]) and np.array_equal(wd2, wd[cols])


# ---------------------------------------------------------------------------
# load-time repack of Q4_0 nibbles for the tensor-core GEMM (the layout the
# GEMM's converter decodes with shifts and masks only)

def _decode_repacked(wr, n, k):
    """Read every element back the way the GEMM converter does: tile
    (row group, 2-block stage) of 4096 bytes, unit 2*row + block of 16 bytes,
    word c holding elements 8c..8c+7, (word >> 4i) & 0x000F000F giving
    elements 8c+2i and 8c+2i+1 in the low and high 16-bit halves."""
    kb = k // QK
    tiles_k = (kb + 1) // 2
    words = wr.view(np.uint32)
    out = np.zeros((n, k), np.int64)
    for r in range(n):
        for b in range(kb):
            tile = (r // 128) * tiles_k + b // 2
            unit = 2 * (r % 128) + b % 2
            base = (tile * 4096 + unit * 16) // 4
            for c in range(4):
                w = int(words[base + c])
                for i in range(4):
                    pair = (w >> (4 * i)) & 0x000F000F
                    out[r, b * QK + 8 * c + 2 * i] = pair & 0xF
                    out[r, b * QK + 8 * c + 2 * i + 1] = pair >> 16
    return out


def test_repack_decodes_with_shifts_and_masks(orc):
    rng = np.random.default_rng(9)
    for (n, k) in [(1, 32), (3, 96), (130, 64), (129, 160)]:
        wq = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
        wr = orc.repack_q4_0_gemm(wq)
        assert wr.size == ((n + 127) // 128) * ((k // QK + 1) // 2) * 4096
        assert np.array_equal(_decode_repacked(wr, n, k), unpack_q4_0(wq)), (n, k)
        assert np.array_equal(orc.unrepack_q4_0_gemm(wr, n, k), wq)


def test_repack_pads_with_value_zero(orc):
    """Rows past n and the block past an odd k/32 hold nibble 8 (value 0)."""
    n, k = 3, 96  # 3 blocks: the second stage has one block; 125 padding rows
    wq = np.zeros((n, k // 2), np.uint8)  # every real nibble 0
    wr = orc.repack_q4_0_gemm(wq)
    words = wr.view(np.uint32).reshape(-1, 4096 // 4)
    real = np.zeros(words.shape, bool)
    for r in range(n):
        for b in range(k // QK):
            unit = 2 * r + b % 2
            real[b // 2, unit * 4:unit * 4 + 4] = True
    assert (words[real] == 0).all() and (words[~real] == 0x88888888).all()


# ---------------------------------------------------------------------------
# Q8_0 weights x Q8_0 activations (the same block on both sides)

def test_q8_0_weight_hand_block(orc):
    g = load_golden("q8_0_q8_0_hand_block.txt")
    w8, wd = orc.quantize_q8_0(floats(g["w"]).astype(np.float32)[None])
    assert np.array_equal(w8[0].astype(np.int64), ints(g["wq"]))
    assert int(wd[0, 0]) == int(g["wd_bits"][0], 0)
    aq, ad = orc.quantize_q8_0(floats(g["x"]).astype(np.float32)[None])
    assert np.array_equal(aq[0].astype(np.int64), ints(g["aq"]))
    assert int(ad[0, 0]) == int(g["ad_bits"][0], 0)
    assert int(orc.block_sums_q8_0(w8, aq)[0, 0, 0]) == int(g["sumi"][0])
    assert float(orc.gemm_q8_0_q8_0(w8, wd, aq, ad)[0, 0]) == float(g["y"][0])
    y64, absterms = orc.gemm_q8_0_q8_0_f64(w8, wd, aq, ad)
    assert float(y64[0, 0]) == float(g["y"][0]) and float(absterms[0, 0]) == abs(float(g["y"][0]))


def test_q8_0_weight_block_sums_vs_integer_einsum(orc):
    for i, (m, n, k) in enumerate(SMALL_SHAPES):
        w, x = _small_case(600 + i, m, n, k)
        w8, _ = orc.quantize_q8_0(w)
        aq, _ = orc.quantize_q8_0(x)
        wv = w8.astype(np.int64).reshape(n, k // QK, QK)
        av = aq.astype(np.int64).reshape(m, k // QK, QK)
        ref = np.einsum("nbj,mbj->mnb", wv, av)
        assert np.array_equal(orc.block_sums_q8_0(w8, aq), ref), (m, n, k)


def test_q8_0_weight_brute_force_dequantize_then_dot(orc):
    for i, (m, n, k) in enumerate(SMALL_SHAPES):
        w, x = _small_case(700 + i, m, n, k)
        w8, wd = orc.quantize_q8_0(w)
        aq, ad = orc.quantize_q8_0(x)
        wf = w8.astype(np.float64) * np.repeat(fp16_bits_to_f64(wd), QK, axis=1)
        af = aq.astype(np.float64) * np.repeat(fp16_bits_to_f64(ad), QK, axis=1)
        y_bf = af @ wf.T
        y64, at = orc.gemm_q8_0_q8_0_f64(w8, wd, aq, ad)
        np.testing.assert_allclose(y64, y_bf, rtol=1e-12, atol=1e-12 * np.abs(y_bf).max())
        y32 = orc.gemm_q8_0_q8_0(w8, wd, aq, ad).astype(np.float64)
        absterms = np.abs(af) @ np.abs(wf).T  # >= the per-block |terms| sum
        assert (np.abs(y32 - y_bf) <= 1e-6 * absterms + 1e-30).all(), (m, n, k)
        assert (at <= absterms * (1 + 1e-12)).all() and (at >= np.abs(y_bf) * (1 - 1e-12)).all()


def test_q8_0_weight_integer_matmul_reduction(orc):
    """With every scale fp16(1.0) the product is the plain integer matmul
    (exact in f32 here: |y| <= 127 * 127 * 256 < 2^24)."""
    rng = np.random.default_rng(4)
    for (m, n, k) in [(1, 5, 64), (3, 17, 96), (7, 33, 256)]:
        w8 = rng.integers(-127, 128, size=(n, k), dtype=np.int64).astype(np.int8)
        aq = rng.integers(-127, 128, size=(m, k), dtype=np.int64).astype(np.int8)
        one = np.uint16(0x3C00)
        wd = np.full((n, k // QK), one, np.uint16)
        ad = np.full((m, k // QK), one, np.uint16)
        ref = aq.astype(np.int64) @ w8.astype(np.int64).T
        y = orc.gemm_q8_0_q8_0(w8, wd, aq, ad)
        assert np.array_equal(y.astype(np.int64), ref)
        assert np.array_equal(orc.block_sums_q8_0(w8, aq).sum(axis=2), ref)
        y64, _ = orc.gemm_q8_0_q8_0_f64(w8, wd, aq, ad)
        assert np.array_equal(y64.astype(np.int64), ref)


def test_q8_0_weight_row_independence(orc):
    w, x = _small_case(8, 6, 23, 128)
    w8, wd = orc.quantize_q8_0(w)
    aq, ad = orc.quantize_q8_0(x)
    y = orc.gemm_q8_0_q8_0(w8, wd, aq, ad)
    rows, cols = [1, 4], [0, 5, 22]
    ys = orc.gemm_q8_0_q8_0(w8[cols], wd[cols], aq[rows], ad[rows])
    assert np.array_equal(ys.view(np.uint32), y[np.ix_(rows, cols)].view(np.uint32))


# ---------------------------------------------------------------------------
# quantizer invariants

def _adversarial_rows(rng, k):
    rows = [rng.standard_normal(k).astype(np.float32)]
    z = np.zeros(k, np.float32)
    rows.append(z)                                        # all-zero row
    r = rng.standard_normal(k).astype(np.float32)
    r[:QK] = 0                                            # one zero block
    r[QK + 3] = 1e4                                       # an outlier
    rows.append(r)
    rows.append((rng.standard_normal(k) * 1e-30).astype(np.float32))  # tiny scales
    rows.append(rng.integers(-3, 4, size=k).astype(np.float32))      # many ties on |x|
    return np.stack(rows)


def test_q8_0_invariants(orc):
    rng = np.random.default_rng(11)
    k = 256
    x = _adversarial_rows(rng, k)
    aq, ad = orc.quantize_q8_0(x)
    q = aq.astype(np.int64).reshape(len(x), -1, QK)
    xb = x.astype(np.float64).reshape(len(x), -1, QK)
    assert (np.abs(q) <= 127).all()
    amax = np.abs(xb).max(axis=2)
    d32 = (amax.astype(np.float32) / np.float32(127)).astype(np.float64)
    for i in range(len(x)):
        for b in range(q.shape[1]):
            if amax[i, b] == 0:
                assert ad[i, b] == 0 and (q[i, b] == 0).all()
                continue
            j = int(np.argmax(np.abs(xb[i, b])))
            assert abs(int(q[i, b, j])) == 127
            assert (np.sign(q[i, b]) * np.sign(xb[i, b]) >= 0).all()
            # |x/d - q| <= 1/2 (+ the rounding of one f32 division)
            err = np.abs(xb[i, b] / d32[i, b] - q[i, b])
            assert (err <= 0.5 + 1e-5).all()
    # the stored scale is the nearest binary16 to the f32 scale
    assert np.array_equal(ad, d32.astype(np.float32).astype(np.float16).view(np.uint16))


def test_q8_0_strided_rows_invariants(orc):
    # rows read with a row stride larger than k: the padding holds values far
    # larger than the rows, so a row read from the wrong place changes the
    # block maxima and breaks the invariants below
    rng = np.random.default_rng(21)
    m, k, ldx = 5, 96, 160
    x = rng.standard_normal((m, k)).astype(np.float32)
    buf = np.full((m, ldx), 1.0e4, np.float32)
    buf[:, :k] = x
    aq, ad = orc.quantize_q8_0_strided(buf, k)
    q = aq.astype(np.int64).reshape(m, -1, QK)
    xb = x.astype(np.float64).reshape(m, -1, QK)
    amax = np.abs(xb).max(axis=2)
    d32 = (amax.astype(np.float32) / np.float32(127)).astype(np.float64)
    assert np.array_equal(ad, d32.astype(np.float32).astype(np.float16).view(np.uint16))
    for i in range(m):
        for b in range(q.shape[1]):
            j = int(np.argmax(np.abs(xb[i, b])))
            assert abs(int(q[i, b, j])) == 127
            assert (np.abs(xb[i, b] / d32[i, b] - q[i, b]) <= 0.5 + 1e-5).all()


def test_q4_0_invariants(orc):
    rng = np.random.default_rng(12)
    k = 256
    w = _adversarial_rows(rng, k) * np.float32(0.02)
    wq, wd = orc.quantize_q4_0(w)
    nib = unpack_q4_0(wq).reshape(len(w), -1, QK)
    wb = w.astype(np.float64).reshape(len(w), -1, QK)
    for i in range(len(w)):
        for b in range(nib.shape[1]):
            blk = wb[i, b]
            if not np.any(blk):
                # d = 0/-8 is a zero (its sign bit follows the division: -0)
                assert fp16_bits_to_f64(wd[i, b]) == 0 and (nib[i, b] == 8).all()
                continue
            j = int(np.argmax(np.abs(blk)))  # argmax: first index on ties
            assert nib[i, b, j] == 0
            d = np.float32(np.float32(blk[j]) / np.float32(-8.0)).astype(np.float64)
            # every element within half a step, except the clamped +8 side
            deq = (nib[i, b] - 8) * d
            ok = (np.abs(blk - deq) <= abs(d) * (0.5 + 1e-5)) | ((nib[i, b] == 15) & (blk / d > 7.5))
            assert ok.all()


def test_q4_0_tie_takes_first_index(orc):
    w = np.zeros((2, 32), np.float32)
    w[0, 3], w[0, 9] = 0.5, -0.5
    w[1, 3], w[1, 9] = -0.5, 0.5
    wq, wd = orc.quantize_q4_0(w)
    d = fp16_bits_to_f64(wd)[:, 0]
    assert d[0] == -0.0625 and d[1] == 0.0625
    nib = unpack_q4_0(wq)
    assert nib[0, 3] == 0 and nib[0, 9] == 15  # -0.5/-0.0625 = 8 -> clamped to 15
    assert nib[1, 3] == 0 and nib[1, 9] == 15


# ---------------------------------------------------------------------------
# ternary path

def test_ternary_identity_and_packing(orc):
    for seed, (m, n, k) in enumerate([(1, 7, 16), (2, 5, 48), (3, 33, 160), (1, 64, 2560)]):
        t, x, absmean = synthetic.bitnet_case(300 + seed, n, k, m)
        tw = orc.pack_ternary(t)
        assert np.array_equal(unpack_ternary(tw) - 1, t.astype(np.int64))
        aq, s, asum = orc.quantize_act_bitnet(x)
        assert np.array_equal(asum.astype(np.int64), aq.astype(np.int64).sum(axis=1))
        direct = aq.astype(np.int64) @ t.astype(np.int64).T
        assert np.array_equal(orc.bitnet_dot(tw, aq, asum).astype(np.int64), direct)


def test_bitnet_act_quant_invariants(orc):
    rng = np.random.default_rng(13)
    x = _adversarial_rows(rng, 160)
    aq, s, asum = orc.quantize_act_bitnet(x)
    for i in range(len(x)):
        amax = float(np.abs(x[i]).max())
        if amax == 0:
            assert s[i] == 0 and asum[i] == 0 and (aq[i] == 0).all()
            continue
        assert float(s[i]) == float(np.float32(127) / np.float32(amax))
        j = int(np.argmax(np.abs(x[i])))
        assert abs(int(aq[i, j])) == 127
        err = np.abs(x[i].astype(np.float64) * float(s[i]) - aq[i])
        assert (err <= 0.5 + 1e-5).all()


def test_bitnet_output_closed_form(orc):
    t, x, absmean = synthetic.bitnet_case(3, 40, 2560, 3)
    x[1] = 0  # a zero row gives scale 0 and y 0
    tw = orc.pack_ternary(t)
    aq, s, asum = orc.quantize_act_bitnet(x)
    y = orc.bitnet_gemv(tw, absmean, aq, s, asum).astype(np.float64)
    dot = (aq.astype(np.int64) @ t.astype(np.int64).T).astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        exact = np.where(s[:, None] != 0, dot * absmean / s[:, None].astype(np.float64), 0.0)
    # two f32 roundings: within 2^-23 relative of the exact quotient
    assert (np.abs(y - exact) <= np.abs(exact) * 2.0 ** -23 + 1e-300).all()
    assert (y[1] == 0).all()


# ---------------------------------------------------------------------------
# the input generator

def test_splitmix64_published_vector():
    # first outputs of SplitMix64 seeded with 1234567 (the generator's
    # published reference sequence)
    z = synthetic.raw_u64(1234567, 0, 5)
    assert [int(v) for v in z] == [6457827717110365317, 3203168211198807973,
                                   9817491932198370423, 4593380528125082431,
                                   16408922859458223821]


def test_generator_counter_form_is_consistent():
    a = synthetic.normal(9, 0, 5000, 1.0)
    b = synthetic.normal(9, 1237, 11, 1.0)
    assert np.array_equal(a[1237:1248], b)
    st = synthetic.Stream(9)
    w = st.normal((10, 50), 0.02)
    x = st.normal((2, 50))
    assert np.array_equal(w.ravel(), synthetic.normal(9, 0, 500, 0.02))
    assert np.array_equal(x.ravel(), synthetic.normal(9, 500, 100, 1.0))
    big = synthetic.normal(1, 0, 400_000, 1.0)
    assert abs(big.mean()) < 0.01 and abs(big.std() - 1) < 0.01
    tern = synthetic.ternary(2, 0, 300_000)
    counts = np.bincount(tern + 1, minlength=3) / tern.size
    assert np.allclose(counts, 1 / 3, atol=0.01)
