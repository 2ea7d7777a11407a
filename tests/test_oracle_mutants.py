"""The oracle's pins must catch plausible mistakes.

Each case below plants one mistake in a private copy of the oracle's C source
(a dropped term, a wrong sign, a swapped index, another rounding mode, a
transposed operand ...), compiles it on the CPU into a temporary directory,
and re-runs the pin battery of tests/test_oracle_pins.py against it.  At
least one pin must fail for every planted mistake.  Nothing here touches a GPU
or the CUDA library.
"""
import importlib.util
import os
import subprocess

import pytest

import test_oracle_pins as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "qmm_oracle.c")

# (name, text to find, replacement, count of occurrences to replace (0 = all))
MUTANTS = [
    ("drop_minus_8_in_gemm",
     "s += (orc_q4_nibble(qs, j) - 8) * (int32_t)qa[j];\n                float scale",
     "s += (orc_q4_nibble(qs, j)) * (int32_t)qa[j];\n                float scale", 1),
    ("no_offset_in_block_sums",
     "s += (orc_q4_nibble(qs, j) - 8) * (int32_t)qa[j];\n                sumi",
     "s += (orc_q4_nibble(qs, j)) * (int32_t)qa[j];\n                sumi", 1),
    ("interleaved_nibble_order",
     "return j < ORC_QK / 2 ? (qs[j] & 0x0f) : (qs[j - ORC_QK / 2] >> 4);",
     "return (j & 1) ? (qs[j / 2] >> 4) : (qs[j / 2] & 0x0f);", 1),
    ("pack_nibbles_swapped",
     "dst[j] = (uint8_t)(q[j] | (q[j + ORC_QK / 2] << 4));",
     "dst[j] = (uint8_t)(q[j + ORC_QK / 2] | (q[j] << 4));", 1),
    ("q8_0_round_half_even",
     "q = roundf(xb[j] / d);", "q = rintf(xb[j] / d);", 1),
    ("q8_0_divides_by_128",
     "float d = amax / 127.0f;", "float d = amax / 128.0f;", 1),
    # (a clamp to -128 instead of -127 is not listed: |x/d| <= 127 + eps for
    # finite inputs, so that clamp can never act and the copy is equivalent)
    ("q8_0_quantizes_with_fp16_scale",
     "q = roundf(xb[j] / d);",
     "q = roundf(xb[j] / orc_fp16_to_fp32(orc_fp32_to_fp16(d)));", 1),
    ("q8_0_row_stride_k",
     "const float *xb = x + i * ldx + b * ORC_QK;", "const float *xb = x + i * k + b * ORC_QK;", 1),
    ("q4_0_positive_divisor",
     "float d = maxv / -8.0f;", "float d = maxv / 8.0f;", 1),
    ("q4_0_last_index_on_ties",
     "if (a > amax) { amax = a; maxv = wb[j]; }",
     "if (a >= amax) { amax = a; maxv = wb[j]; }", 1),
    ("q4_0_unsigned_absmax",
     "if (a > amax) { amax = a; maxv = wb[j]; }",
     "if (a > amax) { amax = a; maxv = a; }", 1),
    ("gemm_reversed_weight_scale_index",
     "float scale = orc_fp16_to_fp32(wd[r * kb + b]) * orc_fp16_to_fp32(ad[i * kb + b]);",
     "float scale = orc_fp16_to_fp32(wd[r * kb + (kb - 1 - b)]) * orc_fp16_to_fp32(ad[i * kb + b]);", 1),
    ("gemm_activation_scale_only",
     "float scale = orc_fp16_to_fp32(wd[r * kb + b]) * orc_fp16_to_fp32(ad[i * kb + b]);",
     "float scale = orc_fp16_to_fp32(ad[i * kb + b]);", 1),
    ("block_activation_stride_16",
     "const int8_t *qa = aq + i * k + b * ORC_QK;\n                int32_t s = 0;\n                for (int j = 0; j < ORC_QK; j++)\n                    s += (orc_q4_nibble(qs, j) - 8) * (int32_t)qa[j];\n                sumi",
     "const int8_t *qa = aq + i * k + b * 16;\n                int32_t s = 0;\n                for (int j = 0; j < ORC_QK; j++)\n                    s += (orc_q4_nibble(qs, j) - 8) * (int32_t)qa[j];\n                sumi", 1),
    ("fp16_ties_away",
     "if (rem > 0x1000u || (rem == 0x1000u && (h & 1u)))",
     "if (rem >= 0x1000u)", 1),
    ("fp16_truncates",
     "if (rem > 0x1000u || (rem == 0x1000u && (h & 1u)))\n            h += 1;",
     "if (0)\n            h += 1;", 1),
    ("fp16_subnormals_flushed",
     "if (ax <= 0x33000000u)", "if (ax < 0x38800000u)", 1),
    ("ternary_bits_msb_first",
     "int32_t code = (int32_t)((word >> (2 * (j % 16))) & 3u);\n                acc += code * (int32_t)aq[i * k + j];\n            }\n            dot",
     "int32_t code = (int32_t)((word >> (2 * (15 - j % 16))) & 3u);\n                acc += code * (int32_t)aq[i * k + j];\n            }\n            dot", 1),
    ("ternary_identity_drops_sum",
     "dot[i * n + r] = acc - act_sum[i];", "dot[i * n + r] = acc;", 1),
    ("ternary_code_offset_2",
     "uint32_t code = (uint32_t)(t[r * k + wi * 16 + i] + 1);",
     "uint32_t code = (uint32_t)(t[r * k + wi * 16 + i] + 2) & 3u;", 1),
    ("bitnet_scale_inverted",
     "if (amax != 0.0f) s = 127.0f / amax;", "if (amax != 0.0f) s = amax / 127.0f;", 1),
    ("bitnet_output_multiplies_scale",
     "out = ((float)d * weight_absmean) / act_scale[i];",
     "out = ((float)d * weight_absmean) * act_scale[i];", 1),
    ("bitnet_sum_skips_clamp",
     "aq[i * k + j] = (int8_t)q;\n            sum += (int32_t)q;",
     "aq[i * k + j] = (int8_t)q;\n            sum += (int32_t)q + (j == 0);", 1),
    # Q8_0 weights x Q8_0 activations
    ("q8w_block_sums_offset_8",
     "s += (int32_t)qw[j] * (int32_t)qa[j];\n                sumi",
     "s += ((int32_t)qw[j] - 8) * (int32_t)qa[j];\n                sumi", 1),
    ("q8w_gemm_weight_row_stride_k_half",
     "const int8_t *qw = w8 + r * k + b * ORC_QK;\n                const int8_t *qa = aq + i * k + b * ORC_QK;\n                int32_t s = 0;\n                for (int j = 0; j < ORC_QK; j++)\n                    s += (int32_t)qw[j] * (int32_t)qa[j];\n                float scale",
     "const int8_t *qw = w8 + r * (k / 2) + b * ORC_QK;\n                const int8_t *qa = aq + i * k + b * ORC_QK;\n                int32_t s = 0;\n                for (int j = 0; j < ORC_QK; j++)\n                    s += (int32_t)qw[j] * (int32_t)qa[j];\n                float scale", 1),
    ("q8w_gemm_reversed_elements",
     "s += (int32_t)qw[j] * (int32_t)qa[j];\n                float scale",
     "s += (int32_t)qw[ORC_QK - 1 - j] * (int32_t)qa[j];\n                float scale", 1),
    ("q8w_gemm_weight_scale_only",
     "float scale = orc_fp16_to_fp32(wd[r * kb + b]) * orc_fp16_to_fp32(ad[i * kb + b]);\n                acc = fmaf((float)s, scale, acc);\n            }\n            y[i * n + r] = acc;\n        }\n}\n\n/* Double-precision product (|sumi| <= 32*127*127",
     "float scale = orc_fp16_to_fp32(wd[r * kb + b]);\n                acc = fmaf((float)s, scale, acc);\n            }\n            y[i * n + r] = acc;\n        }\n}\n\n/* Double-precision product (|sumi| <= 32*127*127", 1),
    ("q8w_f64_block_index_off_by_one",
     "double t = (double)s * (double)orc_fp16_to_fp32(wd[r * kb + b])",
     "double t = (double)s * (double)orc_fp16_to_fp32(wd[r * kb + (b + 1) % kb])", 1),
    ("q8w_absterms_signed",
     "abs_acc += fabs(t);", "abs_acc += t;", 1),
    # load-time repack for the GEMM
    ("repack_halves_swapped",
     "int bit = 4 * i + 16 * h;", "int bit = 4 * i + 16 * (1 - h);", 1),
    ("repack_stages_reversed",  # (every planted mistake stays inside the buffers)
     "return (g * n_tiles_k + j) * 4096 + unit * 16 + c * 4 + bit / 8;",
     "return (g * n_tiles_k + (n_tiles_k - 1 - j)) * 4096 + unit * 16 + c * 4 + bit / 8;", 1),
    ("repack_unit_row_major",
     "int64_t unit = 2 * rr + blk;", "int64_t unit = rr + 128 * blk;", 1),
    ("repack_pads_with_zero_nibbles",
     "for (int64_t i = 0; i < bytes; i++) wr[i] = 0x88;", "for (int64_t i = 0; i < bytes; i++) wr[i] = 0x00;", 1),
]

PIN_FUNCS = [getattr(pins, n) for n in dir(pins)
             if n.startswith("test_") and n not in ("test_splitmix64_published_vector",
                                                    "test_generator_counter_form_is_consistent")]


def _load_mutant(tmp_path, name, find, repl, count):
    src = open(SRC).read()
    assert src.count(find) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(find, repl, count if count else -1)
    assert mutated != src
    csrc = tmp_path / f"{name}.c"
    csrc.write_text(mutated)
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", str(lib), str(csrc), "-lm"], check=True)
    spec = importlib.util.spec_from_file_location(f"oracle_mutant_{name}",
                                                  os.path.join(ROOT, "oracle", "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC, mod._LIB, mod._lib = str(csrc), str(lib), None
    return mod


@pytest.mark.parametrize("name,find,repl,count", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, find, repl, count):
    mod = _load_mutant(tmp_path, name, find, repl, count)
    failed = []
    for fn in PIN_FUNCS:
        try:
            fn(mod)
        except AssertionError:
            failed.append(fn.__name__)
    assert failed, f"no pin caught mutant {name}"


def test_unmutated_copy_passes_all_pins(tmp_path):
    """The harness itself: a copy with an identity 'mutation' passes."""
    mod = _load_mutant(tmp_path, "identity", "#include <math.h>", "#include <math.h>\n", 1)
    for fn in PIN_FUNCS:
        fn(mod)
