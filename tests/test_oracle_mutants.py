"""The pins have teeth: plant one plausible mistake at a time in a copy of the
oracle's C source (on the CPU), build it, and check that at least one pin in
``test_oracle_pins`` fails against the mutant.  The real oracle is untouched."""
import ctypes
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "bit1_oracle.c")

# The binary and ternary row loops share their outer lines; these tails make
# each mutation site unique.
_BIN = "\n                double part = 0.0;\n                for (int64_t k = 128 * g; k < 128 * g + 128; k++) {\n                    double xv"
_TER = "\n                double part = 0.0;\n                for (int64_t k = 128 * g; k < 128 * g + 128; k++) {\n                    int t"
_SCALE = "double s = orc_half_to_double(scales[n * G + g]);"
_SCALE_T = "double s = orc_half_to_double(scales[g * N + n]);"
_XB = "double xv = orc_bf16_to_double(x[b * K + k]);\n                    if (orc_bit"
_XT = "double xv = orc_bf16_to_double(x[b * K + k]);\n                    if (t > 0)"
# The SwiGLU pair's full and selected forms share the gate/up line.
_GU = "double g = y[b * N2 + 2 * n], u = y[b * N2 + 2 * n + 1];"
_GU_SW = "double u = y[b * N2 + 2 * n], g = y[b * N2 + 2 * n + 1];"
_HF = "\n            h[b * (N2 / 2) + n] ="

# (name, text in the source, replacement, pins expected to catch it)
MUTANTS = [
    ("msb_first_bit_order", "return (bits[n * (K / 8) + k / 8] >> (k % 8)) & 1;",
     "return (bits[n * (K / 8) + k / 8] >> (7 - k % 8)) & 1;",
     [lambda o: pins.test_gemv_brute_force_matches_dense(o, 8, 256, 1, 0),
      lambda o: pins.test_closed_form_single_bit(o)]),
    ("sign_polarity", "if (orc_bit(bits, K, n, k))", "if (!orc_bit(bits, K, n, k))",
     [lambda o: pins.test_gemv_brute_force_matches_dense(o, 8, 256, 1, 0),
      lambda o: pins.test_closed_form_all_bits_set_and_clear(o)]),
    ("scale_index_transposed", _SCALE + _BIN, _SCALE_T + _BIN,
     [lambda o: pins.test_gemv_scales_are_per_row_and_group(o)]),
    ("last_group_dropped", "for (int64_t g = 0; g < G; g++) {\n                " + _SCALE + _BIN,
     "for (int64_t g = 0; g < G - 1; g++) {\n                " + _SCALE + _BIN,
     [lambda o: pins.test_gemv_brute_force_matches_dense(o, 5, 256, 3, 1)]),
    ("batch_row_ignored", _XB, _XB.replace("x[b * K + k]", "x[k]"),
     [lambda o: pins.test_gemv_brute_force_matches_dense(o, 5, 256, 3, 1)]),
    ("half_exponent_bias", "v = ldexp((double)(m + 1024), e - 25);",
     "v = ldexp((double)(m + 1024), e - 24);",
     [lambda o: pins.test_half_decode_all_patterns(o)]),
    ("bf16_subnormal_scale", "v = ldexp((double)m, -133);", "v = ldexp((double)m, -126);",
     [lambda o: pins.test_bf16_decode_all_patterns(o)]),
    ("half_rounding_truncates", "n = nearbyint(a / q);", "n = floor(a / q);",
     [lambda o: pins.test_double_to_half_matches_numpy(o)]),
    ("xor_skips_last_byte", "for (int64_t j = 0; j < K / 8; j++)\n            bits[r * (K / 8) + j] ^= 0xFF;",
     "for (int64_t j = 0; j < K / 8 - 1; j++)\n            bits[r * (K / 8) + j] ^= 0xFF;",
     [lambda o: pins.test_xor_patch_flips_listed_rows_only(o)]),
    ("xor_range_error_swallowed", "if (rows[i] < 0 || (int64_t)rows[i] >= N)\n            return ORC_ERANGE;",
     "if (rows[i] < 0 || (int64_t)rows[i] >= N)\n            return ORC_OK;",
     [lambda o: pins.test_xor_patch_range_checked_before_any_change(o)]),
    ("pack_wrong_divisor", "mean = sum / 128.0;", "mean = sum / 127.0;",
     [lambda o: pins.test_pack_scale_is_fp16_of_mean_abs(o), lambda o: pins.test_pack_round_trip(o)]),
    ("pack_zero_is_negative", "if (!(v < 0.0))", "if (v > 0.0)",
     [lambda o: pins.test_pack_bits_are_sign_test_little_endian(o)]),
    ("footprint_scale_bytes", "return N * K / 8 + 2 * N * (K / 128);", "return N * K / 8 + N * (K / 128);",
     [lambda o: pins.test_footprint_is_1_125_bits_per_weight(o)]),
    ("ternary_scale_index_transposed", _SCALE + _TER, _SCALE_T + _TER,
     [lambda o: pins.test_ternary_brute_force_matches_dense(o, 5, 256, 3, 0)]),
    ("ternary_batch_row_ignored", _XT, _XT.replace("x[b * K + k]", "x[k]"),
     [lambda o: pins.test_ternary_brute_force_matches_dense(o, 5, 256, 3, 0)]),
    ("ternary_reads_one_plane", "return (va + vb) / 2;", "return va;",
     [lambda o: pins.test_ternary_brute_force_matches_dense(o, 5, 256, 3, 0),
      lambda o: pins.test_ternary_all_zero_codes_give_exact_zero(o)]),
    ("ternary_zero_subtracts", "else if (t < 0)\n                        part -= xv;",
     "else if (t <= 0)\n                        part -= xv;",
     [lambda o: pins.test_ternary_brute_force_matches_dense(o, 5, 256, 3, 0),
      lambda o: pins.test_ternary_single_code_closed_form(o)]),
    ("ternary_planes_threshold", "if (v >= 0)\n                pa", "if (v > 0)\n                pa",
     [lambda o: pins.test_ternary_planes_match_numpy(o)]),
    ("ternary_codes_unchecked", "if (t[i] < -1 || t[i] > 1)\n            return ORC_ERANGE;\n    memset",
     "if (t[i] < -2 || t[i] > 2)\n            return ORC_ERANGE;\n    memset",
     [lambda o: pins.test_ternary_planes_reject_other_codes(o, 2)]),
    ("ternary_footprint_one_plane", "return 2 * (N * K / 8) + 2 * N * (K / 128);",
     "return (N * K / 8) + 2 * N * (K / 128);",
     [lambda o: pins.test_ternary_footprint_and_printed_sizes(o)]),
    ("t5_digit_order_reversed", "    while (i-- > 0)\n        v /= 3;",
     "    i = (j < 25 ? 4 : 2) - i;\n    while (i-- > 0)\n        v /= 3;",
     [lambda o: pins.test_t5_pack_matches_numpy(o),
      lambda o: pins.test_t5_every_byte_value_decodes_to_its_base3_digits(o)]),
    ("t5_codes_unchecked", "if (t[i] < -1 || t[i] > 1)\n            return ORC_ERANGE;\n    for (int64_t n",
     "if (t[i] < -1 || t[i] > 3)\n            return ORC_ERANGE;\n    for (int64_t n",
     [lambda o: pins.test_t5_rejects_out_of_range(o)]),
    ("t5_group_stride", "int i = (int)(r % 5), v = p[(n * G + g) * 26 + j];",
     "int i = (int)(r % 5), v = p[(n * G + g) * 25 + j];",
     [lambda o: pins.test_t5_pack_matches_numpy(o)]),
    ("t5_last_byte_unchecked", "if (v > (j < 25 ? 242 : 26))", "if (v > 242)",
     [lambda o: pins.test_t5_rejects_out_of_range(o)]),
    ("t5_code_offset", "    return v % 3 - 1;", "    return 1 - v % 3;",
     [lambda o: pins.test_t5_gemv_matches_dense_and_planes(o, 4, 256, 2)]),
    ("t5_footprint_padded", "return N * (K / 128) * 26 + 2 * N * (K / 128);",
     "return N * (K / 128) * 32 + 2 * N * (K / 128);",
     [lambda o: pins.test_t5_footprint_between_ideal_and_slots(o)]),
    ("swiglu_gate_up_swapped", _GU + _HF, _GU_SW + _HF,
     [lambda o: pins.test_swiglu_matches_dense_and_library_silu(o, 6, 256, 2, 1),
      lambda o: pins.test_swiglu_zero_gate_or_zero_up_gives_zero(o)]),
    ("swiglu_sigmoid_sign", _HF + " g / (1.0 + exp(-g)) * u", _HF + " g / (1.0 + exp(g)) * u",
     [lambda o: pins.test_swiglu_closed_form_saturation(o),
      lambda o: pins.test_swiglu_matches_dense_and_library_silu(o, 6, 256, 2, 1)]),
    ("swiglu_sigmoid_without_g", _HF + " g / (1.0 + exp(-g)) * u", _HF + " 1.0 / (1.0 + exp(-g)) * u",
     [lambda o: pins.test_swiglu_zero_gate_or_zero_up_gives_zero(o)]),
    ("swiglu_batch_row_ignored", _HF + " g /", "\n            h[n] = g /",
     [lambda o: pins.test_swiglu_matches_dense_and_library_silu(o, 10, 384, 3, 2)]),
    ("swiglu_odd_rows_accepted", "    if (N2 % 2 != 0)\n        return ORC_ESHAPE;\n    if (!bits || !scales || !x || !h)\n",
     "    if (!bits || !scales || !x || !h)\n",
     [lambda o: pins.test_swiglu_rejects_odd_row_count(o)]),
    ("swiglu_select_batch_row_ignored", "h[b * n_sel + i] = g", "h[i] = g",
     [lambda o: pins.test_swiglu_select_matches_full(o)]),
    ("swiglu_select_gate_up_swapped", _GU + "\n            h[b * n_sel + i] =",
     _GU_SW + "\n            h[b * n_sel + i] =",
     [lambda o: pins.test_swiglu_select_matches_full(o)]),
    ("ternary_swiglu_gate_up_swapped", "double gt = y[b * N2 + 2 * n], up = y[b * N2 + 2 * n + 1];",
     "double up = y[b * N2 + 2 * n], gt = y[b * N2 + 2 * n + 1];",
     [lambda o: pins.test_ternary_swiglu_matches_dense_and_library_silu(o, 8, 256, 2, 1),
      lambda o: pins.test_ternary_swiglu_without_zeros_is_the_binary_pair(o)]),
    ("ternary_swiglu_sigmoid_sign", "gt / (1.0 + exp(-gt)) * up", "gt / (1.0 + exp(gt)) * up",
     [lambda o: pins.test_ternary_swiglu_matches_dense_and_library_silu(o, 8, 256, 2, 1)]),
]


@pytest.mark.parametrize("name,old,new,checks", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, checks):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique/found"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-D_GNU_SOURCE", "-shared", "-fPIC", "-pthread",
                    str(mpath), "-o", str(so), "-lm"], check=True)
    saved = oracle._lib
    oracle._lib = oracle.configure(ctypes.CDLL(str(so)))
    caught = 0
    try:
        for chk in checks:
            try:
                chk(oracle)
            except (AssertionError, oracle.OracleError, pytest.fail.Exception):
                caught += 1
    finally:
        oracle._lib = saved
    assert caught >= 1, f"mutant {name} survived every pin"
