"""Evidence that the oracle pins are strong: plant one plausible mistake at a
time in a copy of the oracle's C source (on the CPU), build it, swap it in, and
check that at least one pin in ``test_oracle_pins.py`` fails.
"""
import ctypes
import os
import shutil
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "cider_oracle.c")
HDR = os.path.join(os.path.dirname(oracle.__file__), "cider_oracle.h")

# (name, original text, planted mistake)
MUTATIONS = [
    ("round_half_away", "float r = nearbyintf(v / scale);", "float r = roundf(v / scale);"),
    ("reciprocal_multiply", "float r = nearbyintf(v / scale);",
     "float r = nearbyintf(v * (1.0f / scale));"),
    ("zero_block_scale", "return (amax == 0.0f) ? 1.0f : amax / qdiv;", "return amax / qdiv;"),
    ("scale_by_128", "float s = block_scale(amax, 127.0f);", "float s = block_scale(amax, 128.0f);"),
    ("int4_qdiv_8", "quantize_weight(W, N, K, group_size, 7.0f, -8, 7, q4, sw);",
     "quantize_weight(W, N, K, group_size, 8.0f, -8, 7, q4, sw);"),
    ("nibble_order", "unsigned lo = (unsigned)(q[n * K + 2 * j] & 0xF);",
     "unsigned lo = (unsigned)(q[n * K + 2 * j + 1] & 0xF);"),
    ("nibble_sign", "return (t < 8u) ? (int)t : (int)t - 16;", "return (t < 8u) ? (int)t : (int)t - 8;"),
    ("gemm_transposed", "s += (int64_t)qa[m * K + k] * (int64_t)qw[n * K + k];",
     "s += (int64_t)qa[m * K + k] * (int64_t)qw[(k % N) * K + n % K];"),
    ("gemm_dropped_term", "for (int64_t j = 0; j < gs; ++j) {\n          int64_t k",
     "for (int64_t j = 1; j < gs; ++j) {\n          int64_t k"),
    ("pg_reversed_order", "for (int64_t g = 0; g < G; ++g) {\n        float scale",
     "for (int64_t g = G - 1; g >= 0; --g) {\n        float scale"),
    ("pc_dropped_weight_scale", "v = v * sw[n];", "v = v * 1.0f;"),
    ("act_amax_signed", "float a = fabsf(widen(row[k]));", "float a = widen(row[k]);"),
    ("bf16_widen_shift", "uint32_t w = (uint32_t)bits << 16;", "uint32_t w = (uint32_t)bits << 15;"),
    ("bf16_read_as_fp16", "quantize_act_rows(x_bf16, M, K, bf16_bits_to_f32, qa, sa);",
     "quantize_act_rows(x_bf16, M, K, f16_bits_to_f32, qa, sa);"),
    ("offset_zero_point_7", "int lo = (int)(src[i] & 0xFu) - 8;", "int lo = (int)(src[i] & 0xFu) - 7;"),
    ("offset_high_nibble_kept", "int hi = (int)(src[i] >> 4) - 8;", "int hi = nibble_value(src[i] >> 4);"),
    ("bf16_truncate", "return (uint16_t)((u + 0x7FFFu + lsb) >> 16);", "return (uint16_t)(u >> 16);"),
    ("bf16_ties_away", "return (uint16_t)((u + 0x7FFFu + lsb) >> 16);",
     "return (uint16_t)((u + 0x8000u) >> 16);"),
    ("clip_rank_n", "const double h = (double)(n - 1) * p / 100.0;",
     "const double h = (double)n * p / 100.0;"),
    ("clip_nearest_lower_rank", "const float t = (float)(h - (double)lo);", "const float t = 0.0f;"),
]

PIN_TESTS = [
    pins.test_quantize_act_hand_worked_cases,
    lambda: pins.test_quantize_act_brute_force_all_fp16_below_amax(3.140625),
    lambda: pins.test_quantize_act_brute_force_all_fp16_below_amax(1000.0),
    lambda: pins.test_quantize_act_brute_force_all_fp16_below_amax(0.0016956329345703125),
    pins.test_quantize_act_zero_row_and_signs,
    pins.test_weight_quant_hand_worked_cases,
    lambda: pins.test_weight_quant_matches_independent_blockwise(64, 8),
    lambda: pins.test_weight_quant_matches_independent_blockwise(0, 4),
    pins.test_int4_nibbles_hand_worked,
    pins.test_int4_unpack_exhaustive_and_pack_roundtrip,
    pins.test_gemm_closed_forms,
    pins.test_gemm_brute_force_python_ints_and_group_sums,
    pins.test_gemm_is_not_transposed,
    pins.test_dequant_pc_special_cases,
    pins.test_dequant_pc_exact_emulation,
    pins.test_dequant_pg_order_hand_worked,
    pins.test_dequant_pg_exact_emulation,
    pins.test_quantize_act_bf16_hand_worked_cases,
    lambda: pins.test_quantize_act_bf16_brute_force_all_bf16_below_amax(0x4049),
    pins.test_quantize_act_bf16_agrees_with_fp16_on_shared_values,
    pins.test_int4_offset_binary_hand_worked,
    pins.test_int4_offset_binary_exhaustive,
    pins.test_bf16_output_rounding_matches_pytorch,
    pins.test_dequant_bf16_special_cases,
    pins.test_clip_percentile_hand_worked_cases,
    lambda: pins.test_clip_percentile_matches_numpy_linear_percentile(128, 99.9),
    lambda: pins.test_clip_percentile_100_is_min_max(64),
]


@pytest.mark.parametrize("name,orig,bad", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, orig, bad):
    src = open(SRC).read()
    assert src.count(orig) >= 1, f"mutation anchor for {name} not found"
    shutil.copy(HDR, tmp_path / "cider_oracle.h")
    (tmp_path / "cider_oracle.c").write_text(src.replace(orig, bad))
    so = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-fPIC", "-shared",
                           "-o", str(so), str(tmp_path / "cider_oracle.c"), "-lm"])
    mutated = oracle._configure(ctypes.CDLL(str(so)))
    saved = oracle._load()
    caught = []
    try:
        oracle._lib = mutated
        for t in PIN_TESTS:
            try:
                t()
            except (AssertionError, OverflowError, ValueError):
                caught.append(getattr(t, "__name__", "lambda"))
    finally:
        oracle._lib = saved
    assert caught, f"no pin caught the planted mistake {name}"
