"""The pins are strong enough: each plausible mistake, planted in a copy of the oracle on
the CPU, makes at least one pin fail.  The mutants are textual edits of the oracle
source, compiled to a temporary library; the pins below are a fast subset of
tests/test_oracle_pins.py run against that library."""
import os
import shutil
import subprocess
import tempfile

import pytest
import torch

import oracle as O
import test_oracle_pins as pins
import test_oracle_pins_bounds as bpins
import test_oracle_pins_next as npins

SRC = os.path.join(os.path.dirname(O.__file__), "ptgq_oracle.cpp")

# (name, original text, mutated text).  Every mutant keeps the oracle's memory accesses in
# bounds: the mutated library runs inside the test process.
MUTANTS = [
    ("amax without abs", "amax = std::fmax(amax, std::fabs(v[i]));", "amax = std::fmax(amax, v[i]);"),
    ("no eps floor", "amax = std::fmax(amax, eps);", ""),
    ("wrong FMAX", "out_dtype == OUT_E4M3 ? 448.0f : 127.0f", "out_dtype == OUT_E4M3 ? 480.0f : 127.0f"),
    ("UE8M0 without round-up", "(b & 0x7FFFFF) != 0 ? 1 : 0", "0"),
    ("e4m3 truncation", "std::nearbyint((2.0 * f - 1.0) * 8.0)", "std::floor((2.0 * f - 1.0) * 8.0)"),
    ("e4m3 ties away", "std::nearbyint(a * 512.0)", "std::round(a * 512.0)"),
    ("no saturation", "if (a > 448.0) a = 448.0;", ""),
    ("silu exp sign", "const float e = exp_f32(-g);", "const float e = exp_f32(g);"),
    ("silu 1 - e", "const float d = 1.0f + e;", "const float d = 1.0f - e;"),
    ("silu association (g * u) / d", "  const float s = g / d;\n  return s * u;",
     "  const float s = g * u;\n  return s / d;"),
    ("reciprocal multiply", "const float y = v[i] / scale;", "const float y = v[i] * (1.0f / scale);"),
    ("col-major transposed", "col * g.mn_pad + row", "row * g.mn_pad + col"),
    ("packed byte order", "<< (8 * j)", "<< (8 * (3 - j))"),
    ("masked rows ignored", "live = masked_m[b];", "live = tokens_pad;"),
    ("no flat zero-fill", "for (int64_t c = 0; c < H; ++c) qb[r * H + c] = 0;",
     "for (int64_t c = 0; c < H; ++c) qb[r * H + c] = qb[r * H + c];"),
    ("int8 without clamp", "if (r > 127.0) r = 127.0;", ""),
    ("fp16 exponent bias", "e - 25", "e - 24"),
    ("UE8M0 float off by one", "return bits_to_float(static_cast<uint32_t>(e) << 23);",
     "return bits_to_float(static_cast<uint32_t>(e + 1) << 23);"),
    ("quotient bound half as wide", "std::ldexp(1.0, ex - 23)", "std::ldexp(1.0, ex - 24)"),
    ("quotient bound twice as wide", "std::ldexp(1.0, ex - 23)", "std::ldexp(1.0, ex - 22)"),
    ("quotient bound ignores the sign of k", "const double b = e + k * u;",
     "const double b = e + (k > 0 ? k : -k) * u;"),
    ("quotient bound ulp of the scale's binade", "std::ilogb(e)", "std::ilogb(s)"),
    # per-token (whole-row) quantization
    ("per-token divides instead of multiplying by the reciprocal", "float y = val(i) * inv;",
     "float y = s == 0.0f ? 0.0f : val(i) / s;"),
    ("per-token zero row unguarded", "const float inv = s == 0.0f ? 0.0f : 1.0f / s;",
     "const float inv = 1.0f / s;"),
    ("per-token max without abs", "m = std::fmax(m, std::fabs(val(i)));", "m = std::fmax(m, val(i));"),
    ("per-token scale with the wrong FMAX", "const float s = m / 448.0f;", "const float s = m / 480.0f;"),
    ("per-token clamp with max first", "y = std::fmax(std::fmin(y, 448.0f), -448.0f);",
     "y = std::fmin(std::fmax(y, -448.0f), 448.0f);"),
    # NaN quotients (infinite amax)
    ("e4m3 NaN saturated", "if (std::isnan(y)) return 0x7F;", "if (std::isnan(y)) return 0x7E;"),
    ("int8 NaN as -128", "if (std::isnan(y)) return 0;", "if (std::isnan(y)) return -128;"),
    # per-token-group -> per-tensor requantization
    ("requant multiplies by the output scale", "const float inv = 1.0f / output_scale;",
     "const float inv = output_scale;"),
    ("requant product order", "const float y = (e4m3_decode(x[i]) * sc) * inv;",
     "const float y = e4m3_decode(x[i]) * (sc * inv);"),
    ("requant ignores masked_m", "int64_t live = masked_m[e];", "int64_t live = M;"),
    ("requant group index from the row", "(k / group_size) * stride_g", "(m / group_size) * stride_g"),
]

# Fast pins: each a callable that raises when the oracle is wrong.
FAST_PINS = [
    pins.test_e4m3_hand_ties_fixture,
    pins.test_int8_encoder_vs_numpy_rint_clip,
    pins.test_ue8m0_closed_forms,
    pins.test_silu_mul_closed_forms_and_error_bound,
    lambda: pins.test_fp16_decode_matches_numpy_all_patterns(),
    lambda: pins.test_vllm_all_zero_worked_example(5),
    pins.test_all_zero_without_floor_closed_form,
    pins.test_mantissa_rounds_up,
    lambda: pins.test_random_rows_vs_library_composition(128, O.OUT_E4M3, O.FMT_FP32),
    lambda: pins.test_scale_layouts_index_and_padding(O.LAYOUT_COL, O.FMT_UE8M0_PACKED),
    lambda: pins.test_scale_layouts_index_and_padding(O.LAYOUT_COL, O.FMT_FP32),
    lambda: pins.test_scale_layouts_index_and_padding(O.LAYOUT_ROW, O.FMT_UE8M0_FP32),
    pins.test_masked_rows_match_flat_and_padding_untouched,
    bpins.test_hand_ties_widen_to_both_neighbours,
    lambda: npins.test_per_token_vs_library_composition(torch.bfloat16, 1076),
    lambda: npins.test_per_token_vs_library_composition(torch.float32, 1368),
    npins.test_per_token_integer_rows_exact,
    npins.test_per_token_midpoint_rounding_and_padded_tail,
    lambda: npins.test_requant_masked_rows_and_k_tail(1152),
    npins.test_requant_vs_library_composition_and_saturation,
    npins.test_per_token_multiplies_by_the_reciprocal,
    npins.test_requant_scales_first_then_the_output_scale,
    npins.test_per_token_reciprocal_overflow_fixture,
    lambda: pins.test_nonfinite_amax_fixture(O.FMT_FP32),
    lambda: pins.test_nonfinite_amax_fixture(O.FMT_UE8M0_PACKED),
    # the slow ones last (several seconds each), so most mutants fail before reaching them
    lambda: pins.test_silu_mul_every_16bit_gate("bf16"),
    pins.test_e4m3_encoder_vs_exhaustive_argmin_and_saturation,
    pins.test_integer_rows_exact_closed_form,
    lambda: _bound_width_pins(),                       # 4M silu values
]


def _bound_width_pins():
    data = bpins.silu_values_data()
    for out in (O.OUT_E4M3, O.OUT_INT8):
        bpins.test_bounds_part_where_a_boundary_is_within_k_ulps(data, out)


def _build_mutant(src_text: str, tmp: str) -> str:
    cpp = os.path.join(tmp, "mutant.cpp")
    lib = os.path.join(tmp, "libmutant.so")
    with open(cpp, "w") as f:
        f.write(src_text)
    subprocess.run(["g++", "-O1", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", "-o", lib, cpp], check=True)
    return lib


def _swap_oracle_lib(lib_path):
    """Point the oracle module at another library (None restores the real one)."""
    O._lib = None
    if lib_path is None:
        O._LIB = os.path.join(os.path.dirname(O.__file__), "libptgq_oracle.so")
        O.build = _REAL_BUILD
        O.lib()
    else:
        O._LIB = lib_path
        O.build = lambda force=False, _p=lib_path: _p   # never rebuild over the mutant
        O.lib()


_REAL_BUILD = O.build


def test_unmutated_source_passes_fast_pins():
    for pin in FAST_PINS:
        pin()


@pytest.mark.parametrize("name,orig,mut", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, orig, mut):
    text = open(SRC).read()
    assert text.count(orig) >= 1, f"mutation point for '{name}' not found"
    tmp = tempfile.mkdtemp()
    try:
        _swap_oracle_lib(_build_mutant(text.replace(orig, mut), tmp))
        caught = None
        for pin in FAST_PINS:
            try:
                pin()
            except Exception as exc:           # any failing pin counts as caught
                caught = exc
                break
        assert caught is not None, f"no pin caught the planted mistake '{name}'"
    finally:
        _swap_oracle_lib(None)
        shutil.rmtree(tmp, ignore_errors=True)
