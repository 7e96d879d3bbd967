"""Pins for the oracle's quotient bounds, which check the fast-math compatibility mode
(sglang PR #34257, "Implementation notes": a fast-math build divides by the scale with a
different rounding; sglang PR #30924, "Risks": about 0.2% of int8 codes then differ by
one).  That mode's division is only known to lie within 2 ulps of the exact quotient
(CUDA Math API, single-precision intrinsics, __fdividef), so the oracle gives, per
element, the codes of the quotient moved k binary32 ulps down and up.

Independent references: numpy's ``spacing`` for the binary32 ulp, torch's fp8 cast and
numpy's rint for the encodings, and hand-worked ties."""
import numpy as np
import pytest
import torch

import oracle as O
from fp8_token_group_gb300 import synth


def _run(x: torch.Tensor, k: int, out_dtype: int, fmt: int = O.FMT_FP32):
    n, H = x.shape
    q = np.zeros(n * H, np.uint8)
    s = np.zeros(O.scale_elems(n, 0, H, 128, fmt, O.LAYOUT_ROW, 0),
                 np.uint32 if fmt == O.FMT_UE8M0_PACKED else np.float32)
    in_dt = O.IN_BF16 if x.dtype == torch.bfloat16 else O.IN_FP16
    O.quant(synth.bits_u16(x), in_dt, n, 0, H, 128, q, out_dtype, s, fmt, O.LAYOUT_ROW, 0, None,
            1e-10, 0, k)
    return q.reshape(n, H), s


def _anchored_grid(vals: np.ndarray, anchor: float) -> np.ndarray:
    """Rows of 128: the anchor (so that s = anchor / FMAX = 1 exactly) and 127 values."""
    per = 127
    ng = -(-len(vals) // per)
    buf = np.zeros(ng * per, np.float32)
    buf[: len(vals)] = vals
    return np.concatenate([np.full((ng, 1), anchor, np.float32), buf.reshape(ng, per)], 1)


def _all_bf16_values(limit: float) -> np.ndarray:
    vals = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    return vals[np.isfinite(vals) & (np.abs(vals) <= limit)]


def test_zero_ulps_is_the_operation():
    x = synth.flat_small()
    for out in (O.OUT_E4M3, O.OUT_INT8):
        q0, s0 = _run(x, 0, out)
        n, H = x.shape
        q = np.zeros(n * H, np.uint8)
        s = np.zeros_like(s0)
        O.quant(synth.bits_u16(x), O.IN_BF16, n, 0, H, 128, q, out, s, O.FMT_FP32, O.LAYOUT_ROW,
                0, None, 1e-10)
        assert np.array_equal(q0.ravel(), q) and np.array_equal(s0, s)


def test_hand_ties_widen_to_both_neighbours():
    """s = 1: an exact e4m3 tie moves to the code on either side; values away from a tie
    keep their code; zero takes -0 below and +0 above."""
    vals = np.array([1.0625, 17.0, -2.0 ** -10, 0.0, 3.0, 448.0], np.float32)
    x = torch.from_numpy(_anchored_grid(vals, 448.0)).to(torch.bfloat16)
    lo, s_lo = _run(x, -2, O.OUT_E4M3)
    hi, s_hi = _run(x, 2, O.OUT_E4M3)
    ex, s_ex = _run(x, 0, O.OUT_E4M3)
    assert np.all(s_lo == 1.0) and np.array_equal(s_lo, s_hi) and np.array_equal(s_lo, s_ex)
    #                         1.0625  17    -2^-10  0     3     448
    assert list(ex[0, 1:7]) == [0x38, 0x58, 0x80, 0x00, 0x44, 0x7E]
    assert list(lo[0, 1:7]) == [0x38, 0x58, 0x81, 0x80, 0x44, 0x7E]
    assert list(hi[0, 1:7]) == [0x39, 0x59, 0x80, 0x00, 0x44, 0x7E]


@pytest.mark.parametrize("k", [-2, 2, -5, 5])
def test_e4m3_bounds_every_bf16_value(k):
    """s = 1, so the exact quotient is v itself and the bound is v + k * ulp(v), which is a
    binary32 value for every bf16 v (8 significant bits): torch's cast of it, after the
    saturation, is the expected code."""
    grid = _anchored_grid(_all_bf16_values(448), 448.0)
    x = torch.from_numpy(grid).to(torch.bfloat16)
    q, s = _run(x, k, O.OUT_E4M3)
    assert np.all(s == 1.0)
    b = grid.astype(np.float64) + k * np.spacing(np.abs(grid)).astype(np.float64)
    assert np.array_equal(b.astype(np.float32).astype(np.float64), b)
    want = torch.from_numpy(np.clip(b, -448, 448).astype(np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, want)


@pytest.mark.parametrize("k", [-2, 2])
def test_int8_bounds_every_bf16_value(k):
    grid = _anchored_grid(_all_bf16_values(127), 127.0)
    x = torch.from_numpy(grid).to(torch.bfloat16)
    q, s = _run(x, k, O.OUT_INT8)
    assert np.all(s == 1.0)
    b = grid.astype(np.float64) + k * np.spacing(np.abs(grid)).astype(np.float64)
    want = np.clip(np.rint(b), -128, 127).astype(np.int8)
    assert np.array_equal(q.view(np.int8), want)
    # the int8 ties (y = m + 1/2) are exactly where the two bounds part
    lo, _ = _run(x, -2, O.OUT_INT8)
    hi, _ = _run(x, 2, O.OUT_INT8)
    half = np.abs(grid - np.trunc(grid)) == 0.5
    assert np.array_equal(lo != hi, half)


def test_bounds_bracket_the_exact_codes_with_general_scales():
    """Random groups (scales not powers of two): lower code <= exact code <= upper code in
    value.  The bounds part only where the quotient lies within 2 ulps of a rounding
    boundary: with bf16 inputs that is about 0.2% of int8 codes, the share of codes the
    pages report changed by a fast-math build, and about 0.6% of e4m3 codes."""
    x = synth.flat_small()
    for out in (O.OUT_E4M3, O.OUT_INT8):
        lo, _ = _run(x, -2, out)
        ex, _ = _run(x, 0, out)
        hi, _ = _run(x, 2, out)
        if out == O.OUT_E4M3:
            val = lambda c: torch.from_numpy(np.ascontiguousarray(c)).view(
                torch.float8_e4m3fn).float().numpy()
        else:
            val = lambda c: c.view(np.int8).astype(np.float32)
        assert np.all(val(lo) <= val(ex)) and np.all(val(ex) <= val(hi))
        assert 0 < (lo != hi).mean() < (1e-2 if out == O.OUT_E4M3 else 4e-3)
