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


def _e4m3_midpoints() -> np.ndarray:
    """The rounding boundaries of the e4m3 encoder: midpoints between neighbouring finite
    values of the format (from its value table), both signs."""
    vals = set()
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            continue
        v = m / 512 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        vals.add(-v if s else v)
    vals = np.array(sorted(vals))
    return (vals[1:] + vals[:-1]) / 2


def silu_values_data():
    """4M fused-silu values, from the oracle as loaded: continuous binary32 quotients,
    unlike the 16-bit inputs, whose quotients lie either within about one ulp of a rounding
    boundary or far from it."""
    T, H = 2048, 2048
    x = synth.normal((T, 2 * H), torch.bfloat16, seed=5)
    xf = x.float().numpy()
    f = O.lib().oracle_silu_mul
    g, u = xf[:, :H].ravel().tolist(), xf[:, H:].ravel().tolist()
    v = np.fromiter((f(a, b) for a, b in zip(g, u)), dtype=np.float64, count=len(g))
    return x, v, T, H


@pytest.fixture(scope="module")
def silu_values():
    return silu_values_data()


@pytest.mark.parametrize("out", [O.OUT_E4M3, O.OUT_INT8])
def test_bounds_part_where_a_boundary_is_within_k_ulps(silu_values, out):
    """Independent of the oracle's bound arithmetic: with the exact quotient y = v / s (in
    binary64, far finer than a binary32 ulp) and the encoder's rounding boundaries (e4m3
    midpoints from the format's value table, or half-integers for int8), the k = 2 bounds
    must part wherever a boundary lies within 1.95 ulps of y and never where it lies beyond
    3.05 ulps (the bound is rounded outward, which can add up to one ulp).  Enough quotients
    fall in both bands that a bound of half or twice the width fails here."""
    x, v, T, H = silu_values
    bits = synth.bits_u16(x)

    def run(k):
        q = np.zeros(T * H, np.uint8)
        s = np.zeros(T * (H // 128), np.float32)
        O.quant(bits, O.IN_BF16, T, 0, H, 128, q, out, s, O.FMT_FP32, O.LAYOUT_ROW, 1, None,
                1e-10, 0, k)
        return q, s

    lo, s = run(-2)
    hi, _ = run(2)
    y = v / np.repeat(s.astype(np.float64), 128)
    ulp = np.spacing(np.abs(y).astype(np.float32)).astype(np.float64)
    if out == O.OUT_E4M3:
        mids = _e4m3_midpoints()
        j = np.searchsorted(mids, y)
        d = np.minimum(np.abs(y - mids[np.clip(j - 1, 0, len(mids) - 1)]),
                       np.abs(y - mids[np.clip(j, 0, len(mids) - 1)]))
    else:
        d = np.abs(y - (np.floor(y) + 0.5))
        d[np.abs(y) > 127.4] = np.inf           # saturated: no boundary to cross
    r = d / ulp
    parted = lo != hi
    near, far = r < 1.95, r > 3.05
    assert ((r > 1) & near).sum() >= 3 and (far & (r < 5)).sum() >= 10
    assert np.all(parted[near]), int((near & ~parted).sum())
    assert not np.any(parted[far]), int((far & parted).sum())
