"""Pins for the CPU oracle: each oracle function is checked against something other
than itself -- the format definitions, closed forms, library routines (torch's fp8
cast, numpy's IEEE binary32 arithmetic, mpmath at 100 bits), exhaustive enumeration
of every 16-bit input, and the worked example printed on the vLLM PR #41326 page.

The mistakes these are meant to catch: a missing abs or eps, a wrong FMAX, UE8M0
without the round-up, ties away from zero instead of to even, a missing saturation,
exp(g) for exp(-g), another rounding order in silu * up, transposed or mis-packed
scale layouts, rows written past masked_m, missing zero-fill.
"""
import os
from fractions import Fraction

import mpmath
import numpy as np
import pytest
import torch

import oracle as O
from fp8_token_group_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32 = np.float32


# ---------------------------------------------------------------- independent references

def e4m3_value_table():
    """Values of the 256 e4m3fn codes from the format definition (NaN for 0x7F, 0xFF)."""
    vals = np.empty(256, dtype=np.float64)
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            vals[c] = np.nan
            continue
        v = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        vals[c] = -v if s else v
    return vals


E4M3_VALUES = e4m3_value_table()


def e4m3_argmin(y: float) -> int:
    """Nearest code by exhaustive search; ties to the even code; clamp to +-448 first."""
    y = min(max(float(y), -448.0), 448.0)
    neg = np.signbit(y)
    best, best_d = None, None
    for c in range(256):
        v = E4M3_VALUES[c]
        if np.isnan(v) or (c >= 128) != neg:
            continue
        d = abs(Fraction(v) - Fraction(y))
        if best is None or d < best_d or (d == best_d and (c & 1) == 0):
            best, best_d = c, d
    return best


def f32_rn(v) -> np.float32:
    """Round an mpmath value to the nearest binary32 (exact comparison of neighbours)."""
    if v >= mpmath.mpf(2) ** 128 - mpmath.mpf(2) ** 103:   # at or past FLT_MAX + ulp/2
        return F32(np.inf)
    c = F32(float(v))
    cands = [np.nextafter(c, F32(-np.inf)), c, np.nextafter(c, F32(np.inf))]
    cands = [x for x in cands if np.isfinite(x)]
    return min(cands, key=lambda f: abs(mpmath.mpf(float(f)) - v))


def all_bf16():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def bf16_values():
    return (all_bf16().astype(np.uint32) << 16).view(np.float32)


def fp16_values():
    return all_bf16().view(np.float16).astype(np.float32)


# ---------------------------------------------------------------- element decoding

def test_bf16_decode_matches_torch_all_patterns():
    ref = torch.from_numpy(all_bf16().view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    got = np.array([O.bf16_to_float(int(h)) for h in all_bf16()], dtype=np.float32)
    assert np.array_equal(got.view(np.uint32)[~np.isnan(ref)], ref.view(np.uint32)[~np.isnan(ref)])
    assert np.all(np.isnan(got[np.isnan(ref)]))


def test_fp16_decode_matches_numpy_all_patterns():
    ref = fp16_values()
    got = np.array([O.fp16_to_float(int(h)) for h in all_bf16()], dtype=np.float32)
    fin = ~np.isnan(ref)
    assert np.array_equal(got.view(np.uint32)[fin], ref.view(np.uint32)[fin])
    assert np.all(np.isnan(got[~fin]))


# ---------------------------------------------------------------- e4m3 / int8 encoders

def test_e4m3_hand_ties_fixture():
    path = os.path.join(GOLDEN, "e4m3_hand_ties.txt")
    n = 0
    for line in open(path):
        if not line.strip() or line.startswith("#"):
            continue
        val, code = line.split()[:2]
        assert O.e4m3_encode(float(val)) == int(code, 16), line
        n += 1
    assert n >= 15


@pytest.mark.parametrize("which", ["bf16", "fp16"])
def test_e4m3_encoder_vs_torch_cast_every_16bit_value(which):
    vals = bf16_values() if which == "bf16" else fp16_values()
    vals = vals[np.isfinite(vals) & (np.abs(vals) <= 448)]
    got = np.array([O.e4m3_encode(float(v)) for v in vals], dtype=np.uint8)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def test_e4m3_encoder_vs_exhaustive_argmin_and_saturation():
    rng = np.random.default_rng(0)
    # every code value, every midpoint between neighbours, random values, out-of-range values
    fin = np.sort(np.unique(E4M3_VALUES[~np.isnan(E4M3_VALUES)]))
    mids = (fin[1:] + fin[:-1]) / 2
    samples = np.concatenate([fin, mids, rng.normal(0, 50, 3000), rng.normal(0, 0.01, 2000),
                              [449.0, 463.9, 464.0, 465.0, 1e6, -1e30, 3.0e38]])
    for y in samples.astype(np.float32):
        assert O.e4m3_encode(float(y)) == e4m3_argmin(float(y)), y


def test_int8_encoder_vs_numpy_rint_clip():
    rng = np.random.default_rng(1)
    halves = np.arange(-260, 261, dtype=np.float32) / 2
    samples = np.concatenate([halves, rng.normal(0, 60, 20000).astype(np.float32), [1e9, -1e9]])
    samples = samples.astype(np.float32)
    ref = np.clip(np.rint(samples.astype(np.float64)), -128, 127).astype(np.int8)
    got = np.array([O.int8_encode(float(v)) for v in samples], dtype=np.int8)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- exp, silu

@pytest.mark.parametrize("which", ["bf16", "fp16"])
def test_exp_correctly_rounded_every_16bit_input(which):
    mpmath.mp.prec = 100
    vals = bf16_values() if which == "bf16" else fp16_values()
    vals = vals[np.isfinite(vals) & (vals > -104) & (vals < 89)]
    bad = []
    for x in vals:
        got = F32(O.exp_f32(float(x)))
        ref = f32_rn(mpmath.exp(mpmath.mpf(float(x))))
        if got.view(np.uint32) != ref.view(np.uint32):
            bad.append((float(x), got, ref))
    assert not bad, bad[:5]


def _silu_mul_ref(g: np.float32, u: np.float32) -> np.float32:
    """Same rounding sequence with exp from mpmath and binary32 steps from numpy."""
    e = f32_rn(mpmath.exp(-mpmath.mpf(float(g))))
    d = F32(1.0) + e
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        return (g / d) * u


@pytest.mark.parametrize("which", ["bf16", "fp16"])
def test_silu_mul_every_16bit_gate(which):
    mpmath.mp.prec = 100
    vals = bf16_values() if which == "bf16" else fp16_values()
    vals = vals[np.isfinite(vals)]
    us = [F32(1.0), F32(-3.0), F32(0.3330078125)]
    bad = 0
    for i, g in enumerate(vals):
        u = us[i % 3]
        got = F32(O.silu_mul(float(g), float(u)))
        ref = _silu_mul_ref(g, u)
        if got.view(np.uint32) != ref.view(np.uint32):
            bad += 1
    assert bad == 0


def test_silu_mul_closed_forms_and_error_bound():
    # silu(0) = 0; silu(g) = g for large g; silu(g) -> -0 for very negative g
    assert O.silu_mul(0.0, 5.0) == 0.0
    assert O.silu_mul(200.0, 1.0) == 200.0
    r = O.silu_mul(-200.0, 1.0)
    assert r == 0.0 and np.signbit(r)
    # against the exact value: within 3 binary32 ulps (4 rounded steps) for typical inputs
    mpmath.mp.prec = 100
    rng = np.random.default_rng(3)
    for g, u in rng.normal(0, 3, (2000, 2)).astype(np.float32):
        got = O.silu_mul(float(g), float(u))
        exact = mpmath.mpf(float(g)) / (1 + mpmath.exp(-mpmath.mpf(float(g)))) * mpmath.mpf(float(u))
        if exact == 0:
            continue
        ulp = np.spacing(F32(abs(float(exact))))
        assert abs(mpmath.mpf(got) - exact) <= 3 * mpmath.mpf(float(ulp))


# ---------------------------------------------------------------- UE8M0

def test_ue8m0_closed_forms():
    assert O.ue8m0_exponent(1.0) == 127                      # 448 / 448
    assert O.ue8m0_exponent(1.5) == 128                      # amax 672: mantissa rounds up
    assert O.ue8m0_exponent(float(F32(8) / F32(448))) == 122 # 0x3C924925 -> 2^-5
    assert O.pow2_from_biased(127) == 1.0 and O.pow2_from_biased(122) == 2.0 ** -5


def test_ue8m0_is_smallest_power_of_two_not_below_s():
    rng = np.random.default_rng(4)
    raw = rng.integers(0x0C000000, 0x7E000000, 20000, dtype=np.uint32)
    raw[:200] &= 0xFF800000  # exact powers of two
    for s in raw.view(np.float32):
        e = O.ue8m0_exponent(float(s))
        fs = Fraction(float(s))
        assert Fraction(2) ** (e - 127) >= fs > Fraction(2) ** (e - 128), s


# ---------------------------------------------------------------- whole pipeline

def _run(x: torch.Tensor, group, out_dtype=O.OUT_E4M3, fmt=O.FMT_FP32, layout=O.LAYOUT_ROW,
         silu=0, masked_m=None, tokens_pad=0, eps=1e-10, flags=0, fill_q=0, fill_s=0):
    in_dtype = O.IN_BF16 if x.dtype == torch.bfloat16 else O.IN_FP16
    masked = masked_m is not None
    if masked:
        E, tp, hin = x.shape
        n, rows = E, tp
        tokens_pad = tp
    else:
        n, hin = x.shape
        rows = tokens_pad or n
    H = hin // 2 if silu else hin
    q = np.full((n if masked else 1) * rows * H, fill_q, dtype=np.uint8)
    ns = O.scale_elems(n, tokens_pad, H, group, fmt, layout, masked)
    s = np.full(ns, fill_s, dtype=np.uint32 if fmt == O.FMT_UE8M0_PACKED else np.uint32)
    if fmt != O.FMT_UE8M0_PACKED:
        s = s.view(np.float32)
    O.quant(synth.bits_u16(x), in_dtype, n, tokens_pad, H, group, q, out_dtype, s, fmt, layout,
            silu, None if masked_m is None else np.asarray(masked_m), eps, flags)
    return q, s


def _worked_example_params():
    p = {}
    for line in open(os.path.join(GOLDEN, "vllm_all_zero_ue8m0.txt")):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            p[k] = v
    return p


@pytest.mark.parametrize("mn", [4, 5])
def test_vllm_all_zero_worked_example(mn):
    """The printed all-zero example: bytes 0x5E with the 1e-10 scale floor, index layout."""
    p = _worked_example_params()
    H, G = int(p["hidden"]), int(p["group_size"])
    x = torch.zeros((mn, H), dtype=torch.bfloat16)
    q, s = _run(x, G, fmt=O.FMT_UE8M0_PACKED, layout=O.LAYOUT_COL,
                flags=O.FLAG_UE8M0_SCALE_FLOOR, fill_q=0xAB, fill_s=0xDEADBEEF)
    assert np.all(q == int(p["expected_code"], 16))
    byte = int(p["expected_exp_byte"], 16)
    ng = H // G
    k_packed = (ng + 3) // 4
    tma_mn = (mn + 3) // 4 * 4
    expected = np.zeros(k_packed * tma_mn, dtype=np.uint32)
    for row in range(mn):
        for g in range(ng):
            expected[(g // 4) * tma_mn + row] |= byte << (8 * (g % 4))
    assert np.array_equal(s, expected)


def test_all_zero_without_floor_closed_form():
    """Without the vLLM floor: s = RN(1e-10 / 448) and the byte is its rounded-up exponent."""
    x = torch.zeros((3, 256), dtype=torch.bfloat16)
    for out, fmax in ((O.OUT_E4M3, 448), (O.OUT_INT8, 127)):
        q, s = _run(x, 128, out_dtype=out, fmt=O.FMT_UE8M0_PACKED, layout=O.LAYOUT_ROW)
        s_exact = Fraction(float(F32(1e-10) / F32(fmax)))
        e = next(e for e in range(0, 255) if Fraction(2) ** (e - 127) >= s_exact)
        assert e == (85 if fmax == 448 else 87)
        assert np.all(q == 0)
        assert np.all(s == (e | (e << 8)))
        q, s = _run(x, 128, out_dtype=out, fmt=O.FMT_FP32)
        assert np.all(s == F32(1e-10) / F32(fmax))


def test_integer_rows_exact_closed_form():
    """Integers in [-8, 8] (the sglang PR #35593 test idea): every value is exact."""
    g = torch.Generator().manual_seed(5)
    k = torch.randint(-8, 9, (16, 512), generator=g)
    k[:, ::128] = 7  # amax of every group is exactly 7 or 8
    k[::2, 1::128] = -8
    x = k.to(torch.bfloat16)
    kk = k.numpy().reshape(16, 4, 128)
    amax = np.abs(kk).max(-1)
    # UE8M0: s = amax/448 -> 2^(e-127) = 2^-6 for amax 7 (7/448 = 1/64 exactly), 2^-5 for 8
    q, s = _run(x, 128, fmt=O.FMT_UE8M0_FP32)
    pow2 = np.where(amax == 7, 2.0 ** -6, 2.0 ** -5)
    assert np.array_equal(s.reshape(16, 4), pow2.astype(np.float32))
    want = np.array([e4m3_argmin(v) for v in (kk / pow2[..., None]).ravel()], dtype=np.uint8)
    assert np.array_equal(q, want)
    # fp32 scale with amax exactly 7: s = 1/64, codes = e4m3(64 k), all representable
    x7 = k.clamp(-7, 7).to(torch.bfloat16)
    q, s = _run(x7, 128)
    assert np.all(s == F32(1 / 64))
    want = torch.from_numpy((64.0 * k.clamp(-7, 7).numpy()).astype(np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy().ravel()
    assert np.array_equal(q, want)


@pytest.mark.parametrize("which", ["bf16", "fp16"])
@pytest.mark.parametrize("fmt", [O.FMT_FP32, O.FMT_UE8M0_FP32])
def test_brute_force_every_16bit_value_in_a_group_with_anchor(which, fmt):
    """Anchor 448 in each group makes s = 1 (both formats), so q(v) = e4m3(v) for every
    16-bit value with |v| <= 448, checked against torch's fp8 cast."""
    vals = bf16_values() if which == "bf16" else fp16_values()
    vals = vals[np.isfinite(vals) & (np.abs(vals) <= 448)]
    per = 127
    ngroups = -(-len(vals) // per)
    buf = np.zeros(ngroups * per, dtype=np.float32)
    buf[: len(vals)] = vals
    grid = np.concatenate([np.full((ngroups, 1), 448, np.float32), buf.reshape(ngroups, per)], 1)
    dt = torch.bfloat16 if which == "bf16" else torch.float16
    x = torch.from_numpy(grid).to(dt)
    q, s = _run(x, 128, fmt=fmt)
    assert np.all(s == 1.0)
    want = torch.from_numpy(grid.ravel()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, want)


def test_brute_force_int8_with_anchor():
    vals = bf16_values()
    vals = vals[np.isfinite(vals) & (np.abs(vals) <= 127)]
    per = 127
    ngroups = -(-len(vals) // per)
    buf = np.zeros(ngroups * per, dtype=np.float32)
    buf[: len(vals)] = vals
    grid = np.concatenate([np.full((ngroups, 1), 127, np.float32), buf.reshape(ngroups, per)], 1)
    x = torch.from_numpy(grid).to(torch.bfloat16)
    q, s = _run(x, 128, out_dtype=O.OUT_INT8)
    assert np.all(s == 1.0)
    want = np.clip(np.rint(grid.ravel().astype(np.float64)), -128, 127).astype(np.int8)
    assert np.array_equal(q.view(np.int8), want)


def test_mantissa_rounds_up():
    """amax 672 -> s = 1.5 -> byte 128, scale 2 ([vllm#41326] test ..._mantissa_rounds_up)."""
    x = torch.zeros((1, 128), dtype=torch.bfloat16)
    x[0, 0] = 672.0
    x[0, 1] = 3.0
    x[0, 2] = -100.0
    q, s = _run(x, 128, fmt=O.FMT_UE8M0_PACKED)
    assert s[0] == 128
    assert q[0] == O.e4m3_encode(336.0) and q[1] == 0x38 + 4 and q[2] == O.e4m3_encode(-50.0)


def _numpy_reference(x: torch.Tensor, G: int, out: int, fmt: int, eps=1e-10):
    """The definition composed from library routines: numpy binary32 max/abs/divide and
    torch's fp8 cast.  Returns codes [T, H] and per-group scale values [T, ng]."""
    v = x.float().numpy()
    T, H = v.shape
    vg = v.reshape(T, H // G, G)
    amax = np.maximum(np.abs(vg).max(-1), F32(eps)).astype(np.float32)
    fmax = F32(448 if out == O.OUT_E4M3 else 127)
    s = (amax / fmax).astype(np.float32)
    if fmt != O.FMT_FP32:
        e = np.ceil(np.log2(s.astype(np.float64)))  # exact for binary32 s in the normal range
        s = np.exp2(e).astype(np.float32)
    y = (vg / s[..., None]).astype(np.float32).reshape(T, H)
    if out == O.OUT_E4M3:
        q = torch.from_numpy(np.clip(y, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    else:
        q = np.clip(np.rint(y), -128, 127).astype(np.int8).view(np.uint8)
    return q, s


@pytest.mark.parametrize("G", [16, 32, 64, 128])
@pytest.mark.parametrize("out", [O.OUT_E4M3, O.OUT_INT8])
@pytest.mark.parametrize("fmt", [O.FMT_FP32, O.FMT_UE8M0_FP32])
def test_random_rows_vs_library_composition(G, out, fmt):
    x = synth.sweep_input(7, 64, 512, torch.bfloat16)
    q, s = _run(x, G, out_dtype=out, fmt=fmt)
    rq, rs = _numpy_reference(x, G, out, fmt)
    assert np.array_equal(q.reshape(64, 512), rq)
    assert np.array_equal(s.reshape(64, 512 // G), rs)


@pytest.mark.parametrize("layout", [O.LAYOUT_ROW, O.LAYOUT_COL])
@pytest.mark.parametrize("fmt", [O.FMT_FP32, O.FMT_UE8M0_PACKED, O.FMT_UE8M0_FP32])
def test_scale_layouts_index_and_padding(layout, fmt):
    """Every group gets a distinct scale, so a transposed index, a wrong pitch or a wrong
    byte order shows; padded rows are zero, the buffer tail is the sentinel."""
    T, tp, H, G = 5, 7, 7 * 128, 128   # ng = 7: the last packed word has one unused byte
    ng = H // G
    x = torch.zeros((T, H), dtype=torch.float32)
    for r in range(T):
        for g in range(ng):
            x[r, g * G] = float(2.0 ** (r * ng + g - 20))  # distinct power-of-two amax
    x = x.to(torch.bfloat16)
    q, s = _run(x, G, fmt=fmt, layout=layout, tokens_pad=tp, fill_q=0xAB, fill_s=0x7FC00001)
    assert np.all(q.reshape(tp, H)[T:] == 0)
    raw = s.view(np.uint32)
    mn_pad = (tp + 3) // 4 * 4
    ncol = (ng + 3) // 4 if fmt == O.FMT_UE8M0_PACKED else ng
    assert raw.size == (tp * ncol if layout == O.LAYOUT_ROW else ncol * mn_pad)
    for r in range(T):
        for g in range(ng):
            sval = F32(2.0 ** (r * ng + g - 20)) / F32(448)
            e = next(e for e in range(256) if Fraction(2) ** (e - 127) >= Fraction(float(sval)))
            col = g // 4 if fmt == O.FMT_UE8M0_PACKED else g
            idx = r * ncol + col if layout == O.LAYOUT_ROW else col * mn_pad + r
            if fmt == O.FMT_UE8M0_PACKED:
                assert (raw[idx] >> (8 * (g % 4))) & 0xFF == e
            elif fmt == O.FMT_UE8M0_FP32:
                assert s[idx] == F32(2.0 ** (e - 127))
            else:
                assert s[idx] == sval
        if fmt == O.FMT_UE8M0_PACKED:  # unused byte of the last word
            idx = r * ncol + ncol - 1 if layout == O.LAYOUT_ROW else (ncol - 1) * mn_pad + r
            assert raw[idx] >> 24 == 0
    srows = tp if layout == O.LAYOUT_ROW else mn_pad
    for r in range(T, srows):
        for c in range(ncol):
            idx = r * ncol + c if layout == O.LAYOUT_ROW else c * mn_pad + r
            assert raw[idx] == 0


def test_masked_rows_match_flat_and_padding_untouched():
    E, tp, H = 4, 48, 256
    x = synth.normal((E, tp, 2 * H), torch.bfloat16, seed=9)
    mm = np.array([0, 1, 17, tp], dtype=np.int32)   # the sglang PR #35593 test's counts
    q, s = _run(x, 128, silu=1, masked_m=mm, fmt=O.FMT_UE8M0_PACKED, layout=O.LAYOUT_COL,
                fill_q=0x7F, fill_s=0xFFFFFFFF)
    q = q.reshape(E, tp, H)
    ncol, mn_pad = 1, 48
    s = s.reshape(E, ncol, mn_pad)
    for e in range(E):
        m = mm[e]
        assert np.all(q[e, m:] == 0x7F) and np.all(s[e, :, m:] == 0xFFFFFFFF)
        if m:
            fq, fs = _run(x[e, :m].contiguous(), 128, silu=1, fmt=O.FMT_UE8M0_PACKED,
                          layout=O.LAYOUT_COL, tokens_pad=m)
            assert np.array_equal(q[e, :m].ravel(), fq)
            assert np.array_equal(s[e, 0, :m], fs[:m])
    # out-of-range counts are clamped to [0, tokens_pad]
    q2, _ = _run(x, 128, silu=1, masked_m=np.array([-5, 0, 1000, 3], np.int32), fill_q=0x7F)
    q2 = q2.reshape(E, tp, H)
    assert np.all(q2[0] == 0x7F) and np.all(q2[1] == 0x7F)
    full, _ = _run(x[2].contiguous(), 128, silu=1)
    assert np.array_equal(q2[2].ravel(), full)


def test_ue8m0_fp32_format_equals_packed_exponents():
    x = synth.flat_outliers(tokens=32, hidden=1024)
    _, sp = _run(x, 128, fmt=O.FMT_UE8M0_PACKED)
    _, sf = _run(x, 128, fmt=O.FMT_UE8M0_FP32)
    bytes_ = sp.view(np.uint8).reshape(32, 8)
    assert np.array_equal(sf.view(np.uint32).reshape(32, 8), bytes_.astype(np.uint32) << 23)


def test_scale_floor_only_affects_tiny_scales():
    x = synth.flat_small()[:8]
    _, a = _run(x, 128, fmt=O.FMT_UE8M0_PACKED)
    _, b = _run(x, 128, fmt=O.FMT_UE8M0_PACKED, flags=O.FLAG_UE8M0_SCALE_FLOOR)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------- infinite amax

@pytest.mark.parametrize("fmt", [O.FMT_FP32, O.FMT_UE8M0_PACKED, O.FMT_UE8M0_FP32])
def test_nonfinite_amax_fixture(fmt):
    """Groups whose amax is +inf (an infinite element; a silu product that overflows
    binary32): the hand-worked codes and scale words of tests/golden/nonfinite_amax.txt,
    in every scale format and output type."""
    from golden_fixtures import nonfinite_amax_cases
    cases = nonfinite_amax_cases()
    assert len(cases) == 4
    key = {O.FMT_FP32: "fp32", O.FMT_UE8M0_PACKED: "packed", O.FMT_UE8M0_FP32: "ue8m0_fp32"}[fmt]
    for c in cases:
        x = torch.from_numpy(c["x"].view(np.int16).copy()).view(torch.bfloat16).reshape(1, -1)
        out = O.OUT_E4M3 if c["out"] == "e4m3" else O.OUT_INT8
        q, s = _run(x, c["group"], out_dtype=out, fmt=fmt, silu=c["silu"])
        assert np.array_equal(q, c["codes"]), (c["name"], q, c["codes"])
        assert np.array_equal(s.view(np.uint32), c[key]), (c["name"], s.view(np.uint32), c[key])
