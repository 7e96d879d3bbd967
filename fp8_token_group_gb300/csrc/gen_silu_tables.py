#!/usr/bin/env python3
"""Generate ``silu_tables.inc``: constant tables for the fused silu(gate) * up prologue.

The kernels evaluate silu(g) = g / (1 + exp(-g)) in binary32 steps with the correctly
rounded binary32 exponential.  Gates are bf16 or fp16 values, so the exponential only
ever sees 16-bit inputs; these tables make it exact without a per-element
double-precision evaluation:

* ``kSiluF16A`` / ``kSiluF16B``  for fp16 gates: with x = -g, exp(x) = exp(x_hi) * exp(x_lo),
  where x_hi keeps the sign, the exponent and the top five mantissa bits of the fp16 x and
  x_lo is the rest (exact).  A holds exp(x_hi) indexed by the top 11 bits of x, B holds
  exp(x_lo) indexed by (sign, exponent, low five mantissa bits), 2048 entries each, every
  value as a pair of binary32 words (hi = RN(v), lo = RN(v - hi)).  The kernel forms
  E = RN(A * B) in double-float (one exact product split by fma), D = RN(1 + E) and
  S = RN(g / D) by the correctly rounded reciprocal plus one fma correction.  This script
  replays those binary32 operations in exact arithmetic for every fp16 gate and checks
  S against the definition; only g <= -88.75 (where exp(-g) overflows binary32, S = -0)
  and g = -0 (S = -0) need the kernel's closed forms.
* ``kSiluBf16``  the full binary32 step sequence E = RN(exp(-g)), D = RN(1 + E),
  S = RN(g / D) for every bf16 g whose exponent field lies in [102, 133]
  (2^-25 <= |g| < 128), indexed by (sign, bits & 0x7FFF): 4096 entries per sign.  Outside that range the
  sequence has closed forms (S = g/2 for |g| < 2^-25; S = g for g >= 128; S = -0 for
  g <= -128), which this script checks for every bf16 value.

Values come from mpmath at 160 bits, rounded to binary32 by exact comparison; the
binary32 steps use numpy (IEEE).  Run from anywhere:
    python gen_silu_tables.py [output path]
"""
import math
import os
import sys
from fractions import Fraction

import mpmath
import numpy as np

F32 = np.float32
mpmath.mp.prec = 160
F16_OVERFLOW_BITS = 0x558C      # fp16 88.75: from x = -g >= 88.75 on, exp(x) overflows binary32
BF16_FIELD_LO, BF16_FIELD_HI = 102, 133
BF16_SPAN = (BF16_FIELD_HI - BF16_FIELD_LO + 1) * 128   # entries per sign


def rn32(v) -> np.float32:
    """Nearest binary32 to an mpmath value (ties cannot occur for these transcendental values,
    except exactly representable ones, which compare at distance 0)."""
    if v >= mpmath.mpf(2) ** 128 - mpmath.mpf(2) ** 103:
        return F32(np.inf)
    if v <= -(mpmath.mpf(2) ** 128 - mpmath.mpf(2) ** 103):
        return F32(-np.inf)
    c = F32(float(v))
    cands = [np.nextafter(c, F32(-np.inf)), c, np.nextafter(c, F32(np.inf))]
    cands = [x for x in cands if np.isfinite(x)]
    best = min(cands, key=lambda f: abs(mpmath.mpf(float(f)) - v))
    return best


def silu_steps(g: np.float32) -> np.float32:
    e = rn32(mpmath.exp(-mpmath.mpf(float(g))))
    with np.errstate(over="ignore", invalid="ignore", under="ignore"):
        d = F32(1.0) + e
        return g / d


def words(arr) -> list:
    """binary32 bit patterns, zero-padded to a multiple of 4 words (16-byte copies)."""
    ws = [int(x) for x in np.asarray(arr, dtype=np.float32).view(np.uint32)]
    return ws + [0] * (-len(ws) % 4)


def fmt_table(name: str, ws: list, comment: str) -> str:
    lines = [f"// {comment}", f"__device__ __align__(16) const uint32_t {name}[{len(ws)}] = {{"]
    for i in range(0, len(ws), 8):
        lines.append("  " + ", ".join(f"0x{w:08X}u" for w in ws[i:i + 8]) + ",")
    lines.append("};")
    return "\n".join(lines) + "\n"


def rn32_exact(v: Fraction) -> float:
    """Nearest binary32 (ties to even) to an exact rational, with subnormals and overflow."""
    if v == 0:
        return 0.0
    s = -1.0 if v < 0 else 1.0
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (max(e, -126) - 23)
    q = a / ulp
    n = q.numerator // q.denominator
    r = q - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    res = n * ulp
    return s * math.inf if res >= Fraction(2) ** 128 else s * float(res)


def mpf_fraction(v) -> Fraction:
    man, ex = v.man_exp
    return Fraction(int(man)) * Fraction(2) ** int(ex)


def hi_lo_exact(v):
    """(RN(v), RN(v - RN(v))) of an mpmath value, both binary32; (inf, 0) on overflow."""
    fv = mpf_fraction(v)
    h = rn32_exact(fv)
    if not math.isfinite(h):
        return math.inf, 0.0
    return h, rn32_exact(fv - Fraction(h))


def fp16_value(bits: int) -> float:
    return float(np.array([bits], dtype=np.uint16).view(np.float16)[0])


def f16_tables():
    """The two exp tables of the fp16 path, as lists of (hi, lo) pairs."""
    ta = [(0.0, 0.0)] * 2048
    tb = [(0.0, 0.0)] * 2048
    for sx in (0, 1):
        for ex in range(31):
            for m5 in range(32):
                top = (sx << 15) | (ex << 10) | (m5 << 5)
                ta[top >> 5] = hi_lo_exact(mpmath.exp(mpmath.mpf(fp16_value(top))))
                x_lo = (-1 if sx else 1) * m5 * Fraction(2) ** (max(ex, 1) - 25)
                tb[(sx << 10) | (ex << 5) | m5] = hi_lo_exact(mpmath.exp(mpmath.mpf(x_lo.numerator) / x_lo.denominator))
    return ta, tb


def check_f16_path(ta, tb) -> None:
    """Replay the kernel's binary32 operations exactly for every finite fp16 gate."""
    def fin(*v):
        return all(math.isfinite(x) for x in v)

    def mul(a, b):
        return rn32_exact(Fraction(a) * Fraction(b)) if fin(a, b) else math.nan

    def fma(a, b, c):
        return rn32_exact(Fraction(a) * Fraction(b) + Fraction(c)) if fin(a, b, c) else math.nan

    def add(a, b):
        return rn32_exact(Fraction(a) + Fraction(b)) if fin(a, b) else math.nan

    for h in range(65536):
        g = fp16_value(h)
        if not math.isfinite(g):
            continue
        if g == 0:
            want = g / 2
        else:
            e = rn32_exact(mpf_fraction(mpmath.exp(-mpmath.mpf(g))))
            d = add(1.0, e) if math.isfinite(e) else math.inf
            want = rn32_exact(Fraction(g) / Fraction(d)) if math.isfinite(d) else math.copysign(0.0, g)
        hx = h ^ 0x8000
        if hx < 0x8000 and hx >= F16_OVERFLOW_BITS:
            got = -0.0                                    # closed form: exp(-g) overflows
        elif (h & 0x7FFF) == 0:
            got = g                                       # closed form: +-0 keeps its sign
        else:
            ah, al = ta[hx >> 5]
            bh, bl = tb[((hx >> 5) & 0x7E0) | (hx & 0x1F)]
            p = mul(ah, bh)
            t = fma(ah, bh, -p)
            t = fma(al, bh, t)
            t = fma(ah, bl, t)
            d = add(1.0, add(p, t))
            r = rn32_exact(Fraction(1) / Fraction(d))
            q0 = mul(g, r)
            res = fma(-q0, d, g)
            got = fma(res, r, q0)
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), \
            (hex(h), g, got, want)


def pair_words(pairs) -> list:
    return [int(w) for hl in pairs for w in np.array(hl, dtype=np.float32).view(np.uint32)]


def main(out_path: str) -> None:
    ta, tb = f16_tables()
    check_f16_path(ta, tb)

    bits = np.arange(65536, dtype=np.uint32)
    gates = (bits << 16).view(np.float32)
    table = np.zeros(2 * BF16_SPAN, dtype=np.float32)
    for b, g in zip(bits, gates):
        if not np.isfinite(g):
            continue
        s = silu_steps(g)
        field = (int(b) >> 7) & 0xFF
        sign = int(b) >> 15
        if BF16_FIELD_LO <= field <= BF16_FIELD_HI:
            table[sign * BF16_SPAN + (int(b) & 0x7FFF) - (BF16_FIELD_LO << 7)] = s
            continue
        # closed forms outside the table
        if field < BF16_FIELD_LO:
            want = g / F32(2.0)
        elif g > 0:
            want = g
        else:
            want = F32(-0.0)
        assert want.view(np.uint32) == s.view(np.uint32), (hex(int(b)), g, s, want)

    body = [
        "// Generated by gen_silu_tables.py -- do not edit.",
        "// Constants of the fused silu(gate) * up prologue (see the generator's docstring).",
        f"#define PTGQ_SILU_BF16_FIELD_LO {BF16_FIELD_LO}",
        f"#define PTGQ_SILU_BF16_FIELD_HI {BF16_FIELD_HI}",
        f"#define PTGQ_SILU_BF16_SPAN {BF16_SPAN}",
        f"#define PTGQ_SILU_F16_OVERFLOW_BITS 0x{F16_OVERFLOW_BITS:04X}",
        "",
        fmt_table("kSiluF16A", pair_words(ta),
                  "exp(x_hi) as (hi, lo) pairs, x_hi = fp16 x = -g with its low 5 mantissa bits cleared, [bits(x) >> 5]"),
        fmt_table("kSiluF16B", pair_words(tb),
                  "exp(x_lo) as (hi, lo) pairs, x_lo = the low 5 mantissa bits of x, [sign][exponent][low 5 bits]"),
        fmt_table("kSiluBf16", words(table),
                  "binary32 silu(g) for bf16 g, [sign][bits & 0x7FFF - (FIELD_LO << 7)]"),
    ]
    with open(out_path, "w") as f:
        f.write("\n".join(body))


if __name__ == "__main__":
    here = os.path.dirname(os.path.abspath(__file__))
    main(sys.argv[1] if len(sys.argv) > 1 else os.path.join(here, "silu_tables.inc"))
