#!/usr/bin/env python3
"""Generate ``silu_tables.inc``: constant tables for the fused silu(gate) * up prologue.

The kernels evaluate silu(g) = g / (1 + exp(-g)) in binary32 steps with the correctly
rounded binary32 exponential.  Gates are bf16 or fp16 values, so the exponential only
ever sees 16-bit inputs; these tables make it exact without a per-element
double-precision evaluation:

* ``kSiluF16``  the same step sequence for every fp16 gate with a non-trivial result,
  indexed by |bits| (positive gates, entries [0, F16_POS)) and F16_POS + |bits| (negative
  gates, |bits| <= 0x558C, i.e. g >= -88.75).  Outside the table the sequence has closed
  forms: S = g for positive gates from F16_POS on (exp(-g) is below half an ulp of 1, so
  D = 1), and S = -0 for g <= -88.75 (exp(-g) overflows binary32), which is also the
  table's last entry, so a kernel can clamp the negative index to it.
* ``kSiluBf16``  the full binary32 step sequence E = RN(exp(-g)), D = RN(1 + E),
  S = RN(g / D) for every bf16 g whose exponent field lies in [102, 133]
  (2^-25 <= |g| < 128), indexed by (sign, bits & 0x7FFF): 4096 entries per sign.  Outside that range the
  sequence has closed forms (S = g/2 for |g| < 2^-25; S = g for g >= 128; S = -0 for
  g <= -128), which this script checks for every bf16 value.

Values come from mpmath at 160 bits, rounded to binary32 by exact comparison; the
binary32 steps use numpy (IEEE).  Every finite 16-bit gate is checked, in the table or
against its closed form.  Run from anywhere:
    python gen_silu_tables.py [output path]
"""
import os
import sys

import mpmath
import numpy as np

F32 = np.float32
mpmath.mp.prec = 160
F16_OVERFLOW_BITS = 0x558C      # fp16 88.75: from -g >= 88.75 on, exp(-g) overflows binary32
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


def fp16_gates() -> np.ndarray:
    """Every fp16 bit pattern's value as binary32 (exact), indexed by the pattern."""
    return np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float32)


def f16_table():
    """(F16_POS, table) of the fp16 path; asserts every closed form it relies on."""
    gates = fp16_gates()
    s = np.array([silu_steps(g) if np.isfinite(g) else F32(0.0) for g in gates], np.float32)
    bits = s.view(np.uint32)
    # F16_POS: the first positive |bits| from which S = g for every finite positive gate
    pos = 0x7C00
    while pos > 0 and bits[pos - 1] == gates[pos - 1].view(np.uint32):
        pos -= 1
    assert 0x4000 < pos < 0x5000, hex(pos)                        # g near 16.6
    neg = np.arange(0x8000, 0x8000 + F16_OVERFLOW_BITS + 1)
    assert np.all(np.isfinite(gates[neg]))
    assert np.all(bits[0x8000 + F16_OVERFLOW_BITS:0xFC00] == 0x80000000)   # -0 from -88.75 on
    assert bits[0x8000 + F16_OVERFLOW_BITS - 1] != 0x80000000              # but not before
    return pos, np.concatenate([s[:pos], s[neg]])


def main(out_path: str) -> None:
    f16_pos, f16 = f16_table()

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
        f"#define PTGQ_SILU_F16_POS 0x{f16_pos:04X}",
        f"#define PTGQ_SILU_F16_OVERFLOW_BITS 0x{F16_OVERFLOW_BITS:04X}",
        f"#define PTGQ_SILU_F16_ENTRIES {len(f16)}",
        "",
        fmt_table("kSiluF16", words(f16),
                  "binary32 silu(g) for fp16 g: [|bits|] (g >= 0, |bits| < POS), [POS + |bits|] (g < 0)"),
        fmt_table("kSiluBf16", words(table),
                  "binary32 silu(g) for bf16 g, [sign][bits & 0x7FFF - (FIELD_LO << 7)]"),
    ]
    with open(out_path, "w") as f:
        f.write("\n".join(body))


if __name__ == "__main__":
    here = os.path.dirname(os.path.abspath(__file__))
    main(sys.argv[1] if len(sys.argv) > 1 else os.path.join(here, "silu_tables.inc"))
