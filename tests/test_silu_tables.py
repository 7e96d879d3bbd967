"""The GPU kernels' silu tables (fp8_token_group_gb300/csrc/silu_tables.inc) are generated
data.  Regenerating them re-runs the generator's own checks: the closed forms outside each
table (S = g/2, g or -0 for bf16; S = g or -0 for fp16) for every 16-bit gate of both types.
The committed file must then match the regenerated one byte for byte.  The tables, read the
way the kernels index them, must also give the oracle's silu for every finite 16-bit gate:
the oracle takes its exponential from libm, the generator from mpmath.  CPU only; no kernel
runs."""
import importlib.util
import os
import re

import numpy as np
import pytest

import oracle as O

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "fp8_token_group_gb300", "csrc")


def test_committed_silu_tables_regenerate_identically(tmp_path):
    pytest.importorskip("mpmath")
    spec = importlib.util.spec_from_file_location("gen_silu_tables",
                                                  os.path.join(CSRC, "gen_silu_tables.py"))
    gen = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(gen)
    out = tmp_path / "silu_tables.inc"
    gen.main(str(out))                       # raises if any generator check fails
    with open(os.path.join(CSRC, "silu_tables.inc")) as f:
        committed = f.read()
    assert out.read_text() == committed


def _inc():
    """The #define constants and a named table (binary32 words) of the committed file."""
    with open(os.path.join(CSRC, "silu_tables.inc")) as f:
        text = f.read()
    defs = {m.group(1): int(m.group(2), 0)
            for m in re.finditer(r"#define (PTGQ_SILU_\w+) (\S+)", text)}

    def table(name):
        body = text[text.index(f"{name}["):]
        body = body[body.index("{") + 1:body.index("};")]
        return np.array([int(w, 16) for w in re.findall(r"0x([0-9A-F]+)u", body)], np.uint32)
    return defs, table


def _oracle_bits(g: np.ndarray) -> np.ndarray:
    """The oracle's binary32 silu(g) (silu(g) * 1 is exact), as bit patterns."""
    return np.array([O.silu_mul(float(v), 1.0) for v in g], np.float32).view(np.uint32)


def test_fp16_table_gives_the_oracle_for_every_gate():
    """The fp16 table read the way the kernel documents it (entry |h| for a positive gate,
    POS + |h| for a negative one clamped to the last entry, S = g for positive gates from
    |h| = POS on) holds the oracle's binary32 silu for every finite fp16 gate, bit for bit
    (signs of zero included).  The oracle takes exp from libm, the generator from mpmath."""
    defs, table = _inc()
    tab = table("kSiluF16")
    pos, entries = defs["PTGQ_SILU_F16_POS"], defs["PTGQ_SILU_F16_ENTRIES"]
    assert len(tab) >= entries
    h = np.arange(65536, dtype=np.uint32)
    g = h.astype(np.uint16).view(np.float16)
    fin = np.isfinite(g)
    h, g = h[fin], g[fin].astype(np.float32)
    mag, neg = h & 0x7FFF, h >> 15
    got = tab[np.minimum(mag + neg * pos, entries - 1)]
    closed = (neg == 0) & (mag >= pos)
    got[closed] = g[closed].view(np.uint32)
    want = _oracle_bits(g)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, [hex(int(h[i])) for i in bad[:8]]


def test_bf16_table_gives_the_oracle_for_every_gate():
    """The bf16 table read the way the kernel documents it (entry sign * SPAN + |h| - (FIELD_LO
    << 7) inside the table; outside it S = g / 2 below the table, g for positive and -0 for
    negative gates above it) holds the oracle's binary32 silu for every finite bf16 gate."""
    defs, table = _inc()
    tab = table("kSiluBf16")
    lo, span = defs["PTGQ_SILU_BF16_FIELD_LO"] << 7, defs["PTGQ_SILU_BF16_SPAN"]
    h = np.arange(65536, dtype=np.uint32)
    g = (h << 16).view(np.float32)
    fin = np.isfinite(g)
    h, g = h[fin], g[fin]
    mag, neg = h & 0x7FFF, h >> 15
    t = (mag - lo).astype(np.int64)
    inside = (t >= 0) & (t < span)
    got = np.where(mag < lo, (g * np.float32(0.5)).view(np.uint32),
                   np.where(neg == 1, np.uint32(0x80000000), g.view(np.uint32)))
    got[inside] = tab[neg[inside] * span + t[inside]]
    want = _oracle_bits(g)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, [hex(int(h[i])) for i in bad[:8]]
