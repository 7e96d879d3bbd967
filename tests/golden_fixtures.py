"""Parsers of the hand-worked fixtures in tests/golden/ (each file documents its
derivation and cites the page it follows)."""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name: str):
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            yield line.split()


def per_token_overflow_rows():
    """[(dtype 'fp32'|'bf16', element bits (uint32 or uint16 array), expected codes)]."""
    rows, cur = [], None
    for tok in _lines("per_token_reciprocal_overflow.txt"):
        if tok[0] == "row":
            dt = tok[1]
            bits = np.array([int(t, 16) for t in tok[2:]],
                            dtype=np.uint32 if dt == "fp32" else np.uint16)
            cur = (dt, bits)
        elif tok[0] == "codes":
            rows.append((cur[0], cur[1], np.array([int(t, 16) for t in tok[1:]], np.uint8)))
            cur = None
    return rows


def nonfinite_amax_cases():
    """[dict(name, group, silu, out, x (uint16 bits of one row), codes, fp32, packed,
    ue8m0_fp32)] with the scale words as uint32 arrays."""
    cases, cur = [], None
    for tok in _lines("nonfinite_amax.txt"):
        key = tok[0]
        if key == "case":
            cur = {"name": tok[1]}
        elif key == "end":
            cases.append(cur)
            cur = None
        elif key in ("group", "silu"):
            cur[key] = int(tok[1])
        elif key == "out":
            cur[key] = tok[1]
        elif key == "x":
            cur[key] = np.array([int(t, 16) for t in tok[1:]], np.uint16)
        elif key == "codes":
            cur[key] = np.array([int(t, 16) for t in tok[1:]], np.uint8)
        else:
            cur[key] = np.array([int(t, 16) for t in tok[1:]], np.uint32)
    return cases
