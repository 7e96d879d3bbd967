"""The C-ABI library without a GPU: it builds, loads, exports every function declared in
include/ptgq.h, and rejects bad arguments with the documented status codes before
touching any device (no compute call is made here)."""
import itertools
import os
import re

import pytest

import oracle as O
import fp8_token_group_gb300 as P
from fp8_token_group_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "ptgq.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return P.lib()


def test_every_declared_function_is_exported(L):
    names = P.header_functions()
    assert set(names) == {"ptgq_quant", "ptgq_quant_ex", "ptgq_scale_elems", "ptgq_strerror",
                          "ptgq_per_token_quant", "ptgq_requant_per_tensor"}
    for n in names:
        assert hasattr(L, n), n


def test_header_constants_match_binding():
    text = open(HEADER).read()
    def val(name):
        return int(re.search(rf"\b{name}\s*=\s*(-?\d+)", text).group(1))
    assert (val("PTGQ_BF16"), val("PTGQ_FP16")) == (P.BF16, P.FP16)
    assert (val("PTGQ_E4M3"), val("PTGQ_INT8")) == (P.E4M3, P.INT8)
    assert (val("PTGQ_SCALE_FP32"), val("PTGQ_SCALE_UE8M0_PACKED"),
            val("PTGQ_SCALE_UE8M0_FP32")) == (P.SCALE_FP32, P.SCALE_UE8M0_PACKED, P.SCALE_UE8M0_FP32)
    assert (val("PTGQ_ROW_MAJOR"), val("PTGQ_COL_MAJOR_TMA")) == (P.ROW_MAJOR, P.COL_MAJOR_TMA)
    assert (val("PTGQ_FLAG_NO_PDL"), val("PTGQ_FLAG_UE8M0_SCALE_FLOOR"),
            val("PTGQ_FLAG_FAST_DIVIDE")) == (P.FLAG_NO_PDL, P.FLAG_UE8M0_SCALE_FLOOR,
                                              P.FLAG_FAST_DIVIDE)


def test_eps_floor_matches_binding_and_keeps_the_scale_positive():
    text = open(HEADER).read()
    m = re.search(r"#define PTGQ_EPS_MIN (\S+)", text).group(1)
    assert float.fromhex(m.rstrip("f")) == P.EPS_MIN == 2.0 ** -140
    import numpy as np
    for fmax in (448, 127):
        assert np.float32(P.EPS_MIN) / np.float32(fmax) > 0


def test_strerror_covers_every_status(L):
    for code in range(-13, 1):
        msg = P.strerror(code)
        assert msg and msg != "unknown status", code
    assert P.strerror(-99) == "unknown status"


@pytest.mark.parametrize("fmt,layout,masked", list(itertools.product([0, 1, 2], [0, 1], [0, 1])))
def test_scale_elems_matches_oracle(L, fmt, layout, masked):
    for n, tp, H, G in [(4096, 0, 7168, 128), (37, 45, 896, 128), (5, 0, 7 * 16, 16),
                        (32, 384, 4096, 128), (3, 7, 2048, 64), (0, 9, 1024, 32)]:
        if masked and tp == 0:
            continue
        assert P.scale_elems(n, tp, H, G, fmt, layout, masked) == \
            O.scale_elems(n, tp, H, G, fmt, layout, masked)


def _call(L, **kw):
    a = dict(x=32, dtype=0, n=4, tokens_pad=0, hidden=256, group=128, q=16, out=0, s=4, fmt=0,
             layout=0, silu=0, mm=None, eps=1e-10, stream=None, flags=0, expected_m=0,
             errors=None)
    a.update(kw)
    return L.ptgq_quant_ex(a["x"], a["dtype"], a["n"], a["tokens_pad"], a["hidden"], a["group"],
                           a["q"], a["out"], a["s"], a["fmt"], a["layout"], a["silu"], a["mm"],
                           a["eps"], a["stream"], a["flags"], a["expected_m"], a["errors"])


def test_validation_codes(L):
    assert _call(L, dtype=2) == -2
    assert _call(L, out=2) == -3
    assert _call(L, group=100) == -4
    assert _call(L, group=256) == -4
    assert _call(L, hidden=200) == -5
    assert _call(L, hidden=0) == -5
    assert _call(L, n=-1) == -6
    assert _call(L, n=8, tokens_pad=4) == -6
    assert _call(L, mm=64, n=5000) == -6
    assert _call(L, x=48) == -7
    assert _call(L, q=8) == -7
    assert _call(L, s=2) == -7
    assert _call(L, fmt=3) == -8
    assert _call(L, layout=2) == -9
    for eps in (0.0, -1.0, 2.0 ** -141, 1e-45, float("inf"), float("nan")):
        assert _call(L, eps=eps) == -10
    assert _call(L, silu=2) == -11
    assert _call(L, flags=8) == -11
    assert _call(L, mm=64, tokens_pad=8, expected_m=-1) == -6
    assert _call(L, mm=64, n=4, tokens_pad=8, errors=2) == -7   # masked_m_errors 4-byte aligned
    assert _call(L, x=0) == -1
    assert _call(L, q=0) == -1
    assert _call(L, s=0) == -1
    assert _call(L, n=2 ** 31, hidden=16 * 128, group=16) == -12


def test_nothing_to_do_returns_ok_without_device(L):
    # no rows anywhere: returns before any CUDA call
    assert _call(L, x=0, q=0, s=0, n=0) == 0
    assert _call(L, x=0, q=0, s=0, n=0, mm=64, tokens_pad=0) == 0
    assert _call(L, x=0, q=0, s=0, n=0, mm=64, tokens_pad=16) == 0


def test_per_token_and_requant_validation(L):
    assert L.ptgq_per_token_quant(16, 3, 4, 64, 16, 16, None) == -2
    assert L.ptgq_per_token_quant(16, 0, 4, 66, 16, 16, None) == -5
    assert L.ptgq_per_token_quant(16, 0, -1, 64, 16, 16, None) == -6
    assert L.ptgq_per_token_quant(0, 0, 4, 64, 16, 16, None) == -1
    assert L.ptgq_per_token_quant(8, 0, 4, 64, 16, 16, None) == -7     # 16-byte rows need 16 B
    assert L.ptgq_per_token_quant(0, 0, 0, 64, 0, 0, None) == 0        # nothing to do
    rq = L.ptgq_requant_per_tensor
    assert rq(16, 16, 1, 1, 1, None, 16, 16, 2, 4, 256, 100, None) == -4
    assert rq(16, 16, 1, 1, 1, None, 16, 16, 2, 4, 200, 128, None) == -5
    assert rq(16, 16, 1, 1, 1, None, 16, 16, -1, 4, 256, 128, None) == -6
    assert rq(0, 16, 1, 1, 1, None, 16, 16, 2, 4, 256, 128, None) == -1
    assert rq(8, 16, 1, 1, 1, None, 16, 16, 2, 4, 256, 128, None) == -7
    assert rq(0, 0, 1, 1, 1, None, 0, 0, 0, 4, 256, 128, None) == 0
