"""GPU parity of the fast-math compatibility mode (PTGQ_FLAG_FAST_DIVIDE): each element
quotient is CUDA's approximate division, known only to lie within 2 ulps of the exact
quotient, so each code must lie between the oracle's codes for the quotient moved 2 ulps
down and up, and equal them wherever the two agree (every dead row, padding byte and
code away from a rounding boundary).  Scales are the exact ones, bit for bit; the UE8M0
formats divide by a power of two exactly, so there the flag changes nothing."""
import numpy as np
import pytest
import torch

import fp8_token_group_gb300 as P
from fp8_token_group_gb300 import synth
from parity_util import Case, assert_same, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

FAST = P.FLAG_FAST_DIVIDE


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    P.lib()


def _values(codes: np.ndarray, out_dtype: int) -> np.ndarray:
    if out_dtype == P.E4M3:
        return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).float().numpy()
    return codes.view(np.int8).astype(np.float32)


def check_fast(x, c: Case, masked_m=None):
    """Returns (codes that differ from the exact mode, codes whose bounds part)."""
    fast = Case(**{**c.__dict__, "flags": c.flags | FAST})
    gq, gs = run_gpu(x, fast, masked_m)
    eq, es = run_oracle(x, c, masked_m)
    lo, ls = run_oracle(x, c, masked_m, quot_ulps=-2)
    hi, hs = run_oracle(x, c, masked_m, quot_ulps=2)
    assert np.array_equal(ls, es) and np.array_equal(hs, es)
    what = f"{tuple(x.shape)} {x.dtype} {c}"
    assert np.array_equal(gs, es), f"{what}: scales differ from the exact ones"
    agree = lo == hi
    assert np.array_equal(gq[agree], lo[agree]), \
        f"{what}: {int((gq[agree] != lo[agree]).sum())} codes differ where the bounds agree"
    part = ~agree
    v, vl, vh = (_values(a[part], c.out_dtype) for a in (gq, lo, hi))
    assert np.all((vl <= v) & (v <= vh)), f"{what}: code outside the quotient bounds"
    return int((gq != eq).sum()), int(part.sum())


def test_flat_small_e4m3_and_int8():
    for out in (P.E4M3, P.INT8):
        check_fast(synth.flat_small(), Case(out_dtype=out))


def test_flat_outliers_int8_col_major_changes_some_codes():
    """Full benchmark shape, int8, fp32 column-major scales.  The bounds part on about 0.2%
    of the codes; the approximate division must land on the other side of the boundary
    for some of them, or the flag did not take effect."""
    diff, part = check_fast(synth.flat_outliers(), Case(out_dtype=P.INT8, layout=P.COL_MAJOR_TMA,
                                                         tokens_pad=4100))
    assert part > 0 and 0 < diff <= part, (diff, part)


def test_flat_fp16_e4m3_ragged():
    x = synth.normal((333, 2048), torch.float16, seed=11)
    for g in (16, 32, 64, 128):
        check_fast(x, Case(group=g, tokens_pad=340))


def test_silu_flat_e4m3_and_int8():
    x = synth.silu_flat(tokens=1024, hidden=2048)
    for out in (P.E4M3, P.INT8):
        check_fast(x, Case(out_dtype=out, silu=True, layout=P.COL_MAJOR_TMA))


def test_silu_fp16():
    check_fast(synth.silu_flat(tokens=257, hidden=1024, dtype=torch.float16),
               Case(silu=True, group=64))


def test_masked_silu_dead_rows_untouched():
    x, mm = synth.masked_silu(experts=8, tokens_pad=96, hidden=2048)
    for out in (P.E4M3, P.INT8):
        check_fast(x, Case(out_dtype=out, silu=True, layout=P.COL_MAJOR_TMA), masked_m=mm.numpy())


@pytest.mark.parametrize("fmt", [P.SCALE_UE8M0_PACKED, P.SCALE_UE8M0_FP32])
def test_flag_is_a_no_op_for_ue8m0(fmt):
    x = synth.flat_outliers(tokens=512, hidden=7168)
    c = Case(scale_fmt=fmt, layout=P.COL_MAJOR_TMA, tokens_pad=515, flags=FAST)
    gq, gs = run_gpu(x, c)
    oq, os_ = run_oracle(x, Case(scale_fmt=fmt, layout=P.COL_MAJOR_TMA, tokens_pad=515))
    assert_same(gq, gs, oq, os_, "ue8m0 with the fast-divide flag")
