"""Shared helpers for the GPU parity tests: run one configuration through the CUDA library
(via the C ABI binding) and through the CPU oracle on the same seeded input, with guard
bands around every device output buffer, and compare."""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

import oracle as O
import fp8_token_group_gb300 as P
from fp8_token_group_gb300 import synth

GUARD = 4096          # bytes of canary before and after each output buffer
CANARY = 0xA5
# Sentinels no kernel output can equal in rows the kernel must leave alone: e4m3 0x7F is
# NaN (emitted only for an infinite element of a group whose amax is infinite), int8 0x80
# = -128 is unreachable (|y| <= 127), float scale 0x7FC00001 is a NaN payload no scale
# has, and a packed word of 0xFFFFFFFF holds exponent byte 255 in all four bytes.
SENT_Q = {P.E4M3: 0x7F, P.INT8: 0x80}
SENT_S_FLOAT = 0x7FC00001
SENT_S_PACKED = 0xFFFFFFFF


@dataclass
class Case:
    group: int = 128
    out_dtype: int = P.E4M3
    scale_fmt: int = P.SCALE_FP32
    layout: int = P.ROW_MAJOR
    silu: bool = False
    tokens_pad: int = 0
    eps: float = 1e-10
    flags: int = 0
    expected_m: int = 0


def _guarded(nbytes: int, fill: int, device="cuda"):
    buf = torch.full((GUARD + nbytes + GUARD,), CANARY, dtype=torch.uint8, device=device)
    body = buf[GUARD:GUARD + nbytes]
    body.fill_(fill) if isinstance(fill, int) and fill < 256 else None
    return buf, body


def _fill_words(body: torch.Tensor, word: int):
    body.view(torch.int32).fill_(np.array(word, dtype=np.uint32).view(np.int32).item())


def shapes(x: torch.Tensor, c: Case, masked: bool):
    if masked:
        E, tp, hin = x.shape
        n, rows, tokens_pad = E, tp, tp
    else:
        n, hin = x.shape
        tokens_pad = c.tokens_pad
        rows = tokens_pad or n
    H = hin // 2 if c.silu else hin
    qn = (n if masked else 1) * rows * H
    sn = P.scale_elems(n, tokens_pad, H, c.group, c.scale_fmt, c.layout, masked)
    assert sn == O.scale_elems(n, tokens_pad, H, c.group, c.scale_fmt, c.layout, masked)
    return n, rows, tokens_pad, H, qn, sn


def run_gpu(x: torch.Tensor, c: Case, masked_m=None, stream=None):
    """Returns (codes uint8 [qn], scales uint32 [sn]) as numpy, after checking the guards."""
    masked = masked_m is not None
    n, rows, tokens_pad, H, qn, sn = shapes(x, c, masked)
    qbuf, qbody = _guarded(qn, SENT_Q[c.out_dtype])
    sbuf, sbody = _guarded(4 * sn, 0)
    _fill_words(sbody, SENT_S_PACKED if c.scale_fmt == P.SCALE_UE8M0_PACKED else SENT_S_FLOAT)
    xd = x.cuda()
    mm = None if masked_m is None else torch.as_tensor(masked_m, dtype=torch.int32).cuda()
    qt = qbody.view(torch.float8_e4m3fn if c.out_dtype == P.E4M3 else torch.int8)
    st = sbody.view(torch.int32 if c.scale_fmt == P.SCALE_UE8M0_PACKED else torch.float32)
    P.quant(xd, qt, st, c.group, out_dtype=c.out_dtype, scale_fmt=c.scale_fmt,
            scale_layout=c.layout, fuse_silu=c.silu, masked_m=mm, eps=c.eps,
            tokens_pad=tokens_pad, flags=c.flags, expected_m=c.expected_m, stream=stream)
    torch.cuda.synchronize()
    qh, sh = qbuf.cpu().numpy(), sbuf.cpu().numpy()
    assert np.all(qh[:GUARD] == CANARY) and np.all(qh[GUARD + qn:] == CANARY), "out_q guard hit"
    assert np.all(sh[:GUARD] == CANARY) and np.all(sh[GUARD + 4 * sn:] == CANARY), "out_s guard hit"
    return qh[GUARD:GUARD + qn].copy(), sh[GUARD:GUARD + 4 * sn].view(np.uint32).copy()


def run_oracle(x: torch.Tensor, c: Case, masked_m=None, quot_ulps: int = 0):
    """The oracle on the same input; ``quot_ulps`` != 0 gives the codes of the quotient bounds
    instead (see oracle.quant)."""
    masked = masked_m is not None
    n, rows, tokens_pad, H, qn, sn = shapes(x, c, masked)
    q = np.full(qn, SENT_Q[c.out_dtype], dtype=np.uint8)
    s = np.full(sn, SENT_S_PACKED if c.scale_fmt == P.SCALE_UE8M0_PACKED else SENT_S_FLOAT,
                dtype=np.uint32)
    sarg = s if c.scale_fmt == P.SCALE_UE8M0_PACKED else s.view(np.float32)
    in_dtype = O.IN_BF16 if x.dtype == torch.bfloat16 else O.IN_FP16
    flags = O.FLAG_UE8M0_SCALE_FLOOR if c.flags & P.FLAG_UE8M0_SCALE_FLOOR else 0
    O.quant(synth.bits_u16(x), in_dtype, n, tokens_pad, H, c.group, q, c.out_dtype, sarg,
            c.scale_fmt, c.layout, int(c.silu), None if masked_m is None else np.asarray(masked_m),
            c.eps, flags, quot_ulps)
    return q, s


# ---------------------------------------------------------------- comparison

def _e4m3_step(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in representable steps between two e4m3 codes (signed-magnitude order)."""
    def order(c):
        c = c.astype(np.int32)
        mag = c & 0x7F
        return np.where(c & 0x80, -mag, mag)
    return np.abs(order(a) - order(b))


def assert_same(gq, gs, oq, os_, what=""):
    if not np.array_equal(gq, oq):
        bad = np.flatnonzero(gq != oq)
        raise AssertionError(f"{what}: {bad.size} code bytes differ, first at {bad[:8]}: "
                             f"gpu {gq[bad[:8]]} oracle {oq[bad[:8]]}")
    if not np.array_equal(gs, os_):
        bad = np.flatnonzero(gs != os_)
        raise AssertionError(f"{what}: {bad.size} scale words differ, first at {bad[:8]}: "
                             f"gpu {[hex(v) for v in gs[bad[:8]]]} oracle {[hex(v) for v in os_[bad[:8]]]}")


def assert_silu_close(gq, gs, oq, os_, c: Case, what=""):
    """The fused-silu tolerance: at most 1 e4m3 step on at most 1e-4 of the codes, scale
    relative error at most 2e-7 (fp32 scales) or the same exponent (UE8M0; e +- 1 only
    where the oracle's raw scale lies within 2 ulps of a power of two, which the packed
    layout does not expose, so exponents must match)."""
    diff = gq != oq
    if diff.any():
        frac = diff.mean()
        assert frac <= 1e-4, f"{what}: {diff.sum()} codes differ ({frac:.2e})"
        if c.out_dtype == P.E4M3:
            assert _e4m3_step(gq[diff], oq[diff]).max() <= 1, f"{what}: code off by >1 step"
        else:
            d = np.abs(gq[diff].view(np.int8).astype(int) - oq[diff].view(np.int8).astype(int))
            assert d.max() <= 1, f"{what}: int8 code off by >1"
    if c.scale_fmt == P.SCALE_FP32:
        g = gs.view(np.float32).astype(np.float64)
        o = os_.view(np.float32).astype(np.float64)
        same = gs == os_
        fin = np.isfinite(o) & (o != 0)
        rel = np.abs(g - o)[fin & ~same] / np.abs(o[fin & ~same])
        assert rel.size == 0 or rel.max() <= 2e-7, f"{what}: scale rel err {rel.max():.3e}"
        assert np.array_equal(gs[~fin], os_[~fin]), f"{what}: padding/sentinel scales differ"
    else:
        assert np.array_equal(gs, os_), f"{what}: UE8M0 exponents differ"


def compare(x, c: Case, masked_m=None, exact_silu=True):
    gq, gs = run_gpu(x, c, masked_m)
    oq, os_ = run_oracle(x, c, masked_m)
    what = f"{tuple(x.shape)} {x.dtype} {c}"
    if c.silu and not exact_silu:
        assert_silu_close(gq, gs, oq, os_, c, what)
    else:
        assert_same(gq, gs, oq, os_, what)
    return gq, gs
