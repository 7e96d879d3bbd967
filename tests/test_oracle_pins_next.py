"""Pins for the oracle's per-token FP8 quantization (sglang PR #34257, "Key source
snippets": the per-token kernels) and its per-token-group -> per-tensor FP8 requant
(sglang PR #35593, "Key source snippets": the requant kernel and its test)."""
import numpy as np
import pytest
import torch

import oracle as O
from fp8_token_group_gb300 import synth

F32 = np.float32


def e4m3_bytes(v: np.ndarray) -> np.ndarray:
    """torch's float8_e4m3fn cast of values already inside [-448, 448]."""
    return torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_matches_torch_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    got = np.array([O.e4m3_decode(int(c)) for c in codes], dtype=np.float32)
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin].view(np.uint32), ref[fin].view(np.uint32))
    assert np.all(np.isnan(got[~fin])) and (~fin).sum() == 2


# ---------------------------------------------------------------- per-token

def _pt(x: torch.Tensor, out_rows=None, fill=0xAB):
    T, H = x.shape
    rows = out_rows or T
    q = np.full(rows * H, fill, np.uint8)
    s = np.full(rows, np.nan, np.float32)
    if x.dtype == torch.float32:
        O.per_token_quant(np.ascontiguousarray(x.numpy()), O.IN_FP32, q, s)
    else:
        O.per_token_quant(synth.bits_u16(x).reshape(T, H),
                          O.IN_BF16 if x.dtype == torch.bfloat16 else O.IN_FP16, q, s)
    return q.reshape(rows, H), s


def _pt_reference(x: torch.Tensor):
    """The page's kernel loop from library routines: numpy binary32 max / divide /
    multiply, torch's fp8 cast."""
    v = x.float().numpy()
    m = np.abs(v).max(1).astype(np.float32)
    s = (m / F32(448)).astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(s == 0, F32(0), (F32(1) / s)).astype(np.float32)
    y = np.clip((v * inv[:, None]).astype(np.float32), -448, 448)
    return e4m3_bytes(y).reshape(v.shape), s


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16, torch.float32])
@pytest.mark.parametrize("hidden", [1076, 1368, 4096])
def test_per_token_vs_library_composition(dt, hidden):
    g = torch.Generator().manual_seed(hidden)
    x = (torch.rand((39, hidden), generator=g) * 4 - 2).to(dt)
    x[5] = 0                                   # zero row: scale 0, codes 0 (guarded path)
    q, s = _pt(x)
    rq, rs = _pt_reference(x)
    assert np.array_equal(q, rq) and np.array_equal(s.view(np.uint32), rs.view(np.uint32))
    assert s[5] == 0 and np.all(q[5] == 0)


def test_per_token_integer_rows_exact():
    g = torch.Generator().manual_seed(1)
    k = torch.randint(-7, 8, (16, 512), generator=g)
    k[:, 0] = 7
    q, s = _pt(k.to(torch.bfloat16))
    assert np.all(s == F32(1 / 64))
    assert np.array_equal(q, e4m3_bytes(64.0 * k.numpy()).reshape(16, 512))


def test_per_token_midpoint_rounding_and_padded_tail():
    # s = 448 / 448 = 1 and inv = 1, so the codes are e4m3(x) at exact midpoints
    mids = [1.0625, 1.1875, 17.0, 19.0, 0.0029296875, 0.0009765625, 248.0]
    want = [0x38, 0x3A, 0x58, 0x5A, 0x02, 0x00, 0x78]
    x = torch.zeros((2, 8), dtype=torch.float32)
    x[:, 0] = 448.0
    x[:, 1:] = torch.tensor(mids)
    q, s = _pt(x, out_rows=5, fill=0xAB)
    assert np.all(s[:2] == 1.0) and np.all(np.isnan(s[2:]))
    assert list(q[0, 1:]) == want and np.all(q[2:] == 0xAB)


# ---------------------------------------------------------------- requant

def _requant_case(E, M, K, seed, group=128):
    """The page's construction: integers in [-8, 8] (exact in e4m3) and power-of-two group
    scales 2^{-1,0,1}, so every value is exact; output scale 2."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randint(-8, 9, (E, M, K), generator=g).float()
    exps = torch.randint(-1, 2, (E, M, K // group), generator=g)
    xs = torch.pow(2.0, exps.float())
    return x, xs


@pytest.mark.parametrize("K", [7168, 3584, 1152])
def test_requant_masked_rows_and_k_tail(K):
    E, M = 4, 48
    masked = np.array([0, 1, 17, M], np.int32)
    x, xs = _requant_case(E, M, K, seed=K)
    codes = e4m3_bytes(x.numpy()).reshape(E, M, K)
    sentinel = e4m3_bytes(np.array([0.375], np.float32))[0]
    out = np.full((E, M, K), sentinel, np.uint8)
    # column-major [E, M, K/128] scales: strides (M*K/128, 1, M)
    xs_cm = np.ascontiguousarray(xs.permute(0, 2, 1).numpy())          # [E, K/128, M]
    O.requant_per_tensor(codes, xs_cm, (M * (K // 128), 1, M), masked, 2.0, out)
    ref = e4m3_bytes((x * xs.repeat_interleave(128, dim=2) * 0.5).numpy()).reshape(E, M, K)
    for e, valid in enumerate(masked):
        assert np.array_equal(out[e, :valid], ref[e, :valid])
        assert np.all(out[e, valid:] == sentinel)


def test_requant_vs_library_composition_and_saturation():
    g = torch.Generator().manual_seed(3)
    E, M, K = 3, 20, 512
    codes = torch.randint(0, 256, (E, M, K), generator=g, dtype=torch.uint8).numpy()
    codes[(codes & 0x7F) == 0x7F] = 0x00                 # no NaN inputs
    xs = (torch.rand((E, M, K // 128), generator=g) * 8 + 0.01).numpy().astype(np.float32)
    out = np.zeros((E, M, K), np.uint8)
    mm = np.array([20, 7, 25], np.int32)
    O.requant_per_tensor(codes, np.ascontiguousarray(xs), (M * (K // 128), K // 128, 1), mm,
                         0.37, out)
    v = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    inv = F32(1) / F32(0.37)
    y = ((v * np.repeat(xs, 128, axis=2)).astype(np.float32) * inv).astype(np.float32)
    ref = e4m3_bytes(np.clip(y, -448, 448)).reshape(E, M, K)
    assert np.array_equal(out[0], ref[0]) and np.array_equal(out[2], ref[2])
    assert np.array_equal(out[1, :7], ref[1, :7]) and np.all(out[1, 7:] == 0)
    assert (np.abs(y) > 448).any()                        # saturation was exercised


# ---------------------------------------------------------------- operation order

def _bits_plus(a: np.ndarray, d: int) -> np.ndarray:
    return (np.asarray(a, np.float32).view(np.int32) + np.int32(d)).view(np.float32)


def test_per_token_multiplies_by_the_reciprocal():
    """The page's per-token kernel multiplies by inv = RN(1/s); a division by s gives other
    codes for some inputs.  Rows are built (seeded search, binary32 numpy arithmetic) from
    values within a few ulps of e4m3 midpoints times s, kept where the two orders part;
    the oracle must follow the reciprocal order on every one of them."""
    rng = np.random.default_rng(7)
    ties = np.array([1.0625, 1.1875, 2.125, 17.0, 19.0, 0.0029296875, 104.0, 208.0, 3.25, 6.5])
    rows = []
    while len(rows) < 8:
        m = F32(rng.uniform(1, 1000))
        s = F32(m / F32(448))
        inv = F32(F32(1) / s)
        cand = np.concatenate([_bits_plus((ties * np.float64(s)).astype(np.float32), d)
                               for d in (-2, -1, 0, 1, 2)])
        a = e4m3_bytes(np.clip(cand * inv, -448, 448))
        b = e4m3_bytes(np.clip(cand / s, -448, 448))
        keep = cand[a != b]
        if keep.size:
            rows.append(np.concatenate([[m], keep[:7], np.zeros(7 - min(7, keep.size), np.float32)]))
    x = torch.from_numpy(np.stack(rows).astype(np.float32))
    q, s = _pt(x)
    rq, rs = _pt_reference(x)                       # x * RN(1/s), numpy binary32
    assert np.array_equal(q, rq) and np.array_equal(s.view(np.uint32), rs.view(np.uint32))
    v = x.numpy()
    by_division = e4m3_bytes(np.clip(v / rs[:, None], -448, 448)).reshape(v.shape)
    assert (by_division != q).sum() >= 8             # the rows do tell the two orders apart


def test_requant_scales_first_then_the_output_scale():
    """The page's requant forms (v * x_scale) * (1 / output_scale); the other association,
    v * (x_scale * (1 / output_scale)), gives other codes for some inputs.  Groups are built
    by a seeded search aiming v * x_scale / output_scale at e4m3 midpoints, kept where the
    two orders part; the oracle must follow the page's order."""
    rng = np.random.default_rng(11)
    vals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    mags = np.unique(np.abs(vals[np.isfinite(vals)]))
    mids = (mags[1:] + mags[:-1]) / 2
    nz = [c for c in range(1, 127) if np.isfinite(vals[c]) and vals[c] != 0]
    os_ = F32(2.243415355682373)
    inv = F32(F32(1) / os_)
    picks = []
    while len(picks) < 8:
        c = int(rng.choice(nz))
        sc0 = F32(float(rng.choice(mids)) * float(os_) / float(vals[c]))
        for d in range(-3, 4):
            sc = _bits_plus(np.array([sc0]), d)
            a = e4m3_bytes(np.clip((vals[c] * sc).astype(np.float32) * inv, -448, 448))
            b = e4m3_bytes(np.clip(vals[c] * (sc * inv).astype(np.float32), -448, 448))
            if a[0] != b[0]:
                picks.append((c, float(sc[0])))
                break
    G, M = 128, len(picks)
    codes = np.zeros((1, M, G), np.uint8)
    xs = np.zeros((1, M, 1), np.float32)
    for r, (c, sc) in enumerate(picks):
        codes[0, r, :] = c
        xs[0, r, 0] = sc
    out = np.zeros_like(codes)
    O.requant_per_tensor(codes, xs, (M, 1, 1), np.array([M], np.int32), float(os_), out)
    v = vals[codes.astype(np.int64)]
    page = e4m3_bytes(np.clip((v * xs).astype(np.float32) * inv, -448, 448)).reshape(codes.shape)
    other = e4m3_bytes(np.clip(v * (xs * inv).astype(np.float32), -448, 448)).reshape(codes.shape)
    assert np.array_equal(out, page)
    assert (other != out).sum() >= 8 * G


# ---------------------------------------------------------------- reciprocal overflow

def test_per_token_reciprocal_overflow_fixture():
    """Rows whose reciprocal 1/s overflows to +inf (max below about 1.3e-36) and one whose
    s is subnormal with a finite reciprocal: the hand-worked codes of
    tests/golden/per_token_reciprocal_overflow.txt (the page's clamp, min first, with
    IEEE minNum / maxNum, so 0 * inf = NaN clamps to +448)."""
    from golden_fixtures import per_token_overflow_rows
    rows = per_token_overflow_rows()
    assert len(rows) == 3
    for dt, bits, want in rows:
        H = bits.size
        q = np.full(H, 0xAB, np.uint8)
        s = np.full(1, np.nan, np.float32)
        if dt == "fp32":
            vals = bits.view(np.float32)
            O.per_token_quant(vals.reshape(1, H).copy(), O.IN_FP32, q, s)
        else:
            vals = (bits.astype(np.uint32) << 16).view(np.float32)
            O.per_token_quant(bits.reshape(1, H).copy(), O.IN_BF16, q, s)
        m = np.abs(vals).max().astype(np.float32)
        assert s[0].view(np.uint32) == (m / F32(448)).astype(np.float32).view(np.uint32)
        assert np.array_equal(q, want), (dt, q, want)
