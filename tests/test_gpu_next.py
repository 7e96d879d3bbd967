"""GPU parity of the per-token FP8 quantizer and the per-token-group -> per-tensor FP8
requant (the two neighbouring operations) against the oracle, bit for bit, through the
C ABI."""
import numpy as np
import pytest
import torch

import oracle as O
import fp8_token_group_gb300 as P
from fp8_token_group_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    P.lib()


def _per_token_both(x: torch.Tensor, out_rows: int):
    T, H = x.shape
    xd = x.cuda()
    q = torch.full((out_rows, H), 0x7F, dtype=torch.uint8, device="cuda")
    s = torch.full((out_rows,), float("nan"), dtype=torch.float32, device="cuda")
    P.per_token_quant(xd, q, s)
    torch.cuda.synchronize()
    oq = np.full(out_rows * H, 0x7F, np.uint8)
    os_ = np.full(out_rows, np.nan, np.float32)
    if x.dtype == torch.float32:
        O.per_token_quant(np.ascontiguousarray(x.numpy()), O.IN_FP32, oq, os_)
    else:
        O.per_token_quant(synth.bits_u16(x).reshape(T, H),
                          O.IN_BF16 if x.dtype == torch.bfloat16 else O.IN_FP16, oq, os_)
    return q.cpu().numpy().ravel(), s.cpu().numpy(), oq, os_


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16, torch.float32])
@pytest.mark.parametrize("hidden", [4, 128, 1076, 1368, 4096, 7168, 16384])
@pytest.mark.parametrize("T", [1, 39, 1000, 2432, 4096])
def test_per_token_vs_oracle(dt, hidden, T):
    """Token counts below and at 16 x SMs (the pages' warp/CTA dispatch threshold) and the
    benchmarked 4096, row lengths that are multiples of 4 but not 8, zero rows, integer
    rows, padded output.  The launch shapes cover one CTA per row (8 warps for T <= 4 x SMs,
    4 warps for T <= 12 x SMs with rows up to 16 KB; rows of 16-byte multiples, including rows
    longer than the CTA keeps in registers), one buffer per warp (one round of rows) and two
    (several rounds)."""
    x = synth.sweep_input(hidden + T, T, hidden, torch.float32)
    x[::7] = 0
    x = x.to(dt)
    gq, gs, oq, os_ = _per_token_both(x, T + 3)
    assert np.array_equal(gq, oq)
    assert np.array_equal(gs.view(np.uint32), os_.view(np.uint32))


def test_per_token_midpoints_and_extremes():
    x = torch.zeros((4, 8), dtype=torch.float32)
    x[:, 0] = 448.0
    x[0, 1:] = torch.tensor([1.0625, 1.1875, 17.0, 19.0, 0.0029296875, 0.0009765625, 248.0])
    x[1, :] = -0.0
    x[2, :] = 3.0e38
    x[3, 1:] = 1e-40
    gq, gs, oq, os_ = _per_token_both(x, 4)
    assert np.array_equal(gq, oq) and np.array_equal(gs.view(np.uint32), os_.view(np.uint32))


def _requant_both(codes, xs, strides, masked, out_scale, group=128, sentinel=0x2C):
    E, M, K = codes.shape
    xd = torch.from_numpy(codes).cuda()
    sd = torch.as_strided(torch.from_numpy(xs.ravel().copy()).cuda(),
                          (E, M, K // group), strides)
    mm = None if masked is None else torch.from_numpy(masked).cuda()
    osc = torch.tensor([out_scale], dtype=torch.float32, device="cuda")
    out = torch.full((E, M, K), sentinel, dtype=torch.uint8, device="cuda")
    P.requant_per_tensor(xd, sd, mm, osc, out, group_size=group)
    torch.cuda.synchronize()
    ref = np.full((E, M, K), sentinel, np.uint8)
    O.requant_per_tensor(codes, xs.ravel().copy(), strides,
                         masked if masked is not None else np.full(E, M, np.int32),
                         out_scale, ref, group)
    return out.cpu().numpy(), ref


@pytest.mark.parametrize("K", [7168, 3584, 1152])
def test_requant_masked_rows_and_k_tail(K):
    """The page's test: integers in [-8, 8], power-of-two group scales, output scale 2,
    masked {0, 1, 17, m}, column-major [E, M, K/128] scales, sentinel 0.375 in padding."""
    E, M = 4, 48
    g = torch.Generator().manual_seed(K)
    x = torch.randint(-8, 9, (E, M, K), generator=g).float()
    exps = torch.randint(-1, 2, (E, M, K // 128), generator=g)
    xs = torch.pow(2.0, exps.float()).permute(0, 2, 1).contiguous().numpy()   # [E, K/128, M]
    codes = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    masked = np.array([0, 1, 17, M], np.int32)
    got, ref = _requant_both(codes, xs, (M * (K // 128), 1, M), masked, 2.0)
    assert np.array_equal(got, ref)
    assert np.all(got[0] == 0x2C) and np.all(got[2, 17:] == 0x2C)


@pytest.mark.parametrize("group", [16, 128])
def test_requant_random_codes_scales_and_saturation(group):
    g = torch.Generator().manual_seed(group)
    E, M, K = 8, 1024, 3584
    codes = torch.randint(0, 256, (E, M, K), generator=g, dtype=torch.uint8).numpy()
    codes[(codes & 0x7F) == 0x7F] = 0
    xs = (torch.rand((E, M, K // group), generator=g) * 4 + 1e-3).numpy().astype(np.float32)
    masked = synth.masked_counts(E, M, seed=7).numpy()
    got, ref = _requant_both(codes, xs, (M * (K // group), K // group, 1), masked, 0.61, group)
    assert np.array_equal(got, ref)
    got, ref = _requant_both(codes, xs, (M * (K // group), K // group, 1), None, 0.61, group)
    assert np.array_equal(got, ref)


def test_per_token_row_sizes_in_any_order():
    """The staged kernel's shared-memory size depends on the row length; calls with a long
    row, then a short one, then the long one again must all launch."""
    for hidden in (4096, 512, 4096, 1024, 3072):
        x = synth.sweep_input(hidden, 64, hidden, torch.float32)
        gq, gs, oq, os_ = _per_token_both(x, 64)
        assert np.array_equal(gq, oq) and np.array_equal(gs.view(np.uint32), os_.view(np.uint32))


def test_per_token_reciprocal_overflow_fixture_and_tiny_rows():
    """Rows whose reciprocal scale overflows (max below about 1.3e-36) take the page's clamp
    (0 * inf = NaN clamps to +448); the hand-worked fixture rows, then random tiny rows of
    every dtype through the CTA-per-row kernel (hidden 512) and the register kernel (hidden
    4, 1076), mixed with ordinary rows in the same call."""
    from golden_fixtures import per_token_overflow_rows
    for dt, bits, want in per_token_overflow_rows():
        if dt == "fp32":
            x = torch.from_numpy(bits.view(np.float32).copy()).reshape(1, -1)
        else:
            x = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).reshape(1, -1)
        # the fixture row, tiled to a 16-byte multiple so both kernels can take it
        xx = x.repeat(1, 8)
        gq, gs, oq, os_ = _per_token_both(xx, 1)
        assert np.array_equal(oq[: want.size], want)
        assert np.array_equal(gq, oq) and np.array_equal(gs.view(np.uint32), os_.view(np.uint32))
    g = torch.Generator().manual_seed(9)
    for dt in (torch.float32, torch.bfloat16):
        for hidden in (4, 512, 1076):
            x = torch.randn((24, hidden), generator=g)
            tiny = torch.tensor([1e-37, 2.0 ** -133, 1.5e-36, 3e-39, 1e-36, 1e-38])
            for i in range(12):
                x[2 * i] *= tiny[i % tiny.numel()]
            x[1::6] = 0
            x[3, : hidden // 2] = 0
            x[4, 0] = 0
            x = x.to(dt)
            gq, gs, oq, os_ = _per_token_both(x, 24)
            assert np.array_equal(gq, oq), (dt, hidden)
            assert np.array_equal(gs.view(np.uint32), os_.view(np.uint32)), (dt, hidden)


def test_requant_chunk_widths_many_experts_and_unaligned_views():
    """32 codes per lane (rows a multiple of 32 codes, 32-byte aligned) and 16 (k = 16 * odd,
    or x / out views offset by 16 bytes); more than 32 experts (live counts read per lane
    instead of shuffled); out-of-range live counts; no masked_m."""
    g = torch.Generator().manual_seed(3)
    for E, M, K, group, off in [(3, 40, 1040, 16, 0), (40, 12, 512, 64, 0), (5, 33, 1024, 16, 0),
                                (4, 20, 2048, 128, 16), (2, 7, 96, 32, 16)]:
        codes = torch.randint(0, 256, (E, M, K), generator=g, dtype=torch.uint8).numpy()
        codes[(codes & 0x7F) == 0x7F] = 0
        xs = (torch.rand((E, M, K // group), generator=g) * 4 + 1e-3).numpy().astype(np.float32)
        masked = torch.randint(-3, M + 4, (E,), generator=g, dtype=torch.int32).numpy()
        masked[0] = M
        strides = (M * (K // group), K // group, 1)
        if off == 0:
            for mm in (masked, None):
                got, ref = _requant_both(codes, xs, strides, mm, 0.37, group)
                assert np.array_equal(got, ref), (E, M, K, group)
            continue
        # x and out as views 16 bytes into larger buffers
        xbig = torch.zeros(E * M * K + 64, dtype=torch.uint8, device="cuda")
        xv = xbig[off:off + E * M * K].view(E, M, K)
        xv.copy_(torch.from_numpy(codes))
        obig = torch.full((E * M * K + 64,), 0x2C, dtype=torch.uint8, device="cuda")
        ov = obig[off:off + E * M * K].view(E, M, K)
        sd = torch.as_strided(torch.from_numpy(xs.ravel().copy()).cuda(), (E, M, K // group), strides)
        osc = torch.tensor([0.37], dtype=torch.float32, device="cuda")
        P.requant_per_tensor(xv, sd, torch.from_numpy(masked).cuda(), osc, ov, group_size=group)
        torch.cuda.synchronize()
        ref = np.full((E, M, K), 0x2C, np.uint8)
        O.requant_per_tensor(codes, xs.ravel().copy(), strides, masked, 0.37, ref, group)
        ob = obig.cpu().numpy()
        assert np.array_equal(ob[off:off + E * M * K].reshape(E, M, K), ref)
        assert np.all(ob[:off] == 0x2C) and np.all(ob[off + E * M * K:] == 0x2C)
