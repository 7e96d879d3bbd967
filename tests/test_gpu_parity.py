"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle, element by
element, on the same seeded inputs.  Non-silu variants must match bit for bit (codes
and scales, including padding and masked rows); the fused-silu variants are held to the
stated tolerance (<= 1 e4m3 step on <= 1e-4 of codes, scale relative error <= 2e-7) and,
separately, checked for the exactness the kernel's correctly rounded exp gives."""
import itertools

import numpy as np
import pytest
import torch

import fp8_token_group_gb300 as P
from fp8_token_group_gb300 import synth
from parity_util import Case, assert_same, compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

FMTS = [P.SCALE_FP32, P.SCALE_UE8M0_PACKED, P.SCALE_UE8M0_FP32]
LAYOUTS = [P.ROW_MAJOR, P.COL_MAJOR_TMA]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    P.lib()


# ---------------------------------------------------------------- the five workloads

def test_flat_small_bf16_64x4096_fp32_rowmajor():
    compare(synth.flat_small(), Case())


def test_flat_outliers_4096x7168_ue8m0_packed_colmajor():
    """The benchmarked workload, at full size, in the launch configuration bench.py times."""
    compare(synth.flat_outliers(), Case(scale_fmt=P.SCALE_UE8M0_PACKED, layout=P.COL_MAJOR_TMA))


def test_silu_flat_8192x2x2048_fp32_colmajor():
    x = synth.silu_flat()
    c = Case(silu=True, layout=P.COL_MAJOR_TMA)
    compare(x, c, exact_silu=False)
    compare(x, c, exact_silu=True)


def test_masked_silu_32x384x2x4096_ue8m0_packed_colmajor():
    x, mm = synth.masked_silu()
    c = Case(silu=True, scale_fmt=P.SCALE_UE8M0_PACKED, layout=P.COL_MAJOR_TMA)
    compare(x, c, masked_m=mm.numpy(), exact_silu=False)
    compare(x, c, masked_m=mm.numpy(), exact_silu=True)


SMALL_SWEEP = [cs for cs in synth.sweep_cases() if cs[1] <= 4096]


@pytest.mark.parametrize("idx,T,H,dt,G,out", SMALL_SWEEP,
                         ids=[f"{c[1]}x{c[2]}-{str(c[3])[6:]}-G{c[4]}-{c[5]}" for c in SMALL_SWEEP])
def test_sweep(idx, T, H, dt, G, out):
    x = synth.sweep_input(idx, T, H, dt)
    compare(x, Case(group=G, out_dtype=P.E4M3 if out == "e4m3" else P.INT8))


# 32768 tokens: every hidden size and dtype, with (G=128, e4m3) and (G=16, int8); the
# other group/output pairs are covered at every smaller token count.
LARGE_SWEEP = [cs for cs in synth.sweep_cases() if cs[1] > 4096
               and (cs[4], cs[5]) in ((128, "e4m3"), (16, "int8"))]


@pytest.mark.parametrize("idx,T,H,dt,G,out", LARGE_SWEEP,
                         ids=[f"{c[1]}x{c[2]}-{str(c[3])[6:]}-G{c[4]}-{c[5]}" for c in LARGE_SWEEP])
def test_sweep_32768_tokens_sampled_rows(idx, T, H, dt, G, out):
    """Full-size launch; the oracle checks a sample of rows (rows are independent)."""
    x = synth.sweep_input(idx, T, H, dt)
    c = Case(group=G, out_dtype=P.E4M3 if out == "e4m3" else P.INT8)
    gq, gs = run_gpu(x, c)
    rng = np.random.default_rng(idx)
    rows = np.unique(np.concatenate([[0, 1, 2, 3, T - 1], rng.choice(T, 252, replace=False)]))
    oq, os_ = run_oracle(x[torch.from_numpy(rows)].contiguous(), c)
    ng = H // G
    assert_same(gq.reshape(T, H)[rows].ravel(), gs.reshape(T, ng)[rows].ravel(), oq, os_,
                f"sweep {idx} sampled rows")


# ---------------------------------------------------------------- the pages' shape grid

@pytest.mark.parametrize("silu", [False, True])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("T", [1, 7, 64, 333])
@pytest.mark.parametrize("H", [128, 2048, 4096])
@pytest.mark.parametrize("fmt", [P.SCALE_FP32, P.SCALE_UE8M0_PACKED])
def test_naive_scheduler_grid(silu, dt, T, H, fmt):
    """96 flat cases: vanilla and fused silu x bf16/fp16 x T x H x float/UE8M0 scales."""
    x = synth.normal((T, 2 * H if silu else H), dt, seed=T * 7 + H)
    compare(x, Case(silu=silu, scale_fmt=fmt, layout=P.COL_MAJOR_TMA), exact_silu=True)


@pytest.mark.parametrize("E,H,tp", list(itertools.product([2, 5], [2048, 4096], [128, 384])))
def test_masked_scheduler_grid(E, H, tp):
    """8 masked cases: UE8M0 + silu, [E, tokens_pad, 2H]."""
    x = synth.normal((E, tp, 2 * H), torch.bfloat16, seed=E * 1000 + tp)
    mm = synth.masked_counts(E, tp, seed=E + tp)
    compare(x, Case(silu=True, scale_fmt=P.SCALE_UE8M0_PACKED, layout=P.COL_MAJOR_TMA),
            masked_m=mm.numpy())


@pytest.mark.parametrize("T", [1024, 4096])
@pytest.mark.parametrize("fmt,layout", [(P.SCALE_FP32, P.ROW_MAJOR), (P.SCALE_UE8M0_PACKED, P.COL_MAJOR_TMA),
                                        (P.SCALE_UE8M0_FP32, P.COL_MAJOR_TMA)])
@pytest.mark.parametrize("out", [P.E4M3, P.INT8])
def test_flat_light_and_standard_flavours(T, fmt, layout, out):
    """Plain flat calls of at most about 8 tasks per warp run the light flavour (one task per
    batch, more warps per SM), larger ones the standard flavour; [1024, 7168] and
    [4096, 7168] fall on either side, in every scale format and output type."""
    x = synth.flat_outliers(tokens=T, hidden=7168)
    compare(x, Case(scale_fmt=fmt, layout=layout, out_dtype=out, tokens_pad=T + 3))


@pytest.mark.parametrize("fmt,layout,out", [(P.SCALE_FP32, P.ROW_MAJOR, P.E4M3),
                                            (P.SCALE_UE8M0_PACKED, P.COL_MAJOR_TMA, P.E4M3),
                                            (P.SCALE_UE8M0_FP32, P.COL_MAJOR_TMA, P.INT8)])
def test_flat_multi_wave_grid(fmt, layout, out):
    """Plain flat calls of more than 16 tasks per warp of one wave run a grid of several
    waves of CTAs with 8 tasks per warp ([8192, 7168] has 23.6 per warp of a wave), padding
    rows included: every output against the oracle."""
    x = synth.flat_outliers(tokens=8192, hidden=7168)
    compare(x, Case(scale_fmt=fmt, layout=layout, out_dtype=out, tokens_pad=8195))


@pytest.mark.parametrize("expected_m", [1, 7, 200, 384, 100000])
def test_masked_expected_m_hint_changes_nothing(expected_m):
    """A hint far below, near or above the live counts sizes the grid differently; the
    grid strides over the live rows either way, so every output matches the oracle."""
    x, mm = synth.masked_silu(experts=32, tokens_pad=384, hidden=2048)
    compare(x, Case(silu=True, scale_fmt=P.SCALE_UE8M0_PACKED, layout=P.COL_MAJOR_TMA,
                    expected_m=expected_m), masked_m=mm.numpy())


@pytest.mark.parametrize("G", [16, 32, 64, 128])
@pytest.mark.parametrize("silu", [False, True])
def test_masked_hint_every_group_size(G, silu):
    """A hinted call guesses each warp's first rows (as if every expert had expected_m live
    rows) and prefetches them before the live counts are read.  The guess must not matter:
    hints below, at and above the live counts, every group size and scale format."""
    x = synth.normal((5, 40, 768 * (2 if silu else 1)), torch.bfloat16, seed=31)
    mm = np.array([3, 0, 40, 3, 17], np.int32)
    for hint in (1, 3, 64):
        for fmt in (P.SCALE_FP32, P.SCALE_UE8M0_PACKED):
            compare(x, Case(group=G, silu=silu, scale_fmt=fmt, layout=P.COL_MAJOR_TMA,
                            expected_m=hint), masked_m=mm)


@pytest.mark.parametrize("fmt", [P.SCALE_UE8M0_PACKED, P.SCALE_FP32])
def test_masked_large_pad_per_expert(fmt):
    """A prefill-sized masked layout: 8 experts of 4096 rows, live counts up to the pad
    (one expert full, one empty), so the row-to-expert buckets use a large shift."""
    x = synth.normal((8, 4096, 2 * 2048), torch.bfloat16, seed=21)
    mm = synth.masked_counts(8, 4096, seed=21).numpy()
    mm[2], mm[5] = 4096, 0
    compare(x, Case(silu=True, scale_fmt=fmt, layout=P.COL_MAJOR_TMA), masked_m=mm)


def test_masked_decode_one_row_per_expert():
    """Decode-sized masked batch: one live row in each of 32 experts of 384, with and
    without the matching hint (most CTAs of the hint-less grid find no work and return)."""
    x, mm = synth.masked_decode()
    for hint in (0, 1):
        compare(x, Case(silu=True, scale_fmt=P.SCALE_UE8M0_PACKED, layout=P.COL_MAJOR_TMA,
                        expected_m=hint), masked_m=mm.numpy())


# ---------------------------------------------------------------- every variant, ragged shapes

@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("out", [P.E4M3, P.INT8])
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("G", [16, 32, 64, 128])
@pytest.mark.parametrize("silu", [False, True])
def test_flat_variants_ragged(dt, out, fmt, layout, G, silu):
    """37 live rows padded to 45, 7 groups per row (a partial packed word)."""
    H = 7 * G
    x = synth.sweep_input(3, 37, 2 * H if silu else H, dt)
    compare(x, Case(group=G, out_dtype=out, scale_fmt=fmt, layout=layout, silu=silu,
                    tokens_pad=45))


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("out", [P.E4M3, P.INT8])
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("G", [16, 128])
@pytest.mark.parametrize("silu", [False, True])
def test_masked_variants(dt, out, fmt, layout, G, silu):
    """The pages' masked counts {0, 1, 17, m} plus out-of-range values, clamped."""
    H = 5 * G
    x = synth.sweep_input(11, 6 * 23, 2 * H if silu else H, dt).reshape(6, 23, -1)
    mm = np.array([0, 1, 17, 23, 40, -3], dtype=np.int32)
    compare(x, Case(group=G, out_dtype=out, scale_fmt=fmt, layout=layout, silu=silu),
            masked_m=mm)


# ---------------------------------------------------------------- exhaustive value checks

@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("out", [P.E4M3, P.INT8])
@pytest.mark.parametrize("fmt", [P.SCALE_FP32, P.SCALE_UE8M0_FP32])
def test_every_16bit_value_with_anchor(dt, out, fmt):
    """Every finite 16-bit value in a group whose anchor makes the scale exactly 1."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = torch.from_numpy(bits.view(np.int16).copy()).view(dt).float()
    anchor = 448.0 if out == P.E4M3 else 127.0
    vals = vals[torch.isfinite(vals) & (vals.abs() <= anchor)]
    n = -(-vals.numel() // 127)
    grid = torch.zeros(n * 127)
    grid[: vals.numel()] = vals
    x = torch.cat([torch.full((n, 1), anchor), grid.view(n, 127)], 1).to(dt)
    compare(x, Case(out_dtype=out, scale_fmt=fmt))


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("out", [P.E4M3, P.INT8])
def test_division_every_quotient_pattern(dt, out):
    """For every amax mantissa of one binade and every value of up to 24 binades below it
    (both signs): the kernel's reciprocal-based division gives the IEEE codes.  Scaling by
    powers of two does not change the rounding, so this covers all normal pairs."""
    mant_bits = 7 if dt == torch.bfloat16 else 10
    step = 2.0 ** -mant_bits
    amaxes = 1.0 + step * np.arange(2 ** mant_bits)
    vals = []
    for e in range(0, 24):
        vals.append((1.0 + step * np.arange(2 ** mant_bits)) * 2.0 ** -e)
    vals = np.concatenate(vals)
    vals = np.concatenate([vals, -vals]).astype(np.float32)
    per = 127
    n_chunks = -(-vals.size // per)
    padded = np.zeros(n_chunks * per, np.float32)
    padded[: vals.size] = vals
    chunks = padded.reshape(n_chunks, per)
    rows = []
    for a in amaxes:
        ok = np.minimum(np.abs(chunks), a)
        rows.append(np.concatenate([np.full((n_chunks, 1), a, np.float32),
                                    np.copysign(ok, chunks)], 1))
    x = torch.from_numpy(np.concatenate(rows)).to(dt)
    x = x.reshape(-1, 128 * 4) if x.shape[0] % 4 == 0 else x
    compare(x, Case(out_dtype=out))


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
def test_silu_every_16bit_gate(dt):
    """Each gate value is the only non-zero product of its group (up = 1): the fp32 scale
    is RN(|silu(g)| / 448), so every silu value the kernel produces is compared."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    g = torch.from_numpy(bits.view(np.int16).copy()).view(dt)
    g = g[torch.isfinite(g.float()) & (g.float().abs() < 1e37)]   # 3 * silu(g) stays finite
    n = g.numel()
    # filler: gate 1.0 with up 0 (product 0), so groups whose tested gate is in the bf16
    # table range take the kernel's table fast path and the others its slow path
    gate = torch.ones((n, 128), dtype=dt)
    up = torch.zeros((n, 128), dtype=dt)
    gate[:, 0] = g
    up[:, 0] = 1.0
    gate[:, 1] = g            # a second copy scaled by up = -3 checks the product
    up[:, 1] = -3.0
    x = torch.cat([gate, up], 1)
    compare(x, Case(silu=True, eps=1e-24), exact_silu=True)


# ---------------------------------------------------------------- edge cases

def test_all_zero_bytes_0x55_and_vllm_floor_0x5e():
    x = torch.zeros((5, 7168), dtype=torch.bfloat16)
    c = Case(scale_fmt=P.SCALE_UE8M0_PACKED, layout=P.COL_MAJOR_TMA)
    gq, gs = compare(x, c)
    assert np.all(gq == 0) and np.all(gs.reshape(14, 8)[:, :5] == 0x55555555)
    assert np.all(gs.reshape(14, 8)[:, 5:] == 0)
    c.flags = P.FLAG_UE8M0_SCALE_FLOOR
    gq, gs = compare(x, c)
    assert np.all(gs.reshape(14, 8)[:, :5] == 0x5E5E5E5E)


@pytest.mark.parametrize("eps", [2.0 ** -140, 1e-38, 1.1754943508222875e-38, 1e-30, 1e-24,
                                 1e-10, 1e-4, 1.0, 1e20])
def test_eps_range(eps):
    """eps from the smallest accepted (2^-140, where an all-zero group's scale is a
    subnormal) through FLT_MIN and 1e-30 to large values; groups of zeros and of tiny
    values (bf16 subnormals included) take the kernel's IEEE-division path below an amax of
    1e-24, in the same warps as ordinary groups."""
    x = synth.sweep_input(5, 64, 1024, torch.bfloat16)
    x[3] = 0
    x[5, :128] = 1e-30
    x[6, 128:256] = 2.0 ** -133
    x[7, 256:384] = torch.linspace(-1e-36, 1e-36, 128)
    x[8, :16] = 0
    for fmt in FMTS:
        for out in (P.E4M3, P.INT8):
            compare(x, Case(eps=eps, scale_fmt=fmt, out_dtype=out, group=16 if fmt == 0 else 128))
    compare(x, Case(eps=eps, flags=P.FLAG_UE8M0_SCALE_FLOOR, scale_fmt=P.SCALE_UE8M0_PACKED,
                    layout=P.COL_MAJOR_TMA))
    xs = torch.cat([x, x.flip(0)], 1)
    compare(xs, Case(eps=eps, silu=True, scale_fmt=P.SCALE_UE8M0_PACKED), exact_silu=True)


@pytest.mark.parametrize("fmt", FMTS)
def test_nonfinite_amax_fixture_and_overflowing_silu(fmt):
    """Groups whose amax is +inf (an infinite element, or a silu product of finite gates
    and ups that overflows binary32): the hand-worked fixture of tests/golden/, then a
    larger call that mixes such groups with ordinary ones in every warp, flat and masked,
    bf16 and fp16, e4m3 and int8."""
    from golden_fixtures import nonfinite_amax_cases
    key = {P.SCALE_FP32: "fp32", P.SCALE_UE8M0_PACKED: "packed", P.SCALE_UE8M0_FP32: "ue8m0_fp32"}[fmt]
    for c in nonfinite_amax_cases():
        x = torch.from_numpy(c["x"].view(np.int16).copy()).view(torch.bfloat16).reshape(1, -1)
        case = Case(group=c["group"], silu=bool(c["silu"]), scale_fmt=fmt,
                    out_dtype=P.E4M3 if c["out"] == "e4m3" else P.INT8)
        gq, gs = compare(x, case)
        assert np.array_equal(gq, c["codes"]) and np.array_equal(gs, c[key]), c["name"]
    g = torch.Generator().manual_seed(17)
    for dt in (torch.bfloat16, torch.float16):
        big = torch.finfo(dt).max
        gate = torch.randn((96, 1024), generator=g)
        up = torch.randn((96, 1024), generator=g)
        rows = torch.randint(0, 96, (40,), generator=g)
        cols = torch.randint(0, 1024, (40,), generator=g)
        gate[rows, cols] = big          # silu(g) = g, and g * up overflows unless |up| < 1
        up[rows, cols] = big * torch.sign(torch.randn(40, generator=g))
        x = torch.cat([gate, up], 1).to(dt)
        for out in (P.E4M3, P.INT8):
            compare(x, Case(silu=True, scale_fmt=fmt, out_dtype=out, group=64), exact_silu=True)
        xi = torch.randn((64, 2048), generator=g)
        xi[torch.randint(0, 64, (30,), generator=g), torch.randint(0, 2048, (30,), generator=g)] = \
            float("inf")
        xi[5, 7] = -float("inf")
        xi = xi.to(dt)
        for out in (P.E4M3, P.INT8):
            compare(xi, Case(scale_fmt=fmt, out_dtype=out, layout=P.COL_MAJOR_TMA))
            compare(xi.reshape(4, 16, 2048), Case(scale_fmt=fmt, out_dtype=out),
                    masked_m=np.array([16, 3, 0, 9], np.int32))


@pytest.mark.parametrize("T,H", [(64, 2048), (4096, 2048), (8192, 4096), (16384, 4096)])
@pytest.mark.parametrize("fmt", [P.SCALE_FP32, P.SCALE_UE8M0_PACKED])
def test_nonfinite_and_tiny_eps_on_every_flat_flavour(T, H, fmt):
    """The plain flat launch shapes (light, light with the next-batch prefetch, one
    persistent wave, several waves): groups with an infinite element (amax = +inf, handled
    by selects in the e4m3 instances and by the warp vote in the int8 ones), and the same
    input with eps = 1e-30 over zeroed groups (the checked instances)."""
    g = torch.Generator().manual_seed(T + H)
    x = torch.randn((T, H), generator=g)
    n = max(8, T // 64)
    x[torch.randint(0, T, (n,), generator=g), torch.randint(0, H, (n,), generator=g)] = float("inf")
    x[1, 3] = -float("inf")
    x[2, :256] = 0.0
    x = x.to(torch.bfloat16)
    for out in (P.E4M3, P.INT8):
        compare(x, Case(scale_fmt=fmt, out_dtype=out, layout=P.COL_MAJOR_TMA))
    xz = x.clone()
    xz[torch.isinf(xz)] = 0.0
    xz[5, 128:512] = 1e-30
    compare(xz, Case(scale_fmt=fmt, eps=1e-30, layout=P.COL_MAJOR_TMA))


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("silu", [False, True])
def test_tiny_eps_masked(dt, silu):
    """eps below 1e-24 in masked calls (the checked masked instances), decode-sized and
    larger, with all-zero and tiny groups among ordinary ones."""
    for E, rows, mm in [(32, 8, [1] * 32), (8, 512, [512, 3, 0, 200, 511, 77, 1, 300])]:
        H = 1024
        x = synth.sweep_input(E + rows, E * rows, 2 * H if silu else H, dt).reshape(E, rows, -1)
        x[0, 0, :128] = 0
        x[3, 0, 128:256] = 1e-30 if dt == torch.bfloat16 else 0
        for fmt in (P.SCALE_FP32, P.SCALE_UE8M0_PACKED):
            compare(x, Case(eps=2.0 ** -140, scale_fmt=fmt, silu=silu),
                    masked_m=np.array(mm, np.int32))


def test_extreme_values():
    dt = torch.bfloat16
    x = torch.zeros((8, 256), dtype=dt)
    x[0, :] = torch.finfo(dt).max
    x[1, ::2] = -torch.finfo(dt).max
    x[2, :] = torch.finfo(dt).tiny
    x[3, :] = 2.0 ** -133              # smallest bf16 subnormal
    x[4, :] = -0.0
    x[5, 0] = 3e38
    x[5, 1:] = 1e-30
    x[6, :] = torch.linspace(-500, 500, 256).to(dt)
    x[7, 1::2] = -0.0
    for out in (P.E4M3, P.INT8):
        for fmt in FMTS:
            compare(x, Case(out_dtype=out, scale_fmt=fmt))
    # silu: extreme gates with up = 1 (gate * up must stay finite)
    xs = torch.cat([x, torch.ones_like(x)], 1)
    for fmt in FMTS:
        compare(xs, Case(silu=True, scale_fmt=fmt), exact_silu=True)


def test_flat_zero_tokens_only_zero_fills_padding():
    x = torch.zeros((0, 1024), dtype=torch.bfloat16)
    for fmt in FMTS:
        for layout in LAYOUTS:
            compare(x, Case(scale_fmt=fmt, layout=layout, tokens_pad=9))
    # the silu instances copy their table before they know there is no task
    for dt in (torch.bfloat16, torch.float16):
        compare(torch.zeros((0, 2048), dtype=dt), Case(silu=True, tokens_pad=9))


def test_masked_all_empty_and_zero_experts():
    x = synth.normal((3, 16, 256), torch.bfloat16, seed=1)
    compare(x, Case(), masked_m=np.zeros(3, np.int32))
    gq, gs = run_gpu(synth.normal((0, 16, 256), torch.bfloat16), Case(),
                     masked_m=np.zeros(0, np.int32))
    assert gq.size == 0 and gs.size == 0


@pytest.mark.parametrize("E", [1, 2, 31, 32, 33])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("silu", [False, True])
@pytest.mark.parametrize("size", ["decode", "large"])
def test_masked_expert_lookup_around_32_experts(E, dt, silu, size):
    """Masked calls of at most 32 experts scan masked_m per warp; decode-sized ones (at most
    one task per warp) look the expert up by shuffles, larger ones through the shared-memory
    buckets, and more than 32 experts take the block-wide prefix.  Short rows (H = 128 at
    G = 128: four rows per warp task; H = 256 at G = 16 packed: two) make tasks cross experts,
    with empty experts, negative counts and counts past the pad in between."""
    rng = np.random.default_rng(E * 10 + silu + (size == "large") * 100)
    if size == "decode":
        rows = 8
        mm = rng.integers(0, 3, E)
    else:
        rows = max(8, 32768 // E)
        mm = rng.integers(rows // 2, rows + 4, E)
    mm[rng.random(E) < 0.2] = 0
    if E > 2:
        mm[1] = -4
        mm[2] = rows + 9
    mm = mm.astype(np.int32)
    for H, c in [(128, Case(silu=silu)),
                 (256, Case(group=16, silu=silu, scale_fmt=P.SCALE_UE8M0_PACKED,
                            layout=P.COL_MAJOR_TMA))]:
        x = synth.sweep_input(E + 7, E * rows, 2 * H if silu else H, dt).reshape(E, rows, -1)
        compare(x, c, masked_m=mm)
        if size == "decode":
            c.expected_m = 1
            compare(x, c, masked_m=mm)


@pytest.mark.parametrize("E", [6, 32, 33, 1000])
@pytest.mark.parametrize("silu", [False, True])
def test_masked_m_error_counter(E, silu):
    """The optional masked_m_errors counter of ptgq_quant_ex: each call adds the number of
    experts whose masked_m lies outside [0, tokens_pad], for the warp-scanned (E <= 32) and
    the block-wide (E > 32) prefix, decode-sized and larger calls; the outputs stay those of
    the clamped counts (oracle), and a second call adds again."""
    rng = np.random.default_rng(E + 7 * silu)
    tp, H = 23, 256
    mm = rng.integers(0, tp + 1, E)
    bad = rng.random(E) < 0.25
    mm[bad] = np.where(rng.random(int(bad.sum())) < 0.5, -rng.integers(1, 5, int(bad.sum())),
                       tp + rng.integers(1, 40, int(bad.sum())))
    mm[0] = -1
    mm = mm.astype(np.int32)
    want = int(((mm < 0) | (mm > tp)).sum())
    x = synth.sweep_input(E + 3, E * tp, 2 * H if silu else H, torch.bfloat16).reshape(E, tp, -1)
    xd = x.cuda()
    md = torch.from_numpy(mm).cuda()
    errs = torch.zeros(1, dtype=torch.int32, device="cuda")
    for hint in (0, 1):
        q, sc = P.alloc_outputs(xd, 128, scale_fmt=P.SCALE_UE8M0_PACKED, fuse_silu=silu, masked=True)
        P.quant(xd, q, sc, 128, scale_fmt=P.SCALE_UE8M0_PACKED, fuse_silu=silu, masked_m=md,
                expected_m=hint, masked_m_errors=errs)
    torch.cuda.synchronize()
    assert int(errs.item()) == 2 * want
    compare(x, Case(silu=silu, scale_fmt=P.SCALE_UE8M0_PACKED), masked_m=mm)


def test_many_experts():
    E = 1000
    x = synth.normal((E, 4, 256), torch.bfloat16, seed=2)
    mm = synth.masked_counts(E, 4, seed=5).numpy()
    compare(x, Case(scale_fmt=P.SCALE_UE8M0_PACKED, layout=P.COL_MAJOR_TMA), masked_m=mm)


# ---------------------------------------------------------------- launch behaviour

def test_pdl_and_plain_launch_agree_and_repeat():
    x = synth.flat_outliers(512, 7168)
    c = Case(scale_fmt=P.SCALE_UE8M0_PACKED, layout=P.COL_MAJOR_TMA)
    a = run_gpu(x, c)
    c.flags = P.FLAG_NO_PDL
    b = run_gpu(x, c)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_back_to_back_launches_and_cuda_graph():
    x = synth.silu_flat(1024, 2048).cuda()
    q, s = P.alloc_outputs(x, 128, fuse_silu=True)
    P.quant(x, q, s, 128, fuse_silu=True)
    torch.cuda.synchronize()
    ref_q, ref_s = q.clone(), s.clone()
    q2, s2 = torch.empty_like(q), torch.empty_like(s)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for _ in range(20):
            P.quant(x, q2, s2, 128, fuse_silu=True)
    torch.cuda.synchronize()
    assert torch.equal(q2.view(torch.uint8), ref_q.view(torch.uint8)) and torch.equal(s2, ref_s)
    q3, s3 = torch.zeros_like(q), torch.zeros_like(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(3):
            P.quant(x, q3, s3, 128, fuse_silu=True)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(q3.view(torch.uint8), ref_q.view(torch.uint8)) and torch.equal(s3, ref_s)


def test_masked_calls_and_error_counter_in_a_cuda_graph():
    """A masked call with the masked_m error counter (two kernels per call) captured in a CUDA
    graph with its masked_m and replayed: the outputs match an eager call, and the counter
    grows by the out-of-range count on every replay."""
    x, mm = synth.masked_silu(experts=8, tokens_pad=64, hidden=512)
    mm = mm.clone()
    mm[1], mm[5] = -2, 90
    xd, md = x.cuda(), mm.cuda()
    q, sc = P.alloc_outputs(xd, 128, fuse_silu=True, masked=True, scale_fmt=P.SCALE_UE8M0_PACKED)
    q.view(torch.uint8).fill_(0x2C)
    sc.fill_(0x2C2C2C2C)
    P.quant(xd, q, sc, 128, fuse_silu=True, masked_m=md, scale_fmt=P.SCALE_UE8M0_PACKED)
    torch.cuda.synchronize()
    ref_q, ref_s = q.clone(), sc.clone()
    q2, s2 = q.clone().fill_(0), sc.clone().fill_(0)
    q2.view(torch.uint8).fill_(0x2C)
    s2.fill_(0x2C2C2C2C)
    errs = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        P.quant(xd, q2, s2, 128, fuse_silu=True, masked_m=md, scale_fmt=P.SCALE_UE8M0_PACKED,
                masked_m_errors=errs)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(q2.view(torch.uint8), ref_q.view(torch.uint8)) and torch.equal(s2, ref_s)
    assert int(errs.item()) == 3 * 2


def test_device_arguments_rejected_before_launch():
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")
    q, s = P.alloc_outputs(x, 128)
    L = P.lib()
    stream = torch.cuda.current_stream().cuda_stream
    rc = L.ptgq_quant(x.data_ptr() + 2, 0, 4, 0, 256, 128, q.data_ptr(), 0, s.data_ptr(), 0, 0,
                      0, None, 1e-10, stream)
    assert rc == -7
    rc = L.ptgq_quant(x.data_ptr(), 0, 4, 0, 256, 128, q.data_ptr() + 8, 0, s.data_ptr(), 0, 0,
                      0, None, 1e-10, stream)
    assert rc == -7
    rc = L.ptgq_quant(x.data_ptr(), 0, 4, 2, 256, 128, q.data_ptr(), 0, s.data_ptr(), 0, 0, 0,
                      None, 1e-10, stream)
    assert rc == -6


def test_concurrent_calls_from_threads_on_their_own_streams():
    """Eight host threads, each on its own stream and with its own variant (scale format,
    layout, output type, silu), call the library repeatedly at once: the launcher's shared
    occupancy and attribute caches are hit concurrently, and every result still matches
    the oracle bit for bit."""
    import threading
    cases = [Case(scale_fmt=FMTS[i % 3], layout=LAYOUTS[i % 2], out_dtype=(P.E4M3, P.INT8)[(i // 2) % 2],
                  silu=bool(i & 4), group=(128, 64, 32, 16)[i % 4]) for i in range(8)]
    xs = [synth.normal((96 + 8 * i, 2048 if c.silu else 1024), torch.bfloat16, seed=50 + i)
          for i, c in enumerate(cases)]
    results, errors = [None] * len(cases), []

    def work(i):
        try:
            c, xd = cases[i], xs[i].cuda()
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                q, s = P.alloc_outputs(xd, c.group, out_dtype=c.out_dtype, scale_fmt=c.scale_fmt,
                                       scale_layout=c.layout, fuse_silu=c.silu)
                for _ in range(25):
                    P.quant(xd, q, s, c.group, out_dtype=c.out_dtype, scale_fmt=c.scale_fmt,
                            scale_layout=c.layout, fuse_silu=c.silu)
            stream.synchronize()
            results[i] = (q.view(torch.uint8).cpu().numpy().ravel(),
                          s.view(torch.int32).cpu().numpy().view(np.uint32).ravel())
        except Exception as exc:           # reported below, on the main thread
            errors.append(exc)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(cases))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for i, c in enumerate(cases):
        oq, os_ = run_oracle(xs[i], c)
        assert_same(results[i][0], results[i][1], oq, os_, f"thread {i} {c}")


def test_binding_rejects_short_buffers_before_launch():
    """The library sees raw pointers; the binding checks that the outputs hold what a call
    writes, so a short buffer raises instead of being written past its end.  Nothing is
    launched: the sentinel contents stay."""
    x = synth.flat_small()
    xd = x.cuda()
    kw = dict(scale_fmt=P.SCALE_UE8M0_PACKED, scale_layout=P.COL_MAJOR_TMA)
    q, s = P.alloc_outputs(xd, 128, **kw)
    q.view(torch.uint8).fill_(0x7F)
    s.fill_(-1)
    with pytest.raises(ValueError, match="out_s"):
        P.quant(xd, q, s[:-1], 128, **kw)
    with pytest.raises(ValueError, match="out_q"):
        P.quant(xd, q[:-1], s, 128, **kw)
    with pytest.raises(ValueError, match="out_q"):
        P.quant(xd, q, s, 128, tokens_pad=80, **kw)           # padding rows need more room
    xm, mm = synth.masked_silu(experts=4, tokens_pad=32, hidden=256)
    xmd, mmd = xm.cuda(), mm.cuda()
    qm, sm = P.alloc_outputs(xmd, 128, fuse_silu=True, masked=True, **kw)
    with pytest.raises(ValueError, match="masked_m"):
        P.quant(xmd, qm, sm, 128, fuse_silu=True, masked_m=mmd[:3], **kw)
    with pytest.raises(ValueError, match="out_s"):
        P.quant(xmd, qm, sm[:-1], 128, fuse_silu=True, masked_m=mmd, **kw)
    xo = torch.zeros((4, 2 * 256 + 1), dtype=torch.bfloat16, device="cuda")    # odd width
    with pytest.raises(ValueError, match="fuse_silu"):
        P.quant(xo, q, s, 128, fuse_silu=True, **kw)
    with pytest.raises(ValueError, match="fuse_silu"):
        P.alloc_outputs(torch.zeros((4, 257), dtype=torch.bfloat16, device="cuda"), 128,
                        fuse_silu=True)
    xt = torch.randn(16, 512, device="cuda").to(torch.bfloat16)
    qt = torch.empty((16, 512), dtype=torch.float8_e4m3fn, device="cuda")
    st = torch.empty(16, dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError, match="out_q"):
        P.per_token_quant(xt, qt, st[:15])
    with pytest.raises(ValueError, match="num_tokens"):
        P.per_token_quant(xt, qt, st, num_tokens=17)
    codes = torch.zeros((2, 8, 256), dtype=torch.uint8, device="cuda")
    xs = torch.ones((2, 8, 2), dtype=torch.float32, device="cuda")
    osc = torch.ones(1, dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError, match="out must hold"):
        P.requant_per_tensor(codes, xs, None, osc,
                             torch.empty(2 * 7 * 256, dtype=torch.uint8, device="cuda"))
    with pytest.raises(ValueError, match="x_scale"):         # one group's scales, two groups
        P.requant_per_tensor(codes, torch.ones((2, 8, 1), device="cuda"), None, osc,
                             torch.empty_like(codes))
    torch.cuda.synchronize()
    assert bool((q.view(torch.uint8) == 0x7F).all()) and bool((s == -1).all())


def test_masked_4096_experts_mostly_empty():
    """The largest expert count, with many empty and one-row experts: exercises the
    row-to-expert buckets across runs of empty experts.  With fused silu on fp16 input it is
    also the largest shared-memory footprint: the fp16 silu table plus 4096 experts' prefix
    sums and the buckets."""
    E, tp = 4096, 3
    x = synth.normal((E, tp, 256), torch.bfloat16, seed=4)
    g = torch.Generator().manual_seed(11)
    mm = torch.randint(0, 4, (E,), generator=g, dtype=torch.int32)
    mm[torch.rand(E, generator=g) < 0.7] = 0          # 70% of experts empty
    mm[-1] = 3
    for fmt in FMTS:
        compare(x, Case(scale_fmt=fmt, layout=P.COL_MAJOR_TMA), masked_m=mm.numpy())
    compare(torch.cat([x, x], 2), Case(silu=True, scale_fmt=P.SCALE_UE8M0_PACKED,
                                       layout=P.COL_MAJOR_TMA), masked_m=mm.numpy())
    xh = synth.normal((E, tp, 512), torch.float16, seed=6)
    compare(xh, Case(silu=True, scale_fmt=P.SCALE_UE8M0_PACKED, layout=P.COL_MAJOR_TMA),
            masked_m=mm.numpy())


def test_pinned_host_buffers_in_place():
    """Pinned host tensors are device-accessible (unified addressing): quantizing them in
    place gives the same bytes as device buffers."""
    x = synth.flat_outliers(256, 7168)
    c = Case(scale_fmt=P.SCALE_UE8M0_PACKED, layout=P.COL_MAJOR_TMA)
    gq, gs = run_gpu(x, c)
    xh = x.pin_memory()
    qh = torch.empty((256, 7168), dtype=torch.float8_e4m3fn).pin_memory()
    sh = torch.empty(P.scale_elems(256, 0, 7168, 128, c.scale_fmt, c.layout, False),
                     dtype=torch.int32).pin_memory()
    P.quant(xh, qh, sh, 128, scale_fmt=c.scale_fmt, scale_layout=c.layout)
    torch.cuda.synchronize()
    assert np.array_equal(qh.view(torch.uint8).numpy().ravel(), gq)
    assert np.array_equal(sh.numpy().view(np.uint32), gs)
