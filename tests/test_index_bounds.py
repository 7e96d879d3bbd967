"""Bounds of the kernel's computed indices, on the CPU.  Each test restates one piece of the
index arithmetic of fp8_token_group_gb300/csrc/ptgq_kernel.cuh and ptgq_math.cuh with
numpy and checks, over every 16-bit value or a sweep of launch parameters, that every
shared-memory or global address it forms lies inside its buffer and equals the plain
per-element index.  They cover the three places where an index is computed from data or
from a guess rather than from the loop counters: the bf16 silu table offsets (formed for
both gates of a word at once, behind a range test), the fp16 silu table indices (two per
word, clamped with min.u16x2), and the rows prefetched on an expected_m hint.  No kernel
runs."""
import itertools
import os
import re

import numpy as np

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "fp8_token_group_gb300", "csrc")


def _defs():
    with open(os.path.join(CSRC, "silu_tables.inc")) as f:
        text = f.read()
    return {m.group(1): int(m.group(2), 0)
            for m in re.finditer(r"#define (PTGQ_SILU_\w+) (\S+)", text)}


def _words(lo: np.ndarray, hi: np.ndarray) -> np.ndarray:
    return (lo.astype(np.uint64) | (hi.astype(np.uint64) << 16)).astype(np.uint32)


# Partner halves: each half of a word must come out the same whatever the other half holds.
PARTNERS = np.array([0x0000, 0x0001, 0x3300, 0x7FFF, 0x8000, 0xB2FF, 0xFFFF], np.uint32)


def test_bf16_silu_offsets_behind_the_range_test():
    """Both gates of a word are offset at once: t = ((w | 0x80008000) - base2) ^ 0x80008000.
    A half passes the range test when t has no bit at 12 or above in it; the byte offset is
    then 4 * (sign * SPAN + |h| - base), at most 0x7FFC of the 32 KB table, and a half
    passes exactly when the gate lies in the table."""
    d = _defs()
    base, span = d["PTGQ_SILU_BF16_FIELD_LO"] << 7, d["PTGQ_SILU_BF16_SPAN"]
    assert span == 4096
    table_bytes = 2 * span * 4
    base2 = np.uint32(base | (base << 16))
    h = np.arange(65536, dtype=np.uint32)
    mag, sign = h & 0x7FFF, h >> 15
    in_table = (mag >= base) & (mag < base + span)
    want = 4 * (sign * span + mag - base)
    for p in PARTNERS:
        for w, half in ((_words(h, np.full_like(h, p)), 0), (_words(np.full_like(h, p), h), 1)):
            t = ((w | np.uint32(0x80008000)) - base2) ^ np.uint32(0x80008000)
            if half == 0:
                passes = (t & 0xF000) == 0
                o = ((t << 2) & 0x3FFC) | ((w >> 1) & 0x4000)
            else:
                passes = (t & 0xF0000000) == 0
                o = ((t >> 14) & 0x3FFC) | ((w >> 17) & 0x4000)
            assert np.array_equal(passes, in_table)
            assert np.all(o[passes] <= table_bytes - 4)
            assert np.array_equal(o[passes], want[passes])


def test_fp16_silu_indices_two_per_word():
    """idx = (w & 0x7FFF7FFF) + ((w >> 15) & 0x00010001) * POS, then min.u16x2 with
    ENTRIES - 1 in both halves: each half is min(|h| + sign * POS, ENTRIES - 1), inside the
    table, whatever the other half holds (no carry crosses the halves)."""
    d = _defs()
    pos, entries = d["PTGQ_SILU_F16_POS"], d["PTGQ_SILU_F16_ENTRIES"]
    assert pos + 0x7FFF < 0x10000 and entries <= 0x10000
    h = np.arange(65536, dtype=np.uint32)
    want = np.minimum((h & 0x7FFF) + (h >> 15) * pos, entries - 1)
    for p in PARTNERS:
        for lo, hi, half in ((h, np.full_like(h, p), 0), (np.full_like(h, p), h, 1)):
            w = _words(lo, hi)
            idx = ((w & np.uint32(0x7FFF7FFF)) +
                   ((w >> 15) & np.uint32(0x00010001)) * np.uint32(pos)).astype(np.uint32)
            got = np.minimum((idx >> (16 * half)) & 0xFFFF, entries - 1)   # min.u16x2, one half
            assert np.array_equal(got, want)
            assert np.all(got < (entries + 3) // 4 * 4)


def _udiv(n, d, magic):
    q = (n * magic) >> 32
    return q + (n - q * d >= d)


def test_hint_prefetch_stays_inside_x():
    """Every masked CTA guesses the rows of its warps' first tasks (each expert taken to have
    min(expected_m, tokens_pad) live rows with a hint, one without: hint 0 below) and
    prefetches them.  Over shapes, group sizes, scale formats, silu, hints, both task
    dealings and more warps than tasks, every prefetched 32-byte chunk (gate and, with silu,
    up) lies inside x = [E, tokens_pad, H_in]."""
    for E, rows, H, G, packed, silu, hint, rr in itertools.product(
            [1, 3, 32], [1, 5, 40], [128, 384, 2048], [16, 32, 64, 128], [0, 1], [0, 1],
            [0, 1, 3, 7, 1000], [0, 24, 32]):
        if H % G:
            continue
        hint = hint or 1                  # no hint: one live row per expert
        lg_log2 = {16: 0, 32: 1, 64: 2, 128: 3}[G]
        ug_log2 = 2 if packed else 0
        ng = H // G
        upr = (ng + (1 << ug_log2) - 1) >> ug_log2
        in_row = 2 * H if silu else H
        rows_hint = min(hint, rows)
        upr_magic = 0xFFFFFFFF if upr == 1 else (1 << 32) // upr
        hint_magic = 0xFFFFFFFF if rows_hint <= 1 else (1 << 32) // rows_hint
        lu = lg_log2 + ug_log2
        grid, warps = 6, rr if rr else 8
        b, w, lane = np.meshgrid(np.arange(grid), np.arange(warps), np.arange(32), indexing="ij")
        b, w, lane = b.ravel().astype(np.int64), w.ravel().astype(np.int64), lane.ravel()
        first = b + grid * w if rr else b * warps + w
        local = lane & ((1 << lu) - 1)
        u = (first << (5 - lu)) + (lane >> lu)
        R = _udiv(u, upr, upr_magic)
        assert np.array_equal(R, u // upr)
        e = _udiv(R, rows_hint, hint_magic)
        assert np.array_equal(e, R // rows_hint)
        g = ((u - R * upr) << ug_log2) + (local >> lg_log2)
        go = (e < E) & (g < ng)
        row = R - e * rows_hint
        off = (e * rows + row) * in_row + (g << (4 + lg_log2)) + (local & ((1 << lg_log2) - 1)) * 16
        end = off + (H if silu else 0) + 16
        assert np.all(row[go] < rows) and np.all(end[go] <= E * rows * in_row)


def _magic(d: int) -> int:
    return 0xFFFFFFFF if d == 1 else (1 << 32) // d


def test_requant_chunks_stay_inside_and_cover_every_live_row_once():
    """ptgq_next.cu, requant_kernel: lane chunks are numbered over row slots S = r * E + e
    (row-major over (row, expert)), and a warp's task loop ends at the tasks that can hold
    the first max(masked_m) * E slots.  Over shapes, group sizes, chunk widths, live counts
    (empty, partial, full, out of range) and grids smaller and larger than the work: every
    live chunk's code range and scale indices lie inside x / x_scale, and the live chunks
    are exactly the chunks of rows r < clamp(masked_m[e], 0, m), each taken once."""
    rng = np.random.default_rng(5)
    for E, m, k, G, V, grid_warps in itertools.product(
            [1, 3, 8, 33], [1, 5, 64], [16, 48, 128, 1152, 3584], [16, 32, 64, 128], [16, 32],
            [8, 200]):
        if k % G or k % V:
            continue
        mm = rng.integers(-2, m + 3, E).astype(np.int64)
        mm[0] = m
        live = np.clip(mm, 0, m)
        max_live = int(live.max())
        cpr = k // V
        live_chunks = max_live * E * cpr
        tasks = (live_chunks + 31) >> 5
        # every chunk index a warp forms: tasks t < tasks, lanes 0..31 (any grid covers
        # t = warp + j * grid_warps for all t < tasks)
        t = np.arange(tasks, dtype=np.int64)
        assert np.array_equal(np.unique(np.concatenate(
            [np.arange(w, tasks, grid_warps) for w in range(min(grid_warps, max(tasks, 1)))] or
            [np.zeros(0, np.int64)])), t)
        c = ((t[:, None] << 5) + np.arange(32)).ravel()
        assert c.max(initial=0) < 2 ** 32
        S = _udiv(c, cpr, _magic(cpr))
        assert np.array_equal(S, c // cpr)
        col = c - S * cpr
        r = _udiv(S, E, _magic(E))
        assert np.array_equal(r, S // E)
        e = S - r * E
        ok = (c < live_chunks) & (r < live[np.minimum(e, E - 1)]) & (e < E)
        off = (e * m + r) * k + col * V
        assert np.all(off[ok] >= 0) and np.all(off[ok] + V <= E * m * k)
        assert np.all(off[ok] % V == 0)
        g = (col * V) >> int(np.log2(G))
        g1 = g + (1 if (V == 32 and G == 16) else 0)
        assert np.all(g1[ok] < k // G)
        got = np.sort(off[ok])
        want = np.sort(np.concatenate([(ee * m + rr) * k + np.arange(cpr) * V
                                       for ee in range(E) for rr in range(int(live[ee]))] or
                                      [np.zeros(0, np.int64)]))
        assert np.array_equal(got, want), (E, m, k, G, V)


def test_requant_speculative_prefetch_stays_inside_x_and_x_scale():
    """ptgq_next.cu, requant_kernel: before the dependency wait each lane prefetches its
    chunk of the warp's first task as if every row were live (c0 = warp * 32 + lane, with
    the slot and row from the same 32-bit divisions as the loop), and that chunk's group
    scale; after the wait it loads the same chunk and its scale(s) before masked_m is
    known.  Over shapes, group sizes, chunk widths and grids: whenever r0 < m, the code
    chunk lies inside x = [E, m, k] and the scale indices (g0, and g0 + 1 when a 32-code
    chunk spans two groups of 16) inside the [E, m, k/G] grid."""
    for E, m, k, G, V, grid_ctas in itertools.product(
            [1, 3, 8, 33], [1, 5, 64, 1024], [16, 48, 128, 3584], [16, 32, 64, 128], [16, 32],
            [1, 7, 456]):
        if k % G or k % V:
            continue
        cpr = k // V
        c0 = np.arange(grid_ctas * 8 * 32, dtype=np.int64)
        S0 = _udiv(c0, cpr, _magic(cpr))
        assert np.array_equal(S0, c0 // cpr)
        r0 = _udiv(S0, E, _magic(E))
        assert np.array_equal(r0, S0 // E)
        ok = r0 < m
        e0 = S0 - r0 * E
        col0 = c0 - S0 * cpr
        off = (e0 * m + r0) * k + col0 * V
        assert np.all(e0[ok] < E) and np.all(off[ok] >= 0) and np.all(off[ok] + V <= E * m * k)
        g0 = (col0 * V) >> int(np.log2(G))
        assert np.all(g0[ok] < k // G)
        if V == 32 and G == 16:
            assert np.all(g0[ok] + 1 < k // G)


def test_flat_first_batch_prefetch_stays_inside_x():
    """ptgq_kernel.cuh: before the dependency wait every flat warp prefetches its first
    batch (the first task and, with two-task batches or in a light call of at most three
    tasks per warp, the task a grid stride further): units
    below the call's units, groups below the row's groups.  Over shapes, group sizes, scale
    formats, silu, batch sizes, both dealings and grids larger and smaller than the work,
    every prefetched chunk (gate and, with silu, up) lies inside x = [T, H_in]."""
    for T, H, G, packed, silu, kB, rr, grid in itertools.product(
            [1, 7, 64, 333], [128, 384, 2048], [16, 32, 64, 128], [0, 1], [0, 1], [1, 2, "light"],
            [0, 1], [1, 6, 600]):
        light = kB == "light"
        if light:
            kB = 1
            if silu or rr:
                continue                  # the light flavour is plain flat, tasks in blocks
        if H % G:
            continue
        lg_log2 = {16: 0, 32: 1, 64: 2, 128: 3}[G]
        ug_log2 = 2 if packed else 0
        ng = H // G
        upr = (ng + (1 << ug_log2) - 1) >> ug_log2
        in_row = 2 * H if silu else H
        units = T * upr
        lu = lg_log2 + ug_log2
        upw_log2 = 5 - lu
        tasks = (units + (1 << upw_log2) - 1) >> upw_log2
        warps = 32 if rr else 8
        stride = grid * warps
        b, w, lane = np.meshgrid(np.arange(grid), np.arange(warps), np.arange(32), indexing="ij")
        b, w, lane = b.ravel().astype(np.int64), w.ravel().astype(np.int64), lane.ravel()
        use_rr = rr and tasks < stride
        t0 = b + grid * w if use_rr else b * warps + w
        nb = 1 if (kB > 1 and tasks <= stride) else kB
        if light and tasks <= 3 * stride:
            nb = 2                        # the light flavour's second task, for <= 3 per warp
        local = lane & ((1 << lu) - 1)
        for bb in range(nb):
            u = ((t0 + bb * stride) << upw_log2) + (lane >> lu)
            ok = u < units
            R = _udiv(u, upr, 0xFFFFFFFF if upr == 1 else (1 << 32) // upr)
            assert np.array_equal(R[ok], (u // upr)[ok])
            g = ((u - R * upr) << ug_log2) + (local >> lg_log2)
            ok &= g < ng
            off = R * in_row + (g << (4 + lg_log2)) + (local & ((1 << lg_log2) - 1)) * 16
            end = off + (H if silu else 0) + 16
            assert np.all(R[ok] < T) and np.all(end[ok] <= T * in_row)


def test_flat_next_batch_prefetch_stays_inside_x():
    """ptgq_kernel.cuh: on a grid of several waves (plain flat calls with p.prefetch_next),
    each batch of KB tasks starting at task t prefetches the chunks of tasks t + (KB + i) *
    stride, i < KB, computed in 64 bits: units below the call's units, groups below the row's
    groups.  Over shapes, group sizes, scale formats, batch sizes and grids of one wave down to
    grids that leave 8 or more tasks per warp, for every batch every warp runs, every
    prefetched chunk lies inside x = [T, H] and is the chunk that task's load reads."""
    for T, H, G, packed, kB, grid in itertools.product(
            [7, 333, 1031], [128, 384, 2048], [16, 32, 64, 128], [0, 1], [1, 2], [1, 3, 40]):
        if H % G:
            continue
        lg_log2 = {16: 0, 32: 1, 64: 2, 128: 3}[G]
        ug_log2 = 2 if packed else 0
        ng = H // G
        upr = (ng + (1 << ug_log2) - 1) >> ug_log2
        units = T * upr
        lu = lg_log2 + ug_log2
        upw_log2 = 5 - lu
        tasks = (units + (1 << upw_log2) - 1) >> upw_log2
        warps = 8
        stride = grid * warps
        if tasks <= stride:
            continue                      # one-task batches without the prefetch
        b, w, lane = np.meshgrid(np.arange(grid), np.arange(warps), np.arange(32), indexing="ij")
        b, w, lane = b.ravel().astype(np.int64), w.ravel().astype(np.int64), lane.ravel()
        first = b * warps + w
        local = lane & ((1 << lu) - 1)
        gj = local >> lg_log2
        kk = local & ((1 << lg_log2) - 1)
        magic = 0xFFFFFFFF if upr == 1 else (1 << 32) // upr
        t = first.copy()
        while np.any(t < tasks):
            live = t < tasks
            for i in range(kB):
                tn = t + (kB + i) * stride
                un = (tn << upw_log2) + (lane >> lu)
                ok = live & (un < units)
                R = _udiv(np.where(ok, un, 0), upr, magic)
                assert np.array_equal(R[ok], (un // upr)[ok])
                g = ((un - R * upr) << ug_log2) + gj
                ok &= g < ng
                off = R * H + g * G + kk * 16
                assert np.all(R[ok] < T) and np.all(off[ok] + 16 <= T * H)
                assert np.array_equal(off[ok], ((un // upr) * H + g * G + kk * 16)[ok])
            t = t + kB * stride


def test_masked_warp_lookup_finds_the_owner_of_every_live_row():
    """ptgq_kernel.cuh, masked calls of at most 32 experts: each warp scans the clamped
    masked_m with shuffles (w_key[e] = exclusive prefix for e < n, all ones past n), and a
    lane with live row R takes the largest e with w_key[e] <= R by a five-step search over
    lanes lo + 16, 8, 4, 2, 1.  Over expert counts 1..32 and live counts with empty experts,
    negatives and counts past the pad: the search reads lanes 0..31 only, and for every live
    row R it returns the expert that owns R and the row R - w_key[e] < masked_m[e]."""
    rng = np.random.default_rng(11)
    for n in range(1, 33):
        for rows in [1, 3, 384]:
            for _ in range(20):
                mm = rng.integers(-3, rows + 4, n)
                mm[rng.random(n) < 0.3] = 0
                c = np.clip(mm, 0, rows).astype(np.int64)
                incl = np.cumsum(c)
                key = np.full(32, 0xFFFFFFFF, np.int64)
                key[:n] = incl - c
                live = int(incl[-1])
                R = np.arange(live, dtype=np.int64)
                lo = np.zeros(live, np.int64)
                base = np.zeros(live, np.int64)
                for step in [16, 8, 4, 2, 1]:
                    src = lo + step
                    assert src.max(initial=0) <= 31
                    v = key[src]
                    take = v <= R
                    lo = np.where(take, src, lo)
                    base = np.where(take, v, base)
                owner = np.repeat(np.arange(n), c)
                assert np.array_equal(lo, owner)
                assert np.array_equal(R - base, R - (incl - c)[owner])
                assert np.all(R - base < c[owner])
