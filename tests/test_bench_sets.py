"""bench.py's buffer sets on the CPU (no kernel runs): the view-based sets of the masked
decode workload stay inside their buffers, and their live rows, code rows and scale words
are distinct between sets, so each timed call reads and writes memory of its own."""
import numpy as np
import pytest
import torch

import bench
import fp8_token_group_gb300 as P


@pytest.fixture(scope="module")
def decode_sets():
    P.lib()
    wl = bench.workloads()["masked_decode"]
    x, mm = wl.inputs()
    sets = bench.build_view_sets(P, wl, x, mm, "cpu", 400)
    return wl, x, mm, sets


def test_view_sets_shapes_and_bounds(decode_sets):
    wl, x, mm, sets = decode_sets
    E, tp, hin = x.shape
    H = hin // 2
    ns = P.scale_elems(E, tp, H, wl.group, wl.fmt, wl.layout, True)
    assert len(sets) == 400
    for xd, q, s, m in sets:
        assert xd.shape == (E, tp, hin) and xd.is_contiguous()
        assert q.shape == (E, tp, H) and q.is_contiguous()
        assert s.numel() == ns and s.is_contiguous()
        for t in (xd, q, s):       # inside the storage it views
            assert t.storage_offset() + t.numel() <= t.untyped_storage().nbytes() // t.element_size()
        assert xd.data_ptr() % 32 == 0 and q.data_ptr() % 16 == 0 and s.data_ptr() % 4 == 0


def test_view_sets_touch_distinct_memory(decode_sets):
    wl, x, mm, sets = decode_sets
    E, tp, hin = x.shape
    H = hin // 2
    live = mm.numpy()
    seen_x, seen_q = set(), set()
    for xd, q, s, m in sets:
        for e in range(E):
            for r in range(int(live[e])):
                kx = (xd.untyped_storage().data_ptr(), xd.data_ptr() + (e * tp + r) * hin * 2)
                kq = (q.untyped_storage().data_ptr(), q.data_ptr() + (e * tp + r) * H)
                assert kx not in seen_x and kq not in seen_q
                seen_x.add(kx)
                seen_q.add(kq)
    # scale words written: column-major packed [E, ncol, tp], row r of expert e, column c
    ncol = (H // wl.group + 3) // 4
    words = set()
    for xd, q, s, m in sets:
        base = (s.untyped_storage().data_ptr(), s.data_ptr())
        for e in range(E):
            for c in range(ncol):
                for r in range(int(live[e])):
                    k = (base[0], base[1] + 4 * (e * ncol * tp + c * tp + r))
                    assert k not in words
                    words.add(k)


def test_full_copies_for_other_masked_workloads():
    wl = bench.workloads()["masked_silu"]
    x, mm = wl.inputs()
    per = wl.bytes_per_call(x, mm)
    nsets = max(2, min(bench.GRAPH_CALLS, -(-int(2.5 * bench.L2_BYTES) // per)))
    assert nsets * x.numel() * 2 <= 8 * 2 ** 30      # below the view-set threshold


@pytest.mark.parametrize("nsets", [2, 4, 5, 8, 200, 400])
def test_graph_plan_runs_exact_calls_on_alternating_sets(nsets):
    """bench.py runs exactly the requested calls, and within a timed region no call reads the
    buffer set the call before it read (so each reads from HBM): over call counts below, at
    and above the graph size.  Between regions bench.py flushes L2."""
    for calls in [1, 2, 3, 5, 19, 20, 21, 399, 400, 401, 1003, 60000]:
        g, reps, r = bench.graph_plan(calls, nsets)
        assert r + reps * g == calls and g % nsets == 0 and g <= bench.GRAPH_CALLS
        seq = [(nsets - r + i) % nsets for i in range(r)] + [i % nsets for i in range(g)] * reps
        assert len(seq) == calls
        assert all(a != b for a, b in zip(seq, seq[1:]))
        assert seq[-1] == nsets - 1
