#!/usr/bin/env python3
"""Benchmark of per-token-group 8-bit quantization on GB300.

One step = one ptgq_quant call over one batch of the benchmarked workload:
flat bf16 x [4096, 7168] (N(0,1), 0.1% outliers x100, 1% all-zero groups), G = 128,
e4m3 codes, UE8M0 exponents packed four per int32 in the TMA-aligned column-major layout.

Prints one JSON line.  ``value`` is the achieved HBM throughput in GB/s (algorithmic bytes:
input read + codes written + scale words written, per call, over the device time of the
timed steps, summed over ranks).  Timing: W warm-up calls, then five timed regions of
exactly K calls each, replayed from CUDA graphs, each bracketed by an L2 flush, a barrier and
a synchronize and timed with CUDA events on the launching stream; the median region (max
over ranks) is reported.  Inputs rotate over buffer sets that together exceed 2.5x L2, so
each call reads from HBM, not L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the CPU oracle (test infrastructure, single-threaded C++) on a
bounded sample of the same workload and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s (% of GB300 peak) and µs/call, per_token_group_quant FP8 G=128"
WORKLOAD = "flat bf16 x[4096,7168] N(0,1)+0.1% outliers x100+1% zero groups, G=128, e4m3, " \
           "UE8M0 packed int32 col-major (mn padded to 4, pads zero-filled)"
T, H, G = 4096, 7168, 128
GRAPH_CALLS = 400                      # most calls captured in one CUDA graph
REPEATS = 5                            # timed regions; the median is reported
KERNEL_SOURCES = ["ptgq_kernel.cuh", "ptgq_math.cuh", "ptgq_api.cu", "ptgq_internal.h",
                  "ptgq_inst_bf16_flat.cu", "ptgq_inst_bf16_masked.cu", "ptgq_inst_fp16_flat.cu",
                  "ptgq_inst_fp16_masked.cu", "ptgq_device.cuh", "ptgq_next.cu",
                  "silu_tables.inc"]


def algorithmic_bytes(tokens: int = T, hidden: int = H, group: int = G) -> int:
    ng = hidden // group
    words = (ng + 3) // 4 * ((tokens + 3) // 4 * 4)
    return tokens * hidden * 2 + tokens * hidden + words * 4


def kernel_source_sha() -> str:
    """Hash of the kernel sources with comments and blank space removed, so a recorded DRAM
    traffic figure stays valid across comment-only edits and no longer."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "fp8_token_group_gb300", "csrc", f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def recorded_traffic(workload: str):
    """Steady-state DRAM bytes per launch of a workload's kernel from the committed ncu
    record (mean over back-to-back launches), if it was taken on the current sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_sha") != kernel_source_sha():
        return None
    w = d.get("workloads", {}).get(workload)
    return None if w is None else w.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def start(self):
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        self.proc.wait()
        self.tmp.flush()
        rows = []
        with open(self.tmp.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.tmp.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("PTGQ_BENCH_BACKEND", "nccl")
        dist.init_process_group(backend)
    return world, rank, local


def reduce_max(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(bytes_per_step: int, steps: int, world: int, max_elapsed_s: float) -> float:
    """Whole-job GB/s: every rank processed `steps` calls of `bytes_per_step`."""
    return world * steps * bytes_per_step / max_elapsed_s / 1e9


# ---------------------------------------------------------------- CPU oracle timing

def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_rate(x_cpu, rows_per_step: int, steps: int, warmup: int, threads: int = 1):
    """Seconds and GB/s of the oracle on `rows_per_step` rows of the workload.  With
    threads > 1 the rows are split into that many blocks of whole rows, each quantized by
    its own oracle call on its own thread (the calls release the GIL), as independent
    problems with their own scale buffers; the oracle itself is unchanged."""
    import numpy as np
    import oracle as O
    from fp8_token_group_gb300 import synth
    nb = max(1, min(threads, rows_per_step))
    edges = [rows_per_step * i // nb for i in range(nb + 1)]
    blocks = []
    for i in range(nb):
        r = edges[i + 1] - edges[i]
        if r == 0:
            continue
        bits = synth.bits_u16(x_cpu[edges[i]:edges[i + 1]].contiguous())
        q = np.empty(r * H, np.uint8)
        s = np.empty(O.scale_elems(r, 0, H, G, O.FMT_UE8M0_PACKED, O.LAYOUT_COL, 0), np.uint32)
        blocks.append((bits, r, q, s))

    def one(b):
        bits, r, q, s = b
        O.quant(bits, O.IN_BF16, r, 0, H, G, q, O.OUT_E4M3, s, O.FMT_UE8M0_PACKED,
                O.LAYOUT_COL, 0, None, 1e-10)

    pool = None
    if len(blocks) > 1:
        from concurrent.futures import ThreadPoolExecutor
        pool = ThreadPoolExecutor(len(blocks))
        run = lambda: list(pool.map(one, blocks))
    else:
        run = lambda: one(blocks[0])
    try:
        for _ in range(warmup):
            run()
        t0 = time.perf_counter()
        for _ in range(steps):
            run()
        el = time.perf_counter() - t0
    finally:
        if pool is not None:
            pool.shutdown()
    nbytes = sum(algorithmic_bytes(b[1]) for b in blocks) * steps
    return el, nbytes / el / 1e9


def cpu_baseline(x_cpu, budget_s: float = 8.0) -> dict:
    """The oracle on the host: all cores (one row block per thread), and one core."""
    import oracle as O
    O.build()
    cores = host_cores()
    rows1, rowsn = 64, 64 * cores
    el, _ = oracle_rate(x_cpu, rows1, 1, 1)
    reps1 = max(1, int(budget_s / max(el, 1e-6)))
    el1, gbs1 = oracle_rate(x_cpu, rows1, reps1, 0)
    el, _ = oracle_rate(x_cpu, rowsn, 1, 1, threads=cores)
    repsn = max(1, int(budget_s / max(el, 1e-6)))
    eln, gbsn = oracle_rate(x_cpu, rowsn, repsn, 0, threads=cores)
    return {"value": round(gbsn, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "single_core_value": round(gbs1, 4),
            "sample": f"{rowsn} rows x {H} of the benchmarked input in {cores} row blocks on "
                      f"{cores} threads, {repsn} repetitions ({eln:.1f} s); one core: {rows1} "
                      f"rows, {reps1} repetitions ({el1:.1f} s); C++ oracle"}


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import oracle as O
    O.build()
    wl = workloads()["flat_outliers"]
    x, _ = wl.inputs()
    # size each step so the whole run stays within about a minute
    cores = host_cores()
    el1, _ = oracle_rate(x, cores, 2, 1, threads=cores)
    per_row = el1 / 2 / cores              # wall seconds per row with all cores busy
    rows = int(max(cores, min(T, 60.0 / max(args.steps + args.warmup, 1) / max(per_row, 1e-7))))
    el, gbs = oracle_rate(x, rows, args.steps, args.warmup, threads=cores)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": bench_config(wl, x, None, world),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: {rows} of the workload's {T} rows x {H}, in "
                                   f"{cores} row blocks on {cores} threads, C++ oracle"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- workloads

L2_BYTES = 129 * 2 ** 20


class Workload:
    """One configuration: seeded CPU input, quantization arguments, algorithmic bytes."""

    def __init__(self, name, desc, make, *, silu=False, fmt=0, layout=0, group=G, out=0,
                 expected_m=0):
        self.name, self.desc, self.make = name, desc, make
        self.silu, self.fmt, self.layout, self.group, self.out = silu, fmt, layout, group, out
        self.expected_m = expected_m

    def inputs(self):
        r = self.make()
        return r if isinstance(r, tuple) else (r, None)

    def live_rows(self, x, mm) -> int:
        if mm is None:
            return x.shape[0]
        return int(mm.clamp(0, x.shape[1]).sum())

    def bytes_per_call(self, x, mm) -> int:
        hin = x.shape[-1]
        h = hin // 2 if self.silu else hin
        live = self.live_rows(x, mm)
        ng = h // self.group
        if self.fmt == 1:   # packed UE8M0: int32 words, column pitch round_up(rows, 4)
            ncol = (ng + 3) // 4
            rows = x.shape[1] if mm is not None else (x.shape[0] + 3) // 4 * 4
            sbytes = 4 * ncol * (live if mm is not None else rows)
        else:
            sbytes = 4 * ng * live
        return live * hin * 2 + live * h + sbytes

    def call(self, P, xd, q, s, mm=None):
        P.quant(xd, q, s, self.group, out_dtype=self.out, scale_fmt=self.fmt,
                scale_layout=self.layout, fuse_silu=self.silu, masked_m=mm,
                expected_m=self.expected_m)

    def alloc(self, P, xd, mm):
        return P.alloc_outputs(xd, self.group, out_dtype=self.out, scale_fmt=self.fmt,
                               scale_layout=self.layout, fuse_silu=self.silu,
                               masked=mm is not None)


class PerTokenWorkload(Workload):
    """Per-token (whole-row) FP8 quantization: x [T, hidden] -> e4m3 codes + one scale/row."""

    def __init__(self, name, desc, tokens, hidden):
        super().__init__(name, desc, None)
        self.tokens, self.hidden = tokens, hidden

    def inputs(self):
        from fp8_token_group_gb300 import synth
        import torch
        return synth.normal((self.tokens, self.hidden), torch.bfloat16, seed=4), None

    def live_rows(self, x, mm):
        return x.shape[0]

    def bytes_per_call(self, x, mm):
        return x.shape[0] * x.shape[1] * 3 + x.shape[0] * 4

    def alloc(self, P, xd, mm):
        import torch
        return (torch.empty(xd.shape, dtype=torch.float8_e4m3fn, device=xd.device),
                torch.empty(xd.shape[0], dtype=torch.float32, device=xd.device))

    def call(self, P, xd, q, s, mm=None):
        P.per_token_quant(xd, q, s)


class RequantWorkload(Workload):
    """Per-token-group FP8 -> per-tensor FP8 requant over [E, M, K] with masked rows."""

    def __init__(self, name, desc, experts, m, k, live_per_expert):
        super().__init__(name, desc, None)
        self.experts, self.m, self.k, self.live = experts, m, k, live_per_expert

    def inputs(self):
        import torch
        g = torch.Generator().manual_seed(6)
        x = torch.randint(-8, 9, (self.experts, self.m, self.k), generator=g).float()
        codes = x.to(torch.float8_e4m3fn).view(torch.uint8)
        mm = torch.full((self.experts,), self.live, dtype=torch.int32)
        return codes, mm

    def live_rows(self, x, mm):
        return int(mm.clamp(0, x.shape[1]).sum())

    def bytes_per_call(self, x, mm):
        live = self.live_rows(x, mm)
        return live * self.k * 2 + live * (self.k // 128) * 4

    def alloc(self, P, xd, mm):
        import torch
        E, M, K = xd.shape
        g = torch.Generator(device="cpu").manual_seed(7)
        exps = torch.randint(-1, 2, (E, K // 128, M), generator=g).float()
        xs = torch.pow(2.0, exps).to(xd.device).permute(0, 2, 1)     # column-major [E, M, K/128]
        out = torch.empty_like(xd)
        self._scale = torch.tensor([2.0], dtype=torch.float32, device=xd.device)
        return out, xs

    def call(self, P, xd, out, xs, mm=None):
        P.requant_per_tensor(xd, xs, mm, self._scale, out, group_size=128)


def _sweep_index(T: int, H: int, dt: str) -> int:
    """The sweep case index whose seeded input the [T, H] shape of dtype dt uses (its G = 16,
    e4m3 case, as in large_sweep)."""
    from fp8_token_group_gb300 import synth
    return {(c[1], c[2], str(c[3])[6:], c[4], c[5]): c[0]
            for c in synth.sweep_cases()}[(T, H, dt, 16, "e4m3")]


def workloads():
    from fp8_token_group_gb300 import synth
    import torch
    return {
        "flat_outliers": Workload("flat_outliers", WORKLOAD, synth.flat_outliers, fmt=1, layout=1),
        "flat_small": Workload("flat_small", "flat bf16 x[64,4096] N(0,1), G=128, e4m3, fp32 "
                               "row-major scales [64,32]", synth.flat_small),
        "silu_flat": Workload("silu_flat", "fused silu*up, bf16 [8192, 2x2048] -> e4m3 "
                              "[8192,2048], G=128, fp32 column-major scales [16,8192]",
                              synth.silu_flat, silu=True, layout=1),
        "masked_silu": Workload("masked_silu", "masked EP-MoE bf16 [32,384,2x4096], masked_m "
                                "uniform in [0,384], fused silu, G=128, e4m3, UE8M0 packed "
                                "column-major", synth.masked_silu, silu=True, fmt=1, layout=1),
        "silu_flat_fp16": Workload("silu_flat_fp16", "fused silu*up, fp16 [8192, 2x2048] -> "
                                   "e4m3 [8192,2048], G=128, fp32 column-major scales",
                                   lambda: synth.silu_flat(dtype=torch.float16), silu=True,
                                   layout=1),
        "masked_silu_fp16": Workload("masked_silu_fp16", "masked EP-MoE fp16 [32,384,2x4096], "
                                     "masked_m uniform in [0,384], fused silu, G=128, e4m3, "
                                     "UE8M0 packed column-major",
                                     lambda: synth.masked_silu(dtype=torch.float16), silu=True,
                                     fmt=1, layout=1),
        "masked_decode": Workload("masked_decode", "masked EP-MoE decode: bf16 [32,384,2x4096] "
                                  "buffer, 1 live row per expert (masked_m = 1), fused silu, "
                                  "G=128, e4m3, UE8M0 packed column-major, no expected_m hint",
                                  synth.masked_decode, silu=True, fmt=1, layout=1),
        "masked_decode_hint": Workload("masked_decode_hint", "as masked_decode, with the "
                                       "expected_m = 1 hint", synth.masked_decode, silu=True,
                                       fmt=1, layout=1, expected_m=1),
        "sweep_big": Workload("sweep_big", "flat bf16 [32768,7168] N(0,1), G=128, e4m3, fp32 "
                              "row-major", lambda: synth.normal((32768, 7168), torch.bfloat16,
                                                                seed=1)),
        "flat_mid": Workload("flat_mid", "flat bf16 [4096,2048] (the shape sweep's input recipe), "
                             "G=128, e4m3, fp32 row-major: the sweep's smallest large shape",
                             lambda: synth.sweep_input(_sweep_index(4096, 2048, "bfloat16"), 4096,
                                                       2048, torch.bfloat16)),
        "per_token": PerTokenWorkload("per_token", "per-token FP8 quant, bf16 [4096,4096] "
                                      "N(0,1) -> e4m3 + fp32 scale per row", 4096, 4096),
        "requant": RequantWorkload("requant", "per-token-group -> per-tensor FP8 requant, e4m3 "
                                   "[8 experts, 1024, 3584], 128 live rows per expert (1024 "
                                   "live rows), column-major group scales", 8, 1024, 3584, 128),
    }


# ---------------------------------------------------------------- GPU timing

def nsets_for(per_set: int) -> int:
    """Buffer sets (each with its own input) that together exceed 2.5x the L2 size; a
    divisor of GRAPH_CALLS."""
    nsets = max(2, min(GRAPH_CALLS, -(-int(2.5 * L2_BYTES) // max(per_set, 1))))
    while GRAPH_CALLS % nsets:
        nsets += 1
    return nsets


def build_sets(P, wl, x_cpu, mm_cpu, device):
    """Enough buffer sets (each with its own input copy) that together they exceed L2 2.5x."""
    nsets = nsets_for(wl.bytes_per_call(x_cpu, mm_cpu))
    mm = None if mm_cpu is None else mm_cpu.to(device)
    if mm is not None and x_cpu.shape[1] > VIEW_SETS_PER_BUFFER and \
            nsets * x_cpu.numel() * 2 > 8 * 2 ** 30:
        return build_view_sets(P, wl, x_cpu, mm, device, nsets)
    sets = []
    for _ in range(nsets):
        xd = x_cpu.to(device)
        q, s = wl.alloc(P, xd, mm)
        sets.append((xd, q, s, mm))
    return sets


VIEW_SETS_PER_BUFFER = 200


def build_view_sets(P, wl, x_cpu, mm, device, nsets):
    """Masked sets with few live rows (decode): a full copy of the [E, tokens_pad, .] buffers
    per set would take hundreds of GB.  Instead set j of a buffer views it from row j on,
    so expert e's live rows of set j are rows e * tokens_pad + j + [0, masked_m[e]):
    distinct between sets while j + masked_m[e] <= tokens_pad, which holds for the
    decode counts this is used with.  The scale view is shifted by j words, which moves
    the written words of the column-major layout by j rows."""
    import torch
    E, tp, hin = x_cpu.shape
    H = hin // 2 if wl.silu else hin
    assert int(mm.max()) + VIEW_SETS_PER_BUFFER <= tp
    nbuf = -(-nsets // VIEW_SETS_PER_BUFFER)
    ns = P.scale_elems(E, tp, H, wl.group, wl.fmt, wl.layout, True)
    qdt = torch.int8 if wl.out == 1 else torch.float8_e4m3fn
    sdt = torch.int32 if wl.fmt == 1 else torch.float32
    flat = x_cpu.reshape(E * tp, hin)
    extra = VIEW_SETS_PER_BUFFER
    sets = []
    for b in range(nbuf):
        xb = torch.cat([flat.roll(b * 1009, 0), flat[:extra]]).to(device)
        qb = torch.empty(((E * tp + extra) * H,), dtype=qdt, device=device)
        sb = torch.empty((ns + extra,), dtype=sdt, device=device)
        for j in range(VIEW_SETS_PER_BUFFER):
            if len(sets) == nsets:
                break
            xd = xb[j:j + E * tp].view(E, tp, hin)
            q = qb[j * H:(j + E * tp) * H].view(E, tp, H)
            s = sb[j:j + ns]
            sets.append((xd, q, s, mm))
    return sets


def graph_plan(calls: int, nsets: int, cap: int = GRAPH_CALLS):
    """How `calls` consecutive calls are replayed: (g, reps, r) with calls = r + reps * g.
    The main graph holds g calls, a multiple of nsets (set i % nsets for call i), so it
    starts at set 0 and ends at set nsets - 1; the remainder graph of r calls runs first
    and uses sets (nsets - r + i) % nsets, so it also ends at set nsets - 1.  Consecutive
    calls therefore always read different buffer sets."""
    g = min(calls, cap) // nsets * nsets
    if g == 0:
        return 0, 0, calls
    return g, calls // g, calls % g


class GraphRunner:
    """CUDA graphs of calls over rotating buffer sets, captured on demand by size."""

    def __init__(self, P, wl, sets, stream):
        self.P, self.wl, self.sets, self.stream = P, wl, sets, stream
        self.graphs = {}

    def _graph(self, n: int, first_set: int):
        import torch
        key = (n, first_set)
        if key not in self.graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                for i in range(n):
                    self.wl.call(self.P, *self.sets[(first_set + i) % len(self.sets)])
            self.graphs[key] = g
        return self.graphs[key]

    def enqueue(self, calls: int):
        """Enqueue exactly `calls` calls on the runner's stream."""
        nsets = len(self.sets)
        g, reps, r = graph_plan(calls, nsets)
        if r:
            self._graph(r, (nsets - r) % nsets).replay()
        for _ in range(reps):
            self._graph(g, 0).replay()

    def prepare(self, calls: int):
        nsets = len(self.sets)
        g, reps, r = graph_plan(calls, nsets)
        if r:
            self._graph(r, (nsets - r) % nsets)
        if reps:
            self._graph(g, 0)


def flush_l2(device):
    """Overwrite a buffer twice the L2 size so the next region starts with a cold cache."""
    import torch
    buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    buf.fill_(1)
    del buf


def time_graph(P, wl, sets, steps: int, warmup: int, world: int, sampler=None,
               repeats: int = REPEATS):
    """`warmup` untimed calls, then `repeats` timed regions of exactly `steps` calls each
    (CUDA graphs over rotating buffer sets), each region bracketed by an L2 flush, a
    barrier and a synchronize, timed with CUDA events on the launching stream.  Returns the
    per-region elapsed seconds (max over ranks) and the clock record."""
    import torch
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for i in range(min(8, len(sets))):
            wl.call(P, *sets[i])
    torch.cuda.synchronize()
    runner = GraphRunner(P, wl, sets, stream)
    runner.prepare(steps)
    runner.prepare(warmup)
    with torch.cuda.stream(stream):
        runner.enqueue(warmup)
    torch.cuda.synchronize()
    device = torch.cuda.current_device()
    if sampler:
        sampler.start()
    regions = []
    for _ in range(repeats):
        flush_l2(device)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            # keep the GPU busy while the host enqueues the region, so the first call
            # follows the start event without a launch gap
            if hasattr(torch.cuda, "_sleep"):
                torch.cuda._sleep(200_000)
            start.record(stream)
            runner.enqueue(steps)
            end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        regions.append(reduce_max(start.elapsed_time(end) / 1e3, world,
                                  torch.device("cuda", device)))
    clocks = sampler.stop() if sampler else None
    runner.graphs.clear()
    return regions, clocks


def time_e2e(P, wl, x_cpu, mm_cpu, steps: int, device):
    """Public API with host buffers.  Every step copies its input from pinned host memory to
    the device, quantizes it, and copies codes and scales back to pinned host memory.
    Steps are double-buffered on three streams (H2D, compute, D2H) so the copy of step i+1
    overlaps the quantization and read-back of step i."""
    import torch
    xh = x_cpu.pin_memory()
    mm = None if mm_cpu is None else mm_cpu.to(device)
    bufs = []
    for _ in range(2):
        xd = torch.empty_like(xh, device=device)
        q, s = wl.alloc(P, xd, mm)
        qh = torch.empty(q.shape, dtype=q.dtype).pin_memory()
        sh = torch.empty(s.shape, dtype=s.dtype).pin_memory()
        bufs.append((xd, q, s, qh, sh))
    h2d, comp, d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    copied = [ev(), ev()]     # input of buffer b is on the device
    quantized = [ev(), ev()]  # outputs of buffer b are ready
    returned = [ev(), ev()]   # outputs of buffer b are back on the host
    consumed = [ev(), ev()]   # buffer b's input was consumed by its quantization
    for e in returned + consumed:
        e.record(torch.cuda.current_stream())

    def step(i):
        b = i % 2
        xd, q, s, qh, sh = bufs[b]
        h2d.wait_event(consumed[b])
        with torch.cuda.stream(h2d):
            xd.copy_(xh, non_blocking=True)
            copied[b].record(h2d)
        comp.wait_event(copied[b])
        comp.wait_event(returned[b])
        with torch.cuda.stream(comp):
            wl.call(P, xd, q, s, mm)
            consumed[b].record(comp)
            quantized[b].record(comp)
        d2h.wait_event(quantized[b])
        with torch.cuda.stream(d2h):
            qh.copy_(q, non_blocking=True)
            sh.copy_(s, non_blocking=True)
            returned[b].record(d2h)

    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        step(i)
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    h2d_b = xh.numel() * xh.element_size()
    qh, sh = bufs[0][3], bufs[0][4]
    d2h_b = qh.numel() * qh.element_size() + sh.numel() * sh.element_size()
    return el, h2d_b, d2h_b


def time_e2e_zero_copy(P, wl, x_cpu, mm_cpu, steps: int, device):
    """Public API with host buffers used in place: x, codes and scales live in pinned host
    memory, which the GPU reads and writes directly over the host link (unified
    addressing).  Every step moves its input from the host and its results back to the host
    inside the quantization call itself.  Two buffer sets alternate."""
    import torch
    mm = None if mm_cpu is None else mm_cpu.to(device)
    sets = []
    for _ in range(2):
        xh = x_cpu.pin_memory()
        qd, sd = wl.alloc(P, torch.empty(x_cpu.shape, dtype=x_cpu.dtype, device=device), mm)
        qh = torch.empty(qd.shape, dtype=qd.dtype).pin_memory()
        sh = torch.empty(sd.shape, dtype=sd.dtype).pin_memory()
        del qd, sd
        sets.append((xh, qh, sh))
    for i in range(4):
        wl.call(P, sets[i % 2][0], sets[i % 2][1], sets[i % 2][2], mm)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        wl.call(P, sets[i % 2][0], sets[i % 2][1], sets[i % 2][2], mm)
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    xh, qh, sh = sets[0]
    return el, xh.numel() * xh.element_size(), qh.numel() * qh.element_size() + sh.numel() * sh.element_size()


def measure_device(P, wl, device, steps: int, inputs=None, repeats: int = 3) -> dict:
    """One workload timed like the benchmark line (median of `repeats` regions)."""
    import torch
    x, mm = inputs if inputs is not None else wl.inputs()
    sets = build_sets(P, wl, x, mm, device)
    regions, _ = time_graph(P, wl, sets, steps, 100, 1, repeats=repeats)
    nb = wl.bytes_per_call(x, mm)
    us = statistics.median(regions) / steps * 1e6
    del sets
    torch.cuda.empty_cache()
    peak, _ = measured_peak()
    return {"desc": wl.desc, "us_per_call": round(us, 3), "bytes_per_call": nb,
            "gbs": round(nb / us / 1e3, 1), "pct_of_peak": round(100 * nb / us / 1e3 / peak, 1),
            "live_rows": wl.live_rows(x, mm)}


class CopyWorkload(Workload):
    """A streaming elementwise kernel from torch (bitwise_not over int32 words) that reads
    half a call's algorithmic bytes and writes the other half, so it moves the same total:
    the memory system's floor for one launch moving that much, as a reference point beside
    the quantizer.  (A captured copy_ is not used: inside a CUDA graph a device-to-device
    memcpy can run on a copy engine at a fraction of HBM bandwidth.)"""

    def __init__(self, nbytes: int):
        super().__init__("copy_reference", f"torch bitwise_not of {nbytes // 2 // 16 * 16} bytes "
                         f"into another buffer (reads + writes {nbytes // 32 * 32} bytes)", None)
        self.nbytes = nbytes

    def inputs(self):
        import torch
        return torch.zeros(self.nbytes // 2 // 16 * 16, dtype=torch.uint8), None

    def live_rows(self, x, mm):
        return 0

    def bytes_per_call(self, x, mm):
        return 2 * x.numel()

    def alloc(self, P, xd, mm):
        import torch
        return torch.empty_like(xd), None

    def call(self, P, xd, q, s, mm=None):
        import torch
        torch.bitwise_not(xd.view(torch.int32), out=q.view(torch.int32))


# The large-token shapes of the sweep timed in the benchmark line: T in {4096, 32768} x H in
# {2048, 4096, 7168} x G in {16, 128}, bf16 -> e4m3, plus one fp16 and one int8 shape per T;
# fp32 row-major scales.
LARGE_SWEEP = ([(T, H, "bfloat16", G, "e4m3") for T in (4096, 32768) for H in (2048, 4096, 7168)
                for G in (16, 128)] +
               [(T, 4096, "float16", 64, "e4m3") for T in (4096, 32768)] +
               [(T, 2048, "bfloat16", 32, "int8") for T in (4096, 32768)])


def large_sweep(P, device, steps: int, copy_reference: bool = True):
    """The LARGE_SWEEP shapes (inputs of the sweep's recipe, drawn with the seed of the
    shape's G = 16, e4m3 case and shared by its group sizes), each with the quantizer's time
    and, for T = 4096, a copy of equal traffic as the floor reference."""
    import torch
    from fp8_token_group_gb300 import synth
    peak, _ = measured_peak()
    index = {(T, H, str(dt)[6:], G, out): i for i, T, H, dt, G, out in synth.sweep_cases()}
    rows, inputs = [], {}
    for T, H, dt, G, out in LARGE_SWEEP:
        key = (T, H, dt)
        if key not in inputs:
            inputs.clear()
            inputs[key] = synth.sweep_input(index[(T, H, dt, 16, "e4m3")], T, H,
                                            getattr(torch, dt))
        x = inputs[key]
        name = f"{T}x{H}-{dt}-G{G}-{out}"
        wl = Workload(name, name, None, group=G, out=0 if out == "e4m3" else 1)
        r = measure_device(P, wl, device, steps, inputs=(x, None))
        line = {"tokens": T, "hidden": H, "dtype": dt, "group": G, "out": out,
                "us_per_call": r["us_per_call"], "gbs": r["gbs"], "pct_of_peak": r["pct_of_peak"]}
        if copy_reference and T == 4096:
            c = measure_device(P, CopyWorkload(r["bytes_per_call"]), device, steps)
            line["copy_reference"] = {"us_per_call": c["us_per_call"], "gbs": c["gbs"],
                                      "pct_of_peak": c["pct_of_peak"]}
        rows.append(line)
    pcts = [r["pct_of_peak"] for r in rows]
    summary = {"configs": len(rows), "min_pct": min(pcts), "median_pct": statistics.median(pcts),
               "at_or_above_75_pct": sum(p >= 75 for p in pcts),
               "peak_gbs": peak, "timing": f"median of 3 regions of {steps} calls each"}
    return rows, summary


def bench_config(wl, x, mm, world: int) -> dict:
    """The `config` object of the JSON line (shared by both arms)."""
    bpc = wl.bytes_per_call(x, mm)
    nsets = nsets_for(bpc)
    return {"workload": wl.desc, "global_batch": wl.live_rows(x, mm) * world,
            "group_size": wl.group, "input": "bf16", "output": "e4m3",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": f"{nsets} rotating buffer sets, each with its own input, together "
                  f"{nsets * bpc / 1e6:.0f} MB > 2.5x the 129 MB L2; L2 flushed before "
                  f"each timed region",
            "timing": f"median of {REPEATS} timed regions of exactly `steps` calls, CUDA "
                      f"graphs of up to {GRAPH_CALLS} calls, CUDA events on the launching "
                      f"stream"}


def run_ours(args, world, rank, local):
    import torch
    import fp8_token_group_gb300 as P

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    P.lib()
    wls = workloads()
    wl = wls[args.workload]
    x, mm = wl.inputs()
    sets = build_sets(P, wl, x, mm, device)
    sampler = ClockSampler(local) if rank == 0 else None
    regions, clocks = time_graph(P, wl, sets, args.steps, args.warmup, world, sampler)
    del sets
    torch.cuda.empty_cache()
    steps = args.steps
    el = statistics.median(regions)               # max over ranks, median over regions
    bpc = wl.bytes_per_call(x, mm)
    value = aggregate(bpc, steps, world, el)
    us = el / steps * 1e6
    peak, peak_kind = measured_peak()
    achieved = bpc / (el / steps) / 1e9

    e2e_steps = max(3, min(args.steps, 50))
    copy_el, h2d, d2h = time_e2e(P, wl, x, mm, e2e_steps, device)
    copy_el = reduce_max(copy_el, world, device)
    zc_el = None
    if type(wl) is Workload:
        zc_el, _, _ = time_e2e_zero_copy(P, wl, x, mm, e2e_steps, device)
        zc_el = reduce_max(zc_el, world, device)
    e2e_mode = "zero-copy" if zc_el is not None and zc_el < copy_el else "copies"
    e2e_el = zc_el if e2e_mode == "zero-copy" else copy_el
    e2e_gbs = lambda t: None if t is None else round(world * e2e_steps * bpc / t / 1e9, 2)
    others, sweep_rows, sweep_summary, copy_ref = {}, None, None, None
    if rank == 0 and not args.no_extra:
        c = measure_device(P, CopyWorkload(bpc), device, 4000)
        copy_ref = {"us_per_call": c["us_per_call"], "gbs": c["gbs"],
                    "pct_of_peak": c["pct_of_peak"], "desc": c["desc"]}
        for name, other in wls.items():
            if name != wl.name:
                r = measure_device(P, other, device, 4000)
                c = measure_device(P, CopyWorkload(r["bytes_per_call"]), device, 4000)
                r["copy_reference"] = {"us_per_call": c["us_per_call"], "gbs": c["gbs"],
                                       "pct_of_peak": c["pct_of_peak"]}
                others[name] = r
        sweep_rows, sweep_summary = large_sweep(P, device, 2000)
    base = cpu_baseline(x) if (rank == 0 and world == 1 and not args.no_cpu
                               and wl.name == "flat_outliers") else None
    live = wl.live_rows(x, mm)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": round(el / steps * 1e3, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": bench_config(wl, x, mm, world),
            "us_per_call": round(us, 3),
            "tokens_per_s": round(world * live * steps / el, 1),
            "pct_of_peak": round(100 * achieved / peak, 2),
            "regions_ms": [round(r * 1e3, 5) for r in regions],
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                         if peak_kind == "measured" else "fallback 6.8 TB/s",
                         "traffic": recorded_traffic(wl.name),
                         "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum "
                                           "per launch, mean over back-to-back launches "
                                           "(profiles/traffic.json), when taken on the "
                                           "current kernel sources",
                         "algorithmic_bytes_per_launch": bpc},
            "clocks": clocks,
            "gpu_launches": steps,
            "e2e": {"value": e2e_gbs(e2e_el), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "mode": e2e_mode, "copies_gbs": e2e_gbs(copy_el),
                    "zero_copy_gbs": e2e_gbs(zc_el),
                    "path": ("per step: fp8_token_group_gb300.quant on pinned host x, codes "
                             "and scales, read and written by the GPU over the host link "
                             "(zero-copy), wall clock over all steps")
                    if e2e_mode == "zero-copy" else
                    ("per step: pinned host x -> device, fp8_token_group_gb300.quant, codes "
                     "and scales -> pinned host; double-buffered on H2D/compute/D2H streams, "
                     "wall clock over all steps")},
            "cpu_baseline": base,
            "copy_reference": copy_ref,
            "other_workloads": others,
            "large_sweep": sweep_rows,
            "large_sweep_summary": sweep_summary,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_sweep(args, out_path=None):
    """Every configuration of the shape sweep (T in {1, 7, 64, 333, 4096, 32768} x H in
    {128, 2048, 4096, 7168} x {fp16, bf16} x G in {16, 32, 64, 128} x {e4m3, int8}, fp32
    row-major scales), each timed like the other workloads (graph replay, rotating buffer
    sets beyond L2).  Prints one JSON line per configuration and a summary line; the large
    configurations (T >= 4096 and H >= 2048) are the ones held to the HBM roofline."""
    import torch
    import fp8_token_group_gb300 as P
    from fp8_token_group_gb300 import synth
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    P.lib()
    peak, peak_kind = measured_peak()
    rows, large = [], []
    for idx, T, H, dt, G, out in synth.sweep_cases():
        if args.sweep_min_tokens and T < args.sweep_min_tokens:
            continue
        x = synth.sweep_input(idx, T, H, dt)
        name = f"{T}x{H}-{str(dt)[6:]}-G{G}-{out}"
        wl = Workload(name, name, None, group=G, out=0 if out == "e4m3" else 1)
        r = measure_device(P, wl, device, args.sweep_steps, inputs=(x, None))
        pct = r["pct_of_peak"]
        line = {"sweep": idx, "tokens": T, "hidden": H, "dtype": str(dt)[6:], "group": G,
                "out": out, "us_per_call": r["us_per_call"], "gbs": r["gbs"],
                "pct_of_peak": pct}
        print(json.dumps(line), flush=True)
        rows.append(line)
        if T >= 4096 and H >= 2048:
            large.append(pct)
    summary = {"sweep_summary": {"configs": len(rows), "peak_gbs": peak, "peak_source": peak_kind,
                                 "large_configs": len(large),
                                 "large_min_pct": min(large) if large else None,
                                 "large_median_pct": statistics.median(large) if large else None}}
    print(json.dumps(summary), flush=True)
    if out_path:
        with open(out_path, "w") as f:
            for line in rows:
                f.write(json.dumps(line) + "\n")
            f.write(json.dumps(summary) + "\n")
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="flat_outliers",
                    choices=["flat_outliers", "flat_small", "silu_flat", "masked_silu",
                             "silu_flat_fp16", "masked_silu_fp16", "masked_decode",
                             "masked_decode_hint", "sweep_big", "flat_mid", "per_token", "requant"],
                    help="workload of the JSON line (default: the "
                    "benchmarked flat_outliers)")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--sweep", action="store_true", help="time every shape-sweep configuration "
                    "(one JSON line each, then a summary) instead of the benchmark line")
    ap.add_argument("--sweep-steps", type=int, default=2000)
    ap.add_argument("--sweep-min-tokens", type=int, default=0)
    ap.add_argument("--sweep-out", default=None, help="also write the sweep lines to this file")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.sweep:
        return run_sweep(args, args.sweep_out)
    if args.impl == "reference":
        # the CPU oracle: rank 0 alone runs it, other ranks exit without work
        return run_reference(args, int(os.environ.get("WORLD_SIZE", str(args.gpus))),
                             int(os.environ.get("RANK", "0")))
    world, rank, local = dist_setup(args.gpus)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
