"""Benchmark of the partial MXFP8 cast hot path on GB300.

Workload: 16384x6144 FP32 master weight (per-row scale 10^U(-4,1) times
N(0, 0.02), seed 0), one full fragment, bidirectional MXFP8 (E4M3 data, E8M0
32-value block scales), model dtype BF16.  One step = one pass of the whole hot
path through the public API: partial amax into the packed amax slot -> packed
MAX reduction over the slots (one slot: one rank) fused with the scale update ->
partial cast (three kernels).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  `value` is whole-job HBM throughput in GB/s of
algorithmic bytes (every kernel's compulsory reads and writes) over exactly K timed
steps with the input resident in device memory (no events inside them).  `kernels`
gives each kernel's device time per call -- the median of 256 in-step samples taken
with CUDA events around every phase of a sampling region after the timed steps --
with its GB/s and fraction of the measured HBM peak, both from that median;
`roofline` the dominant kernel against that peak (with the ncu DRAM traffic recorded
for the current kernel code under profiles/).  `clocks` comes from nvidia-smi samples
over at least a second of continuous load around the timed region.  `e2e` runs the
same four-step flow on pinned host buffers (copy-in, per-chunk partial amax, MAX
reduction + scales, per-chunk partial cast storing into the pinned outputs, all inside its
timed region; its staged-copy form beside it);
`e2e_one_pass` the one-pass kernel reading and writing the pinned host buffers directly
(its staged-copy pipeline beside it), over its own bytes; both give per-step spreads and
the flow its measured copy-engine bound.  Outside the timed
steps: `fused_whole_blocks` (the one-pass kernel on the same weight), `sharded_batch`
(the multi-fragment driver on the config-5 batch in four emulated shards, with its
phases) and `other_configs` (configs 1-3, and the headline weight bidirectional and row-only,
each kernel alone in CUDA graphs of repeated calls, median of 7 rounds: the pages' method).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload (the reference arm of this benchmark).
N > 1 (torchrun): every rank runs its own replica of the workload on its GPU.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

ROWS, COLS = 16384, 6144
METRIC = "MXFP8 partial amax+cast µs/call and HBM GB/s (% of GB300 roofline), 1 GPU"
WORKLOAD = ("16384x6144 FP32 master (per-row scale 10^U(-4,1) x N(0,0.02), seed 0), full fragment, "
            "bidirectional MXFP8 E4M3 / E8M0 32-value blocks, model dtype BF16")
PAGES_GB200_US = {"amax": 110.395, "cast": 210.154}  # context only: other hardware
# The pages' whole table ("Support row-only MXFP8 distributed master-weight casts", section
# "Bidirectional kernel performance": GB200, full input, both directions, median µs per
# call over graph replays): (rows, cols, input dtype) -> (amax µs, cast µs).  Context only.
PAGES_GB200_TABLE = {
    (160, 96, "bf16"): (3.278, 7.578), (1024, 1024, "bf16"): (3.690, 7.894),
    (4096, 4096, "bf16"): (20.099, 24.784), (16384, 6144, "bf16"): (113.376, 202.658),
    (160, 96, "f32"): (2.953, 7.378), (1024, 1024, "f32"): (3.362, 7.870),
    (4096, 4096, "f32"): (19.556, 35.254), (16384, 6144, "f32"): (110.395, 210.154),
}
FALLBACK_HBM_GBS = 6800.0


def algorithmic_bytes(n: int, s_in: int = 4, colwise: bool = True) -> dict:
    """Compulsory HBM bytes per call of each kernel for an n-element fragment (one slot)."""
    dirs = 2 if colwise else 1
    blocks = dirs * n // 32            # amax / scale entries
    return {
        "amax": n * s_in + blocks * s_in,                 # read x, write amax
        "reduce": 2 * blocks * s_in,                      # read 1 slot, write reduced
        "scales": blocks * s_in + blocks,                 # read amax, write E8M0 bytes
        "reduce_scales": 2 * blocks * s_in + blocks,      # read 1 slot, write reduced + E8M0
        "cast": n * s_in + blocks + dirs * n,             # read x and scales, write E4M3
    }


def sharded_phase_bytes(specs, num_slots: int, packed_entries: int, s_in: int = 4,
                        slot_entries_read: int | None = None) -> dict:
    """Compulsory HBM bytes of one multi-fragment driver step by phase: every fragment's
    input and block maxima (amax); the slot entries the reduction reads and the reduced
    amax + E8M0 bytes it writes (reduce_scales); every fragment's input, scales and E4M3
    outputs (cast).  The reduction reads every slot in full (num_slots * packed_entries
    entries) unless `slot_entries_read` gives the entries the slots hold (the ranged
    reduction reads a slot only where its shard's amax wrote)."""
    amax = cast = 0
    for sp in specs:
        n = sp.rows * sp.cols
        dirs = 2 if sp.colwise else 1
        blocks = dirs * n // 32
        amax += n * s_in + blocks * s_in
        cast += n * s_in + blocks + dirs * n
    reads = num_slots * packed_entries if slot_entries_read is None else slot_entries_read
    red = reads * s_in + packed_entries * s_in + packed_entries
    return {"amax": amax, "reduce_scales": red, "cast": cast}


def sharded_step_bytes(specs, num_slots: int, packed_entries: int, s_in: int = 4,
                       slot_entries_read: int | None = None) -> int:
    """Total of sharded_phase_bytes."""
    return sum(sharded_phase_bytes(specs, num_slots, packed_entries, s_in, slot_entries_read).values())


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def read_traffic(kernel: str):
    """ncu DRAM bytes per launch recorded under profiles/, or None unless the record was
    taken with the current kernel sources (digest of the device code only: host-side
    edits of the C ABI do not invalidate it)."""
    path = os.path.join(ROOT, "profiles", "traffic_16384x6144_f32.txt")
    if not os.path.exists(path):
        return None
    from mxfp8_master_weight_gb300 import build as libbuild
    digest = libbuild.kernel_digest()
    for line in open(path):
        parts = dict(p.split("=", 1) for p in line.split() if "=" in p)
        if parts.get("kernel") == kernel and parts.get("kernel_sources_sha256") == digest:
            return int(parts["dram_bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples (every 100 ms) taken while the GPU is under the
    bench's load: the sampler runs across a load window of steps before the timed region,
    the timed region itself and a load window after it."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._reader = None

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self

        def read():
            for line in self.proc.stdout:
                self.lines.append(line)

        self._reader = threading.Thread(target=read, daemon=True)
        self._reader.start()
        return self

    def wait_started(self, timeout_s: float = 5.0) -> bool:
        """Wait until the sampler has produced its first line (nvidia-smi takes a moment
        to start); False when it never does."""
        t0 = time.perf_counter()
        while self.proc is not None and not self.lines and time.perf_counter() - t0 < timeout_s:
            time.sleep(0.02)
        return bool(self.lines)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
            if self._reader is not None:
                self._reader.join(timeout=5)
        self.out = "".join(self.lines)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in (getattr(self, "out", None) or "".join(self.lines)).splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus: int):
    import torch
    if n_gpus <= 1 or "RANK" not in os.environ:
        return 0, 1, 0
    import torch.distributed as dist
    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    dist.init_process_group("nccl")
    return dist.get_rank(), dist.get_world_size(), local


def aggregate_over_ranks(elapsed_s: float, units: float, world: int, device=None):
    """(max elapsed over ranks, sum of units over ranks) via torch.distributed."""
    if world <= 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":", 1)[0].strip().lower() == "model name":
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.split(":", 1)[0].strip().lower() in ("model name", "cpu model"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_sample_run(data: np.ndarray, row0: int, rows: int):
    """Time the CPU oracle (as it stands, one thread) on rows [row0, row0+rows) of the
    workload (whole 32-row bands, so every block is complete): amax -> scales -> cast.
    Returns (seconds, algorithmic bytes)."""
    import oracle
    x = np.ascontiguousarray(data[row0 * COLS:(row0 + rows) * COLS])
    t0 = time.perf_counter()
    oracle.full_cast(x, rows, COLS, True)
    dt = time.perf_counter() - t0
    b = algorithmic_bytes(rows * COLS)
    return dt, b["amax"] + b["scales"] + b["cast"]


def _band_worker(args):
    """Worker process: the unchanged oracle on rows [row0, row0 + rows) of the sample
    file (memory-mapped); returns its seconds and algorithmic bytes."""
    path, row0, rows, cols = args
    import oracle
    oracle.build()
    data = np.load(path, mmap_mode="r")
    x = np.ascontiguousarray(data[row0 * cols:(row0 + rows) * cols])
    t0 = time.perf_counter()
    oracle.full_cast(x, rows, cols, True)
    dt = time.perf_counter() - t0
    b = algorithmic_bytes(rows * cols)
    return dt, b["amax"] + b["scales"] + b["cast"]


def cpu_all_cores_run(data: np.ndarray, rows: int, procs: int):
    """The oracle as it stands, run on every host core at once: the sample's 32-row bands
    are split over `procs` worker processes (started with spawn, so they are safe after
    CUDA use), each running the single-threaded oracle on its bands.  Returns (wall
    seconds of the parallel run, algorithmic bytes, processes used)."""
    import multiprocessing as mp
    import tempfile

    bands = rows // 32
    procs = max(1, min(procs, bands))
    per = [bands // procs + (1 if k < bands % procs else 0) for k in range(procs)]
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "sample.npy")
        np.save(path, np.ascontiguousarray(data[:rows * COLS]))
        tasks, row0 = [], 0
        for nb in per:
            tasks.append((path, row0, nb * 32, COLS))
            row0 += nb * 32
        ctx = mp.get_context("spawn")
        with ctx.Pool(procs) as pool:
            pool.map(_band_worker, [(path, 0, 32, COLS)] * procs)  # start and build first
            t0 = time.perf_counter()
            res = pool.map(_band_worker, tasks)
            wall = time.perf_counter() - t0
    return wall, sum(b for _, b in res), procs


def run_reference(args):
    rank = int(os.environ.get("RANK", 0))
    if rank != 0:
        return  # the CPU reference arm runs on rank 0 only
    import oracle
    from mxfp8_master_weight_gb300 import workloads as wl
    oracle.build()
    data = wl.cfg4_headline(rows=ROWS, cols=COLS).data
    rows = 32  # one 32-row band per step: the whole run stays within a few minutes
    bands = ROWS // rows
    for k in range(args.warmup):
        cpu_sample_run(data, (k % bands) * rows, rows)
    tot_t, tot_b = 0.0, 0
    for k in range(args.steps):
        dt, b = cpu_sample_run(data, (k % bands) * rows, rows)
        tot_t += dt
        tot_b += b
    gbs = tot_b / tot_t / 1e9
    sample = (f"one {rows}-row band ({rows * COLS} elements) of the workload per step, bands in "
              f"order: amax, scales, cast")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_t / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample_rows_per_step": rows},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


def graph_us_per_call(call, stream, elems: int, rounds: int = 7, replays: int = 20) -> float:
    """Median over `rounds` of the µs per call of a CUDA graph holding G calls (G = 50 for
    fragments of at most 4M elements, else 10), replayed `replays` times per round."""
    import torch

    g_calls = 50 if elems <= 4 * 2 ** 20 else 10
    side = torch.cuda.Stream(stream.device)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for _ in range(3):
            call.call(side)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for _ in range(g_calls):
            call.call(side)
    graph.replay()
    torch.cuda.synchronize()
    per_round = []
    for _ in range(rounds):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(replays):
            graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        per_round.append(a.elapsed_time(b) * 1e3 / (replays * g_calls))
    return statistics.median(per_round)


def measure_configs(x_headline, dev) -> dict:
    """amax and cast µs per call, each kernel alone, on configs 1-3 and on the headline weight
    (bidirectional and row-only), the pages' timing method: graphs of repeated calls, 7
    rounds, median.  Configs 1-3 fit in L2 (126 MB), so their figures are L2-warm, not HBM
    measurements; the headline weight's are HBM figures, with GB/s and peak fraction."""
    import torch

    from mxfp8_master_weight_gb300 import api
    from mxfp8_master_weight_gb300 import workloads as wl

    stream = torch.cuda.current_stream(dev)
    w1, w2, w3 = wl.cfg1_tiny(), wl.cfg2_bf16_outliers(), wl.cfg3_square()
    cases = [  # name, weight shape, flat device data, fragment start/length, colwise, memory
        ("cfg1 160x96 FP32 full bidirectional", w1, 0, w1.numel, True, "L2-warm"),
        ("cfg2 1024x1024 BF16 [17, +262144) bidirectional", w2, 17, w2.numel // 4, True, "L2-warm"),
        ("cfg2 1024x1024 BF16 [17, +262144) row-only", w2, 17, w2.numel // 4, False, "L2-warm"),
        ("cfg3 4096x4096 FP32 full bidirectional", w3, 0, w3.numel, True, "L2-warm"),
        ("cfg3 4096x4096 FP32 [17, +n/4) bidirectional", w3, 17, w3.numel // 4, True, "L2-warm"),
        ("cfg4 16384x6144 FP32 full bidirectional", None, 0, ROWS * COLS, True, "HBM"),
        ("cfg4 16384x6144 FP32 full row-only", None, 0, ROWS * COLS, False, "HBM"),
    ]
    peak, peak_kind = measured_peak()
    out = {}
    for name, w, start, length, colwise, mem in cases:
        if w is None:
            rows, cols, flat = ROWS, COLS, x_headline
        else:
            rows, cols = w.rows, w.cols
            if w.data.dtype == np.uint16:
                flat = torch.from_numpy(w.data.view(np.int16)).to(dev).view(torch.bfloat16)
            else:
                flat = torch.from_numpy(w.data).to(dev)
        frag = flat[start:start + length]
        (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
        ar = torch.zeros((rr, rc), dtype=frag.dtype, device=dev)
        ac = torch.zeros((cr, cc), dtype=frag.dtype, device=dev) if colwise else None
        sr = torch.empty((rr, rc), dtype=torch.uint8, device=dev)
        scl = torch.empty((cr, cc), dtype=torch.uint8, device=dev) if colwise else None
        qr = torch.empty(rows * cols, dtype=torch.uint8, device=dev)
        qc = torch.empty(rows * cols, dtype=torch.uint8, device=dev) if colwise else None
        amax = api.prepare_partial_amax(frag, ar, ac, rows, cols, start)
        amax.call(stream)
        api.mxfp8_update_scales(ar, ac, sr, scl, rows, cols)
        cast = api.prepare_partial_cast(frag, sr, scl, qr, qc, rows, cols, start)
        rec = {"amax_us": round(graph_us_per_call(amax, stream, length), 3),
               "cast_us": round(graph_us_per_call(cast, stream, length), 3), "memory": mem}
        if mem == "HBM":  # larger than L2: HBM figures against the measured peak
            ab = algorithmic_bytes(length, frag.element_size(), colwise)
            for k in ("amax", "cast"):
                gbs = ab[k] / (rec[k + "_us"] * 1e-6) / 1e9
                rec[k + "_gbs"] = round(gbs, 1)
                rec[k + "_frac_of_" + peak_kind + "_peak"] = round(gbs / peak, 4)
        out[name] = rec
    return out


def measure_pages_table(dev) -> dict:
    """Every case of the pages' kernel table on this GPU, by the pages' method (each kernel
    alone, full input, both directions, graph replays, median of 7 rounds): amax and cast
    µs per call beside the pages' GB200 figures.  Inputs: N(0, 0.02) draws (seed 0) of the
    shape, rounded to BF16 for the BF16 rows."""
    import torch

    from mxfp8_master_weight_gb300 import api
    from mxfp8_master_weight_gb300 import workloads as wl

    stream = torch.cuda.current_stream(dev)
    out = {}
    for (rows, cols, dt), (p_amax, p_cast) in PAGES_GB200_TABLE.items():
        n = rows * cols
        x = torch.from_numpy(wl.normal_f32(np.random.default_rng(0), n)).to(dev)
        if dt == "bf16":
            x = x.to(torch.bfloat16)
        (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
        ar = torch.zeros((rr, rc), dtype=x.dtype, device=dev)
        ac = torch.zeros((cr, cc), dtype=x.dtype, device=dev)
        sr = torch.empty((rr, rc), dtype=torch.uint8, device=dev)
        scl = torch.empty((cr, cc), dtype=torch.uint8, device=dev)
        qr = torch.empty(n, dtype=torch.uint8, device=dev)
        qc = torch.empty(n, dtype=torch.uint8, device=dev)
        amax = api.prepare_partial_amax(x, ar, ac, rows, cols, 0)
        amax.call(stream)
        api.mxfp8_update_scales(ar, ac, sr, scl, rows, cols)
        cast = api.prepare_partial_cast(x, sr, scl, qr, qc, rows, cols, 0)
        a_us = graph_us_per_call(amax, stream, n)
        c_us = graph_us_per_call(cast, stream, n)
        out[f"{rows}x{cols} {dt.upper()}"] = {
            "amax_us": round(a_us, 3), "cast_us": round(c_us, 3),
            "pages_gb200_amax_us": p_amax, "pages_gb200_cast_us": p_cast,
            "pages_over_ours_amax": round(p_amax / a_us, 2), "pages_over_ours_cast": round(p_cast / c_us, 2)}
        del x, ar, ac, sr, scl, qr, qc, amax, cast
    return out


def sample_phases(step, n: int, nphases: int = 3):
    """Per-phase device time of `n` steps, each bracketed by CUDA events on the launching
    stream (events around every phase; recorded only in this sampling region, so the
    timed steps run without them).  Returns a list per phase of n durations in µs."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n)]
    for e in evs:
        step(events=e)
    torch.cuda.synchronize()
    bounds = ((0, 1), (1, 3), (3, 4))[:nphases]
    return [[e[a].elapsed_time(e[b]) * 1e3 for e in evs] for a, b in bounds]


def marginal_costs(phases, stream, n: int = 200, rounds: int = 3) -> dict:
    """What each phase adds to a step of back-to-back steps: the µs per step of the whole
    step minus that of the step without the phase (the library calls of the other phases,
    in order, n times; median of `rounds` rounds each).  A short kernel bracketed by events
    also pays its launch and loses its programmatic overlap with the kernel before; this
    figure does not."""
    import torch

    def loop(keep):
        calls = [c for k, cs in enumerate(phases) if k in keep for c in cs]
        for _ in range(5):
            for c in calls:
                c.call(stream)
        torch.cuda.synchronize()
        per = []
        for _ in range(rounds):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(n):
                for c in calls:
                    c.call(stream)
            b.record(stream)
            torch.cuda.synchronize()
            per.append(a.elapsed_time(b) * 1e3 / n)
        return statistics.median(per)

    present = [k for k, cs in enumerate(phases) if cs]
    full = loop(set(present))
    return {k: full - loop(set(present) - {k}) for k in present}, full


def run_for(step, seconds: float, stream) -> int:
    """Run steps back to back for about `seconds` of device time (the clock sampler's
    load window); returns the number of steps run."""
    import torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(20):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    per = max(a.elapsed_time(b) / 20 / 1e3, 1e-6)
    k = max(1, int(seconds / per))
    for _ in range(k):
        step()
    torch.cuda.synchronize()
    return k + 20


def stats(samples) -> dict:
    return {"median": statistics.median(samples), "mean": statistics.fmean(samples),
            "min": min(samples), "max": max(samples), "n": len(samples)}


KERNEL_SAMPLES = 256  # in-step samples per kernel, whatever --steps is
FUSED_SAMPLES, FUSED_GROUP = 32, 8  # one-pass kernel: samples of back-to-back calls


def spread(ms) -> dict:
    """Median, 10th and 90th percentile and maximum of per-step milliseconds."""
    v = sorted(ms)
    if not v:
        return {}
    return {"median": round(statistics.median(v), 4), "p10": round(v[len(v) // 10], 4),
            "p90": round(v[(9 * len(v)) // 10], 4), "max": round(v[-1], 4)}


def copy_engine_rates(host_in, dev_in, host_out, dev_out, stream, reps: int = 4, rounds: int = 5) -> dict:
    """GB/s of pinned-host <-> device copies on this GPU: host->device alone, device->host
    alone, and each direction while the other runs (equal byte counts on two streams, each
    timed to its own end); the best of `rounds` rounds of `reps` copies each, so that the
    bound built from them is the lowest the engines have shown.  `host_in` and `dev_in` hold
    the same bytes, so the copies leave the workload unchanged."""
    import torch

    dev = stream.device
    nin = host_in.numel() * host_in.element_size()
    nout = host_out.numel() * host_out.element_size()
    m = min(nin, nout)
    hin8, din8 = host_in.view(torch.uint8)[:m], dev_in.view(torch.uint8)[:m]

    def timed(fn, nbytes):
        fn()
        torch.cuda.synchronize()
        best = 0.0
        for _ in range(rounds):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            best = max(best, nbytes * reps / (a.elapsed_time(b) / 1e3) / 1e9)
        return round(best, 1)

    h2d = timed(lambda: dev_in.copy_(host_in, non_blocking=True), nin)
    d2h = timed(lambda: host_out.copy_(dev_out, non_blocking=True), nout)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    hout8, dout8 = host_out.view(torch.uint8)[:m], dev_out.view(torch.uint8)[:m]
    c_in = c_out = 0.0
    for _ in range(rounds):
        start = torch.cuda.Event(enable_timing=True)
        e_in, e_out = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start.record(stream)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for _ in range(reps):
            with torch.cuda.stream(s_in):
                din8.copy_(hin8, non_blocking=True)
            with torch.cuda.stream(s_out):
                hout8.copy_(dout8, non_blocking=True)
        e_in.record(s_in)
        e_out.record(s_out)
        torch.cuda.synchronize()
        c_in = max(c_in, m * reps / (start.elapsed_time(e_in) / 1e3) / 1e9)
        c_out = max(c_out, m * reps / (start.elapsed_time(e_out) / 1e3) / 1e9)
    stream.wait_stream(s_in)
    stream.wait_stream(s_out)
    return {"h2d_gbs": h2d, "d2h_gbs": d2h, "concurrent_h2d_gbs": round(c_in, 1),
            "concurrent_d2h_gbs": round(c_out, 1)}


def copy_bound_s(h2d_bytes: int, d2h_bytes: int, link: dict) -> float:
    """Seconds the copy engines need for one step's copies at the measured rates, with the
    two directions overlapped as far as they go: both run together at their concurrent
    rates until the shorter one ends, then the longer one runs alone at its own rate."""
    r_in_c, r_out_c = link["concurrent_h2d_gbs"] * 1e9, link["concurrent_d2h_gbs"] * 1e9
    r_in, r_out = link["h2d_gbs"] * 1e9, link["d2h_gbs"] * 1e9
    if h2d_bytes / r_in_c >= d2h_bytes / r_out_c:
        t = d2h_bytes / r_out_c
        return t + (h2d_bytes - t * r_in_c) / r_in
    t = h2d_bytes / r_in_c
    return t + (d2h_bytes - t * r_out_c) / r_out


def nvfp4_algorithmic_bytes(n: int, s_in: int = 4, colwise: bool = True) -> dict:
    """Compulsory HBM bytes per call of the NVFP4 kernels for an n-element fragment: F32
    1x16 / 16x1 block amaxes, E4M3 block scales, two E2M1 codes per byte."""
    dirs = 2 if colwise else 1
    blocks = dirs * n // 16
    return {"amax": n * s_in + 4 * blocks,                # read x, write F32 block amaxes
            "scales": 4 * blocks + blocks,                # read block amaxes, write E4M3 bytes
            "cast": n * s_in + blocks + dirs * n // 2}    # read x and scales, write codes


def measure_nvfp4(x, dev, peak: float, frac_key: str, samples: int = 256, steps: int = 100) -> dict:
    """The NVFP4 step on the headline weight (16384x6144 FP32, both directions): tensor amax
    reset, partial amax, scale update, partial cast.  Each kernel's time is the median of
    `samples` in-step samples (events around every phase), as for the MXFP8 step: the scale
    update reads the block amaxes its predecessor just wrote, as it does in a real step
    (timed alone its 63 MB would stay in L2).  The whole step is also timed over `steps`
    back-to-back steps without events."""
    import torch

    from mxfp8_master_weight_gb300 import api

    (rr, rc), (cr, cc) = api.nvfp4_block_shapes(ROWS, COLS)
    ar = torch.zeros((rr, rc), device=dev)
    ac = torch.zeros((cr, cc), device=dev)
    at = torch.zeros(1, device=dev)
    sr = torch.empty((rr, rc), dtype=torch.uint8, device=dev)
    scl = torch.empty((cr, cc), dtype=torch.uint8, device=dev)
    qr = torch.empty(ROWS * COLS // 2, dtype=torch.uint8, device=dev)
    qc = torch.empty(ROWS * COLS // 2, dtype=torch.uint8, device=dev)
    amax = api.prepare_nvfp4_partial_amax(x, ar, ac, at, ROWS, COLS, 0)
    scales = api.prepare_nvfp4_update_scales(ar, ac, at, sr, scl, ROWS, COLS)
    cast = api.prepare_nvfp4_partial_cast(x, sr, scl, at, qr, qc, ROWS, COLS, 0)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        at.zero_()
        amax.call(stream)
        if ev:
            ev[1].record(stream)
        scales.call(stream)
        if ev:
            ev[2].record(stream)
        cast.call(stream)
        if ev:
            ev[3].record(stream)

    for _ in range(5):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    step_us = a.elapsed_time(b) * 1e3 / steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(samples)]
    for e in evs:
        step(e)
    torch.cuda.synchronize()

    class _Reset:  # the tensor-amax reset as a call of the amax phase
        def call(self, s):
            with torch.cuda.stream(s):
                at.zero_()

    marg, marg_full = marginal_costs([[_Reset(), amax], [scales], [cast]], stream)
    nb = nvfp4_algorithmic_bytes(ROWS * COLS)
    step_bytes = sum(nb.values())
    out = {"workload": "16384x6144 FP32 headline weight, full fragment, rowwise+columnwise NVFP4 "
                       "(E2M1, 16-value blocks with E4M3 scales, F32 tensor scale)",
           "method": f"median of {samples} in-step samples per kernel (events around each phase; "
                     "the amax phase includes the 4-byte tensor-amax reset); step: "
                     f"{steps} back-to-back steps without events; marginal_us_in_step as for the "
                     f"MXFP8 kernels (full step {marg_full:.2f} µs this way)",
           "us_per_step": round(step_us, 2), "algorithmic_bytes_per_step": step_bytes,
           "step_gbs": round(step_bytes / (step_us * 1e-6) / 1e9, 1),
           "step_" + frac_key: round(step_bytes / (step_us * 1e-6) / 1e9 / peak, 4)}
    for k, nm in enumerate(("amax", "scales", "cast")):
        us = statistics.median(e[k].elapsed_time(e[k + 1]) * 1e3 for e in evs)
        gbs = nb[nm] / (us * 1e-6) / 1e9
        out[nm] = {"us_per_call": round(us, 3), "algorithmic_bytes": nb[nm], "gbs": round(gbs, 1),
                   frac_key: round(gbs / peak, 4), "marginal_us_in_step": round(marg[k], 3),
                   "marginal_gbs": round(nb[nm] / (marg[k] * 1e-6) / 1e9, 1)}
    return out


def run_ours(args):
    import torch

    from mxfp8_master_weight_gb300 import build as libbuild
    libbuild.build()
    from mxfp8_master_weight_gb300 import driver
    from mxfp8_master_weight_gb300 import workloads as wl

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    n = ROWS * COLS
    w = wl.cfg4_headline(rows=ROWS, cols=COLS)
    host = torch.from_numpy(w.data).pin_memory()
    x = host.to(dev)
    sc = driver.ShardedCast([driver.WeightSpec(ROWS, COLS, True)], [0, n], dev,
                            fuse_reduce_scales=True)
    stream = torch.cuda.current_stream(dev)
    names = ("amax", "reduce_scales", "cast")
    abytes = algorithmic_bytes(n)
    step_bytes = sum(abytes[nm] for nm in names)

    def step(events=None):
        sc.step([x], events=events)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # The clock sampler runs over a load window of steps (about half a second), the timed
    # region and the kernel-sampling region, and another load window: at least a second of
    # continuous load, so that the line carries its own clock record.
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        clocks.wait_started()
        load_steps = run_for(step, args.clock_window_s / 2, stream)
        # timed region: exactly K steps, no events inside
        barrier(world)
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(args.steps):
            step()
        stop.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        # per-kernel durations: a fixed number of in-step samples, events around each phase
        per_kernel = dict(zip(names, sample_phases(step, KERNEL_SAMPLES)))
        # phases of the driver's step: amax, reduction (+ fused scales), scales (empty), cast
        marg, marg_full = marginal_costs(sc._prepared([x]), stream)
        load_steps += run_for(step, args.clock_window_s / 2, stream)
    elapsed = start.elapsed_time(stop) / 1e3
    t_max, total_bytes = aggregate_over_ranks(elapsed, step_bytes * args.steps, world, dev)

    # the one-pass path for fragments made of whole blocks (a single rank owns the whole
    # weight here, so it applies): same outputs, reported beside the four-step flow
    from mxfp8_master_weight_gb300 import api as mx_api
    fused_call = mx_api.prepare_quantize_whole_blocks_batched(
        [(x, None, None, sc.scales[0][0], sc.scales[0][1], sc.outputs[0][0], sc.outputs[0][1],
          ROWS, COLS, 0)])
    for _ in range(max(3, args.warmup)):
        fused_call.call(stream)
    torch.cuda.synchronize()
    # throughput of back-to-back calls, as a training loop makes them: 32 samples of 8
    # calls each between two events (consecutive launches overlap through the
    # programmatic launch; an event between every two calls would prevent that)
    fused_samples = []
    for _ in range(FUSED_SAMPLES):
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(FUSED_GROUP):
            fused_call.call(stream)
        f1.record(stream)
        fused_samples.append((f0, f1))
    torch.cuda.synchronize()
    fused_st = stats([a.elapsed_time(b) * 1e3 / FUSED_GROUP for a, b in fused_samples])
    fused_us = fused_st["median"]
    fused_bytes = n * 4 + 2 * n // 32 + 2 * n  # read x, write E8M0 scales and E4M3 data

    # the multi-fragment driver on the sharded mixed batch: 7 weights (8192x8192 and
    # 4096x4096 / 2048x8192, row-only and bidirectional), 4 emulated shards in their own
    # buffers (one boundary inside a 32-value block, one empty shard), one packed MAX
    # reduction per step
    batch = wl.cfg5_sharded_batch(seed=0)
    bspecs = [driver.WeightSpec(w_.rows, w_.cols, w_.colwise) for w_ in batch.weights]
    bsc = driver.ShardedCast(bspecs, batch.bounds, dev)
    bshards = [torch.from_numpy(np.ascontiguousarray(batch.shard(s_))).to(dev)
               for s_ in range(bsc.num_shards)]
    for _ in range(max(3, min(args.warmup, 10))):
        bsc.step(bshards)
    b_steps = 100
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    g0.record(stream)
    for _ in range(b_steps):
        bsc.step(bshards)
    g1.record(stream)
    torch.cuda.synchronize()
    b_us = g0.elapsed_time(g1) * 1e3 / b_steps
    held = sum(e - a for _, a, e in bsc.ranges) if bsc.ranged else None
    b_bytes = sharded_step_bytes(bspecs, bsc.num_shards, bsc.layout.total, slot_entries_read=held)
    b_phase_bytes = sharded_phase_bytes(bspecs, bsc.num_shards, bsc.layout.total,
                                        slot_entries_read=held)
    bsc_launches = bsc.launches_per_step()
    bsc_ranged, bsc_slots, bsc_packed = bsc.ranged, bsc.num_shards, bsc.layout.total
    # per-phase split of the sharded step (events around the phases of sampled steps)
    phase_samples = sample_phases(lambda events=None: bsc.step(bshards, events=events), 64)
    b_phases = {}
    for nm, v in zip(("amax", "reduce_scales", "cast"), phase_samples):
        med = statistics.median(v)
        b_phases[nm] = {"us_median": round(med, 2), "algorithmic_bytes": b_phase_bytes[nm],
                        "gbs": round(b_phase_bytes[nm] / (med * 1e-6) / 1e9, 1)}
    del bshards, bsc, batch
    configs = measure_configs(x, dev)
    pages_table = measure_pages_table(dev)
    peak, peak_kind = measured_peak()
    nvfp4 = measure_nvfp4(x, dev, peak, "frac_of_" + peak_kind + "_peak")

    # End to end through the public API with host buffers, every step copying the 402.7 MB
    # input in from pinned host memory and both E4M3 outputs and both scale grids back.
    # (1) the four-step partial flow (partial amax per chunk as it lands, MAX reduction +
    # scales, partial cast per chunk, copies out) -- the same work as the timed step;
    # (2) the one-pass pipeline (chunks quantised by the one-pass kernel) over its own bytes.
    from mxfp8_master_weight_gb300.host import HostPartialFlow, HostQuantizer, ZeroCopyQuantizer
    out_r, out_c = sc.outputs[0]
    s_r, s_c = sc.scales[0]
    host_q = [torch.empty(out_r.shape, dtype=torch.uint8).pin_memory() for _ in range(2)]
    host_s = [torch.empty(s_r.shape, dtype=torch.uint8).pin_memory(),
              torch.empty(s_c.shape, dtype=torch.uint8).pin_memory()]
    e2e_steps = max(1, min(args.steps, 50))
    h2d = n * 4
    d2h = 2 * n + s_r.numel() + s_c.numel()

    def time_host_path(run):
        """Seconds for e2e_steps back-to-back calls, and each call's milliseconds (events
        recorded on the caller's stream after every call: a call's copy-in does not wait
        for that stream, so the events do not serialise consecutive calls)."""
        for _ in range(3):
            run()
        barrier(world)
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps + 1)]
        ev[0].record(stream)
        for i in range(e2e_steps):
            run()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return ev[0].elapsed_time(ev[-1]) / 1e3, [ev[i].elapsed_time(ev[i + 1]) for i in range(e2e_steps)]

    link = copy_engine_rates(host, x, host_q[0], out_r, stream)
    bound_s = copy_bound_s(h2d, d2h, link)
    flow = HostPartialFlow(ROWS, COLS, True, device=dev, chunk_rows=args.e2e_chunk_rows, direct_out=True)
    flow_t, flow_per = time_host_path(lambda: flow.run(host, host_q[0], host_q[1], host_s[0], host_s[1]))
    flow_t, flow_bytes = aggregate_over_ranks(flow_t, step_bytes * e2e_steps, world, dev)
    flow_launches = flow.launches_per_run()
    flow_chunks = len(flow.chunks)
    del flow
    sflow = HostPartialFlow(ROWS, COLS, True, device=dev, chunk_rows=args.e2e_chunk_rows, direct_out=False)
    sflow_t, sflow_per = time_host_path(lambda: sflow.run(host, host_q[0], host_q[1], host_s[0], host_s[1]))
    sflow_t, sflow_bytes = aggregate_over_ranks(sflow_t, step_bytes * e2e_steps, world, dev)
    del sflow
    zc = ZeroCopyQuantizer(ROWS, COLS, True, device=dev)
    zc_t, zc_per = time_host_path(lambda: zc.run(host, host_q[0], host_q[1], host_s[0], host_s[1]))
    zc_t, zc_bytes = aggregate_over_ranks(zc_t, fused_bytes * e2e_steps, world, dev)
    hq = HostQuantizer(ROWS, COLS, True, device=dev, chunk_rows=1024, depth=3)
    hq_t, hq_per = time_host_path(lambda: hq.run(host, host_q[0], host_q[1], host_s[0], host_s[1]))
    hq_t, hq_bytes = aggregate_over_ranks(hq_t, fused_bytes * e2e_steps, world, dev)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peak()
    frac_key = "frac_of_" + peak_kind + "_peak"
    kernels = {}
    for nm in names:
        st = stats(per_kernel[nm])
        gbs = abytes[nm] / (st["median"] * 1e-6) / 1e9
        kernels[nm] = {"us_per_call_median": round(st["median"], 3),
                       "us_per_call_mean": round(st["mean"], 3), "samples": st["n"],
                       "algorithmic_bytes": abytes[nm], "gbs": round(gbs, 1),
                       frac_key: round(gbs / peak, 4)}
    for nm, k in zip(names, (0, 1, 3)):  # the driver's phase index of each kernel
        mu = marg[k]
        kernels[nm]["marginal_us_in_step"] = round(mu, 3)
        kernels[nm]["marginal_gbs"] = round(abytes[nm] / (mu * 1e-6) / 1e9, 1)
    dom = "cast"
    achieved = kernels[dom]["gbs"]

    cpu = None
    if world == 1 or rank == 0:
        import oracle
        oracle.build()
        cpu_rows = args.cpu_rows
        dt, b = cpu_sample_run(w.data, 0, cpu_rows)
        cpu = {"value": b / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"first {cpu_rows} rows ({cpu_rows * COLS} elements) of the workload: "
                         f"amax, scales, cast; {dt:.1f} s single-threaded",
               "cpu_model": cpu_model()}
        try:
            wall, pb, used = cpu_all_cores_run(w.data, cpu_rows, os.cpu_count() or 1)
            cpu["all_cores"] = {"value": pb / wall / 1e9, "unit": "GB/s", "cores": used,
                                "sample": f"the same rows in 32-row bands over {used} processes "
                                          f"running the single-threaded oracle; {wall:.2f} s wall"}
        except Exception as exc:  # the single-core figure stands on its own
            cpu["all_cores"] = {"unavailable": f"{type(exc).__name__}: {exc}"[:200]}

    value = total_bytes / t_max / 1e9
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_max / args.steps * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "rows": ROWS, "cols": COLS, "fragment": "full (offset 0)",
                   "directions": "rowwise+columnwise", "emulated_shards": 1,
                   "l2": "inputs larger than L2 (402.7 MB FP32 fragment vs 126 MB L2); no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "us_per_call": {nm: kernels[nm]["us_per_call_median"] for nm in names},
        "kernels": kernels,
        "kernel_timing": f"median of {KERNEL_SAMPLES} in-step samples per kernel: CUDA events on "
                         "the launching stream around each phase of every step of a sampling "
                         "region that follows the timed steps (the timed steps carry no events); "
                         "marginal_us_in_step: µs per step of 200 back-to-back steps of the "
                         "library calls minus the same without that kernel (median of 3 rounds; "
                         f"the full step {marg_full:.2f} µs this way), free of the launch and lost "
                         "overlap an event-bracketed short kernel pays",
        "pages_gb200_us_per_call": PAGES_GB200_US,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": read_traffic(dom),
                     "achieved_from": f"algorithmic bytes / median in-step duration ({KERNEL_SAMPLES} samples)"},
        "fused_whole_blocks": {
            "note": "one-pass amax+scales+cast (mxfp8_quantize_whole_blocks), same outputs; "
                    "applies when a rank owns whole blocks, as here",
            "us_per_call": round(fused_us, 3), "us_per_call_mean": round(fused_st["mean"], 3),
            "samples": fused_st["n"],
            "timing": f"median over {FUSED_SAMPLES} samples of {FUSED_GROUP} back-to-back calls",
            "algorithmic_bytes": fused_bytes,
            "gbs": round(fused_bytes / (fused_us * 1e-6) / 1e9, 1),
            frac_key: round(fused_bytes / (fused_us * 1e-6) / 1e9 / peak, 4),
            "traffic": read_traffic("fused"),
            "speedup_vs_step": round(t_max / args.steps * 1e6 / fused_us, 3)},
        "sharded_batch": {
            "workload": "7 FP32 weights (8192x8192; 4096x4096 / 2048x8192, 3 row-only, 4 "
                        "bidirectional; 167.8M elements), 4 emulated shards in own buffers",
            "launches_per_step": bsc_launches, "steps": b_steps,
            "reduction": (f"ranged: reads the {held} slot entries the shards' amax wrote "
                          f"(of {bsc_slots} x {bsc_packed}); slots never zeroed"
                          if bsc_ranged else "whole slots, zeroed before each step"),
            "us_per_step": round(b_us, 2), "phases": b_phases, "algorithmic_bytes": b_bytes,
            "gbs": round(b_bytes / (b_us * 1e-6) / 1e9, 1),
            frac_key: round(b_bytes / (b_us * 1e-6) / 1e9 / peak, 4)},
        "e2e": {"value": round(flow_bytes / flow_t / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(flow_t / e2e_steps * 1e3, 4), "steps": e2e_steps,
                "ms_per_step_spread": spread(flow_per),
                "algorithmic_bytes_per_step": step_bytes,
                "path": f"HostPartialFlow: input copied in by chunks ({flow_chunks} of "
                        f"{args.e2e_chunk_rows} rows), partial amax per chunk as it lands, MAX "
                        "reduction + scales, partial cast per chunk storing straight into the "
                        "pinned host outputs, scale grids copied out; device input double-buffered",
                "gpu_launches_per_step": flow_launches,
                "link_gbs": round((h2d + d2h) * e2e_steps / flow_t / 1e9, 1),
                "copy_engines": dict(link, bound_ms=round(bound_s * 1e3, 4),
                                     note="the least time the step's bytes need through the copy "
                                          "engines alone; the flow's output stores bypass them"),
                "staged_copies": {
                    "path": "the same flow with the casts into device staging buffers and the "
                            "E4M3 bytes copied out by the copy engine",
                    "value": round(sflow_bytes / sflow_t / 1e9, 1),
                    "ms_per_step": round(sflow_t / e2e_steps * 1e3, 4),
                    "ms_per_step_spread": spread(sflow_per),
                    "copy_gbs": round((h2d + d2h) * e2e_steps / sflow_t / 1e9, 1),
                    "frac_of_copy_bound": round(bound_s * e2e_steps / sflow_t, 4)}},
        "e2e_one_pass": {"value": round(zc_bytes / zc_t / 1e9, 1), "unit": "GB/s",
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "ms_per_step": round(zc_t / e2e_steps * 1e3, 4), "steps": e2e_steps,
                         "ms_per_step_spread": spread(zc_per),
                         "algorithmic_bytes_per_step": fused_bytes,
                         "path": "ZeroCopyQuantizer: one launch of the one-pass kernel reading the "
                                 "pinned input and writing the pinned outputs over the CPU-GPU link "
                                 "(the byte counts are those loads and stores; no copy engines)",
                         "gpu_launches_per_step": 1,
                         "link_gbs": round((h2d + d2h) * e2e_steps / zc_t / 1e9, 1),
                         "staged_copies": {
                             "path": f"HostQuantizer: {len(hq.chunks)} chunks of {hq.chunk_rows} rows, "
                                     "3 streams, one-pass kernel per chunk",
                             "value": round(hq_bytes / hq_t / 1e9, 1),
                             "ms_per_step": round(hq_t / e2e_steps * 1e3, 4),
                             "ms_per_step_spread": spread(hq_per),
                             "copy_gbs": round((h2d + d2h) * e2e_steps / hq_t / 1e9, 1),
                             "frac_of_copy_bound": round(bound_s * e2e_steps / hq_t, 4)}},
        "nvfp4": nvfp4,
        "other_configs": {
            "method": "CUDA graph of 50 calls (fragments <= 4M elements) else 10, 20 replays per "
                      "round, 7 rounds, median us per call (the pages' method: their GB200 figures "
                      "for the headline weight bidirectional are in pages_gb200_us_per_call); "
                      "outputs checked bitwise in the tests",
            "cases": configs},
        "pages_table": {
            "method": "each kernel alone, full input, both directions, CUDA graph of 50 calls "
                      "(<= 4M elements) else 10, 20 replays per round, 7 rounds, median; the pages' "
                      "figures are GB200 (context only: other hardware)",
            "cases": pages_table},
        "gpu_launches": sc.launches_per_step() * args.steps,
        "clocks": dict(clocks.summary(), window=f"{load_steps} load steps around the timed region "
                                               f"and {KERNEL_SAMPLES} sampled steps"),
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-chunk-rows", type=int, default=4096,
                    help="rows per chunk of the four-step host-buffer (e2e) leg")
    ap.add_argument("--cpu-rows", type=int, default=8192,
                    help="rows of the workload the CPU-oracle baseline runs on")
    ap.add_argument("--clock-window-s", type=float, default=1.2,
                    help="seconds of load steps around the timed region for the clock samples")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
