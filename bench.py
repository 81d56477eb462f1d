#!/usr/bin/env python3
"""Benchmark of the fused decode-batch QKV front on GB300.

One step = one qkv_front call (projection + q/k RMS norm + RoPE + y store +
paged K/V insert) over one batch of synthetic tokens.  Prints ONE JSON line
(rank 0).  Metric: achieved HBM GB/s = algorithmic bytes of a call
(W + x read, out + K/V written) / time per call; the line also carries
us_per_call.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on the same workload

Timing: W is rotated over R device copies with R x |W| >= 10 x L2, so every
call streams its weights from HBM (checked by DRAM bytes per call over a
range of back-to-back calls); calls are captured in CUDA graphs (their
PDL edges kept) and timed with CUDA events on the launching stream.  A timed
region is exactly --steps calls, bracketed by a barrier and a device
synchronize on both sides; a short spin kernel queued ahead of the region's
start event covers the host's graph launch, as GPU benchmark harnesses do.
Regions repeat until at least --min-seconds of timed GPU work; the line
reports the median region (p10 / p90 beside it), the max over ranks, and the
SM clocks nvidia-smi saw during the regions.  `per_config` repeats the
measurement (back-to-back graph replays) on every workload of the metric's
M = 1..16 range.  Multi-GPU runs are independent replicas (each rank one
tensor-parallel shard of KV heads; no collective on the data path).
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from kv_insert_gb300 import workloads as wl  # noqa: E402

METRIC = "µs/call and achieved HBM GB/s (fraction of GB300 peak) at M=1..16, 1 GPU"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
# the files that define each op's kernel (qkv_front.cu also holds the shared
# device helpers); a traffic record counts only for the source it was taken on
OP_SOURCES = {
    "qkv_front": ("qkv_front.cu",),
    "qknorm_rope_kv_insert": ("qkv_front.cu", "qknorm_rope_kv_insert.cuh"),
    "layer_front": ("qkv_front.cu", "layer_front.cuh"),
    "attn2": ("qkv_front.cu", "attn2.cuh"),
    "attn2_split_kv": ("qkv_front.cu", "attn2.cuh"),
}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")
# every workload of the metric's range, each measured in the same run
PER_CONFIG = (["m1_nkv1_n1152", "m8_nkv8_n9216", "m16_nkv8_n9216_consecutive"]
              + [f"sweep_m{m}_nkv8_n9216" for m in wl.SWEEP_M] + ["m8_nkv16_n18432"])
SPIN_CYCLES = 100_000   # ~50 us at 2 GHz: the region's graph is queued before it starts
# rotated input copies span this many L2 sizes (set by --l2-multiple): at 3
# back-to-back calls still found ~10 % of W in L2 (per-call DRAM reads over a
# range of calls), at 10 ~3 % (with 3 stages of L2 prefetch per CTA), at 30
# every call reads all of its W from DRAM
L2_MULTIPLE = 30


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=96)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="repeat the timed region of --steps calls until this much timed GPU work")
    ap.add_argument("--per-config-seconds", type=float, default=0.3,
                    help="timed GPU work per workload of the per_config records (0: skip them)")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--op", choices=("qkv_front", "qknorm_rope_kv_insert", "chain", "attn2"),
                    default="qkv_front",
                    help="qkv_front: the fused decode front (the headline); qknorm_rope_kv_insert: "
                         "the standalone epilogue on a prefill chunk; chain: layer_front then "
                         "qkv_front, PDL-linked, against each alone; attn2: verify-step paged "
                         "attention reading the cache")
    ap.add_argument("--workload", default=None,
                    choices=sorted(wl.WORKLOADS) + sorted(wl.EPI_WORKLOADS) + sorted(wl.ATTN_WORKLOADS))
    ap.add_argument("--graph-calls", type=int, default=96,
                    help="calls per captured CUDA graph (a multiple of the W copies is used)")
    ap.add_argument("--front-stages", type=int, default=0,
                    help="chain op: run the front at this ring depth (0: the library's choice)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--engine", choices=("cluster", "split_kv"), default="split_kv",
                    help="attn2 engine: clusters merging over DSMEM (the attn2 entry point, no "
                         "workspace) or split-KV over the whole GPU with partials in a workspace")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--l2-multiple", type=float, default=30.0,
                    help="the rotated copies of the streamed input (W, qkv or the cache) span at least "
                         "this many L2 sizes")
    ap.add_argument("--ncu-range", type=int, default=0,
                    help="after warm-up, run this many calls (direct launches, inputs rotated as in "
                         "the timed region) between cudaProfilerStart and cudaProfilerStop, print "
                         "one line and exit: the range an `ncu --replay-mode app-range` capture "
                         "measures, so that DRAM bytes include the write-backs later calls cause")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=90.0,
                    help="target duration of the whole --impl reference run")
    a = ap.parse_args(argv)
    defaults = {"qknorm_rope_kv_insert": wl.EPI_BENCH_WORKLOAD, "attn2": wl.ATTN_BENCH_WORKLOAD}
    tables = {"qknorm_rope_kv_insert": wl.EPI_WORKLOADS, "attn2": wl.ATTN_WORKLOADS}
    if a.workload is None:
        a.workload = defaults.get(a.op, wl.BENCH_WORKLOAD)
    table = tables.get(a.op, wl.WORKLOADS)
    if a.workload not in table:
        ap.error(f"workload {a.workload} is not a {a.op} workload")
    if a.op != "qkv_front" and a.impl == "reference":
        ap.error("the reference arm times the fused front only")
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    if a.steps < 1:
        ap.error("--steps must be >= 1")
    return a


# ---- distributed plumbing (host side) ------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(backend: str):
    world, rank, _ = dist_env()
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)
    return world, rank


def barrier():
    if torch.distributed.is_initialized():
        torch.distributed.barrier()


def max_over_ranks(value: float, device=None) -> float:
    """The maximum of a per-rank float over all ranks (the job's wall time)."""
    if not torch.distributed.is_initialized():
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate(bytes_per_step: int, steps: int, world: int, seconds_max: float) -> dict:
    """Whole-job throughput: units all ranks processed / the slowest rank's time."""
    us = seconds_max / steps * 1e6
    gbs = bytes_per_step * steps * world / seconds_max / 1e9
    return {"value": gbs, "us_per_call": us, "ms_per_step": us / 1e3}


# ---- peaks, traffic, clocks --------------------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            v = float(json.load(fh)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def source_digest(op: str) -> str:
    """sha256 over the op's kernel sources (the .cu / .cuh files that make its
    kernels; the C header only declares them)."""
    h = hashlib.sha256()
    for f in OP_SOURCES[op]:
        with open(os.path.join(ROOT, "kv_insert_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(op: str, workload: str):
    """DRAM bytes per launch from the committed ncu record, if it was taken on
    this exact kernel source, op and workload; else None."""
    try:
        with open(TRAFFIC_FILE) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        return None
    per = rec.get("records", {}).get(f"{op}/{workload}")
    if per is None or per.get("source_sha256") != source_digest(op):
        return None
    return float(per["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the GPU works.
    Every sample carries nvidia-smi's own timestamp, so a summary can keep
    only the samples taken inside a timed window (host wall-clock times from
    `now()`)."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None
        self.rows = []

    @staticmethod
    def now() -> datetime.datetime:
        return datetime.datetime.now()

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        """Ends sampling and parses the samples (kept for `summary`)."""
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        text = self.file.read()
        self.file.close()
        os.unlink(self.file.name)
        self.rows = self.parse(text)

    @classmethod
    def parse(cls, text: str) -> list:
        rows = []
        for line in text.strip().splitlines():
            r = [c.strip() for c in line.split(",")]
            if len(r) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f")
                sm, mx = float(r[2]), float(r[3])
            except ValueError:
                continue
            reasons = {n for n, f in zip(cls.REASONS, r[6:10]) if f.lower() == "active"}
            rows.append((ts, sm, mx, reasons))
        return rows

    def summary(self, t0=None, t1=None):
        """Median SM clock, max clock and throttle reasons of the samples
        taken in [t0, t1] (all samples when no window is given), or None."""
        rows = [r for r in self.rows if (t0 is None or r[0] >= t0) and (t1 is None or r[0] <= t1)]
        if not rows:
            return None
        sm = [r[1] for r in rows]
        reasons = set().union(*[r[3] for r in rows])
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[2] for r in rows),
                "sm_mhz_min": min(sm), "reasons": sorted(reasons), "samples": len(rows),
                "window": "samples taken while the timed work ran"}


def spin(stream):
    """A short device-side spin queued ahead of a timed region (outside it),
    so the region's start event fires only after the host has queued the
    region's work: the region measures the GPU, not the host's launch."""
    with torch.cuda.stream(stream):
        torch.cuda._sleep(SPIN_CYCLES)


def profile_range(call, calls: int, stream, dev) -> dict:
    """`calls` calls of call(i) on `stream` inside one profiler range."""
    torch.cuda.synchronize(dev)
    torch.cuda.profiler.start()
    with torch.cuda.stream(stream):
        for i in range(calls):
            call(i)
    torch.cuda.synchronize(dev)
    torch.cuda.profiler.stop()
    return {"ncu_range_calls": calls}


def time_regions(region, stream, dev, min_seconds: float, min_regions: int = 3,
                 max_regions: int = 100000):
    """Times `region()` (which queues exactly one region's calls on `stream`)
    repeatedly: each time bracketed by a barrier and a device synchronize on
    both sides, with CUDA events on `stream` right around the region.  Runs
    `min_regions` first to size the count, then as many as make
    `min_seconds` of timed GPU work (the same count on every rank).  Returns
    (seconds of each region, wall-clock window of the timed regions)."""
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def one():
        barrier()
        torch.cuda.synchronize(dev)
        spin(stream)
        with torch.cuda.stream(stream):
            start.record(stream)
            region()
            end.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        return start.elapsed_time(end) / 1e3

    est = statistics.median([one() for _ in range(min_regions)])
    n = int(min(max_regions, max(min_regions, math.ceil(min_seconds / max(est, 1e-9)))))
    n = int(max_over_ranks(float(n), dev))
    t0 = ClockSampler.now()
    times = [one() for _ in range(n)]
    return times, (t0, ClockSampler.now())


def region_stats(times: list, steps: int) -> dict:
    """Median, p10 and p90 of the regions in microseconds per call."""
    q = np.percentile(np.asarray(times), [10, 50, 90]) / steps * 1e6
    return {"us_per_call_p10": float(q[0]), "us_per_call_median": float(q[1]),
            "us_per_call_p90": float(q[2]), "regions": len(times),
            "timed_seconds": float(sum(times))}


# ---- the CPU oracle (baseline and reference arm) ---------------------------

def shard_rows(nkv: int, g: int) -> np.ndarray:
    """The rows of W that KV head g owns ([q heads 8g..8g+7 | k head g | v
    head g | gate heads 8g..8g+7]): one tensor-parallel shard, itself a front
    with one KV head."""
    heads = (list(range(8 * g, 8 * g + 8)) + [8 * nkv + g, 9 * nkv + g]
             + list(range(10 * nkv + 8 * g, 10 * nkv + 8 * g + 8)))
    return np.concatenate([np.arange(h * 64, h * 64 + 64) for h in heads])


def oracle_unit_inputs(inp: dict, w: wl.Workload, t: int, g: int):
    """One token and one KV-head group of the workload: KV head g's shard of
    W and token t."""
    Wb = wl.bits(inp["W"])[shard_rows(w.num_kv_heads, g)]
    return (wl.bits(inp["x"])[t: t + 1], np.ascontiguousarray(Wb),
            inp["positions"].numpy()[t: t + 1], np.array([0], np.int64))


def time_oracle_units(inp, w, units: int):
    """Run `units` (token, KV group) oracle calls; returns seconds."""
    import oracle
    cs = inp["cos_sin"].numpy()
    cache = np.zeros((1, 1, 16, 128), np.uint16)
    n_units = w.M * w.num_kv_heads
    prepared = [oracle_unit_inputs(inp, w, u % w.M, (u // w.M) % w.num_kv_heads)
                for u in range(min(units, n_units))]
    t0 = time.perf_counter()
    for u in range(units):
        x, Wb, pos, sl = prepared[u % len(prepared)]
        _, err = oracle.qkv_front(x, Wb, pos, sl, cs, cache, 1)
        if err:
            raise RuntimeError(f"oracle error {err}")
    return time.perf_counter() - t0


def cpu_model() -> str:
    """The host CPU's name as /proc/cpuinfo gives it (x86 model name, or the
    Arm implementer / part numbers), else the machine type."""
    try:
        fields = {}
        for line in open("/proc/cpuinfo"):
            k, _, v = line.partition(":")
            fields.setdefault(k.strip(), v.strip())
        if "model name" in fields:
            return fields["model name"]
        if "CPU part" in fields:
            return f"{platform.machine()} CPU implementer {fields.get('CPU implementer', '?')} part {fields['CPU part']}"
    except OSError:
        pass
    return platform.machine()


def cpu_baseline(inp, w, seconds: float) -> dict:
    """The oracle, as it stands, on host cores: whole calls of the workload
    until `seconds` of CPU work (at least one)."""
    import oracle
    cs = inp["cos_sin"].numpy()
    xb, Wb = wl.bits(inp["x"]), wl.bits(inp["W"])
    pos, sl = inp["positions"].numpy(), inp["slots"].numpy()
    cache = wl.bits(inp["kv_cache"]).copy()
    calls, t0 = 0, time.perf_counter()
    while True:
        _, err = oracle.qkv_front(xb, Wb, pos, sl, cs, cache, w.num_kv_heads)
        if err:
            raise RuntimeError(f"oracle error {err}")
        calls += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": w.roofline_bytes() * calls / el / 1e9, "unit": UNIT, "cores": 1,
            "kind": "oracle",
            "sample": f"{calls} whole calls of {w.name} (single-threaded C oracle), {el:.1f} s, "
                      f"on {cpu_model()} ({os.cpu_count()} cores visible)"}


def oracle_shard_call(xb, w_shard, pos, cs, cache):
    """One KV head's shard of a call through the oracle, tokens t -> slots t
    of a one-page cache (M <= 16): the same arithmetic, per column, as the
    whole call."""
    import oracle
    slots = np.arange(xb.shape[0], dtype=np.int64)
    out, err = oracle.qkv_front(xb, w_shard, pos, slots, cs, cache, 1)
    if err:
        raise RuntimeError(f"oracle error {err}")
    return out


def cpu_baseline_all_cores(inp, w, seconds: float) -> dict:
    """The same oracle on every host core: each whole call split into its
    KV-head shards, the shards of several calls run side by side in threads
    (the oracle's C call releases the GIL). Each output column is computed
    exactly as in the whole call."""
    from concurrent.futures import ThreadPoolExecutor
    threads = os.cpu_count() or 1
    nkv = w.num_kv_heads
    cs = inp["cos_sin"].numpy()
    xb, pos = wl.bits(inp["x"]), inp["positions"].numpy()
    Wall = wl.bits(inp["W"])
    shards = [np.ascontiguousarray(Wall[shard_rows(nkv, g)]) for g in range(nkv)]
    per_wave = max(1, -(-threads // nkv))   # whole calls in flight together
    tasks = per_wave * nkv
    caches = [np.zeros((1, 1, 16, 128), np.uint16) for _ in range(tasks)]

    def task(i):
        oracle_shard_call(xb, shards[i % nkv], pos, cs, caches[i])

    calls = 0
    with ThreadPoolExecutor(min(threads, tasks)) as ex:
        t0 = time.perf_counter()
        while True:
            list(ex.map(task, range(tasks)))
            calls += per_wave
            el = time.perf_counter() - t0
            if el >= seconds:
                break
    return {"value": w.roofline_bytes() * calls / el / 1e9, "unit": UNIT,
            "cores": min(threads, tasks), "kind": "oracle",
            "sample": f"{calls} whole calls of {w.name} as {nkv} KV-head shards each, "
                      f"{min(threads, tasks)} threads, {el:.1f} s, on {cpu_model()}"}


def run_reference(args, w: wl.Workload):
    world, rank = dist_init("gloo")
    if rank != 0:
        return None
    inp = wl.make_inputs(w)
    n_units = w.M * w.num_kv_heads
    unit_bytes = w.roofline_bytes() / n_units
    t_unit = time_oracle_units(inp, w, 1)
    units_per_step = int(max(1, min(n_units, args.ref_seconds / ((args.steps + args.warmup) * t_unit))))
    time_oracle_units(inp, w, units_per_step * args.warmup)
    el = time_oracle_units(inp, w, units_per_step * args.steps)
    value = unit_bytes * units_per_step * args.steps / el / 1e9
    sample = (f"each step: {units_per_step} of the {n_units} (token, KV-head group) units of "
              f"{w.name} through the single-threaded C oracle, on {cpu_model()}")
    cfg = w.describe()
    cfg.update({"l2": "n/a (host)", "units_per_step": units_per_step})
    return {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ---- our arm ----------------------------------------------------------------

def front_setup(qf, w: wl.Workload, dev, stream, graph_calls: int, inp=None):
    """Device inputs of a front workload, W rotated over enough copies to
    exceed 3 x L2, and a capture helper.  Returns a dict of the pieces."""
    inp = wl.make_inputs(w) if inp is None else inp
    g = {k: v.to(dev) for k, v in inp.items()}
    qf.prepare(w.N, w.num_kv_heads)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    w_bytes = w.N * wl.HIDDEN * 2
    copies = max(2, math.ceil(L2_MULTIPLE * l2 / w_bytes))
    Ws = [g["W"]] + [g["W"].clone() for _ in range(copies - 1)]
    torch.cuda.synchronize(dev)   # W is read before the PDL wait: no writer may be in flight
    out = torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev)
    per_graph = max(copies, (graph_calls // copies) * copies)

    def call(i):
        qf.launch(g["x"], Ws[i % copies], g["positions"], g["slots"], g["cos_sin"],
                  g["kv_cache"], out)

    def capture(n, start=0):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(n):
                call(start + i)
        return graph

    return {"inp": inp, "g": g, "Ws": Ws, "copies": copies, "out": out, "call": call,
            "capture": capture, "per_graph": per_graph, "l2": l2, "w_bytes": w_bytes}


def per_config_records(qf, dev, stream, sampler, seconds: float, graph_calls: int) -> list:
    """Every workload of the metric's range measured the same way: a CUDA
    graph of PDL-linked calls (W rotated past L2) replayed back to back, each
    replay timed by CUDA events on the stream, until `seconds` of timed work;
    the median replay per call, its p10 / p90, GB/s and fraction of the
    measured copy peak.  Each record keeps its wall-clock window, for the
    clocks sampled while its replays ran (filled in once sampling stops)."""
    peak, peak_kind = hbm_peak()
    recs = []
    for name in PER_CONFIG:
        w = wl.WORKLOADS[name]
        f = front_setup(qf, w, dev, stream, graph_calls)
        with torch.cuda.stream(stream):
            for i in range(8):
                f["call"](i)
        stream.synchronize()
        graph = f["capture"](f["per_graph"])
        with torch.cuda.stream(stream):
            graph.replay()
        stream.synchronize()
        if qf.status():
            raise RuntimeError(f"device status raised during the warm-up of {name}")
        # size the run from one replay
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        reps = int(min(5000, max(20, math.ceil(seconds / max(e0.elapsed_time(e1) / 1e3, 1e-6)))))
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        t0 = sampler.now()
        with torch.cuda.stream(stream):
            evs[0].record(stream)
            for k in range(reps):
                graph.replay()
                evs[k + 1].record(stream)
        torch.cuda.synchronize(dev)
        t1 = sampler.now()
        if qf.status():
            raise RuntimeError(f"device status raised while timing {name}")
        per_replay = np.asarray([evs[k].elapsed_time(evs[k + 1]) for k in range(reps)]) / 1e3
        q = np.percentile(per_replay, [10, 50, 90]) / f["per_graph"] * 1e6
        gbs = w.roofline_bytes() / (q[1] * 1e-6) / 1e9
        recs.append({
            "workload": name, "M": w.M, "N": w.N, "num_kv_heads": w.num_kv_heads,
            "variant": qf.variant_full(w.N, w.M),
            "us_per_call": float(q[1]), "us_per_call_p10": float(q[0]),
            "us_per_call_p90": float(q[2]), "bytes_per_call": w.roofline_bytes(), "gbs": gbs,
            "frac": gbs / peak, "frac_of_measured_peak": gbs / peak, "peak_kind": peak_kind,
            "frac_of_nominal_8tbs": gbs / NOMINAL_HBM_GBS,
            "traffic": recorded_traffic("qkv_front", name),
            "calls": reps * f["per_graph"], "graph_calls": f["per_graph"],
            "l2": f"W rotated over {f['copies']} copies of {f['w_bytes'] / 1e6:.1f} MB",
            "clocks": None, "window": (t0, t1)})
        del f, graph
        torch.cuda.empty_cache()
    return recs


def run_ours(args, w: wl.Workload):
    from kv_insert_gb300 import qkv_front as qf

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (the product path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init("nccl")
    qf.load()

    stream = torch.cuda.Stream(device=dev)
    f = front_setup(qf, w, dev, stream, args.graph_calls)
    inp, g, Ws, copies, out = f["inp"], f["g"], f["Ws"], f["copies"], f["out"]
    M, N = w.M, w.N
    variant = qf.variant_full(N, M)
    per_graph = f["per_graph"]

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            f["call"](i)
    stream.synchronize()
    assert qf.status() == 0, "device status raised during warm-up"
    if args.ncu_range:
        return dict(profile_range(f["call"], args.ncu_range, stream, dev), workload=w.name)
    full, rem = divmod(args.steps, per_graph)
    g_full = f["capture"](per_graph) if full else None
    g_rem = f["capture"](rem) if rem else None
    # graph upload before timing (part of set-up, not a timed step)
    with torch.cuda.stream(stream):
        if g_full:
            g_full.replay()
        if g_rem:
            g_rem.replay()
    stream.synchronize()

    def region():
        for _ in range(full):
            g_full.replay()
        if g_rem:
            g_rem.replay()

    sampler = ClockSampler(local)
    sampler.start()
    times, (t0, t1) = time_regions(region, stream, dev, args.min_seconds)
    st = qf.status()
    if st:
        raise RuntimeError(f"device status {st:#x} raised in the timed region")
    el_med = statistics.median(times)
    el_max = max_over_ranks(el_med, dev)
    res = aggregate(w.roofline_bytes(), args.steps, world, el_max)
    stats = region_stats(times, args.steps)

    # the same calls on one W copy (the warm case: whatever of W the L2 keeps
    # between calls is not re-read), outside the timed region, labelled
    warm_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(warm_graph, stream=stream):
        for _ in range(per_graph):
            qf.launch(g["x"], Ws[0], g["positions"], g["slots"], g["cos_sin"], g["kv_cache"], out)
    with torch.cuda.stream(stream):
        warm_graph.replay()
    stream.synchronize()
    w_start, w_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    warm_reps = 20
    with torch.cuda.stream(stream):
        w_start.record(stream)
        for _ in range(warm_reps):
            warm_graph.replay()
        w_end.record(stream)
    torch.cuda.synchronize(dev)
    warm_us = w_start.elapsed_time(w_end) * 1e3 / (warm_reps * per_graph)

    # end to end through the public API: pinned host inputs -> device, the call,
    # device -> pinned host result, every step
    e2e = None
    if not args.no_e2e:
        xh = inp["x"].pin_memory()
        ph = inp["positions"].pin_memory()
        sh = inp["slots"].pin_memory()
        oh = torch.empty(M, N, dtype=torch.bfloat16).pin_memory()
        staging = torch.empty(qf.staging_bytes(M, N), dtype=torch.uint8, device=dev)

        def e2e_step(i):
            # one library call: host x / positions / slots in, the front, out back to host
            qf.qkv_front_from_host(xh, ph, sh, oh, Ws[i % copies], g["cos_sin"], g["kv_cache"],
                                   staging, stream=stream)

        for i in range(args.warmup):
            e2e_step(i)
        stream.synchronize()

        def e2e_region():
            for i in range(args.steps):
                e2e_step(i)

        e_times, _ = time_regions(e2e_region, stream, dev, args.min_seconds / 2)
        if qf.status():
            raise RuntimeError("device status raised in the end-to-end leg")
        e_el = max_over_ranks(statistics.median(e_times), dev)
        e_res = aggregate(w.roofline_bytes(), args.steps, world, e_el)
        e2e = {"value": e_res["value"], "unit": UNIT, "us_per_call": e_res["us_per_call"],
               "h2d_bytes_per_step": xh.numel() * 2 + ph.numel() * 8 + sh.numel() * 8,
               "d2h_bytes_per_step": oh.numel() * 2,
               "timing": f"median of {len(e_times)} regions of {args.steps} library calls from "
                         "pinned host buffers"}

    per_config = None
    if args.per_config_seconds > 0 and rank == 0:
        del warm_graph, g_full, g_rem
        torch.cuda.empty_cache()
        per_config = per_config_records(qf, dev, stream, sampler, args.per_config_seconds,
                                        args.graph_calls)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    for r in per_config or []:   # the samples are parsed once sampling has stopped
        r["clocks"] = sampler.summary(*r.pop("window"))

    if rank != 0:
        return None
    peak, peak_kind = hbm_peak()
    bytes_call = w.roofline_bytes()
    achieved = bytes_call / (el_max / args.steps) / 1e9
    traffic = recorded_traffic("qkv_front", w.name)
    line = {
        "metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
        "us_per_call": res["us_per_call"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(w.describe(), **{
            "variant": variant,
            "l2": f"inputs larger than L2: W rotated over {copies} copies of {f['w_bytes'] / 1e6:.1f} MB "
                  f"(L2 {f['l2'] / 1e6:.1f} MB)",
            "graph_calls": per_graph, "parallelism": f"replicas x{world}"}),
        "timing": dict(stats, **{
            "region": f"exactly {args.steps} calls between CUDA events, barrier + synchronize on "
                      "both sides, a spin kernel queued ahead of the start event",
            "reported": "median region (max over ranks)"}),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "frac_of_measured_peak": achieved / peak,
                     "peak_kind": peak_kind, "traffic": traffic, "bytes_per_launch": bytes_call,
                     "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "e2e": e2e,
        "warm_same_w": {"us_per_call": warm_us, "calls": warm_reps * per_graph,
                        "note": "one W copy for every call, timed after and apart from the "
                                "headline; not the headline"},
        "per_config": per_config,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, w, args.cpu_seconds)
        line["cpu_baseline_all_cores"] = cpu_baseline_all_cores(inp, w, args.cpu_seconds)
    return line


EPI_METRIC = "qknorm_rope_kv_insert achieved HBM GB/s on a prefill chunk, 1 GPU"


def run_epilogue(args, w):
    """The standalone epilogue on a prefill chunk: in place on qkv copies
    rotated past L2, CUDA-graph replays, CUDA events."""
    from kv_insert_gb300 import qkv_front as qf

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (the product path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init("nccl")
    qf.load()
    inp = wl.make_epi_inputs(w)
    g = {k: v.to(dev) for k, v in inp.items()}
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    q_bytes = g["qkv"].numel() * 2
    copies = max(2, math.ceil(L2_MULTIPLE * l2 / q_bytes))
    qs = [g["qkv"]] + [g["qkv"].clone() for _ in range(copies - 1)]
    torch.cuda.synchronize(dev)
    stream = torch.cuda.Stream(device=dev)
    per_graph = max(copies, (args.graph_calls // copies) * copies)

    def call(i):
        qf.qknorm_rope_kv_insert(qs[i % copies], g["positions"], g["slots"], g["cos_sin"],
                                 g["kv_cache"])

    def capture(n):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(n):
                call(i)
        return graph

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            call(i)
    stream.synchronize()
    if args.ncu_range:
        return dict(profile_range(call, args.ncu_range, stream, dev), workload=w.name)
    full, rem = divmod(args.steps, per_graph)
    g_full = capture(per_graph) if full else None
    g_rem = capture(rem) if rem else None
    with torch.cuda.stream(stream):
        for gr in (g_full, g_rem):
            if gr:
                gr.replay()
    stream.synchronize()
    def region():
        for _ in range(full):
            g_full.replay()
        if g_rem:
            g_rem.replay()

    sampler = ClockSampler(local)
    sampler.start()
    times, (t0, t1) = time_regions(region, stream, dev, args.min_seconds)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    el_max = max_over_ranks(statistics.median(times), dev)
    if qf.status():
        raise RuntimeError("device status raised in the timed region")
    res = aggregate(w.roofline_bytes(), args.steps, world, el_max)
    if rank != 0:
        return None
    peak, peak_kind = hbm_peak()
    achieved = w.roofline_bytes() / (el_max / args.steps) / 1e9
    return {"metric": EPI_METRIC, "timing": region_stats(times, args.steps), "value": res["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
            "us_per_call": res["us_per_call"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(w.describe(), **{
                "l2": f"inputs larger than L2: qkv rotated over {copies} copies of "
                      f"{q_bytes / 1e6:.1f} MB (L2 {l2 / 1e6:.1f} MB)",
                "graph_calls": per_graph, "parallelism": f"replicas x{world}"}),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "traffic": recorded_traffic("qknorm_rope_kv_insert", w.name),
                         "bytes_per_launch": w.roofline_bytes()},
            "gpu_launches": args.steps, "clocks": clocks, "e2e": None}


ATTN_METRIC = "attn2 achieved HBM GB/s (verify-step paged attention), 1 GPU"


def run_attn2(args, w):
    """attn2 over cache copies rotated past L2, CUDA-graph replays, events."""
    from kv_insert_gb300 import qkv_front as qf

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (the product path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init("nccl")
    qf.load()
    inp = wl.make_attn_inputs(w)
    g = {k: v.to(dev) for k, v in inp.items()}
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    c_bytes = g["kv_cache"].numel() * 2
    copies = max(2, math.ceil(L2_MULTIPLE * l2 / c_bytes))
    caches = [g["kv_cache"]] + [g["kv_cache"].clone() for _ in range(copies - 1)]
    out = torch.empty(8 * w.R, 512 * w.num_kv_heads, dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize(dev)
    stream = torch.cuda.Stream(device=dev)
    per_graph = max(copies, (args.graph_calls // copies) * copies)
    if args.engine == "split_kv":
        splits = qf.attn2_split_kv_splits(w.R, w.num_kv_heads, w.max_blocks(), w.window)
        ws = torch.zeros(qf.attn2_split_kv_workspace_bytes(w.R, w.num_kv_heads, splits),
                         dtype=torch.uint8, device=dev)

        def call(i):
            qf.attn2_split_kv(g["qkv"], caches[i % copies], g["block_table"], g["context_lens"], ws,
                              out=out, window=w.window, splits=splits)
    else:
        splits = qf.attn2_splits(w.R, w.num_kv_heads, w.max_blocks(), w.window)

        def call(i):
            qf.attn2(g["qkv"], caches[i % copies], g["block_table"], g["context_lens"], out=out,
                     window=w.window)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            call(i)
    stream.synchronize()
    if args.ncu_range:
        return dict(profile_range(call, args.ncu_range, stream, dev), workload=w.name)
    full, rem = divmod(args.steps, per_graph)
    graphs = []
    for n in ([per_graph] if full else []) + ([rem] if rem else []):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(n):
                call(i)
        graphs.append(graph)
    with torch.cuda.stream(stream):
        for gr in graphs:
            gr.replay()
    stream.synchronize()
    def region():
        for _ in range(full):
            graphs[0].replay()
        if rem:
            graphs[-1].replay()

    sampler = ClockSampler(local)
    sampler.start()
    times, (t0, t1) = time_regions(region, stream, dev, args.min_seconds)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    el_max = max_over_ranks(statistics.median(times), dev)
    if qf.status():
        raise RuntimeError("device status raised in the timed region")
    res = aggregate(w.roofline_bytes(), args.steps, world, el_max)
    if rank != 0:
        return None
    peak, peak_kind = hbm_peak()
    achieved = w.roofline_bytes() / (el_max / args.steps) / 1e9
    return {"metric": ATTN_METRIC, "timing": region_stats(times, args.steps), "value": res["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
            "us_per_call": res["us_per_call"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(w.describe(), **{
                "engine": args.engine, "splits": splits,
                "l2": f"inputs larger than L2: cache rotated over {copies} copies of "
                      f"{c_bytes / 1e6:.1f} MB (L2 {l2 / 1e6:.1f} MB)",
                "graph_calls": per_graph, "parallelism": f"replicas x{world}"}),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "traffic": recorded_traffic(
                             "attn2" if args.engine == "cluster" else "attn2_split_kv", w.name),
                         "bytes_per_launch": w.roofline_bytes()},
            "gpu_launches": args.steps * (2 if args.engine == "split_kv" and splits > 1 else 1), "clocks": clocks,
            "e2e": None}


CHAIN_METRIC = "µs per first-layer front step: layer_front then qkv_front, PDL-linked, 1 GPU"


def run_chain(args, w: wl.Workload):
    """layer_front (embedded tokens -> residual stream + normed x) followed by
    qkv_front on its output, PDL-linked on one stream: µs per step, against
    the two kernels timed alone in the same way; the difference is the time
    the front's weight prefetch hides under its predecessor."""
    from kv_insert_gb300 import qkv_front as qf

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (the product path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init("nccl")
    qf.load()
    inp = wl.make_inputs(w)
    lf = wl.make_layer_front_inputs(w)
    g = {k: v.to(dev) for k, v in inp.items()}
    g.update({k: v.to(dev) for k, v in lf.items()})
    stream_buf = torch.empty(w.M, wl.HIDDEN, device=dev)
    x_attn = torch.empty(w.M, wl.HIDDEN, dtype=torch.bfloat16, device=dev)
    out = torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev)
    qf.prepare(w.N, w.num_kv_heads)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    w_bytes = w.N * wl.HIDDEN * 2
    copies = max(2, math.ceil(L2_MULTIPLE * l2 / w_bytes))
    Ws = [g["W"]] + [g["W"].clone() for _ in range(copies - 1)]
    torch.cuda.synchronize(dev)
    s = torch.cuda.Stream(device=dev)
    per_graph = max(copies, (args.graph_calls // copies) * copies)

    def lf_call():
        qf.layer_front(g["x_embed"], stream_buf, x_attn, weight=g["norm_weight"])

    v = qf.variant_full(w.N, w.M)

    def front_call(i):
        if args.front_stages:
            qf.launch_variant(x_attn, Ws[i % copies], g["positions"], g["slots"], g["cos_sin"],
                              g["kv_cache"], out, v["splits"], args.front_stages, kb=v["kb"])
        else:
            qf.launch(x_attn, Ws[i % copies], g["positions"], g["slots"], g["cos_sin"],
                      g["kv_cache"], out)

    legs = {"chain": lambda i: (lf_call(), front_call(i)),
            "chain_no_pdl": lambda i: (lf_call(), front_call(i)),
            "layer_front": lambda i: lf_call(),
            "qkv_front": front_call}
    timings = {}
    for name, fn in legs.items():
        qf.set_pdl(name != "chain_no_pdl")
        with torch.cuda.stream(s):
            for i in range(args.warmup):
                fn(i)
        s.synchronize()
        full, rem = divmod(args.steps, per_graph)
        graphs = []
        for n in ([per_graph] if full else []) + ([rem] if rem else []):
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=s):
                for i in range(n):
                    fn(i)
            graphs.append(graph)
        with torch.cuda.stream(s):
            for gr in graphs:
                gr.replay()
        s.synchronize()
        def region():
            for _ in range(full):
                graphs[0].replay()
            if rem:
                graphs[-1].replay()

        times, _ = time_regions(region, s, dev, args.min_seconds / 2)
        timings[name] = max_over_ranks(statistics.median(times), dev) / args.steps * 1e6
    qf.set_pdl(True)
    if qf.status():
        raise RuntimeError("device status raised in the timed region")
    if rank != 0:
        return None
    return {"metric": CHAIN_METRIC, "value": timings["chain"], "unit": "µs/step", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": timings["chain"] / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": dict(w.describe(), **{
                "l2": f"inputs larger than L2: W rotated over {copies} copies",
                "front_variant": dict(v, stages=args.front_stages or v["stages"]),
                "graph_calls": per_graph, "parallelism": f"replicas x{world}"}),
            "layer_front_alone_us": timings["layer_front"],
            "qkv_front_alone_us": timings["qkv_front"],
            "sum_alone_us": timings["layer_front"] + timings["qkv_front"],
            "hidden_by_overlap_us": timings["layer_front"] + timings["qkv_front"] - timings["chain"],
            "chain_without_pdl_us": timings["chain_no_pdl"],
            "pdl_gain_us": timings["chain_no_pdl"] - timings["chain"],
            "gpu_launches": 2 * args.steps, "e2e": None}  # launches of the PDL chain leg


def main(argv=None):
    global L2_MULTIPLE
    args = parse_args(argv)
    L2_MULTIPLE = args.l2_multiple
    if args.op == "chain":
        line = run_chain(args, wl.WORKLOADS[args.workload])
    elif args.op == "attn2":
        line = run_attn2(args, wl.ATTN_WORKLOADS[args.workload])
    elif args.op == "qknorm_rope_kv_insert":
        line = run_epilogue(args, wl.EPI_WORKLOADS[args.workload])
    else:
        w = wl.WORKLOADS[args.workload]
        line = run_reference(args, w) if args.impl == "reference" else run_ours(args, w)
    if line is not None:
        print(json.dumps(line), flush=True)
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
