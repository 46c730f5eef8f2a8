"""Benchmark of the fused reduce + residual + RMSNorm step on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...      # the CPU oracle, timed on host cores
    python bench.py --sweep                   # SM-budget x token-count table (many lines)
    python bench.py --corun                   # split pipelined against a GEMM (many lines)
    python bench.py --offset-sweep [--sm-budget k]   # timed offset sweep -> lookup table
    python bench.py --link                    # host-link copy bandwidth (e2e bytes)

A step is one pass of the hot path over one batch: the wave-aware split plan
and the fused step over the batch, prefix on one stream, suffix on another
(at T=1024 the plan keeps the batch whole). Eager steps make one C call,
tw_run_wave_split, which computes the plan on the host every step and
launches the halves; graph mode plans with tw_wave_split and replays the
graph captured for that plan.
The default workload is the Llama-3.3-70B layer shape, T=1024 tokens, H=8192,
N=8 partial buffers. Inputs rotate among enough seeded sets to exceed 4x the
L2 cache, so no step reads inputs the previous step left in L2.

Rank 0 prints ONE JSON line. ``value`` is whole-job algorithmic GB/s:
(N+3)*T*H*2 + H*2 bytes per step, times the steps of all ranks, over the
slowest rank's device time. With torchrun (N>1) every rank runs its own
replica of the workload (the step has no cross-GPU exchange on one node's
replicas), and the timing is the max over ranks. Besides the timed region the
line carries the step timed per launch and right after the row-parallel GEMM
(``roofline``), a compact sweep over T and SM budgets (``sweep``), the
unfused baseline, the end-to-end leg from host buffers (``e2e``, with the
same copies timed without the step as its host-link bound) and the CPU
oracle (``cpu_baseline``).
"""

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused reduce+RMSNorm GB/s and % of GB300 HBM peak; tokens/s at T=1K–16K"
PLANNER_SMS = 148  # SMs the planner models for the compute kernels (split workload)
FALLBACK_HBM_GBS = 6800.0
KERNEL_SRC = os.path.join(ROOT, "reduce_rmsnorm_gb300", "csrc", "fused_kernel.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "fused_kernel_traffic.json")


# ------------------------------------------------------------------ small helpers


def peak_hbm():
    """(GB/s, source) of the HBM roofline denominator."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sha(path=None):
    """Fingerprint of the kernel's code: its source with comments removed and
    whitespace runs collapsed, so that editing prose keeps the ncu record
    while any change to the code orphans it."""
    with open(path or KERNEL_SRC) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return hashlib.sha256(" ".join(src.split()).encode()).hexdigest()[:16]


def ncu_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    summary is for another kernel revision or workload."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("kernel_sha") != kernel_sha():
        return None
    w = d.get("workloads", {}).get(workload)
    return None if w is None else int(w["dram_bytes_per_launch"])


def ctas_unsplit(T, H):
    """CTA count of the row-parallel projection the split plan models:
    128-token x 128-column tiles, 8 ranks: ceil(T/128) * (H/128) / 8."""
    return math.ceil(T / 128) * (H // 128) // 8


SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class NvmlSource:
    """Read-only NVML device queries (libnvidia-ml, which ships with the
    driver) through ctypes: SM clock, maximum SM clock, power draw and the
    active clock-event reasons. Nothing is set."""

    CLOCK_SM = 1
    REASON_BITS = ((0x4, "sw_power_cap"), (0x8, "hw_slowdown"),
                   (0x20, "sw_thermal_slowdown"), (0x40, "hw_thermal_slowdown"))
    name = "nvml"

    def __init__(self, uuid, index):
        import ctypes
        self.ct = ctypes
        L = ctypes.CDLL("libnvidia-ml.so.1")
        if L.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        h = ctypes.c_void_p()
        by_uuid = bool(uuid) and L.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0
        if not by_uuid and L.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) != 0:
            L.nvmlShutdown()
            raise OSError("no NVML handle for the device")
        self.L, self.h = L, h
        self.reasons_fn = (getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or
                           getattr(L, "nvmlDeviceGetCurrentClocksThrottleReasons", None))

    def sample(self):
        ct, L, h = self.ct, self.L, self.h
        clk, mx, mw, bits = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if (L.nvmlDeviceGetClockInfo(h, self.CLOCK_SM, ct.byref(clk)) != 0 or
                L.nvmlDeviceGetMaxClockInfo(h, self.CLOCK_SM, ct.byref(mx)) != 0):
            return None
        power = mw.value / 1000.0 if L.nvmlDeviceGetPowerUsage(h, ct.byref(mw)) == 0 else 0.0
        reasons = []
        if self.reasons_fn is not None and self.reasons_fn(h, ct.byref(bits)) == 0:
            reasons = [name for bit, name in self.REASON_BITS if bits.value & bit]
        return {"sm": float(clk.value), "max": float(mx.value), "power": power,
                "reasons": reasons}

    def close(self):
        self.L.nvmlShutdown()


class SmiSource:
    """One `nvidia-smi --query-gpu` call per sample (used where NVML cannot
    be loaded)."""

    name = "nvidia-smi"

    def __init__(self, index):
        self.index = index

    def sample(self):
        try:
            out = subprocess.run(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + SMI_FIELDS,
                                  "--format=csv,noheader,nounits"], capture_output=True, text=True,
                                 timeout=10).stdout
        except Exception:
            return None
        rows = [r for r in map(clock_row, out.splitlines()) if r]
        return rows[0] if rows else None

    def close(self):
        pass


class ClockSampler:
    """SM clock, power and clock-event reasons sampled DURING a timed region.

    Construct it before the warm-up, so that starting it does not leave the
    GPU idle (and its clock falling) just before the region. A background
    thread samples every period_ms. take_now() adds a sample from the
    caller: taken right after the region's steps are enqueued, while the GPU
    still runs them, it gives a region shorter than the period a sample from
    inside it. begin() and end() mark the region on the host clock (end()
    after the synchronise that closes it); stop() summarises the samples
    taken between the marks."""

    def __init__(self, source, period_ms=20):
        import threading
        self.source = source
        self.samples = []
        self.edges = {}
        self.lock = threading.Lock()
        self.t0 = self.t1 = None
        self.halt = threading.Event()
        self.period = period_ms / 1e3
        self.thread = threading.Thread(target=self._loop, daemon=True)
        self.thread.start()

    @classmethod
    def for_device(cls, dev, index):
        """NVML for torch device `dev` (matched by UUID, else NVML index
        `index`), else nvidia-smi; None if neither works."""
        import torch
        try:
            uuid = str(torch.cuda.get_device_properties(dev).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            uuid = None
        for make in (lambda: NvmlSource(uuid, index), lambda: SmiSource(index)):
            try:
                src = make()
            except Exception:
                continue
            try:
                if src.sample() is not None:
                    return cls(src)
            except Exception:
                pass
            src.close()
        return None

    def _take(self):
        t = time.perf_counter()
        r = self.source.sample()
        if r is not None:
            r["t"] = t
            with self.lock:
                self.samples.append(r)

    def _loop(self):
        while not self.halt.wait(self.period):
            self._take()

    def take_now(self):
        self._take()

    def take_edge(self, name):
        """One sample reported on its own (not in the region's summary): taken
        right before the region, while the warm-up steps still run, or right
        after it."""
        r = self.source.sample()
        if r is not None:
            self.edges[name] = {"sm_mhz": r["sm"], "reasons": r["reasons"]}

    def begin(self):
        self.t0 = time.perf_counter()

    def end(self):
        self.t1 = time.perf_counter()

    def stop(self):
        self.halt.set()
        self.thread.join(timeout=10)
        self.source.close()
        with self.lock:
            rows = [r for r in self.samples if self.t0 is not None and self.t1 is not None and
                    self.t0 <= r["t"] <= self.t1]
        out = summarise_clocks(rows)
        if out is not None:
            out["source"] = self.source.name
            out["window"] = "timed region (%.1f ms)" % ((self.t1 - self.t0) * 1e3)
            if self.edges:
                out["edges"] = self.edges
        return out


def clock_row(line):
    """One `nvidia-smi --query-gpu=<SMI_FIELDS> --format=csv,noheader,nounits`
    line as a sample dict, or None."""
    f = [x.strip() for x in line.split(",")]
    if len(f) < 9:
        return None
    try:
        row = dict(sm=float(f[1]), max=float(f[2]), power=float(f[3]))
    except ValueError:
        return None
    row["reasons"] = [name for k, name in ((5, "hw_slowdown"), (6, "hw_thermal_slowdown"),
                                           (7, "sw_thermal_slowdown"), (8, "sw_power_cap"))
                      if f[k].lower().startswith("active")]
    return row


def summarise_clocks(rows):
    """Median SM clock, max clock, max power, and the clock-event reasons seen
    active in any sample; None without samples."""
    if not rows:
        return None
    return {"sm_mhz": statistics.median(r["sm"] for r in rows),
            "sm_max_mhz": max(r["max"] for r in rows),
            "power_w_max": max(r["power"] for r in rows),
            "samples": len(rows),
            "reasons": sorted({name for r in rows for name in r["reasons"]})}


def parse_clock_lines(lines):
    """Summary of nvidia-smi sample lines (see clock_row)."""
    return summarise_clocks([r for r in map(clock_row, lines) if r])


# ------------------------------------------------------------------ distributed plumbing


def dist_setup():
    """(rank, world). Initialises torch.distributed when launched by torchrun."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """Max of a float over ranks (the slowest rank sets the job's time)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, elapsed_s_max, world):
    """Whole-job rate: the units all ranks processed over the slowest rank's time."""
    return units_per_rank * world / elapsed_s_max


# ------------------------------------------------------------------ the GPU arm


def make_sets(name, T_override, l2_bytes, device, N_override=0, H_override=0):
    import torch
    import synth
    w = dict(synth.WORKLOADS[name])
    if T_override:
        w["T"] = T_override
    if N_override:
        w["N"] = N_override
    if H_override:
        w["H"] = H_override
    T, H, N = w["T"], w["H"], w["N"]
    per_set = (N + 2) * T * H * 2 + H * 2  # resident bytes of one set (inputs + output)
    nsets = max(1, math.ceil(4 * l2_bytes / per_set))
    sets = []
    for k in range(nsets):
        p, r, g = synth.make_inputs(seed=k, **w)
        P = p.to(device)
        sets.append(dict(P=P, plist=[P[i] for i in range(N)], R=r.to(device), G=g.to(device),
                         out=torch.empty((T, H), dtype=torch.bfloat16, device=device)))
    torch.cuda.synchronize()
    return T, H, N, sets, per_set


NOMINAL_HBM_GBS = 8000.0  # GB300's nominal HBM3e bandwidth, about 8 TB/s
PRIME_CYCLES = 400_000     # ~0.2 ms at 2 GHz: the queue-priming delay before a timed region


def _median(xs):
    xs = sorted(xs)
    return xs[len(xs) // 2]


def after_gemm(tw, sets, eps, stream, H, N, reps=30):
    """The fused step timed right after its real predecessor in a layer: the
    row-parallel down projection of one rank, [T, 4H/N] x [4H/N, H] in bf16
    (torch.matmul, cuBLAS), writing partial 0 of the set the step then reads.
    Per rep, events around GEMM + fused step and, in a separate pass, around
    the GEMM alone; the step's time is the difference of the medians."""
    import torch
    T = sets[0]["R"].shape[0]
    K = 4 * H // N
    dev = sets[0]["R"].device
    gen = torch.Generator(device=dev).manual_seed(7)
    x = torch.randn((T, K), generator=gen, device=dev).to(torch.bfloat16)
    w = (torch.randn((K, H), generator=gen, device=dev) * K ** -0.5).to(torch.bfloat16)
    fcalls = [tw.FusedCall(s["plist"], s["R"], s["G"], eps, s["out"], stream=stream) for s in sets]

    def gemm(k):
        torch.matmul(x, w, out=sets[k % len(sets)]["P"][0])

    def timed(fused):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        with torch.cuda.stream(stream):
            for k in range(3):
                gemm(k)
                if fused:
                    fcalls[k % len(fcalls)]()
            for k in range(reps):
                evs[k][0].record(stream)
                gemm(k)
                if fused:
                    fcalls[k % len(fcalls)]()
                evs[k][1].record(stream)
        torch.cuda.synchronize()
        return _median(a.elapsed_time(b) * 1e3 for a, b in evs)

    pair_us = timed(True)
    gemm_us = timed(False)
    return {"pair_us": round(pair_us, 3), "gemm_us": round(gemm_us, 3),
            "fused_us": round(pair_us - gemm_us, 3),
            "gemm": "[%d,%d]x[%d,%d] bf16 torch.matmul" % (T, K, K, H), "reps": reps}


def compact_sweep(tw, dev, l2, peak, reps=20):
    """The rest of the metric in the default line: GB/s and tokens/s at
    T = 1024 / 4096 / 16384 on the whole GPU, and GB/s per SM at SM budgets
    2 / 4 / 8 / 16 for T = 8192 (H = 8192, N = 8), plus N = 2 and N = 12 at
    an 8-SM budget (T = 4096), and two small batches on the whole GPU that
    take the direct form: T = 128 (H = 8192, N = 8; one row per CTA) and
    T = 304 (H = 4096, N = 8; one CTA per row, two per SM). Inputs are made on the
    device from a seeded generator with the workload's distributions (this
    measures time only; parity runs on the synthetic CPU inputs). Each cell
    times `reps` prepared launches back to back between one event pair, and
    the median of per-launch event pairs over the same launches; inputs
    rotate over enough sets to exceed 4x the L2, or one set is already larger
    than that."""
    import torch
    eps = 1e-5
    gen = torch.Generator(device=dev).manual_seed(0)

    def make(T, N, H):
        per_set = (N + 2) * T * H * 2
        out = []
        for _ in range(max(1, math.ceil(4 * l2 / per_set))):
            P = torch.empty((N, T, H), dtype=torch.bfloat16, device=dev)
            for r in range(N):
                P[r] = torch.randn((T, H), generator=gen, device=dev) * 0.02
            R = torch.randn((T, H), generator=gen, device=dev).to(torch.bfloat16)
            G = (torch.randn((H,), generator=gen, device=dev) * 0.1 + 1).to(torch.bfloat16)
            out.append(dict(P=P, R=R, G=G, out=torch.empty_like(R)))
        return out

    stream = torch.cuda.Stream(dev)
    stream.wait_stream(torch.cuda.current_stream(dev))

    def cell(sets, T, N, H, budget):
        calls = [tw.FusedCall(s["P"], s["R"], s["G"], eps, s["out"], stream=stream,
                              sm_budget=budget) for s in sets]
        with torch.cuda.stream(stream):
            for k in range(3):
                calls[k % len(calls)]()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for k in range(reps):
                calls[k % len(calls)]()
            b.record(stream)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(reps)]
            for k in range(reps):
                evs[k][0].record(stream)
                calls[k % len(calls)]()
                evs[k][1].record(stream)
        torch.cuda.synchronize()
        b2b = a.elapsed_time(b) * 1e3 / reps
        per = _median(x.elapsed_time(y) * 1e3 for x, y in evs)
        nbytes = tw.bytes_per_call(T, H, N)
        shape = tw.tw_launch_shape(T, H, N, budget)
        used = min(shape["grid"], tw_sms)
        form = {256: "direct", 288: "ring", 544: "two pipelines"}.get(shape["threads"], "?")
        gbs = nbytes / b2b / 1e3
        return {"T": T, "H": H, "N": N, "sm_budget": budget or "full", "sms_used": used,
                "ctas": shape["grid"], "form": form,
                "us_b2b": round(b2b, 2), "GB_s": round(gbs, 1), "frac": round(gbs / peak, 4),
                "GB_s_per_sm": round(gbs / used, 2), "tokens_per_s": round(T / b2b * 1e6, 1),
                "us_per_launch": round(per, 2),
                "GB_s_per_launch": round(nbytes / per / 1e3, 1)}

    tw_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    cells = []
    # N = 8 over T and budgets; N = 2 and 12 under an 8-SM budget, where the
    # launch takes the two-pipeline forms; two small batches in the direct form
    for T, N, H, budgets in ((1024, 8, 8192, (0,)), (4096, 8, 8192, (0,)),
                             (16384, 8, 8192, (0,)), (8192, 8, 8192, (2, 4, 8, 16, 0)),
                             (4096, 2, 8192, (8,)), (4096, 12, 8192, (8,)),
                             (128, 8, 8192, (0,)), (304, 8, 4096, (0,))):
        sets = make(T, N, H)
        torch.cuda.synchronize()
        for budget in budgets:
            cells.append(cell(sets, T, N, H, budget))
        del sets
    torch.cuda.current_stream(dev).wait_stream(stream)
    torch.cuda.empty_cache()
    return {"reps": reps, "cells": cells,
            "timing": "us_b2b: launches back to back between one event pair (GB_s, frac, "
                      "GB_s_per_sm, tokens_per_s); us_per_launch: median of an event pair "
                      "around each launch (launch latency included)"}


def gpu_arm(args, rank, world):
    import torch
    import reduce_rmsnorm_gb300 as tw
    from reduce_rmsnorm_gb300 import build

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    build.build()
    tw.lib()
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    l2 = props.L2_cache_size
    T, H, N, sets, per_set = make_sets(args.workload, args.tokens, l2, dev)
    eps = 1e-5
    C = ctas_unsplit(T, H)
    bytes_step = tw.bytes_per_call(T, H, N)
    sa = torch.cuda.Stream(dev)  # launching stream (a created stream, so graphs can capture it)
    sb = torch.cuda.Stream(dev)
    calls = [tw.SplitCall(s["plist"], s["R"], s["G"], eps, s["out"], sa, sb, args.sm_budget)
             for s in sets]
    # eager steps: one C call plans the split (every step) and runs it
    planned = [tw.PlannedSplitCall(C, PLANNER_SMS, s["plist"], s["R"], s["G"], eps, s["out"], sa,
                                   sb, args.sm_budget) for s in sets]
    graphs = {}

    planner = tw.WaveSplitCall(C, PLANNER_SMS)

    def plan():
        return planner(T)[0]

    def step_eager(k):
        planned[k % len(planned)]()

    def step_graph(k):
        # the plan is computed every step; the graph captured for this input
        # set and this plan is replayed (captured on first use)
        key = (k % len(calls), plan())
        g = graphs.get(key)
        if g is None:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=sa):
                calls[key[0]](key[1])
            graphs[key] = g
        g.replay()

    step = step_graph if args.mode == "graph" else step_eager
    # started before the warm-up: starting it later would idle the GPU
    clocks = ClockSampler.for_device(dev, local) if rank == 0 else None
    sa.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(sa):
        for k in range(max(args.warmup, len(calls))):
            step_eager(k)
        # graph mode captures one graph per input set on first use: warm every
        # set's graph here, so no capture falls inside the timed region
        for k in range(max(args.warmup, len(calls)) if args.mode == "graph" else args.warmup):
            step(k)
    if clocks:
        clocks.take_edge("before")  # the warm-up steps are still running
    torch.cuda.synchronize()
    prefix, suffix = tw.tw_wave_split(T, C, PLANNER_SMS)
    launches_per_step = (1 if prefix > 0 else 0) + (1 if suffix > 0 else 0)

    # timed region: K steps back to back, events on the launching stream only
    barrier(world)
    torch.cuda.synchronize()
    graphs_before = len(graphs)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if clocks:
        clocks.begin()
    with torch.cuda.stream(sa):
        # A device-side delay ahead of the first event primes the launch queue:
        # while it runs the host enqueues the first steps, so the region times
        # the device running K steps back to back, not the host's first enqueue
        # of an idle GPU (a short region otherwise carries ~10-20 us of it).
        torch.cuda._sleep(PRIME_CYCLES)
        t_start.record(sa)
        for k in range(args.steps):
            step(args.warmup + k)
        t_end.record(sa)
    if clocks and not t_end.query():
        clocks.take_now()  # the GPU is still running the timed steps
    torch.cuda.synchronize()
    if clocks:
        clocks.end()
        clocks.take_edge("after")
    barrier(world)
    clk = clocks.stop() if clocks else None
    elapsed_ms = t_start.elapsed_time(t_end)
    elapsed_ms_max = max_over_ranks(elapsed_ms, world)
    captures_in_region = len(graphs) - graphs_before
    value_gbs = job_throughput(bytes_step * args.steps, elapsed_ms_max / 1e3, world) / 1e9
    mean_step_ms = elapsed_ms / args.steps

    # per-step distribution (separate pass: events between steps would
    # serialise the programmatic launch of the next step)
    n_dist = min(max(args.steps, 50), 500)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_dist)]
    with torch.cuda.stream(sa):
        for k in range(n_dist):
            evs[k][0].record(sa)
            step(k)
            evs[k][1].record(sa)
    torch.cuda.synchronize()
    step_us = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)

    # the unfused baseline (reduce -> HBM -> residual add + RMSNorm) on the same
    # rotating sets, timed the same way, for the fusion ratio
    unfused = None
    if not args.no_unfused:
        ucalls = [tw.UnfusedCall(s["plist"], s["R"], s["G"], eps, s["out"], sa) for s in sets]
        n_u = min(args.steps, 2000)
        with torch.cuda.stream(sa):
            for k in range(max(args.warmup, len(ucalls))):
                ucalls[k % len(ucalls)]()
            u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            u0.record(sa)
            for k in range(n_u):
                ucalls[k % len(ucalls)]()
            u1.record(sa)
        torch.cuda.synchronize()
        u_ms = u0.elapsed_time(u1) / n_u
        u_bytes = (N + 5) * T * H * 2 + H * 2
        unfused = {"us_per_step": round(u_ms * 1e3, 3), "steps": n_u, "launches_per_step": 2,
                   "hbm_bytes_per_step": u_bytes,
                   "GB_s_on_fused_bytes": round(bytes_step / (u_ms / 1e3) / 1e9, 2),
                   "GB_s_on_own_bytes": round(u_bytes / (u_ms / 1e3) / 1e9, 2),
                   "fused_speedup": round(u_ms / mean_step_ms, 4)}
    peak, peak_src = peak_hbm()
    gemm_pair = sweep_block = None
    if rank == 0 and not args.no_extras:
        gemm_pair = after_gemm(tw, sets, eps, sa, H, N)
        sweep_block = compact_sweep(tw, dev, l2, peak)
    assert tw.tw_device_status(reset=True) == 0, "a kernel gave up on a bounded wait"

    achieved = bytes_step / (mean_step_ms / 1e3) / 1e9
    per_launch_us = step_us[len(step_us) // 2]
    traffic = ncu_traffic(args.workload if not args.tokens else None)

    result = None
    if rank == 0:
        e2e = e2e_arm(args, tw, T, H, N, eps, C, dev, sa, sb)
        cpu = None if args.no_cpu_baseline or world > 1 else cpu_baseline(args.workload, args.tokens)
        cpu_procs = None
        if cpu is not None:
            cpu_procs = cpu_baseline_procs(args.workload, args.tokens, cpu.pop("t_row_s"))
        result = {
            "metric": METRIC, "value": round(value_gbs, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(elapsed_ms_max / args.steps, 6), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16",
            "data": "synthetic (seeded N(0,sigma^2) partials, N(0,1) residual, N(1,0.1^2) gamma)",
            "config": {"workload": args.workload, "T": T, "H": H, "N": N, "eps": eps,
                       "sm_budget": args.sm_budget, "plan": [prefix, suffix],
                       "launch": "cuda graph per (input set, plan); plan computed every step"
                                 if args.mode == "graph" else
                                 "eager prepared calls, programmatic dependent launch",
                       "graph_captures_in_region": captures_in_region,
                       "queue": "a device-side delay before the first event primes the launch "
                                "queue (the region times device execution of the K steps)",
                       "planner": {"ctas_unsplit": C, "num_sms": PLANNER_SMS},
                       "parallelism": "replicas" if world > 1 else "single-gpu",
                       "l2": "rotating %d input sets, %.1f MB total (L2 %.1f MB): inputs larger "
                             "than 4x L2" % (len(sets), len(sets) * per_set / 1e6, l2 / 1e6)},
            "tokens_per_s": round(T * args.steps * world / (elapsed_ms_max / 1e3), 1),
            "hbm_frac": round(value_gbs / peak, 4),
            "hbm_frac_nominal": round(value_gbs / NOMINAL_HBM_GBS, 4),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                         "peak_source": peak_src, "per": "launch (one fused call per step)"
                         if launches_per_step == 1 else "step (%d concurrent launches)"
                         % launches_per_step,
                         "algorithmic_bytes": bytes_step,
                         "duration": "mean over the timed region's %d steps" % args.steps,
                         "frac_per_launch": round(bytes_step / per_launch_us / 1e3 / peak, 4),
                         "frac_per_launch_note": "median of an event pair around each step "
                                                 "(step_us), launch latency included",
                         "frac_after_gemm": None if gemm_pair is None else
                         round(bytes_step / gemm_pair["fused_us"] / 1e3 / peak, 4),
                         "after_gemm": gemm_pair,
                         "nominal_peak": NOMINAL_HBM_GBS,
                         "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4)},
            "step_us": {"median": round(step_us[len(step_us) // 2], 3),
                        "p10": round(step_us[len(step_us) // 10], 3),
                        "p90": round(step_us[(9 * len(step_us)) // 10], 3),
                        "n": n_dist, "note": "events around each step (separate pass)"},
            "unfused": unfused, "cpu_baseline": cpu, "cpu_baseline_procs": cpu_procs, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "sweep": sweep_block,
        }
    return result


def e2e_arm(args, tw, T, H, N, eps, C, dev, sa, sb):
    """End to end through the public API with host buffers. Every step copies
    its inputs (N partials, residual, gamma) from pinned host memory, plans,
    runs the fused step, and copies the updated residual and the output back
    to pinned host memory. Steps are pipelined the way a serving loop would
    run them: two device buffer sets, H2D on one stream, compute on another,
    D2H on a third, so step k's D2H overlaps step k+1's H2D (events order
    every reuse of a buffer set)."""
    import torch
    import synth
    w = dict(synth.WORKLOADS[args.workload])
    if args.tokens:
        w["T"] = args.tokens
    p, r, g = synth.make_inputs(seed=100, **w)
    hp, hr, hg = p.pin_memory(), r.pin_memory(), g.pin_memory()
    hr_out = torch.empty_like(hr).pin_memory()
    hy_out = torch.empty_like(hr).pin_memory()
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    bufs = []
    for _ in range(2):
        P = torch.empty_like(p, device=dev)
        R = torch.empty_like(r, device=dev)
        G = torch.empty_like(g, device=dev)
        out = torch.empty_like(R)
        bufs.append(dict(P=P, R=R, G=G, out=out,
                         call=tw.PlannedSplitCall(C, PLANNER_SMS, [P[i] for i in range(N)], R,
                                                  G, eps, out, sa, sb, args.sm_budget),
                         loaded=torch.cuda.Event(), computed=torch.cuda.Event(),
                         drained=torch.cuda.Event()))
    steps = max(3, min(args.e2e_steps, args.steps))

    def step(k):
        b = bufs[k % 2]
        s_h2d.wait_event(b["drained"])        # the set's previous results are back on the host
        with torch.cuda.stream(s_h2d):
            b["P"].copy_(hp, non_blocking=True)
            b["R"].copy_(hr, non_blocking=True)
            b["G"].copy_(hg, non_blocking=True)
            b["loaded"].record(s_h2d)
        sa.wait_event(b["loaded"])
        b["call"]()
        b["computed"].record(sa)
        s_d2h.wait_event(b["computed"])
        with torch.cuda.stream(s_d2h):
            hr_out.copy_(b["R"], non_blocking=True)
            hy_out.copy_(b["out"], non_blocking=True)
            b["drained"].record(s_d2h)

    for b in bufs:
        b["drained"].record(s_d2h)
    for k in range(3):
        step(k)
    torch.cuda.synchronize()
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_h2d)
    for k in range(steps):
        step(k)
    s_h2d.wait_stream(s_d2h)
    e.record(s_h2d)
    torch.cuda.synchronize()
    ms = a.elapsed_time(e) / steps

    def copies_only(k):
        # the same transfers in the same pipeline, without the fused step
        b = bufs[k % 2]
        s_h2d.wait_event(b["drained"])
        with torch.cuda.stream(s_h2d):
            b["P"].copy_(hp, non_blocking=True)
            b["R"].copy_(hr, non_blocking=True)
            b["G"].copy_(hg, non_blocking=True)
            b["loaded"].record(s_h2d)
        s_d2h.wait_event(b["loaded"])
        with torch.cuda.stream(s_d2h):
            hr_out.copy_(b["R"], non_blocking=True)
            hy_out.copy_(b["out"], non_blocking=True)
            b["drained"].record(s_d2h)

    for k in range(3):
        copies_only(k)
    torch.cuda.synchronize()
    a.record(s_h2d)
    for k in range(steps):
        copies_only(k)
    s_h2d.wait_stream(s_d2h)
    e.record(s_h2d)
    torch.cuda.synchronize()
    link_ms = a.elapsed_time(e) / steps
    h2d = (N + 1) * T * H * 2 + H * 2
    d2h = 2 * T * H * 2
    return {"value": round(tw.bytes_per_call(T, H, N) / (ms / 1e3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(ms, 4),
            "pipeline": "2 device buffer sets; H2D, compute and D2H on separate streams",
            "h2d_GB_s": round(h2d / (ms / 1e3) / 1e9, 1),
            "link_bound": {"ms_per_step": round(link_ms, 4),
                           "GB_s": round(tw.bytes_per_call(T, H, N) / (link_ms / 1e3) / 1e9, 2),
                           "frac": round(link_ms / ms, 4),
                           "what": "the same copies in the same pipeline without the fused step"}}


# ------------------------------------------------------------------ the CPU oracle


def _oracle_rows_timer(workload, T_override):
    """Returns (T, H, N, time_rows(n) -> seconds) over the workload's first rows."""
    import synth
    from oracle import fused
    w = dict(synth.WORKLOADS[workload])
    if T_override:
        w["T"] = T_override
    T, H, N = w["T"], w["H"], w["N"]

    def sample(n_rows, seed=0):
        ww = dict(w)
        ww["T"] = n_rows
        p, r, g = synth.make_inputs(seed=seed, **ww)
        return synth.bits(p), synth.bits(r), synth.bits(g)

    def time_bits(bits):
        pb, rb, gb = bits
        t0 = time.perf_counter()
        fused.reduce_residual_rmsnorm(pb, rb, gb, 1e-5)
        fused.residual_fp32_rank_order(pb, rb)
        return time.perf_counter() - t0

    def time_rows(n_rows, seed=0):
        return time_bits(sample(n_rows, seed))

    time_rows.sample = sample
    time_rows.time_bits = time_bits
    return T, H, N, time_rows


def cpu_baseline(workload, T_override, budget_s=10.0):
    """The oracle as it stands, on a bounded sample of the workload's rows."""
    import reduce_rmsnorm_gb300 as tw
    T, H, N, time_rows = _oracle_rows_timer(workload, T_override)
    t1 = time_rows(8) / 8
    rows = int(max(1, min(T, budget_s / max(t1, 1e-6) / 1.2)))
    secs = time_rows(rows)
    gbs = tw.bytes_per_call(rows, H, N) / secs / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "first %d of %d token rows of %s (fp64 NumPy oracle, one process), %.1f s"
                      % (rows, T, workload, secs),
            "t_row_s": secs / rows}


def _oracle_shard_worker(workload, T_override, rows, seed, barrier, queue):
    """One worker of the multi-process oracle timing: builds its shard's
    inputs, waits for the others, then times the oracle on its rows."""
    try:
        import synth
        from oracle import fused
        w = dict(synth.WORKLOADS[workload])
        w["T"] = rows
        p, r, g = synth.make_inputs(seed=seed, **w)
        pb, rb, gb = synth.bits(p), synth.bits(r), synth.bits(g)
        barrier.wait(timeout=600)
        t0 = time.perf_counter()  # CLOCK_MONOTONIC: comparable across processes
        fused.reduce_residual_rmsnorm(pb, rb, gb, 1e-5)
        fused.residual_fp32_rank_order(pb, rb)
        queue.put((t0, time.perf_counter()))
    except Exception as e:  # reported by the parent as a missing figure
        queue.put(("error", repr(e)))


def cpu_baseline_procs(workload, T_override, t_row_s, budget_s=10.0):
    """The oracle over token shards in one spawned process per host core: the
    workload's rows (or as many as fit the budget) split into P contiguous
    shards. Returns None if a worker fails."""
    import multiprocessing as mp
    import queue as queue_mod
    import reduce_rmsnorm_gb300 as tw
    import synth
    w = synth.WORKLOADS[workload]
    T = T_override or w["T"]
    P = len(os.sched_getaffinity(0))
    rows_total = int(max(1, min(T, P * budget_s / max(t_row_s, 1e-6))))
    per = [rows_total // P + (1 if i < rows_total % P else 0) for i in range(P)]
    per = [n for n in per if n > 0]
    ctx = mp.get_context("spawn")  # the parent has a CUDA context: never fork
    bar, q = ctx.Barrier(len(per)), ctx.Queue()
    procs = [ctx.Process(target=_oracle_shard_worker, args=(workload, T_override, n, i, bar, q))
             for i, n in enumerate(per)]
    for pr in procs:
        pr.start()
    spans = []
    try:
        for _ in procs:
            spans.append(q.get(timeout=900))
    except queue_mod.Empty:
        spans.append(("error", "timeout"))
    for pr in procs:
        pr.join(timeout=60)
        if pr.is_alive():
            pr.kill()
    if any(sp[0] == "error" for sp in spans):
        return None
    wall = max(e for _, e in spans) - min(s0 for s0, _ in spans)
    return {"value": round(tw.bytes_per_call(rows_total, w["H"], w["N"]) / wall / 1e9, 4),
            "unit": "GB/s", "cores": len(per), "kind": "oracle",
            "sample": "%d of %d token rows of %s in %d contiguous shards, one spawned process "
                      "per shard (fp64 NumPy oracle), %.2f s wall" % (
                          rows_total, T, workload, len(per), wall)}


def reference_arm(args, rank, world):
    """The oracle timed on the host cores as the reference arm: each step runs
    the oracle on a bounded sample of the workload's rows."""
    if rank != 0:
        return None
    import reduce_rmsnorm_gb300 as tw
    T, H, N, time_rows = _oracle_rows_timer(args.workload, args.tokens)
    # cost of one oracle call on n rows ~ fixed + n * per_row, both measured,
    # so that many short steps also fit the budget
    t8 = time_rows(8)
    t1 = time_rows(1)
    per_row = max((t8 - t1) / 7, 1e-7)
    fixed = max(t1 - per_row, 0.0)
    total_budget_s = 90.0
    per_step = total_budget_s / (args.steps + args.warmup)
    rows = int(max(1, min(T, (per_step - fixed) / per_row)))
    bits = time_rows.sample(rows)   # one sample, timed every step
    for _ in range(args.warmup):
        time_rows.time_bits(bits)
    secs = [time_rows.time_bits(bits) for _ in range(args.steps)]
    total = sum(secs)
    value = tw.bytes_per_call(rows, H, N) * args.steps / total / 1e9
    sample = ("the same %d of %d token rows of %s every step (fp64 NumPy oracle, one process)"
              % (rows, T, args.workload))
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "T": T, "H": H, "N": N, "eps": 1e-5,
                       "rows_per_step": rows},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


# ------------------------------------------------------------------ SM-budget sweep


def sweep(args):
    """GB/s and GB/s per SM for T = 512..16384 and budgets 2/4/8/16/full
    (H=8192, N=8 unless --sweep-hidden / --sweep-partials say otherwise); one
    JSON line per cell. The headline figure per cell is the
    median of per-launch CUDA events (launch latency included); b2b_us and
    graph_us are the mean per launch over the same launches issued back to
    back eagerly and replayed from one CUDA graph. All three launch prepared
    calls (FusedCall), so argument marshalling is not timed."""
    import torch
    import reduce_rmsnorm_gb300 as tw
    from reduce_rmsnorm_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peak, _ = peak_hbm()
    tokens = [int(t) for t in args.sweep_tokens.split(",")]
    budgets = [int(b) for b in args.sweep_budgets.split(",")]
    partials = [int(n) for n in args.sweep_partials.split(",")]
    hiddens = [int(h) for h in args.sweep_hidden.split(",")]
    for T, Nsw, Hsw in [(t, n, h) for h in hiddens for t in tokens for n in partials]:
        T_, H, N, sets, per_set = make_sets("llama70b_t1024_h8192_n8", T, l2, dev, Nsw, Hsw)
        bytes_call = tw.bytes_per_call(T, H, N)
        for budget in budgets:
            reps = args.sweep_reps
            # prepared calls: marshalling and argument checks stay outside the
            # timed regions
            ss = torch.cuda.Stream(dev)
            ss.wait_stream(torch.cuda.current_stream(dev))
            fcalls = [tw.FusedCall(s["plist"], s["R"], s["G"], 1e-5, s["out"], stream=ss,
                                   sm_budget=budget) for s in sets]
            with torch.cuda.stream(ss):
                for k in range(3):
                    fcalls[k % len(fcalls)]()
                torch.cuda.synchronize()
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(reps)]
                for k in range(reps):
                    evs[k][0].record(ss)
                    fcalls[k % len(fcalls)]()
                    evs[k][1].record(ss)
            torch.cuda.synchronize()
            us = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
            med = us[len(us) // 2]
            ctas = tw.tw_launch_shape(T, H, N, budget)["grid"]
            used = min(ctas, sms)  # more CTAs than SMs: one direct CTA per row
            gbs = bytes_call / (med / 1e6) / 1e9
            # launch-overhead context: the same launches back to back (eager,
            # programmatic dependent launch) and replayed from one CUDA graph

            def launch(k):
                fcalls[k % len(fcalls)]()

            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(ss):
                a.record(ss)
                for k in range(reps):
                    launch(k)
                b.record(ss)
                torch.cuda.synchronize()
                b2b_us = a.elapsed_time(b) * 1e3 / reps
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=ss):
                    for k in range(reps):
                        launch(k)
                g.replay()
                torch.cuda.synchronize()
                a.record(ss)
                g.replay()
                b.record(ss)
                torch.cuda.synchronize()
                graph_us = a.elapsed_time(b) * 1e3 / reps
            del g
            torch.cuda.current_stream(dev).wait_stream(ss)
            extra = {"b2b_us": round(b2b_us, 2), "b2b_GB_s": round(bytes_call / b2b_us / 1e3, 1),
                     "graph_us": round(graph_us, 2),
                     "graph_GB_s": round(bytes_call / graph_us / 1e3, 1)}
            if budget == 0:
                ucalls = [tw.UnfusedCall(s["plist"], s["R"], s["G"], 1e-5, s["out"]) for s in sets]
                for k in range(3):
                    ucalls[k % len(ucalls)]()
                torch.cuda.synchronize()
                uevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                        for _ in range(reps)]
                for k in range(reps):
                    uevs[k][0].record()
                    ucalls[k % len(ucalls)]()
                    uevs[k][1].record()
                torch.cuda.synchronize()
                uus = sorted(a.elapsed_time(b) * 1e3 for a, b in uevs)[reps // 2]
                extra.update({"unfused_us_median": round(uus, 2),
                              "fused_speedup": round(uus / med, 3)})
            print(json.dumps({"T": T, "H": H, "N": N, "sm_budget": budget or "full",
                              "sms_used": used, "ctas": ctas, "us_median": round(med, 2),
                              "us_p10": round(us[len(us) // 10], 2),
                              "us_p90": round(us[(9 * len(us)) // 10], 2),
                              "GB_s": round(gbs, 1), "GB_s_per_sm": round(gbs / used, 2),
                              "hbm_frac": round(gbs / peak, 4),
                              "tokens_per_s": round(T / (med / 1e6), 1), "sms": sms, **extra}),
                  flush=True)
        del sets
        torch.cuda.empty_cache()
    assert tw.tw_device_status(reset=True) == 0


# ------------------------------------------------------------------ co-run with a GEMM


class GemmPipeline:
    """One tensor-parallel layer's tail on one GPU: the row-parallel down
    projection of one rank, [T, 4H/N] x [4H/N, H] in bf16 (torch.matmul,
    cuBLAS), writes partial 0; partials 1..N-1 stand for the other ranks'
    contributions already in HBM. forward(prefix) runs, as the pages' guide
    pipelines it:

      stream A (compute):            GEMM(rows [0,p)) -> GEMM(rows [p,T))
      stream B (high priority, k SMs): fused(rows [0,p)) after GEMM(prefix),
                                     fused(rows [p,T)) after GEMM(suffix)

    prefix == T is the unsplit forward: GEMM(T) then the fused step."""

    def __init__(self, T, H=8192, N=8, sm_budget=0, seed=0):
        import torch
        import synth
        dev = torch.device("cuda", 0)
        self.T, self.H, self.N, self.budget, self.eps = T, H, N, sm_budget, 1e-5
        K = 4 * H // N
        p, r, g = synth.make_inputs(T, H, N, 0.02, seed=seed)
        self.P, self.R, self.G = p.to(dev), r.to(dev), g.to(dev)
        gen = torch.Generator(device=dev).manual_seed(seed)
        self.x = torch.randn((T, K), generator=gen, device=dev).to(torch.bfloat16)
        self.w = (torch.randn((K, H), generator=gen, device=dev) * K ** -0.5).to(torch.bfloat16)
        self.out = torch.empty_like(self.R)
        self.sa = torch.cuda.Stream(dev, priority=0)
        self.sb = torch.cuda.Stream(dev, priority=-1)
        self.gemm_shape = "[%d,%d]x[%d,%d] bf16" % (T, K, K, H)
        torch.cuda.synchronize()

    def gemm(self, a, b):
        import torch
        if b > a:
            torch.matmul(self.x[a:b], self.w, out=self.P[0, a:b])

    def forward(self, prefix):
        import torch
        import reduce_rmsnorm_gb300 as tw
        sa, sb = self.sa, self.sb
        e1, e2 = torch.cuda.Event(), torch.cuda.Event()
        sb.wait_stream(sa)
        with torch.cuda.stream(sa):
            self.gemm(0, prefix)
            e1.record(sa)
            self.gemm(prefix, self.T)
            e2.record(sa)
        tw.tw_run_split_after(prefix, self.P, self.R, self.G, self.eps, self.out, sb, e1, e2,
                              sm_budget=self.budget)
        sa.wait_stream(sb)

    def serial(self):
        import torch
        import reduce_rmsnorm_gb300 as tw
        with torch.cuda.stream(self.sa):
            self.gemm(0, self.T)
            tw.tw_fused_reduce_residual_rmsnorm(self.P, self.R, self.G, self.eps, self.out,
                                                stream=self.sa)

    def timed(self, fn, reps):
        """Median microseconds of fn() on stream A (events on A; A joins B)."""
        import torch
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        out = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(self.sa)
            fn()
            b.record(self.sa)
            torch.cuda.synchronize()
            out.append(a.elapsed_time(b) * 1e3)
        return sorted(out)[len(out) // 2]


def corun(args):
    """The split pipelined against the projection that produces the partials
    (one JSON line per token count and SM budget):

      serial    GEMM(T) then the fused step on the whole GPU, one stream
      overlap   GemmPipeline.forward with the planner's split at the budget
      equal     the same with prefix = T/2
      model     T_GEMM(p) + max(T_GEMM(T-p), T_FUSED(p)) + T_FUSED(T-p), the
                overlap formula of the pages' guide, from the pieces timed alone
      gemm_slowdown   GEMM(T) time while a long fused call runs at the budget,
                      over GEMM(T) alone"""
    import torch
    import reduce_rmsnorm_gb300 as tw
    import synth
    from reduce_rmsnorm_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    reps = args.corun_reps
    cover = synth.make_inputs(4096, 8192, 8, 0.02, seed=1)
    Pc, Rc, Gc = cover[0].to(dev), cover[1].to(dev), cover[2].to(dev)
    outc = torch.empty_like(Rc)
    for T in [int(t) for t in args.corun_tokens.split(",")]:
        for budget in [int(b) for b in args.corun_budgets.split(",")]:
            pipe = GemmPipeline(T, sm_budget=budget, seed=T)
            C = ctas_unsplit(T, pipe.H)
            plan_p = tw.tw_wave_split(T, C, PLANNER_SMS)[0]

            def fused_rows(a, b):
                def run():
                    if b > a:
                        tw.tw_fused_reduce_residual_rmsnorm(
                            pipe.P[:, a:b], pipe.R[a:b], pipe.G, pipe.eps, pipe.out[a:b],
                            stream=pipe.sa, sm_budget=budget)
                return run

            def gemm_rows(a, b):
                def run():
                    with torch.cuda.stream(pipe.sa):
                        pipe.gemm(a, b)
                return run

            def gemm_beside_fused():
                pipe.sb.wait_stream(pipe.sa)
                tw.tw_fused_reduce_residual_rmsnorm(Pc, Rc, Gc, pipe.eps, outc, stream=pipe.sb,
                                                    sm_budget=budget)
                with torch.cuda.stream(pipe.sa):
                    pipe.gemm(0, T)

            t_serial = pipe.timed(pipe.serial, reps)
            t_overlap = pipe.timed(lambda: pipe.forward(plan_p), reps)
            t_equal = pipe.timed(lambda: pipe.forward(T // 2), reps)
            g_p, g_s = pipe.timed(gemm_rows(0, plan_p), reps), pipe.timed(gemm_rows(plan_p, T), reps)
            f_p, f_s = pipe.timed(fused_rows(0, plan_p), reps), pipe.timed(fused_rows(plan_p, T), reps)
            g_all = pipe.timed(gemm_rows(0, T), reps)
            g_beside = pipe.timed(gemm_beside_fused, reps) if budget else None
            model = g_p + max(g_s, f_p) + f_s
            print(json.dumps({
                "T": T, "H": pipe.H, "N": pipe.N, "gemm": pipe.gemm_shape,
                "sm_budget": budget or "full", "plan": [plan_p, T - plan_p],
                "serial_us": round(t_serial, 2), "overlap_us": round(t_overlap, 2),
                "equal_split_us": round(t_equal, 2),
                "speedup_vs_serial": round(t_serial / t_overlap, 3),
                "model_us": round(model, 2),
                "pieces_us": {"gemm_prefix": round(g_p, 2), "gemm_suffix": round(g_s, 2),
                              "fused_prefix": round(f_p, 2), "fused_suffix": round(f_s, 2),
                              "gemm_all": round(g_all, 2)},
                "gemm_slowdown": None if g_beside is None else round(g_beside / g_all, 3)}),
                flush=True)
            del pipe
            torch.cuda.empty_cache()
    assert tw.tw_device_status(reset=True) == 0


def offset_sweep(args):
    """The pages' offline selection rule ("Fix one" of the wave-arithmetic
    blog): for each token count, time a forward for every candidate split
    (no split, and half -/+ each offset of the grid below half), keep the
    fastest as the lookup table's entry, and compare it with the planner's
    wave-constraint choice. One JSON line per token count, then the table."""
    import torch
    import reduce_rmsnorm_gb300 as tw
    from reduce_rmsnorm_gb300 import build
    build.build()
    table = {}
    agree = 0
    tokens = [int(t) for t in args.sweep_offsets_tokens.split(",")]
    for T in tokens:
        pipe = GemmPipeline(T, sm_budget=args.sm_budget, seed=T)
        half = T // 2
        cands = [T] + sorted({half - o for o in tw.DEFAULT_OFFSETS if o < half} |
                             {half + o for o in tw.DEFAULT_OFFSETS if o < half})
        times = {p: pipe.timed(lambda p=p: pipe.forward(p), args.corun_reps) for p in cands}
        # fastest; ties (within 0.5%) go to the smaller |p - half|, then the smaller prefix
        best_t = min(times.values())
        best = min((p for p in cands if times[p] <= best_t * 1.005),
                   key=lambda p: (abs(p - half) if p != T else T, p))
        plan = tw.tw_wave_split(T, ctas_unsplit(T, pipe.H), PLANNER_SMS)[0]
        agree += int(plan == best)
        table[T] = best
        print(json.dumps({"T": T, "sm_budget": args.sm_budget or "full",
                          "table_prefix": best, "table_us": round(times[best], 2),
                          "planner_prefix": plan, "planner_us": round(times[plan], 2)
                          if plan in times else None,
                          "planner_loss": round(times[plan] / times[best], 4)
                          if plan in times else None,
                          "equal_us": round(times[half], 2), "unsplit_us": round(times[T], 2),
                          "candidates_us": {str(p): round(t, 2) for p, t in sorted(times.items())}}),
              flush=True)
        del pipe
        torch.cuda.empty_cache()
    print(json.dumps({"table": {str(k): v for k, v in table.items()},
                      "planner_agrees": agree, "of": len(tokens)}), flush=True)
    assert tw.tw_device_status(reset=True) == 0


# ------------------------------------------------------------------ host link


def link_probe(args):
    """Copy-engine bandwidth of the host link for the e2e leg's byte counts at
    the workload's shape: host->device of the inputs, device->host of the two
    outputs, and both at once, each on 1, 2 and 4 streams. One JSON line per
    measurement."""
    import torch
    import synth
    w = dict(synth.WORKLOADS[args.workload])
    if args.tokens:
        w["T"] = args.tokens
    T, H, N = w["T"], w["H"], w["N"]
    dev = torch.device("cuda", 0)
    n_in = (N + 1) * T * H * 2 + H * 2
    n_out = 2 * T * H * 2
    h_in = torch.ones(n_in, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(n_out, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(n_in, dtype=torch.uint8, device=dev)
    d_out = torch.zeros(n_out, dtype=torch.uint8, device=dev)
    streams = [torch.cuda.Stream(dev) for _ in range(8)]
    cur = torch.cuda.current_stream(dev)

    def pieces(n, k):
        step = -(-n // k)
        return [(i * step, min(n, (i + 1) * step)) for i in range(k)]

    def run(k, up, down):
        for i in range(k):
            if up:
                s = streams[i]
                s.wait_stream(cur)
                a, b = pieces(n_in, k)[i]
                with torch.cuda.stream(s):
                    d_in[a:b].copy_(h_in[a:b], non_blocking=True)
            if down:
                s = streams[4 + i]
                s.wait_stream(cur)
                a, b = pieces(n_out, k)[i]
                with torch.cuda.stream(s):
                    h_out[a:b].copy_(d_out[a:b], non_blocking=True)
        for s in streams:
            cur.wait_stream(s)

    reps = max(3, min(args.steps, 20))
    for up, down, what in ((True, False, "h2d"), (False, True, "d2h"), (True, True, "both")):
        for k in (1, 2, 4):
            for _ in range(3):
                run(k, up, down)
            torch.cuda.synchronize()
            a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(cur)
            for _ in range(reps):
                run(k, up, down)
            e.record(cur)
            torch.cuda.synchronize()
            ms = a.elapsed_time(e) / reps
            nbytes = (n_in if up else 0) + (n_out if down else 0)
            print(json.dumps({"link": what, "streams": k, "bytes": nbytes, "us": round(ms * 1e3, 1),
                              "GB_s": round(nbytes / (ms / 1e3) / 1e9, 1), "reps": reps}),
                  flush=True)


# ------------------------------------------------------------------ main


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="llama70b_t1024_h8192_n8")
    ap.add_argument("--tokens", type=int, default=0, help="override the workload's T")
    ap.add_argument("--sm-budget", type=int, default=0)
    ap.add_argument("--mode", choices=("eager", "graph"), default="eager")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-unfused", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the after-GEMM timing and the compact sweep block")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--sweep-tokens", default="512,1024,2048,4096,8192,16384")
    ap.add_argument("--sweep-budgets", default="2,4,8,16,0")
    ap.add_argument("--sweep-reps", type=int, default=50)
    ap.add_argument("--sweep-partials", default="8", help="N values for --sweep")
    ap.add_argument("--sweep-hidden", default="8192", help="H values for --sweep")
    ap.add_argument("--corun", action="store_true")
    ap.add_argument("--corun-tokens", default="1024,2048,4096,8192")
    ap.add_argument("--corun-budgets", default="2,4,8,16,0")
    ap.add_argument("--corun-reps", type=int, default=20)
    ap.add_argument("--offset-sweep", action="store_true")
    ap.add_argument("--link", action="store_true",
                    help="host-link copy bandwidth at the e2e leg's byte counts")
    ap.add_argument("--sweep-offsets-tokens",
                    default="1024,1536,2048,2560,3072,3584,4096,4864,5376,6144,7168,8192,9600")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if args.sweep:
        sweep(args)
        return
    if args.corun:
        corun(args)
        return
    if args.offset_sweep:
        offset_sweep(args)
        return
    if args.link:
        link_probe(args)
        return
    if args.impl == "reference":
        # rank 0 alone times the oracle; other ranks exit without work
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        res = reference_arm(args, rank, world)
        if rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
        return
    rank, world = dist_setup()
    res = gpu_arm(args, rank, world)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
