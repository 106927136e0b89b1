"""Benchmark of the NVFP4 grouped GEMM hot path on GB300.

One step = the whole path over one grouped call: the scale-factor relayout
of every SFA and SFB (one launch) and the grouped GEMM (one launch per 32
groups), issued by one nvfp4_relayout_and_gemm call, inputs resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload all|NAME]
    python bench.py --impl reference ...   # the CPU oracle, timed on host cores

With no --workload every workload runs in one process and ONE JSON line is
printed: its top level is the largest configuration (`square`, 4 groups of
4096^3, the compute-bound case) and `per_config` holds the same figures for
the other four (tiny, moe_gate_up, moe_down, quantized).

Timing (per workload):
* K steps are replayed back to back (a captured CUDA graph per step) and
  bracketed by one pair of CUDA events; the inputs rotate over R resident
  copies of the problem whose inputs total more than twice the L2, so each
  step reads inputs that more than 2 x 129 MB of other data has passed
  through L2 since their last use.  Workloads too small for that (tiny)
  flush the L2 with a 512 MiB write before every step instead, outside the
  events, and time each step alone.
* The GEMM and the relayout are timed alone the same way (their own graphs,
  K launches) for the roofline figures; `isolated` repeats both with an L2
  flush and a pair of events around every single launch.
* A sustained window (>= 1 s of the same step replays) follows, so that
  nvidia-smi sees the GPU busy; its clocks are reported with the line.

The `e2e` figure runs the same step through the public API from pinned host
buffers: every step copies its inputs to the device and its outputs back,
two device problems taking alternate steps so that one step's copies
overlap the neighbouring step's compute.

Under torchrun (N ranks, one GPU each) the ranks share one global grouped
call of N copies of the workload's group list, split by
shard.shard_groups (expert parallel, no collective on the data path; the
host reduces the step time with a max over ranks): each rank keeps about
one workload's FLOPs (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "grouped-call TFLOPS and µs/call; achieved fraction of max(FLOP, HBM) roofline"
UNIT = "TFLOPS"
FLUSH_BYTES = 512 << 20
L2_BYTES = 129 * 10**6
NOMINAL_FP4_OVER_BF16 = 13.5 / 2.25     # dense tensor-core ratio, GB300
HEADLINE = "square"                     # the largest single-GPU configuration
ORDER = ("tiny", "moe_gate_up", "moe_down", "quantized", "square")

# dram__bytes_read.sum + dram__bytes_write.sum per GEMM launch from one ncu
# capture, keyed by workload, valid only for the kernel source it was taken
# on (kernel_source_hash: the GEMM sources without comments).  From profiles/.
NCU_TRAFFIC = {
    "moe_gate_up": {"bytes": 140507136 + 6611456, "kernel_sha": "7f2b5c0684ed3d16",
                    "source": "profiles/gemm_moe_gate_up.md"},
    "moe_down": {"bytes": 68549120 + 4058880, "kernel_sha": "7f2b5c0684ed3d16",
                 "source": "profiles/gemm_moe_down.md"},
    "quantized": {"bytes": 16572928 + 0, "kernel_sha": "7f2b5c0684ed3d16",
                  "source": "profiles/gemm_quantized.md"},
    "square": {"bytes": 75577856 + 88402688, "kernel_sha": "7f2b5c0684ed3d16",
               "source": "profiles/gemm_square.md"},
    "tiny": {"bytes": 141568 + 0, "kernel_sha": "7f2b5c0684ed3d16",
             "source": "profiles/gemm_tiny.md"},
}
KERNEL_SOURCES = ("gemm_kernel.cuh", "gemm_pair_kernel.cuh", "group_gemm.cu", "ptx.cuh")


def kernel_source_hash() -> str:
    """sha256 prefix over the GEMM sources with // comments and blank lines
    dropped (no string in them holds "//"), so that a comment edit keeps the
    recorded counters"""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        text = open(os.path.join(ROOT, "block_scaled_nvfp4_group_gb300", "csrc", f)).read()
        for line in text.splitlines():
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.t:
                self.t.join(timeout=2)

    def summary(self, t0: float, t1: float) -> dict:
        """Median SM clock, max clock and the throttle reasons seen between
        wall times t0 and t1 (all samples if none fall inside)."""
        rows = [l.split(", ") for (ts, l) in self.lines if t0 - 0.05 <= ts <= t1 + 0.05]
        if not rows:
            rows = [l.split(", ") for (_, l) in self.lines]
        sm, pw, mx, reasons = [], [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[2]))
                mx = float(r[3])
                pw.append(float(r[4]))
                for n, v in zip(names, r[6:10]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(pw) if pw else None}


def flops_of(shapes):
    return sum(2 * M * N * K for M, N, K in shapes)


def bytes_of(shapes):
    return sum(M * K // 2 + N * K // 2 + M * K // 16 + N * K // 16 + M * N * 2
               for M, N, K in shapes if M > 0)


def relayout_bytes_of(shapes):
    """Algorithmic bytes of the relayout step: scales read + tiled written."""
    from block_scaled_nvfp4_group_gb300 import ops
    tot = 0
    for M, N, K in shapes:
        if M == 0:
            continue
        tot += M * K // 16 + N * K // 16 + ops.sf_tiled_bytes(M, K) + ops.sf_tiled_bytes(N, K)
    return tot


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int) -> float:
    from block_scaled_nvfp4_group_gb300 import shard
    return shard.max_over_ranks(x, device="cuda") if ws > 1 else x


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def workload_config(name, groups, l2: str, ws: int = 1) -> dict:
    shapes = [(g.M, g.N, g.K) for g in groups]
    from block_scaled_nvfp4_group_gb300 import workloads
    d = {"workload": name, "groups": len(shapes), "M_g": [s[0] for s in shapes],
         "N": shapes[0][1], "K": shapes[0][2], "seed": workloads.describe(name)["seed"], "l2": l2}
    if ws > 1:
        d["parallelism"] = (f"expert parallel: {ws} ranks share one grouped call of {ws} copies of "
                            f"the workload's groups (rank 0's groups listed)")
    return d


# --------------------------------------------------------------------------- #
# CPU oracle timing (reference arm and cpu_baseline)                          #
# --------------------------------------------------------------------------- #

def _groups_of(wl_or_groups):
    return wl_or_groups.groups if hasattr(wl_or_groups, "groups") else list(wl_or_groups)


def oracle_fraction(groups, budget_s: float) -> float:
    """Fraction of every group's output rows the oracle covers in about
    `budget_s` seconds on all host cores (calibrated on a few rows of the
    first non-empty group)."""
    from oracle import oracle
    o = oracle.get()
    cores = os.cpu_count() or 1
    g0 = next(g for g in groups if g.M > 0)
    t = time.perf_counter()
    n = min(cores, g0.M)
    o.gemm_rows(g0.A, g0.SFA, g0.B, g0.SFB, g0.M, g0.N, g0.K, list(range(n)))
    cal = time.perf_counter() - t
    rate = n * 2 * g0.N * g0.K / max(cal, 1e-6)
    total = flops_of([(g.M, g.N, g.K) for g in groups])
    return min(1.0, rate * budget_s / total)


def oracle_sample(groups, frac: float, keep: bool = False):
    """The oracle on an evenly spread `frac` of every group's output rows
    (all N columns).  Returns (flops, rows, seconds, kept): kept is None, or
    with keep=True the results, [(group index, rows, FP16 bits)]."""
    from oracle import oracle
    o = oracle.get()
    t = time.perf_counter()
    done = nrows = 0
    out = []
    for i, g in enumerate(groups):
        if g.M == 0:
            continue
        r = max(1, int(round(g.M * frac)))
        rows = np.unique(np.linspace(0, g.M - 1, r).astype(np.int64))
        ref = o.gemm_rows(g.A, g.SFA, g.B, g.SFB, g.M, g.N, g.K, rows)
        if keep:
            out.append((i, rows, ref))
        done += 2 * rows.size * g.N * g.K
        nrows += rows.size
    return done, nrows, time.perf_counter() - t, (out if keep else None)


def time_oracle(wl_or_groups, budget_s: float, keep: bool = False):
    """Time the oracle on an evenly spread sample of output rows, sized to
    take about `budget_s` seconds on all host cores.  Returns (TFLOPS,
    description, cores, seconds, kept) -- see oracle_sample for kept."""
    groups = _groups_of(wl_or_groups)
    cores = os.cpu_count() or 1
    frac = oracle_fraction(groups, budget_s)
    done, nrows, dt, kept = oracle_sample(groups, frac, keep)
    if dt < 0.5 * budget_s and frac < 1.0:       # fixed per-group costs dominated: grow once
        frac = min(1.0, frac * budget_s / max(dt, 1e-3))
        done, nrows, dt, kept = oracle_sample(groups, frac, keep)
    desc = (f"{nrows} of {sum(g.M for g in groups)} output rows (all N columns) spread evenly "
            f"over the {len(groups)} groups, {done / 1e9:.1f} GFLOP, {dt:.1f} s")
    return done / dt / 1e12, desc, cores, dt, kept


def fp16_mismatches(got_bits: np.ndarray, ref_bits: np.ndarray) -> int:
    """Elements outside |C - C_oracle| <= 1e-3 |C_oracle| + 1e-2 (non-finite
    oracle values must be matched exactly)."""
    g = got_bits.view(np.float16).astype(np.float64)
    r = ref_bits.view(np.float16).astype(np.float64)
    fin = np.isfinite(r)
    bad = int(np.count_nonzero(~(np.abs(g[fin] - r[fin]) <= 1e-3 * np.abs(r[fin]) + 1e-2)))
    bad += int(np.count_nonzero(got_bits[~fin] != ref_bits[~fin]))
    return bad


def run_reference(args):
    """The reference arm: the CPU oracle as it stands, on the host cores, on
    the headline workload (or --workload).  Every step (W untimed, then K
    timed) is the oracle on the same bounded sample of the workload's output
    rows, sized so the whole run takes about --ref-budget-s; ms_per_step is
    the measured wall time of one such step and value its FLOPs / time.
    Under torchrun only rank 0 runs."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from block_scaled_nvfp4_group_gb300 import workloads
    name = HEADLINE if args.workload == "all" else args.workload
    groups = workloads.make_workload(name).groups
    per_step = max(0.3, args.ref_budget_s / max(1, args.steps + args.warmup))
    frac = oracle_fraction(groups, per_step)
    secs, flops, nrows = [], 0, 0
    for i in range(args.warmup + args.steps):
        done, nrows, dt, _ = oracle_sample(groups, frac)
        if i >= args.warmup:
            secs.append(dt)
            flops = done
    ms_per_step = statistics.fmean(secs) * 1e3
    value = flops / (ms_per_step * 1e-3) / 1e12
    cores = os.cpu_count() or 1
    desc = (f"every step: the oracle on {nrows} of {sum(g.M for g in groups)} output rows (all N "
            f"columns) spread evenly over the {len(groups)} groups, {flops / 1e9:.2f} GFLOP; "
            f"{cores} threads")
    cfg = workload_config(name, groups, "host memory (CPU oracle)")
    cfg["sample"] = desc
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- #
# GPU arm                                                                     #
# --------------------------------------------------------------------------- #

MAX_COPIES = 64


def copies_needed(input_bytes: int) -> int:
    """Resident copies of a problem so that between two uses of one copy's
    inputs the other copies' inputs total at least 2 x L2; 0 when that would
    take more than MAX_COPIES (the workload then flushes L2 instead)."""
    r = 1 + -(-2 * L2_BYTES // max(1, input_bytes))
    return r if r <= MAX_COPIES else 0


class Timer:
    """CUDA events on one stream."""

    def __init__(self, stream):
        self.stream = stream

    def span(self, fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(self.stream)
        fn()
        b.record(self.stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    def each(self, fn, n, pre):
        """n launches of fn, each after pre() and bracketed by its own events;
        mean and median in ms"""
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for a, b in evs:
            pre()
            a.record(self.stream)
            fn()
            b.record(self.stream)
        torch.cuda.synchronize()
        t = [a.elapsed_time(b) for a, b in evs]
        return statistics.fmean(t), statistics.median(t)


def capture(fns, stream):
    """One CUDA graph running fns in order (launches issued by the library
    keep their programmatic dependent launch edges inside the graph)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for f in fns:
            f()
    return g


def measure_workload(name, groups, args, dev, ws, sampler):
    """Every figure of one workload on this rank (see the module docstring)."""
    from block_scaled_nvfp4_group_gb300 import _abi, ops
    from block_scaled_nvfp4_group_gb300.device import DeviceProblem

    shapes = [(g.M, g.N, g.K) for g in groups]
    flops, gemm_bytes, rl_bytes = flops_of(shapes), bytes_of(shapes), relayout_bytes_of(shapes)
    stream = torch.cuda.current_stream(dev)
    timer = Timer(stream)
    first = DeviceProblem(groups, device=dev)
    R = copies_needed(int(first.inputs.numel()))
    probs = [first] + [DeviceProblem(groups, device=dev) for _ in range(max(R, 2) - 1)]
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if R == 0 else None
    if R:
        l2 = (f"inputs rotate over {R} resident copies ({R * int(first.inputs.numel()) / 1e6:.0f} MB "
              f"of inputs): between two uses of a copy > 2 x L2 of other inputs pass through; "
              f"steps back to back")
    else:
        l2 = "flushed by a 512 MiB device write before every timed step (outside the events)"
    kind, gemm_launches = ops.group_gemm_plan(descs=first.descs)
    kernel = _abi.KIND_KERNELS[[k for k, v in _abi.KIND_NAMES.items() if v == kind][0]]
    per_step = 1 + gemm_launches

    def pre():
        if flush is not None:
            flush.zero_()

    # warm-up: first-use costs and the library's one-time per-device set-up
    # (which must precede graph capture); every copy's tiled scales exist
    # afterwards, so the GEMM can also run alone
    for _ in range(max(args.warmup, 3)):
        for p in probs:
            pre()
            p.step()
    torch.cuda.synchronize()
    cap = torch.cuda.Stream(dev)
    with torch.cuda.stream(cap):
        probs[0].step()
    torch.cuda.synchronize()

    K = args.steps
    seq = [probs[i % len(probs)] for i in range(K)] if R else [probs[0]] * K

    def graph_of(method):
        if R:
            return capture([getattr(p, method) for p in seq], cap)
        return capture([getattr(probs[0], method)], cap)

    g_step, g_gemm, g_rel = graph_of("step"), graph_of("gemm"), graph_of("relayout")
    for g in (g_step, g_gemm, g_rel):
        pre()
        g.replay()
    torch.cuda.synchronize()

    def run_k(g):
        """ms per launch over exactly K launches"""
        if R:
            return timer.span(g.replay) / K, None
        return timer.each(g.replay, K, pre)

    # ---- the timed region: exactly K steps
    barrier(ws)
    torch.cuda.synchronize()
    w0 = time.time()
    step_ms, _ = run_k(g_step)
    torch.cuda.synchronize()
    barrier(ws)
    step_ms = max_over_ranks(step_ms, ws)
    gemm_ms, _ = run_k(g_gemm)
    rel_ms, _ = run_k(g_rel)
    # sustained window: the same K-step replays for >= --sustain-s
    s0 = time.time()
    n_sus = 0
    ev_a, ev_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_a.record(stream)
    batch = max(1, min(8, int(0.05 / max(step_ms * 1e-3 * (K if R else 1), 1e-6))))
    while time.time() - s0 < args.sustain_s:
        for _ in range(batch):
            pre()
            g_step.replay()
        n_sus += batch
        torch.cuda.synchronize()      # the host waits for every batch: replays are asynchronous
    ev_b.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    # (with per-step flushes the window also holds the flush writes)
    sus_ms = ev_a.elapsed_time(ev_b) / (n_sus * K) if R else None
    # isolated launches: L2 flushed before each, events around each
    iso_flush = flush if flush is not None else torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    n_iso = min(K, 100)
    one = probs[0]
    iso_gemm = timer.each(one.gemm, n_iso, iso_flush.zero_)
    iso_rel = timer.each(one.relayout, n_iso, iso_flush.zero_)
    iso_step = timer.each(one.step, n_iso, iso_flush.zero_)
    del iso_flush
    clocks = sampler.summary(w0, w1)
    rc = ops.last_device_error()
    if rc != 0:
        raise RuntimeError(f"{name}: device error word {rc} after the timed launches")
    rec = {
        "name": name, "shapes": shapes, "groups": groups, "probs": probs, "flops": flops,
        "gemm_bytes": gemm_bytes, "rl_bytes": rl_bytes, "l2": l2, "copies": R,
        "kind": kind, "kernel": kernel, "launches_per_step": per_step,
        "step_ms": step_ms, "gemm_ms": gemm_ms, "rel_ms": rel_ms,
        "sustained": {"steps": n_sus * (K if R else 1), "ms_per_step": sus_ms,
                      "seconds": round(w1 - s0, 2)},
        "isolated_us": {"step_mean": iso_step[0] * 1e3, "gemm_mean": iso_gemm[0] * 1e3,
                        "gemm_median": iso_gemm[1] * 1e3, "relayout_mean": iso_rel[0] * 1e3},
        "clocks": clocks,
    }
    del g_step, g_gemm, g_rel
    return rec


def measure_e2e(rec, args, dev, ws):
    """The step through the public API with host buffers: every step copies
    all inputs (A, B and the row-major scales of every group: one pinned
    buffer) to the device, runs the step and copies all outputs back.  Two
    device problems take alternate steps, so the host->device copy of step
    i+1 (its own stream) overlaps the compute and the device->host read of
    step i, when a step moves >= 8 MiB of inputs; otherwise one problem and
    copies and step in sequence."""
    probs = rec["probs"]
    stream = torch.cuda.current_stream(dev)
    prob = probs[0]
    pipelined = int(prob.inputs.numel()) >= (8 << 20)
    pair = [probs[0], probs[1]] if pipelined else [prob, prob]
    h_in = torch.empty(prob.inputs.shape, dtype=torch.uint8, pin_memory=True)
    h_in.copy_(prob.inputs)
    h_out = [torch.empty(prob.outputs.shape, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    n = max(3, min(args.steps, 50))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_done + ev_out:
        e.record(stream)

    def sequential(i):
        prob.inputs.copy_(h_in, non_blocking=True)
        prob.step()
        h_out[0].copy_(prob.outputs, non_blocking=True)

    def overlapped(i):
        b = i % 2
        p = pair[b]
        s_in.wait_event(ev_done[b])           # step i-2 has read its inputs
        with torch.cuda.stream(s_in):
            p.inputs.copy_(h_in, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])          # step i-2's results have been read back
        p.step()
        ev_done[b].record(stream)
        s_out.wait_event(ev_done[b])
        with torch.cuda.stream(s_out):
            h_out[b].copy_(p.outputs, non_blocking=True)
            ev_out[b].record(s_out)

    step = overlapped if pipelined else sequential
    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    e0.record(stream)
    s_in.wait_event(e0)
    for i in range(n):
        step(i)
    if pipelined:
        stream.wait_event(ev_out[(n - 1) % 2])
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    ms = max_over_ranks(e0.elapsed_time(e1), ws) / n
    return {"value": ws * rec["flops"] / (ms * 1e-3) / 1e12, "unit": UNIT,
            "h2d_bytes_per_step": int(prob.inputs.numel()), "d2h_bytes_per_step": int(prob.outputs.numel()),
            "ms_per_step": ms, "steps": n, "pipelined": pipelined}


def roofline_of(rec, peaks):
    """The GEMM against max(bytes / HBM, FLOPs / FP4 peak): HBM-bound
    workloads report algorithmic bytes per launch / mean launch time against
    the measured copy bandwidth, tensor-bound ones FLOPs / time against the
    measured bf16 peak x the nominal FP4 / bf16 ratio."""
    fp4_peak = peaks["bf16_tflops"] * NOMINAL_FP4_OVER_BF16
    t_mem = rec["gemm_bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_flop = rec["flops"] / (fp4_peak * 1e12)
    bound = "hbm" if t_mem >= t_flop else "tensor"
    gemm_s = rec["gemm_ms"] * 1e-3 / max(1, rec["launches_per_step"] - 1)
    if bound == "hbm":
        achieved, peak, unit = rec["gemm_bytes"] / gemm_s / 1e9, peaks["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = rec["flops"] / gemm_s / 1e12, fp4_peak, "TFLOP/s"
    traffic = None
    ncu = NCU_TRAFFIC.get(rec["name"])
    if ncu and ncu.get("kernel_sha") == kernel_source_hash():
        traffic = ncu["bytes"]
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "traffic": traffic, "kernel": rec["kernel"], "kernel_config": rec["kind"],
            "peak_source": peaks["source"] + (" (hbm_gbs)" if bound == "hbm" else
                                              " (bf16_tflops x 6, nominal fp4/bf16 dense ratio)"),
            "algorithmic_bytes_per_launch": rec["gemm_bytes"], "flops_per_launch": rec["flops"],
            "launch_us": gemm_s * 1e6,
            "roofline_fraction_of_max_time": max(t_mem, t_flop) / gemm_s}


def oracle_check(rec, budget_s):
    """The oracle on a sample of output rows (timed: the CPU baseline) and
    the same rows of the GPU's C in every resident copy (element by element,
    outside every timed region)."""
    v, desc, cores, _, kept = time_oracle(rec["groups"], budget_s, keep=True)
    n_el = n_bad = 0
    try:
        for p in rec["probs"]:
            got = p.outputs_fp16_bits()
            for gi, rows, ref in kept:
                n_el += ref.size
                n_bad += fp16_mismatches(got[gi][rows], ref)
        parity = {"elements": n_el, "mismatches": n_bad, "copies_checked": len(rec["probs"]),
                  "tolerance": "|C - C_oracle| <= 1e-3 |C_oracle| + 1e-2"}
        if n_bad:
            print(f"bench: {rec['name']}: {n_bad} of {n_el} sampled outputs differ from the oracle",
                  file=sys.stderr)
    except Exception as e:          # the check must not cost the measurement its line
        parity = {"error": f"{type(e).__name__}: {e}"}
    return {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}, parity


def summary_of(rec, args, ws, peaks):
    K = args.steps
    return {
        "value": ws * rec["flops"] / (rec["step_ms"] * 1e-3) / 1e12,
        "ms_per_step": rec["step_ms"],
        "config": workload_config(rec["name"], rec["groups"], rec["l2"], ws),
        "us_per_call": {"step": rec["step_ms"] * 1e3,
                        "gemm": rec["gemm_ms"] * 1e3 / max(1, rec["launches_per_step"] - 1),
                        "relayout": rec["rel_ms"] * 1e3},
        "isolated_us": rec["isolated_us"],
        "roofline": roofline_of(rec, peaks),
        "relayout": {"us": rec["rel_ms"] * 1e3, "bytes": rec["rl_bytes"],
                     "gbs": rec["rl_bytes"] / (rec["rel_ms"] * 1e-3) / 1e9,
                     "peak_gbs": peaks["hbm_gbs"],
                     "frac": rec["rl_bytes"] / (rec["rel_ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"]},
        "sustained": rec["sustained"],
        "gpu_launches": rec["launches_per_step"] * K,
        "clocks": rec["clocks"],
    }


def run_ours(args):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from block_scaled_nvfp4_group_gb300 import workloads

    names = ORDER if args.workload == "all" else (args.workload,)
    head = HEADLINE if args.workload == "all" else args.workload
    peaks = load_peaks()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.15)
    out = {}
    try:
        for name in names:
            _, groups = workloads.expert_parallel_groups(name, ws, rank)
            rec = measure_workload(name, groups, args, dev, ws, sampler)
            s = summary_of(rec, args, ws, peaks)
            if name == head:
                s["e2e"] = measure_e2e(rec, args, dev, ws)
            if rank == 0 and ws == 1 and not args.no_cpu_baseline:
                cpu, parity = oracle_check(rec, args.cpu_budget_s if name == head else args.cpu_check_s)
                s["parity"] = parity
                if name == head:
                    s["cpu_baseline"] = dict(cpu, parity=parity)
            del rec
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
            out[name] = s
    finally:
        sampler.stop()
    if rank == 0:
        h = out[head]
        line = {
            "metric": METRIC, "value": h["value"], "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": h["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4",
            "data": "synthetic (seeded uniform / Gaussian-quantised FP4 codes and E4M3 scales)",
            "config": h["config"],
            "launch": ("one nvfp4_relayout_and_gemm call per step (relayout + grouped GEMM "
                       "launches), K steps captured in one CUDA graph"),
        }
        for k in ("us_per_call", "isolated_us", "roofline", "relayout", "e2e", "gpu_launches", "clocks",
                  "sustained", "cpu_baseline", "parity"):
            if k in h:
                line[k] = h[k]
        if len(out) > 1:
            line["per_config"] = {k: v for k, v in out.items() if k != head}
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
def run_profile(args):
    """Minimal launch sequence for an ncu capture: `warmup` steps (flush,
    relayout, GEMM), then one more step; no timing, no oracle."""
    from block_scaled_nvfp4_group_gb300 import workloads
    from block_scaled_nvfp4_group_gb300.device import DeviceProblem
    torch.cuda.set_device(0)
    wl = workloads.make_workload(args.workload)
    prob = DeviceProblem(wl.groups, device="cuda:0")
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda:0")
    for _ in range(args.warmup + 1):
        flush.zero_()
        prob.step()
    torch.cuda.synchronize()
    from block_scaled_nvfp4_group_gb300 import ops
    rc = ops.last_device_error()
    print(json.dumps({"profile": args.workload, "steps": args.warmup + 1, "device_error": rc}))
    if rc != 0:
        sys.exit(1)


def quantize_input(wl, seed: int) -> np.ndarray:
    """The rows the quantisation kernel is timed on: one FP16 matrix holding
    the A operands (activations) of every group of the workload, Gaussian
    values, [sum(M_g), K]."""
    rows = sum(g.M for g in wl.groups)
    K = wl.groups[0].K
    rng = np.random.default_rng(seed)
    return rng.standard_normal((rows, K)).astype(np.float16)


def run_quantize(args):
    """NVFP4 quantisation of the workload's activations: one launch per step
    (FP16 [sum M_g, K] -> codes + tiled scales), inputs resident; K launches
    back to back over rotating copies whose inputs total more than twice the
    L2 (one CUDA graph), and each launch alone after an L2 flush
    (`isolated_us`); HBM roofline."""
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    from block_scaled_nvfp4_group_gb300 import ops, workloads
    wl = workloads.make_workload(args.workload)
    x16 = quantize_input(wl, wl.seed + 104729)
    rows, K = x16.shape
    R = max(2, copies_needed(x16.nbytes) or 2)
    xs = [torch.from_numpy(x16).to(dev) for _ in range(R)]
    codes = [torch.empty((rows, K // 2), dtype=torch.uint8, device=dev) for _ in range(R)]
    tiled = [torch.empty(ops.sf_tiled_bytes(rows, K), dtype=torch.uint8, device=dev) for _ in range(R)]
    x, codes0, tiled0 = xs[0], codes[0], tiled[0]
    nbytes = rows * K * 2 + rows * K // 2 + ops.sf_tiled_bytes(rows, K)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def launch(i):
        ops.quantize(xs[i], codes=codes[i], sf_tiled=tiled[i])

    for _ in range(max(args.warmup, 3)):
        for i in range(R):
            launch(i)
    torch.cuda.synchronize()
    if args.profile:
        print(json.dumps({"profile": "quantize_" + args.workload, "device_error": ops.last_device_error()}))
        return
    cap = torch.cuda.Stream(dev)
    with torch.cuda.stream(cap):
        launch(0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        for k in range(args.steps):
            launch(k % R)
    g.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.15)
    timer = Timer(stream)
    torch.cuda.synchronize()
    w0 = time.time()
    ms_mean = timer.span(g.replay) / args.steps
    s0 = time.time()
    while time.time() - s0 < args.sustain_s:      # sustained window for the clock samples
        g.replay()
        torch.cuda.synchronize()
    w1 = time.time()
    sampler.stop()
    clocks = sampler.summary(w0, w1)
    iso_mean, iso_med = timer.each(lambda: launch(0), min(args.steps, 100), flush.zero_)
    # end to end through the public API: pinned H2D of x, the launch, D2H of
    # codes and tiled scales
    xh = torch.from_numpy(x16).pin_memory()
    ch = torch.empty(codes0.shape, dtype=torch.uint8).pin_memory()
    th = torch.empty(tiled0.shape, dtype=torch.uint8).pin_memory()
    n_e2e = min(args.steps, 100)
    e2e = []
    for _ in range(n_e2e):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        x.copy_(xh, non_blocking=True)
        launch(0)
        ch.copy_(codes0, non_blocking=True)
        th.copy_(tiled0, non_blocking=True)
        b.record(stream)
        b.synchronize()
        e2e.append(a.elapsed_time(b))
    e2e_ms = statistics.median(e2e)
    peaks = load_peaks()
    gbs = nbytes / (ms_mean * 1e-3) / 1e9
    line = {
        "metric": "NVFP4 quantisation GB/s (FP16 in, codes + tiled scales out)", "value": gbs,
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_mean, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"quantize_{args.workload}_activations", "rows": rows, "K": K,
                   "l2": (f"inputs rotate over {R} resident copies ({R * x16.nbytes / 1e6:.0f} MB); "
                          f"launches back to back")},
        "us_per_call": {"mean": ms_mean * 1e3},
        "isolated_us": {"mean": iso_mean * 1e3, "median": iso_med * 1e3,
                        "l2": "flushed by a 512 MiB device write before each launch"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                     "traffic": None, "kernel": "quantize_kernel",
                     "algorithmic_bytes_per_launch": nbytes,
                     "peak_source": peaks["source"] + " (hbm_gbs)"},
        "e2e": {"value": nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": rows * K * 2,
                "d2h_bytes_per_step": codes0.numel() + tiled0.numel(), "ms_per_step": e2e_ms},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        from oracle import oracle
        o = oracle.get()
        sample = min(rows, 256)
        t0 = time.time()
        o.quantize(x16[:sample].view(np.uint16), sample, K)
        dt = time.time() - t0
        line["cpu_baseline"] = {"value": sample * K * (2 + 0.5 + 1 / 16) / dt / 1e9, "unit": "GB/s",
                                "cores": 1, "kind": "oracle",
                                "sample": f"{sample} of {rows} rows, {dt:.2f} s"}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="all",
                    help="all (default: every workload, the largest as the headline) or one name")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--ref-budget-s", type=float, default=60.0)
    ap.add_argument("--cpu-check-s", type=float, default=4.0,
                    help="oracle seconds for the parity sample of each non-headline workload")
    ap.add_argument("--sustain-s", type=float, default=1.0,
                    help="length of each workload's sustained replay window (clock evidence)")
    ap.add_argument("--profile", action="store_true",
                    help="few launches for ncu: W warm-up steps, then one step")
    ap.add_argument("--op", default="gemm", choices=["gemm", "quantize"],
                    help="gemm: the relayout + grouped GEMM step (default); quantize: the "
                         "NVFP4 quantisation of the workload's activations")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.workload == "all" and (args.profile or args.op == "quantize"):
        args.workload = HEADLINE if args.profile else "moe_gate_up"
    if args.op == "quantize":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "op": "quantize",
                              "unavailable": "the reference arm times the GEMM oracle"}))
            return
        run_quantize(args)
    elif args.impl == "reference":
        run_reference(args)
    elif args.profile:
        run_profile(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
