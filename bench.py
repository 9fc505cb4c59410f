"""Benchmark of the fused softmax cross-entropy forward + gradient.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--headline-only]

Prints ONE JSON line.  The headline ``value`` is rows/s of the largest
workload, the ragged stress case (B=16384, C=50257, fp32), processed by the
library's kernels with the inputs resident in HBM; ``workloads`` carries the
same measurement for every workload (all five, in the same run).  A step is
one ``ce_fwd_bwd`` call: the loss and the full gradient of one batch.

Timing: steps run from a CUDA graph (one library call per step, captured
once), cycling through enough buffer sets that every step reads inputs that
are not in L2; CUDA events on the launching stream bracket the timed steps.
``e2e`` times the host-buffer call ce_fwd_bwd_host_grad, eagerly: every step
copies its inputs from pinned host memory and its gradient and loss back.  ``--impl reference`` times
the fp64 CPU oracle (the only reference this path has) on the host cores.

With torchrun (N > 1) every rank runs an independent replica of the workload
(rows are independent; the path has no exchange step), barriers bracket the
timed region and rank 0 reports the max time over ranks.
"""

from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "fused CE fwd+grad rows/s and achieved HBM GB/s vs ~8 TB/s roofline (1×GB300)"
HEADLINE = "stress_16384x50257_f32"
TIMED_PARTS = 5            # the timed region is split into parts for a spread
FALLBACK_HBM_GBS = 6800.0
TARGET_REGION_S = 1.5      # timed work per workload when --steps is not given
HOLD_CYCLES = 400_000      # device-side wait (~0.2 ms) queued ahead of each timed region
CPU_SAMPLE_S = 10.0
MAX_SETS = 64              # a workload this small stays L2-resident (said in the output)


# ------------------------------------------------------------------ helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# The host-side C-ABI layer: argument checks, workspaces and the planner.  Its
# launch decisions are recorded with the traffic (PLAN_KEYS), so the hashes
# cover the device code only: each kernel's own file and the headers every
# kernel includes.
HOST_ONLY_SOURCES = ("ce_api.cu",)
SHARED_DEVICE_SOURCES = ("ce_device.cuh", "ce_launch.h")
KERNEL_SOURCES = {"rows_warp": "ce_rows_warp.cu", "row_split": "ce_row_split.cu",
                  "row_pipe": "ce_row_pipe.cu", "row_twopass": "ce_row_twopass.cu",
                  "stream": "ce_stream.cu", "rows_online": "ce_rows_online.cu"}
PLAN_KEYS = ("path", "split", "ctas", "threads", "smem_bytes")


CSRC = os.path.join(ROOT, "softmax_cross_entropy_row_gb300", "csrc")


def kernel_source_names(kernel: str | None = None) -> list[str]:
    """The csrc files a kernel's device code comes from: its file, a header of
    the same name if it has one, and the shared headers; every csrc file but
    the host-only ones when no kernel is named."""
    if kernel is None:
        return sorted(os.path.basename(p) for p in glob.glob(os.path.join(CSRC, "*"))
                      if os.path.basename(p) not in HOST_ONLY_SOURCES)
    own = KERNEL_SOURCES[kernel]
    header = os.path.splitext(own)[0] + ".h"
    return sorted((own,) + SHARED_DEVICE_SOURCES
                  + ((header,) if os.path.exists(os.path.join(CSRC, header)) else ()))


def source_hash(kernel: str | None = None) -> str:
    """Hash of the files kernel_source_names lists (names and contents)."""
    h = hashlib.sha256()
    for name in kernel_source_names(kernel):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, plan=None):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None if that kernel's sources or its launch (path, split,
    CTAs, threads, shared memory) changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload)
    if not e or e.get("kernel") not in KERNEL_SOURCES:
        return None
    if e.get("source_sha") != source_hash(e["kernel"]):
        return None
    if plan is not None and e.get("plan") != {k: plan.get(k) for k in PLAN_KEYS}:
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="ce_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"samples": 0, "note": "nvidia-smi unavailable"}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r)
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# -------------------------------------------------------------- oracle arm

def time_oracle(inp, budget_s: float = CPU_SAMPLE_S):
    """Rows/s of the fp64 oracle's forward + gradient on a bounded sample of
    the workload's rows, on every host core the process may use; and, on a
    sample of a quarter of the budget, on one thread."""
    import oracle

    oracle.build()
    cores = cpu_cores()
    oracle.set_threads(1)
    one = _time_oracle_threads(inp, 0.25 * budget_s)
    oracle.set_threads(cores)
    res = _time_oracle_threads(inp, 0.75 * budget_s)
    res["one_thread"] = {"value": one["value"], "unit": "rows/s", "cores": 1,
                         "sample": one["sample"]}
    return res


def _time_oracle_threads(inp, budget_s):
    import oracle

    B, C = inp.logits.shape
    # calibrate on a small block, then size the sample to the budget
    probe = max(1, min(B, 64))
    z = np.ascontiguousarray(inp.logits[:probe])
    t = np.ascontiguousarray(inp.targets[:probe])
    g = np.empty_like(z)
    sc = np.empty(probe, dtype=np.float64)
    t0 = time.perf_counter()
    oracle.fwd_bwd(z, t, g, sc)
    per_row = max((time.perf_counter() - t0) / probe, 1e-9)
    rows = int(min(B, max(1, 0.5 * budget_s / per_row)))
    z = np.ascontiguousarray(inp.logits[:rows])
    t = np.ascontiguousarray(inp.targets[:rows])
    g = np.empty_like(z)
    sc = np.empty(rows, dtype=np.float64)
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.fwd_bwd(z, t, g, sc)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s:
            break
    value = rows * reps / dt
    sample = (f"leading {rows} of {B} rows x {C} classes ({inp.workload.dtype}), "
              f"{reps} pass(es), {dt:.1f} s wall-clock on {oracle.threads()} threads")
    return {"value": value, "unit": "rows/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": sample}


# ------------------------------------------------------------------ our arm

def max_over_ranks(value: float, device) -> float:
    """The largest of every rank's `value` (replicas are timed by their
    slowest rank); the value itself when the job has one process."""
    import torch

    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return value
    tt = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
    return float(tt.item())


def replica_rows_per_s(rows_per_rank: int, world: int, seconds_per_step: float) -> float:
    """Whole-job throughput of `world` replicas that each process
    `rows_per_rank` rows per step, timed by the slowest rank."""
    return world * rows_per_rank / seconds_per_step


def device_set(inp, device):
    import torch

    if inp.workload.dtype == "bf16":
        z = torch.from_numpy(inp.logits.view(np.int16)).view(torch.bfloat16).to(device)
    else:
        z = torch.from_numpy(inp.logits).to(device)
    t = torch.from_numpy(inp.targets).to(device)
    return z, t


def bench_workload(w, inp, steps, warmup, device, l2_bytes, hbm_peak, peak_note, sampler_gpu,
                   world, with_e2e=True):
    import torch

    import softmax_cross_entropy_row_gb300 as ce

    plan = ce.ce_query_plan(w.B, w.C, w.dtype_code)
    set_bytes = 2 * w.B * w.C * w.elem_bytes + 4 * w.B
    nsets = 1
    if set_bytes <= 2 * l2_bytes:
        nsets = min(MAX_SETS, int(np.ceil(2 * l2_bytes / set_bytes)) + 1)
    z0, t0 = device_set(inp, device)
    sets = []
    for i in range(nsets):
        z = z0 if i == 0 else z0.clone()
        t = t0 if i == 0 else t0.clone()
        sets.append((z, t, torch.empty(1, dtype=torch.float32, device=device),
                     torch.empty_like(z)))
    s = torch.cuda.Stream(device)
    with torch.cuda.stream(s):
        for i in range(max(warmup, 3)):
            z, t, loss, grad = sets[i % nsets]
            ce.ce_fwd_bwd(z, t, loss, grad, s)
        s.synchronize()
        # one graph runs a whole number of passes over the buffer sets
        per_graph = nsets * max(1, int(np.ceil(64 / nsets)))

        def capture(n):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for i in range(n):
                    z, t, loss, grad = sets[i % nsets]
                    ce.ce_fwd_bwd(z, t, loss, grad, s)
            return g

        graph = capture(per_graph)
        graph.replay()  # warm the graph
        s.synchronize()
        # estimate the step time to size the timed region
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        graph.replay()
        e1.record(s)
        e1.synchronize()
        est = e0.elapsed_time(e1) / 1e3 / per_graph
        if steps is None:
            steps = per_graph * max(1, int(np.ceil(TARGET_REGION_S / (est * per_graph))))
        replays, rest = divmod(steps, per_graph)
        tail = capture(rest) if rest else None
        if tail is not None:
            tail.replay()
        n_steps = steps
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(device)
        # the replays split into TIMED_PARTS parts, an event after each
        cuts = [round(replays * k / TIMED_PARTS) for k in range(TIMED_PARTS + 1)]
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(TIMED_PARTS + 1)]
        part_steps = [(cuts[k + 1] - cuts[k]) * per_graph for k in range(TIMED_PARTS)]
        part_steps[-1] += rest
        sampler = ClockSampler(sampler_gpu)
        with sampler:
            # keep the stream busy while the host submits the timed graphs, so
            # that the start event does not wait on host launch latency
            torch.cuda._sleep(HOLD_CYCLES)
            e0.record(s)
            marks[0] = e0
            for k in range(TIMED_PARTS):
                for _ in range(cuts[k + 1] - cuts[k]):
                    graph.replay()
                if k == TIMED_PARTS - 1 and tail is not None:
                    tail.replay()
                if k < TIMED_PARTS - 1:
                    marks[k + 1].record(s)
            e1.record(s)
            marks[-1] = e1
            e1.synchronize()
        torch.cuda.synchronize(device)
        elapsed = max_over_ranks(e0.elapsed_time(e1) / 1e3, device)
        if world > 1:
            torch.distributed.barrier()
        bad, tmo = ce.ce_get_device_errors(s)
    del graph, tail
    # per-step time of each part of the timed region (events only, no
    # synchronisation between the parts)
    part_ms = [a.elapsed_time(b) / n for a, b, n in zip(marks[:-1], marks[1:], part_steps) if n]
    per_step = elapsed / n_steps
    per_launch = per_step / plan["launches"] if plan["launches"] == 1 else None
    achieved = w.min_bytes / per_step / 1e9
    res = {
        "workload": w.name, "B": w.B, "C": w.C, "logits_dtype": w.dtype,
        "path": plan["path_name"], "split": plan["split"], "ctas": plan["ctas"],
        "threads": plan["threads"], "smem_bytes": plan["smem_bytes"],
        "launches_per_step": plan["launches"], "steps": n_steps, "buffer_sets": nsets,
        "ms_per_step": per_step * 1e3, "rows_per_s": replica_rows_per_s(w.B, world, per_step),
        "achieved_gbs": achieved, "frac_of_peak": achieved / hbm_peak,
        "min_bytes_per_step": w.min_bytes, "device_errors": [bad, tmo],
        "clocks": sampler.summary(),
        "ms_per_step_parts": {"median": statistics.median(part_ms), "min": min(part_ms),
                              "max": max(part_ms), "parts": len(part_ms)} if part_ms else None,
    }
    if per_launch is not None:
        res["kernel_ms_per_launch"] = per_launch * 1e3
    if with_e2e:
        res["e2e"] = bench_e2e(w, inp, device, steps=min(50, max(5, int(0.5 / max(est, 1e-6)))),
                               world=world)
    for z, t, loss, grad in sets:
        del z, t, loss, grad
    torch.cuda.empty_cache()
    return res


def bench_e2e(w, inp, device, steps, world=1):
    """The public call with host buffers, ce_fwd_bwd_host_grad: every step
    copies the pinned logits and targets to the device, runs the kernels and
    copies the gradient and the loss back to pinned host memory (chunk by
    chunk, the copies in and out overlapping)."""
    import torch

    import softmax_cross_entropy_row_gb300 as ce

    if w.dtype == "bf16":
        hz = torch.from_numpy(inp.logits.view(np.int16)).view(torch.bfloat16).pin_memory()
    else:
        hz = torch.from_numpy(inp.logits).pin_memory()
    ht = torch.from_numpy(inp.targets).pin_memory()
    hl = torch.empty(1, dtype=torch.float32).pin_memory()
    hg = torch.empty(hz.shape, dtype=hz.dtype).pin_memory()
    s = torch.cuda.Stream(device)

    def step():
        ce.ce_fwd_bwd_host_grad(hz, ht, hl, hg, s)

    with torch.cuda.stream(s):
        for _ in range(3):
            step()
        s.synchronize()
        if world > 1:
            torch.distributed.barrier()
        # an event after every step as well: the per-step spread (the copies
        # share the host's memory with whatever else runs on the machine)
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        marks[0].record(s)
        for k in range(steps):
            step()
            marks[k + 1].record(s)
        marks[-1].synchronize()
    per_step = max_over_ranks(marks[0].elapsed_time(marks[-1]) / 1e3, device) / steps
    each = [a.elapsed_time(b) for a, b in zip(marks[:-1], marks[1:])]
    h2d = hz.numel() * hz.element_size() + ht.numel() * ht.element_size()
    d2h = hg.numel() * hg.element_size() + hl.numel() * hl.element_size()
    del hg
    # whole-job figures: every replica copies its own inputs and results
    return {"value": replica_rows_per_s(w.B, world, per_step), "unit": "rows/s",
            "h2d_bytes_per_step": int(world * h2d), "d2h_bytes_per_step": int(world * d2h),
            "steps": steps, "ms_per_step": per_step * 1e3,
            "ms_per_step_median": statistics.median(each), "ms_per_step_max": max(each),
            "call": "ce_fwd_bwd_host_grad (pinned host logits, targets, loss and gradient)"}


# The rows beyond the plain fused step, measured the same way: (label, workload,
# call kind).  Bytes per step are those each call must move.
# f16 logits: the 32k-class LM head recipe drawn the same way, narrowed to f16
F16_HEAD = wl.Workload("lm_head_8192x32000_f16", 8192, 32000, "f16", seed=2, sigma=3.0,
                       description="LM head, f16 logits ~ N(0, 3^2)")
wl.WORKLOADS_BY_NAME.setdefault(F16_HEAD.name, F16_HEAD)

NEXT_ROWS = [("f16_logits", "lm_head_8192x32000_f16", "plain"),
             ("loss_only_mean", "classifier_4096x1000_f32", "forward"),
             ("loss_only_mean", "lm_head_8192x32000_bf16", "forward"),
             ("loss_only_mean", "lm_head_4096x128256_bf16_peaked", "forward"),
             ("loss_only_mean", "stress_16384x50257_f32", "forward"),
             ("sum_scalar_upstream", "classifier_4096x1000_f32", "sum"),
             ("none_per_row_upstream", "classifier_4096x1000_f32", "none"),
             ("softmax_forward", "lm_head_8192x32000_bf16", "softmax_fwd"),
             ("softmax_forward", "classifier_4096x1000_f32", "softmax_fwd"),
             ("softmax_backward", "lm_head_8192x32000_bf16", "softmax_bwd"),
             ("softmax_backward", "classifier_4096x1000_f32", "softmax_bwd")]


def next_row_bytes(w, kind):
    n = w.B * w.C * w.elem_bytes
    if kind == "softmax_fwd":  # z in, p out
        return 2 * n
    if kind == "softmax_bwd":  # p and dy in, dx out
        return 3 * n
    read = n + 4 * w.B
    if kind == "plain":
        return w.min_bytes
    if kind == "forward":
        return read + 4
    if kind == "sum":
        return read + w.B * w.C * w.elem_bytes + 4 + 4
    return read + w.B * w.C * w.elem_bytes + 4 * w.B + 4 * w.B  # per-row scale and losses


def bench_next_row(label, w, inp, kind, device, l2_bytes, hbm_peak):
    """Device time per step of one extended call (graph replay over buffer
    sets larger than twice L2, CUDA events on the launching stream)."""
    import torch

    import softmax_cross_entropy_row_gb300 as ce

    nbytes = next_row_bytes(w, kind)
    nsets = 1 if nbytes > 2 * l2_bytes else min(MAX_SETS, int(np.ceil(2 * l2_bytes / nbytes)) + 1)
    z0, t0 = device_set(inp, device)
    sets = []
    for i in range(nsets):
        z = z0 if i == 0 else z0.clone()
        grad = None if kind == "forward" else torch.empty_like(z)
        if kind == "softmax_bwd":  # (p, dy, -, dx, -): probabilities, an upstream gradient
            probs = torch.empty_like(z)
            ce.ce_softmax_fwd(z, probs)
            dy = torch.empty_like(z).normal_() if i == 0 else sets[0][1].clone()
            sets.append((probs, dy, None, torch.empty_like(z), None))
            continue
        loss = torch.empty(w.B if kind == "none" else 1, dtype=torch.float32, device=device)
        up = (torch.linspace(0.5, 1.5, w.B, device=device) if kind == "none"
              else torch.full((1,), 0.5, device=device) if kind == "sum" else None)
        sets.append((z, t0, loss, grad, up))
    red = {"forward": ce.CE_REDUCE_MEAN, "sum": ce.CE_REDUCE_SUM, "none": ce.CE_REDUCE_NONE
           }.get(kind, ce.CE_REDUCE_MEAN)
    s = torch.cuda.Stream(device)

    def call(i):
        z, t, loss, grad, up = sets[i % nsets]
        if kind == "softmax_fwd":
            ce.ce_softmax_fwd(z, grad, s)
        elif kind == "softmax_bwd":
            ce.ce_softmax_bwd(z, t, grad, s)  # (p, dy, dx)
        elif kind == "forward":
            ce.ce_forward(z, t, loss, red, s)
        elif kind == "plain":
            ce.ce_fwd_bwd(z, t, loss, grad, s)
        else:
            ce.ce_fwd_bwd_ex(z, t, loss, grad, red, up, s)

    with torch.cuda.stream(s):
        for i in range(3):
            call(i)
        s.synchronize()
        per_graph = nsets * max(1, int(np.ceil(32 / nsets)))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(per_graph):
                call(i)
        g.replay()
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        g.replay()
        e1.record(s)
        e1.synchronize()
        reps = max(2, min(200, int(0.3 / max(e0.elapsed_time(e1) / 1e3, 1e-6))))
        e0.record(s)
        for _ in range(reps):
            g.replay()
        e1.record(s)
        e1.synchronize()
    per_step = e0.elapsed_time(e1) / 1e3 / (reps * per_graph)
    del g
    gbs = nbytes / per_step / 1e9
    return {"row": label, "workload": w.name, "call": kind, "us_per_step": per_step * 1e6,
            "bytes_per_step": nbytes, "achieved_gbs": gbs, "frac_of_peak": gbs / hbm_peak,
            "rows_per_s": w.B / per_step}


def l2_note(res, w, l2_bytes):
    n = res["buffer_sets"]
    total = n * (2 * w.B * w.C * w.elem_bytes + 4 * w.B)
    if n == 1:
        return f"inputs larger than L2 ({total / 1e6:.0f} MB vs L2 {l2_bytes / 1e6:.0f} MB)"
    if total > 2 * l2_bytes:
        return (f"{n} rotating buffer sets ({total / 1e6:.0f} MB > 2x L2 "
                f"{l2_bytes / 1e6:.0f} MB): every step reads inputs not in L2")
    return f"{n} rotating buffer sets, {total / 1e3:.1f} KB in all: L2-resident (tiny workload)"


# --------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps of the headline workload (default: ~1.5 s of work)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(wl.WORKLOADS_BY_NAME))
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--cpu-sample-s", type=float, default=CPU_SAMPLE_S,
                    help="seconds of oracle timing for cpu_baseline (0: skip)")
    ap.add_argument("--rows", type=int, default=None,
                    help="profiling only: run the workload's recipe with this many rows")
    ap.add_argument("--no-e2e", action="store_true", help="profiling only: skip the e2e leg")
    args = ap.parse_args()

    world, rank, local = dist_env()
    w = wl.WORKLOADS_BY_NAME[args.workload]
    if args.rows:
        import dataclasses

        w = dataclasses.replace(w, B=int(args.rows), name=f"{w.name}_rows{args.rows}")
        wl.WORKLOADS_BY_NAME[w.name] = w
        args.headline_only = True

    if args.impl == "reference":
        if rank != 0:
            return
        inp = wl.make_inputs(w)
        cb = time_oracle(inp, args.cpu_sample_s)
        out = {"metric": METRIC, "value": cb["value"], "unit": "rows/s", "impl": "reference",
               "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
               "dtype": "f64", "data": "synthetic",
               "config": {"workload": w.name, "B": w.B, "C": w.C, "logits_dtype": w.dtype},
               "cpu_baseline": cb,
               "e2e": {"value": cb["value"], "unit": "rows/s", "h2d_bytes_per_step": 0,
                       "d2h_bytes_per_step": 0}}
        print(json.dumps(out))
        return

    import torch

    import softmax_cross_entropy_row_gb300 as ce

    ce.build()
    ce.load_library()
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    device = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    props = torch.cuda.get_device_properties(device)
    l2_bytes = int(getattr(props, "L2_cache_size", 0) or 126 * 2**20)
    hbm_peak, peak_note = measured_peaks()
    sampler_gpu = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(device.index)).split(",")[0]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else device.index

    names = [w.name] if args.headline_only else [w.name] + [x.name for x in wl.WORKLOADS
                                                            if x.name != w.name]
    results = {}
    for name in names:
        ww = wl.WORKLOADS_BY_NAME[name]
        inp = wl.make_inputs(ww)
        steps = args.steps if name == w.name else None
        results[name] = bench_workload(ww, inp, steps, args.warmup, device, l2_bytes, hbm_peak,
                                       peak_note, sampler_gpu, world,
                                       with_e2e=not args.no_e2e)
        if name == w.name and rank == 0:
            head_inp = inp
        del inp

    next_rows = []
    if not args.headline_only and world == 1:
        for label, name, kind in NEXT_ROWS:
            ww = wl.WORKLOADS_BY_NAME[name]
            next_rows.append(bench_next_row(label, ww, wl.make_inputs(ww), kind, device,
                                            l2_bytes, hbm_peak))

    head = results[w.name]
    cpu = None
    if rank == 0 and world == 1 and args.cpu_sample_s > 0:
        cpu = time_oracle(head_inp, args.cpu_sample_s)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    roof = {"bound": "hbm", "achieved": head["achieved_gbs"], "peak": hbm_peak, "unit": "GB/s",
            "frac": head["frac_of_peak"],
            "traffic": recorded_traffic(w.name, {"path": head["path"], "split": head["split"],
                                                 "ctas": head["ctas"], "threads": head["threads"],
                                                 "smem_bytes": head["smem_bytes"]}),
            "peak_source": peak_note,
            "algorithmic_bytes_per_launch": w.min_bytes,
            "kernel": head["path"]}
    out = {
        "metric": METRIC, "value": head["rows_per_s"], "unit": "rows/s", "n_gpus": world,
        "steps": head["steps"], "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "C": w.C, "logits_dtype": w.dtype,
                   "l2": l2_note(head, w, l2_bytes),
                   "launch": "CUDA graph replay, one ce_fwd_bwd per step",
                   "timing": ("CUDA events on the launching stream; a device-side wait is "
                              "queued before the start event so that host submission "
                              "latency stays outside the timed region"),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": ({k: head["e2e"][k] for k in ("value", "unit", "h2d_bytes_per_step",
                                             "d2h_bytes_per_step", "ms_per_step",
                                             "ms_per_step_median", "ms_per_step_max")}
                if "e2e" in head else None),
        "gpu_launches": world * head["steps"] * head["launches_per_step"],
        "ms_per_step_parts": head["ms_per_step_parts"],
        "clocks": head["clocks"],
        "workloads": [dict(results[n], l2=l2_note(results[n], wl.WORKLOADS_BY_NAME[n], l2_bytes))
                      for n in names],
        "next_rows": next_rows,
    }
    print(json.dumps(out))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
