#!/usr/bin/env python3
"""Benchmark of the fused ZeRO-1 distributed-optimizer step on GB300.

One step = the whole fused step over every bucket of the GPT-2-small-shaped
flat buffer (124,439,808 elements, D=8, 40 Mi buckets padded to multiples
of D*64): reduce-scatter of the D bf16 grad replicas (scaled, fp32, rank
order), fp32 main grads through the range map, AdamW with bias correction
on fp32 master/m/v, bf16 write-back and all-gather into the D param
replicas.  The timed steps are dopt_step_counted calls (step number in a
device counter) captured in CUDA graphs and replayed; the same steps as
plain dopt_step calls (one launch each) are timed too and reported under
"direct".  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (plain C, run on every host core over
disjoint windows) on a bounded sample of the same workload.  With N>1 (torchrun, one
rank per GPU) every rank runs its own replica of the workload: the step has
no data exchange between GPUs, so the ranks only meet for the timing
barrier and the max-over-ranks reduction.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from zero_distributed_optimizer_gb300 import workloads as W  # noqa: E402

METRIC = "fused RS+AdamW+gather elements/s and HBM GB/s (% of ~8 TB/s), 1 GB300"
UNIT = "elements/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "dopt_step_kernel_gpt2_small.md")
KERNEL_SOURCES = [os.path.join(ROOT, "zero_distributed_optimizer_gb300", "csrc", f)
                  for f in ("kernels.cuh", "dopt_internal.h")]
CPU_SAMPLE_ELEMS = 1 << 21
GRAPH_STEPS = 8


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


L2_BYTES = 129 * 10 ** 6


def l2_note(working_set_bytes: int) -> str:
    if working_set_bytes > L2_BYTES:
        return "working set %.1f GB > 129 MB L2, no flush" % (working_set_bytes / 1e9)
    return ("working set %.1f MB fits in the 129 MB L2: a latency figure, not a bandwidth one"
            % (working_set_bytes / 1e6))


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank number over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def strip_c_comments(text: str) -> str:
    """C/C++ source without its comments and blank space: the code tokens,
    one space apart (string and character literals kept as written)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            i = text.find("\n", i)
            i = n if i < 0 else i
        elif text.startswith("/*", i):
            i = text.find("*/", i + 2)
            i = n if i < 0 else i + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """Hash of the device code's tokens (comments and layout left out, so a
    comment edit does not void the stored counters; any code change does)."""
    import hashlib

    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, encoding="utf-8") as f:
            h.update(strip_c_comments(f.read()).encode())
    return h.hexdigest()[:16]


def read_profile_traffic():
    """dram bytes per launch of the step kernel from the committed ncu
    summary, or None if there is none or the kernel changed since."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu_index), "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        inside = [p for t, p in self.samples if t0 - 0.05 <= t <= t1 + 0.05]
        note = "samples during the timed region"
        if not inside:
            mid = 0.5 * (t0 + t1)
            inside = [min(self.samples, key=lambda s: abs(s[0] - mid))[1]]
            note = "timed region shorter than the sampling period: nearest sample"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[2]) for p in inside if num(p[2]) is not None]
        smax = [num(p[3]) for p in inside if num(p[3]) is not None]
        power = [num(p[4]) for p in inside if num(p[4]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4)
                          if p[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_mhz_min": min(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": reasons, "samples": len(inside), "note": note}


def cpu_oracle_rate(w: W.Workload, seconds: float = 12.0, max_steps: int = 40, grads_src=None,
                    state_src=None, sample=CPU_SAMPLE_ELEMS, threads: int = 1):
    """Elements/s of the oracle (as it stands) stepping the first `sample`
    buffer elements of the workload, repeated for about `seconds` seconds.
    With threads > 1 the sample is cut into that many disjoint windows and
    each host thread steps one (the oracle's C call releases the GIL and
    every element depends on its own inputs alone)."""
    from concurrent.futures import ThreadPoolExecutor
    from dataclasses import asdict

    import numpy as np
    import torch

    import oracle
    from zero_distributed_optimizer_gb300.binding import AdamConfig

    oracle.build()
    adam = oracle.make_adam(**asdict(AdamConfig(**w.adam_kwargs())))
    sample = min(sample, oracle.range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit).numel)
    if grads_src is None:
        grads_src = W.make_grads(w, sample, 1, "cpu")
        state_src = W.make_state(w, sample, "cpu")

    def host(t):
        t = t[:sample].detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16).copy()
        return t.numpy().copy()

    grads = [host(g) for g in grads_src]
    master, m, v = (host(x) for x in state_src)
    params = [np.zeros(sample, np.uint16) for _ in range(w.D)]
    sizes, wd = list(w.sizes), list(w.wd_mask)
    threads = max(1, min(threads, sample))
    cuts = [sample * i // threads for i in range(threads + 1)]

    def window(i, t):
        a, b = cuts[i], cuts[i + 1]
        oracle.step(sizes, wd, w.D, w.bucket_elems, w.pad_unit, adam, t,
                    [g[a:b] for g in grads], master[a:b], m[a:b], v[a:b],
                    [p[a:b] for p in params], window=(a, b))

    steps = 0
    with ThreadPoolExecutor(threads) as ex:
        t0 = time.perf_counter()
        while steps < max_steps and (time.perf_counter() - t0) < seconds:
            list(ex.map(window, range(threads), [steps + 1] * threads))
            steps += 1
        dt = time.perf_counter() - t0
    return sample * steps / dt, steps, dt, sample


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


WORKLOADS = ("gpt2_small", "toy_1000", "llama_1p3b", "sweep_256m", "moe_many_small")


def workload_by_name(name: str) -> W.Workload:
    """The named workload; the sweep at its D=8, 64 Mi point."""
    if name == "sweep_256m":
        return W.sweep_256m(8, 64)
    return getattr(W, name)()


def workload_config(w: W.Workload, padded_numel: int, n_buckets: int, world: int) -> dict:
    """The `config` object of the JSON line: the workload alone, the same
    for both arms (how each arm runs it is stated outside `config`)."""
    resident = padded_numel * (w.D * w.grad_bytes + 12 + 2 * w.D)
    return {"workload": w.name, "N": w.numel, "padded_numel": padded_numel, "D": w.D,
            "bucket_elems": w.bucket_elems, "pad_unit": w.pad_unit, "n_buckets": n_buckets,
            "grad_dtype": w.grad_dtype, "state_dtype": "f32", "param_dtype": "bf16",
            "bytes_per_element": w.algorithmic_bytes_per_element(),
            "l2": l2_note(resident),
            # device memory of the step's buffers, and the fp32 master/m/v
            # shard each simulated rank owns (12 bytes per element over D
            # ranks: ZeRO-1's optimizer state)
            "resident_bytes": resident,
            "optimizer_state_bytes_per_rank": 12 * padded_numel // w.D,
            "parallelism": "replicas" if world > 1 else "single"}


def run_reference(args):
    """The oracle arm: rank 0 alone times the CPU oracle on a bounded window."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = workload_by_name(args.workload)
    import torch

    threads = args.cpu_threads or host_threads()
    elems = CPU_SAMPLE_ELEMS * threads
    grads_src = W.make_grads(w, elems, 1, "cpu")
    state_src = W.make_state(w, elems, "cpu")
    cpu_oracle_rate(w, seconds=1e9, max_steps=max(1, args.warmup), grads_src=grads_src,
                    state_src=state_src, sample=elems, threads=threads)
    rate, steps, dt, used = cpu_oracle_rate(w, seconds=1e9, max_steps=args.steps,
                                            grads_src=grads_src, state_src=state_src,
                                            sample=elems, threads=threads)
    sample = (f"first {used} elements of the {w.name} buffer (D={w.D}), "
              f"{steps} oracle steps, {threads} host threads on disjoint windows")
    import oracle

    O = oracle.range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit)
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / max(steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": workload_config(w, O.numel, O.n_buckets, world),
        "path": "the CPU oracle (plain C) stepping a bounded sample of the buffer",
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "torch": torch.__version__,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch

    from zero_distributed_optimizer_gb300 import binding as B
    from zero_distributed_optimizer_gb300 import build as libbuild

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())
    if rank == 0:
        libbuild.build()
    if world > 1:
        torch.distributed.barrier()

    w = workload_by_name(args.workload)
    L = B.dopt_build_range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit,
                               list(w.wd_mask)).to_device()
    N = L.padded_numel
    master, m, v = W.make_state(w, N, device)
    params = W.make_params(master, w.D)
    grads = W.make_grads(w, N, 1, device)
    adam = B.AdamConfig(**w.adam_kwargs())
    stream = torch.cuda.current_stream()

    def step(t):
        B.dopt_step(L, adam, t, grads, master, m, v, params, gather=True, stream=stream)

    t = 0
    for _ in range(max(args.warmup, 3)):
        t += 1
        step(t)
    torch.cuda.synchronize()

    # The timed path: dopt_step_counted (the step number lives in a device
    # counter, so the launches do not depend on it) captured GRAPH_STEPS at a
    # time in a CUDA graph, plus one graph for the remainder of K, replayed
    # until exactly K steps are done.  Each step is two launches: a counter
    # kernel of two threads, then the step kernel.
    per = GRAPH_STEPS
    counter = B.step_counter(t + 1, device)
    B.dopt_step_counted(L, adam, counter, grads, master, m, v, params)  # kernels loaded
    torch.cuda.synchronize()
    graphs = {}
    for n in sorted({per, args.steps % per} - {0}):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(n):
                B.dopt_step_counted(L, adam, counter, grads, master, m, v, params)
        graphs[n] = g
    taken = 1
    for _ in range(max(args.warmup, 3)):
        graphs[per].replay()
        taken += per
    torch.cuda.synchronize()

    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    # let the sampler come up and the clocks settle under the same load
    settle_end = time.time() + 0.4
    settled = 0
    s0 = time.time()
    while time.time() < settle_end:
        graphs[per].replay()
        taken += per
        settled += per
        torch.cuda.synchronize()
    est_ms = 1e3 * (time.time() - s0) / max(settled, 1)

    # The timed region: R repeats of exactly K steps, each bracketed by a
    # barrier and a synchronize on both sides and timed with CUDA events;
    # the reported time per step is the median over the repeats.  R is at
    # least 5 and large enough that the repeats cover about
    # --timed-seconds, so that the clock sampler sees the load several times.
    repeats = args.repeats or max(5, min(1000, int(args.timed_seconds /
                                                   max(args.steps * est_ms / 1e3, 1e-6)) + 1))
    rep_ms = []
    h0 = time.time()
    for _ in range(repeats):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(args.steps // per):
            graphs[per].replay()
        if args.steps % per:
            graphs[args.steps % per].replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        rep_ms.append(max_over_ranks(ev0.elapsed_time(ev1), world, device))
        taken += args.steps
    h1 = time.time()
    sampler.stop()
    next_step, status = B.counter_state(counter)
    assert status == 0 and next_step == t + 1 + taken, (next_step, status, t, taken)
    t = next_step - 1
    del graphs
    ms_total = statistics.median(rep_ms)
    ms_per_step = ms_total / args.steps

    elems = w.numel
    value = world * elems * args.steps / (ms_total / 1e3)
    bytes_per_launch = elems * w.algorithmic_bytes_per_element()
    gbs = bytes_per_launch / (ms_per_step / 1e3) / 1e9
    peak, peak_kind = measured_hbm_peak()
    traffic = read_profile_traffic()

    # the same K steps as one dopt_step call each (one launch per step, the
    # step number a host argument), 5 repeats, the median reported
    d_reps = []
    for _ in range(5):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        for _ in range(args.steps):
            t += 1
            step(t)
        d1.record(stream)
        torch.cuda.synchronize()
        d_reps.append(max_over_ranks(d0.elapsed_time(d1), world, device) / args.steps)
    d_ms = statistics.median(d_reps)
    direct = {"ms_per_step": d_ms, "value": world * elems / (d_ms / 1e3), "unit": UNIT,
              "launches_per_step": 1, "repeats": len(d_reps),
              "path": "binding.dopt_step, one call (one kernel launch) per step, each a "
                      "programmatic dependent of the one before"}

    # end to end through the public API: grads from pinned host memory,
    # updated params (replica 0) back to pinned host memory, every step
    e2e = None
    if not args.no_e2e:
        # through the public API with the grads in pinned host memory, both
        # ways the library offers: staged (copy to device, then the step) and
        # zero-copy (the kernel reads the host replicas over the host link)
        host_grads = [g.cpu().pin_memory() for g in grads]
        host_out = torch.empty(N, dtype=torch.bfloat16).pin_memory()
        dev_stage = [torch.empty_like(g) for g in grads]
        k_e2e = max(3, min(args.steps, 20))
        variants = {}
        stepper = B.HostStepper(L, adam, master, m, v, params, host_out, stream=stream)

        def one(name, t):
            if name == "pipelined":
                stepper.step(t, host_grads)
            else:
                B.step_from_host(L, adam, t, host_grads, dev_stage, master, m, v, params,
                                 host_out, stream=stream,
                                 zero_copy=name in ("zero_copy", "in_place_out"),
                                 params_out_in_place=name == "in_place_out")

        for name in ("staged", "zero_copy", "pipelined", "in_place_out"):
            for _ in range(2):
                t += 1
                one(name, t)
            stepper.synchronize()
            torch.cuda.synchronize()
            if world > 1:
                torch.distributed.barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(k_e2e):
                t += 1
                one(name, t)
            stepper.synchronize()  # the last result is on the host inside the timed region
            e1.record(stream)
            torch.cuda.synchronize()
            variants[name] = max_over_ranks(e0.elapsed_time(e1), world, device) / k_e2e
        best = min(variants, key=variants.get)
        e2e = {"value": world * elems / (variants[best] / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in host_grads),
               "d2h_bytes_per_step": host_out.numel() * host_out.element_size(),
               "steps": k_e2e, "ms_per_step": variants[best],
               "path": {"staged": "binding.step_from_host: H2D copy of the D grad replicas, "
                                  "dopt_step, D2H of param replica 0",
                        "zero_copy": "binding.step_from_host(zero_copy): dopt_step reads the "
                                     "pinned host grads in place, D2H of param replica 0",
                        "pipelined": "binding.HostStepper: zero-copy step, param replica 0 "
                                     "staged on the device and copied to the host on a side "
                                     "stream while the next step runs",
                        "in_place_out": "binding.step_from_host(zero_copy, params_out_in_place): "
                                        "dopt_step reads the pinned host grads in place and "
                                        "writes param replica 0 straight into pinned host "
                                        "memory (the other 7 replicas on the device)"}[best],
               "ms_per_step_by_variant": variants}
        del host_grads, host_out, dev_stage

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = args.cpu_threads or host_threads()
        rate1, steps1, dt1, used1 = cpu_oracle_rate(w, seconds=args.cpu_seconds / 2,
                                                    grads_src=grads, state_src=(master, m, v))
        rate, steps_done, dt, used = cpu_oracle_rate(
            w, seconds=args.cpu_seconds / 2, grads_src=grads, state_src=(master, m, v),
            sample=CPU_SAMPLE_ELEMS * threads, threads=threads)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"first {used} elements of the {w.name} buffer, {steps_done} oracle "
                         f"steps in {dt:.1f} s, {threads} host threads on disjoint windows",
               "one_thread": {"value": rate1, "cores": 1,
                              "sample": f"first {used1} elements, {steps1} oracle steps in "
                                        f"{dt1:.1f} s"}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "repeats": repeats,
            "ms_per_step_spread": {"min": min(rep_ms) / args.steps,
                                   "median": ms_per_step,
                                   "max": max(rep_ms) / args.steps,
                                   "note": f"{repeats} repeats of the {args.steps} timed steps, "
                                           "each bracketed by barrier + synchronize; value and "
                                           "ms_per_step use the median repeat"},
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": workload_config(w, N, L.n_buckets, world),
            "path": f"binding.dopt_step_counted, {GRAPH_STEPS} steps per CUDA graph, replayed "
                    "(a counter kernel and the step kernel per step)",
            "hbm_gbs": gbs, "pct_of_8tbs": gbs / NOMINAL_HBM_GBS,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                         "frac": gbs / peak, "peak_kind": peak_kind,
                         "traffic": traffic,
                         "kernel": "dopt_step_kernel (the counter kernel's time is "
                                   "included in the step time it divides by)",
                         "algorithmic_bytes_per_launch": bytes_per_launch},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "direct": direct,
            "gpu_launches": 2 * args.steps * repeats,
            "clocks": sampler.summary(h0, h1),
            "torch": torch.__version__,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="wall time of the CPU-baseline legs (one thread, all threads)")
    ap.add_argument("--cpu-threads", type=int, default=0,
                    help="host threads of the oracle runs (0: every core this process may use)")
    ap.add_argument("--repeats", type=int, default=0,
                    help="repeats of the K timed steps (0: at least 5, enough to cover "
                         "--timed-seconds)")
    ap.add_argument("--timed-seconds", type=float, default=1.0,
                    help="device time the repeats of the timed region should cover")
    ap.add_argument("--workload", choices=WORKLOADS, default="gpt2_small",
                    help="the GPT-2-small layout is the configuration of the reported metric")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
