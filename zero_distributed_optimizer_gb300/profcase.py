"""Run a few launches of the fused step on one workload, for profilers.

    python -m zero_distributed_optimizer_gb300.profcase --workload gpt2_small \
        [--max-elems N] [--warmup W] [--launches K] [--mode MODE]
    python -m zero_distributed_optimizer_gb300.profcase --probe R,W[;R,W...] [--mib M]
    python -m zero_distributed_optimizer_gb300.profcase --workload gpt2_small --ab-stage ROUNDS

--probe times the stream probe (dopt_stream_probe) for each mix of R read
and W write streams of M MiB each: the HBM's ceiling for that mix.

--ab-stage times the step (or the counted step) with direct loads and with
DOPT_STEP_STAGE alternately in one process on the same buffers, ROUNDS
rounds of --launches launches each, and prints the best of each.

--max-elems keeps the leading params of the workload whose total stays
within N elements, so that a profiler capture can run on a smaller buffer of
the same shape mix.  Inputs come from the seeded workload generators.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def truncated(w, max_elems):
    if not max_elems or w.numel <= max_elems:
        return w
    sizes, wd, total = [], [], 0
    for s, d in zip(w.sizes, w.wd_mask):
        if total + s > max_elems:
            if not sizes:  # a single param larger than the cap: cut it
                sizes.append(max_elems)
                wd.append(d)
            break
        sizes.append(s)
        wd.append(d)
        total += s
    return w.with_(name=f"{w.name}_first{sum(sizes)}", sizes=tuple(sizes), wd_mask=tuple(wd))


def main(argv=None):
    import torch

    from zero_distributed_optimizer_gb300 import binding as B
    from zero_distributed_optimizer_gb300 import build as libbuild
    from zero_distributed_optimizer_gb300 import workloads as W

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="gpt2_small",
                    choices=["toy_1000", "gpt2_small", "llama_1p3b", "sweep_256m", "moe_many_small"])
    ap.add_argument("--D", type=int, default=8, help="sweep_256m only")
    ap.add_argument("--bucket-mi", type=int, default=64, help="sweep_256m only")
    ap.add_argument("--max-elems", type=int, default=0)
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--mode", default="step",
                    choices=["step", "gather", "clipped", "buckets", "buckets_graph", "allreduce",
                             "step_allreduce", "counted"],
                    help="the fused step, dopt_gather alone, the clipped step, the step as "
                         "one launch per bucket, dopt_allreduce alone, the step with "
                         "force_all_reduce, or the counted step (step number on the device)")
    ap.add_argument("--streams", type=int, default=1,
                    help="buckets mode: bucket k is launched on stream k mod STREAMS")
    ap.add_argument("--plan", action="store_true",
                    help="step and buckets modes: launch through a StepPlan")
    ap.add_argument("--grad-dtype", choices=["bf16", "fp16", "fp32"], default=None,
                    help="override the workload's grad type")
    ap.add_argument("--param-dtype", choices=["bf16", "fp16"], default="bf16")
    ap.add_argument("--instances", type=int, default=1,
                    help="distributed-optimizer instances (D must divide by it)")
    ap.add_argument("--probe", default="",
                    help="mixes 'R,W;R,W;...' of read and write streams for the stream probe "
                         "(the workload is then not used)")
    ap.add_argument("--mib", type=int, default=256, help="--probe: MiB per stream")
    ap.add_argument("--stage", action="store_true",
                    help="step, counted and buckets modes: read through shared memory with "
                         "bulk copies (DOPT_STEP_STAGE)")
    ap.add_argument("--ab-stage", type=int, default=0, metavar="ROUNDS",
                    help="step and counted modes: alternate direct and staged launches for "
                         "ROUNDS rounds and print the best time of each")
    args = ap.parse_args(argv)

    libbuild.build()
    if args.probe:
        return probe(args)
    if args.workload == "sweep_256m":
        w = W.sweep_256m(args.D, args.bucket_mi)
    else:
        w = getattr(W, args.workload)()
    w = truncated(w, args.max_elems)
    if args.grad_dtype:
        w = w.with_(grad_dtype=args.grad_dtype)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    L = B.dopt_build_range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit,
                               list(w.wd_mask), instances=args.instances).to_device(dev)
    N = L.padded_numel
    master, m, v = W.make_state(w, N, dev)
    params = W.make_params(master, w.D)
    if args.param_dtype == "fp16":
        params = [p.float().half() for p in params]
    grads = W.make_grads(w, N, 1, dev)
    adam = B.AdamConfig(**w.adam_kwargs())
    if args.mode == "clipped":
        main_grad = torch.empty(N, device=dev)
        ws = B.clip_workspace(dev)
    streams = [torch.cuda.current_stream()] + [torch.cuda.Stream(dev) for _ in range(args.streams - 1)]
    plan = B.StepPlan(L, adam, grads, master, m, v, params, stage=args.stage) if args.plan else None

    def bucket_launches(t):
        # fork the side streams off the main one, launch, join them back
        fork = torch.cuda.Event()
        fork.record(streams[0])
        for s_ in streams[1:]:
            s_.wait_event(fork)
        for k in range(L.n_buckets):
            s_ = streams[k % len(streams)]
            if plan is not None:
                plan.step_buckets(t, k, 1, stream=s_)
            else:
                B.dopt_step_buckets(L, adam, t, k, 1, grads, master, m, v, params, stream=s_,
                                    stage=args.stage)
        for s_ in streams[1:]:
            join = torch.cuda.Event()
            join.record(s_)
            streams[0].wait_event(join)

    counter = B.step_counter(1, dev) if args.mode == "counted" else None
    graph = None
    if args.mode == "buckets_graph":
        # the per-bucket launches of one step recorded once and replayed: the
        # replays repeat the same step count (same bias corrections); they
        # time the device side of per-bucket stepping without host submission
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            streams[0] = side
            bucket_launches(1)  # warm-up outside the capture
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                bucket_launches(1)
        torch.cuda.current_stream().wait_stream(side)
        streams[0] = torch.cuda.current_stream()
    torch.cuda.synchronize()
    if args.ab_stage:
        return ab_stage(args, w, L, adam, grads, master, m, v, params, counter)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    t = 0
    for i in range(args.warmup + args.launches):
        if i == args.warmup:
            ev[0].record()
        t += 1
        if args.mode == "gather":
            B.dopt_gather(L, params)
        elif args.mode == "buckets":
            bucket_launches(t)
        elif args.mode == "buckets_graph":
            graph.replay()
        elif args.mode == "allreduce":
            B.dopt_allreduce(L, grads, 1.0)
        elif args.mode == "step_allreduce":
            B.dopt_step_allreduce(L, adam, t, grads, master, m, v, params)
        elif args.mode == "clipped":
            B.dopt_step_clipped(L, adam, t, 1.0, grads, master, m, v, params, main_grad, ws)
        elif args.mode == "counted":
            B.dopt_step_counted(L, adam, counter, grads, master, m, v, params, stage=args.stage)
        elif plan is not None:
            plan.step(t)
        else:
            B.dopt_step(L, adam, t, grads, master, m, v, params, stage=args.stage)
    ev[1].record()
    torch.cuda.synchronize()
    ms = ev[0].elapsed_time(ev[1]) / max(args.launches, 1)
    step_bytes = w.algorithmic_bytes_per_element()
    per_elem = {"gather": 2 * w.D, "step": step_bytes, "buckets": step_bytes,
                "buckets_graph": step_bytes, "counted": step_bytes,
                "clipped": step_bytes + 8, "allreduce": 2 * w.D * w.grad_bytes,
                "step_allreduce": step_bytes + w.D * w.grad_bytes}[args.mode]
    bytes_per = w.numel * per_elem
    print(json.dumps({"workload": w.name, "N": w.numel, "padded_numel": N, "D": w.D,
                      "mode": args.mode, "grad_dtype": w.grad_dtype, "param_dtype": args.param_dtype,
                      "instances": args.instances, "stage": args.stage,
                      "n_buckets": L.n_buckets, "streams": args.streams, "plan": args.plan,
                      "launches": args.launches, "ms_per_launch": ms,
                      "algorithmic_bytes_per_launch": bytes_per,
                      "gbs": bytes_per / (ms / 1e3) / 1e9}))


def ab_stage(args, w, L, adam, grads, master, m, v, params, counter):
    """Direct loads against DOPT_STEP_STAGE, alternating: `warmup` launches
    of each, then `ab_stage` rounds of `launches` launches of each, CUDA
    events around every round; the best round of each is reported."""
    import torch

    from zero_distributed_optimizer_gb300 import binding as B

    if args.mode not in ("step", "counted"):
        raise SystemExit("--ab-stage takes --mode step or counted")
    t = 0

    def launch(stage):
        nonlocal t
        t += 1
        if args.mode == "counted":
            B.dopt_step_counted(L, adam, counter, grads, master, m, v, params, stage=stage)
        else:
            B.dopt_step(L, adam, t, grads, master, m, v, params, stage=stage)

    for stage in (False, True):
        for _ in range(args.warmup):
            launch(stage)
    times = {False: [], True: []}
    for _ in range(args.ab_stage):
        for stage in (False, True):
            torch.cuda.synchronize()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            ev[0].record()
            for _ in range(args.launches):
                launch(stage)
            ev[1].record()
            torch.cuda.synchronize()
            times[stage].append(ev[0].elapsed_time(ev[1]) / args.launches)
    bytes_per = w.numel * w.algorithmic_bytes_per_element()
    out = {"workload": w.name, "N": w.numel, "D": w.D, "mode": args.mode, "grad_dtype": w.grad_dtype,
           "launches": args.launches, "rounds": args.ab_stage}
    for stage, name in ((False, "direct"), (True, "staged")):
        best = min(times[stage])
        out[name] = {"ms_per_launch": best, "gbs": bytes_per / (best / 1e3) / 1e9,
                     "rounds_ms": times[stage]}
    out["staged_over_direct"] = out["staged"]["ms_per_launch"] / out["direct"]["ms_per_launch"]
    print(json.dumps(out), flush=True)


def probe(args):
    """Bandwidth of each read/write stream mix: CUDA events around
    `launches` probe launches captured in a CUDA graph (so that host
    submission never limits short launches), after `warmup` direct ones,
    best of three replays."""
    import torch

    from zero_distributed_optimizer_gb300 import binding as B

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    n = args.mib << 20
    for mix in args.probe.split(";"):
        reads, writes = (int(x) for x in mix.split(","))
        rb = [torch.full((n // 4,), float(i + 1), device=dev) for i in range(reads)]
        wb = [torch.empty(n // 4, device=dev) for _ in range(writes)]
        for _ in range(args.warmup):
            B.dopt_stream_probe(rb, wb)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side), torch.cuda.graph(graph, stream=side):
            for _ in range(args.launches):
                B.dopt_stream_probe(rb, wb)
        torch.cuda.current_stream().wait_stream(side)
        best = float("inf")
        for _ in range(3):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            ev[0].record()
            graph.replay()
            ev[1].record()
            torch.cuda.synchronize()
            best = min(best, ev[0].elapsed_time(ev[1]) / args.launches)
        del graph
        moved = (reads + writes) * n
        print(json.dumps({"mode": "probe", "reads": reads, "writes": writes, "mib_per_stream": args.mib,
                          "ms_per_launch": best, "bytes_per_launch": moved,
                          "gbs": moved / (best / 1e3) / 1e9}), flush=True)
        del rb, wb
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
