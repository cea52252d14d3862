"""Launch order between the library's kernels.

The step, all-reduce and gather kernels let their dependents start while
their last wave runs, and are themselves launched as programmatic
dependents of the kernel before them: their CTAs may become resident early
but must not read or write grads, state or params before that kernel has
completed.  These tests run chains of launches back to back on one stream
(and captured in a CUDA graph), with torch kernels that rewrite the inputs
in between, and require every buffer to equal the same launches with a
device synchronisation after each, bit for bit."""
import pytest
import torch

from zero_distributed_optimizer_gb300 import binding as B
from zero_distributed_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(D=8, seed=0):
    sizes, wd = [300000, 5, 70001, 4096, 123], [1, 0, 1, 1, 0]
    L = B.dopt_build_range_map(sizes, D, 100000, 64, wd).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, 4, "bf16", seed=seed)
    state = [master.to(DEV), m.to(DEV), v.to(DEV)]
    return L, N, state, [p.to(DEV) for p in params], [[g.to(DEV) for g in gs] for gs in grads]


def _clone(xs):
    return [x.clone() for x in xs]


def _equal(xs, ys):
    for x, y in zip(xs, ys):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def _chain(L, N, state, params, grads, sync):
    """Steps, an all-reduce, a step without the gather, the gather and a
    clipped step, with torch kernels rewriting the grads and the state in
    between; `sync` synchronises after every launch."""
    D = L.D
    adam = B.AdamConfig(grad_scale=1.0 / D)
    work = [g.clone() for g in grads[0]]
    mg = torch.zeros(N, device=DEV)
    ws = B.clip_workspace(DEV)
    done = (lambda: torch.cuda.synchronize()) if sync else (lambda: None)
    for t in (1, 2, 3):
        for w, g in zip(work, grads[t]):  # torch kernels: new grads for this step
            w.copy_(g)
        done()
        B.dopt_step(L, adam, t, work, *state, params)
        done()
    state[0].mul_(0.999)  # a torch kernel on the state the next launch reads
    done()
    B.dopt_allreduce(L, work, 1.0 / D)
    done()
    B.dopt_step(L, adam, 4, work, *state, params, gather=False)
    done()
    B.dopt_gather(L, params)
    done()
    B.dopt_step_clipped(L, adam, 5, 0.05, work, *state, params, mg, ws)
    done()
    B.dopt_step(L, adam, 6, work, *state, params, main_grad_out=mg)
    torch.cuda.synchronize()
    return state + params + work + [mg]


def test_back_to_back_launches_equal_synchronised_ones():
    L, N, state, params, grads = _case(seed=1)
    a = _chain(L, N, _clone(state), _clone(params), grads, sync=False)
    b = _chain(L, N, _clone(state), _clone(params), grads, sync=True)
    _equal(a, b)


def test_launch_chain_replayed_from_a_graph():
    """The same chain (fixed step numbers) captured once and replayed twice
    on fresh copies of the inputs gives the eager chain's buffers."""
    L, N, state, params, grads = _case(D=4, seed=2)
    want = _chain(L, N, _clone(state), _clone(params), grads, sync=True)
    s, p = _clone(state), _clone(params)
    _chain(L, N, _clone(state), _clone(params), grads, sync=False)  # warm-up: kernels loaded
    torch.cuda.synchronize()
    s0, p0 = _clone(s), _clone(p)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            out = _graph_chain(L, N, s, p, grads)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        for x, x0 in zip(s + p, s0 + p0):
            x.copy_(x0)
        graph.replay()
        torch.cuda.synchronize()
        _equal(out, want)


def _graph_chain(L, N, state, params, grads):
    """_chain without its final synchronisation (not allowed in a capture)."""
    D = L.D
    adam = B.AdamConfig(grad_scale=1.0 / D)
    work = [torch.empty_like(g) for g in grads[0]]
    mg = torch.zeros(N, device=DEV)
    ws = B.clip_workspace(DEV)
    for t in (1, 2, 3):
        for w, g in zip(work, grads[t]):
            w.copy_(g)
        B.dopt_step(L, adam, t, work, *state, params)
    state[0].mul_(0.999)
    B.dopt_allreduce(L, work, 1.0 / D)
    B.dopt_step(L, adam, 4, work, *state, params, gather=False)
    B.dopt_gather(L, params)
    B.dopt_step_clipped(L, adam, 5, 0.05, work, *state, params, mg, ws)
    B.dopt_step(L, adam, 6, work, *state, params, main_grad_out=mg)
    return state + params + work + [mg]
