"""dopt_step_counted: the step number read from, and advanced in, a device
counter.  It must give dopt_step's results bit for bit at every step
number, replay from a CUDA graph, and refuse bad step numbers on the
device without touching anything."""
from dataclasses import asdict

import numpy as np
import pytest
import torch

import oracle
from parity import assert_bf16_close, assert_f32_close, t2np_bf16, t2np_f32
from zero_distributed_optimizer_gb300 import binding as B
from zero_distributed_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(sizes, wd, D, bucket, pad, grad_dtype="bf16", steps=3, seed=0, instances=1):
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd, instances=instances).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, steps, grad_dtype, seed)
    state = [master.to(DEV), m.to(DEV), v.to(DEV)]
    dparams = [p.to(DEV) for p in params]
    dgrads = [[g.to(DEV) for g in gs] for gs in grads]
    return L, state, dparams, dgrads, (master, m, v, params, grads)


def _clone(state, params):
    return [x.clone() for x in state], [p.clone() for p in params]


def _equal(a, b):
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("D,instances,grad_dtype", [(4, 1, "bf16"), (8, 2, "fp32"), (3, 1, "bf16"),
                                                     (16, 1, "fp32"), (8, 2, "bf16"),
                                                     (16, 4, "fp16")])
def test_counted_equals_host_step(D, instances, grad_dtype):
    L, s, p, g, _ = _case([5000, 1, 7, 300, 20000, 3, 9999], [1, 0, 1, 0, 1, 1, 0], D, 9000, 8,
                          grad_dtype, seed=D, instances=instances)
    s2, p2 = _clone(s, p)
    mg, mg2 = (torch.full((L.padded_numel,), -2.0, device=DEV) for _ in range(2))
    adam = B.AdamConfig(grad_scale=1.0 / D)
    counter = B.step_counter(1)
    for t in range(1, 4):
        B.dopt_step(L, adam, t, g[t - 1], *s, p, main_grad_out=mg)
        B.dopt_step_counted(L, adam, counter, g[t - 1], *s2, p2, main_grad_out=mg2)
    torch.cuda.synchronize()
    _equal(s + p + [mg], s2 + p2 + [mg2])
    assert B.counter_state(counter) == (4, 0)


def test_counted_against_oracle():
    sizes, wd, D, bucket, pad = [4096, 333, 12345, 8, 77777], [0, 1, 1, 0, 1], 6, 20000, 1
    L, s, p, g, host = _case(sizes, wd, D, bucket, pad, "bf16", steps=3, seed=44, instances=3)
    master, m, v, params, grads = host
    h = [master.numpy().copy(), m.numpy().copy(), v.numpy().copy()]
    hp = [t2np_bf16(x).copy() for x in params]
    adam = B.AdamConfig(grad_scale=1.0 / D)
    oadam = oracle.make_adam(**asdict(adam))
    counter = B.step_counter(1)
    for t in range(1, 4):
        B.dopt_step_counted(L, adam, counter, g[t - 1], *s, p, gather=(t != 2))
        oracle.step(sizes, wd, D, bucket, pad, oadam, t, [t2np_bf16(x) for x in grads[t - 1]],
                    *h, hp, gather=(t != 2), instances=3)
    torch.cuda.synchronize()
    for name, x, y in zip(("master", "exp_avg", "exp_avg_sq"), s, h):
        assert_f32_close(t2np_f32(x), y, name)
    for r in range(D):
        assert_bf16_close(t2np_bf16(p[r]), hp[r], f"param{r}")


def test_counted_scalars_at_any_step_number():
    """One step at step number t from the same state, counted vs host step
    number, for t from 1 to 2^62: the device's scalars equal the host's."""
    L, s0, p0, g, _ = _case([3000, 17, 2500], [1, 0, 1], 2, 0, 8, steps=1, seed=3)
    adam = B.AdamConfig(lr=3e-3, beta1=0.85, beta2=0.97, grad_scale=0.5)
    for t in [1, 2, 3, 7, 10, 99, 1000, 12345, 10 ** 6, 10 ** 9, 2 ** 40, 2 ** 62]:
        a, pa = _clone(s0, p0)
        b, pb = _clone(s0, p0)
        counter = B.step_counter(t)
        B.dopt_step(L, adam, t, g[0], *a, pa)
        B.dopt_step_counted(L, adam, counter, g[0], *b, pb)
        torch.cuda.synchronize()
        _equal(a + pa, b + pb)
        assert B.counter_state(counter) == (t + 1, 0), t


def test_counted_graph_replay():
    """One counted step captured in a CUDA graph, replayed 5 times, equals 5
    host steps; the counter ends at 6."""
    L, s, p, g, _ = _case([65536, 1000, 65536, 3], [1, 0, 1, 0], 8, 0, 64, steps=1, seed=8)
    s2, p2 = _clone(s, p)
    adam = B.AdamConfig(grad_scale=1.0 / 8)
    # warm-up on scratch copies, so that every kernel is loaded before capture
    ws, wp = _clone(s, p)
    B.dopt_step_counted(L, adam, B.step_counter(1), g[0], *ws, wp)
    torch.cuda.synchronize()
    counter = B.step_counter(1)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        B.dopt_step_counted(L, adam, counter, g[0], *s2, p2)
    assert B.counter_state(counter) == (1, 0)  # capture ran nothing
    for _ in range(5):
        graph.replay()
    for t in range(1, 6):
        B.dopt_step(L, adam, t, g[0], *s, p)
    torch.cuda.synchronize()
    _equal(s + p, s2 + p2)
    assert B.counter_state(counter) == (6, 0)


@pytest.mark.parametrize("bad", [0, -5, -(2 ** 63), 2 ** 62 + 1])
def test_counted_bad_step_number_changes_nothing(bad):
    L, s, p, g, _ = _case([700, 300], None, 4, 0, 1, steps=1, seed=1)
    before = [x.clone() for x in s + p]
    mg = torch.full((L.padded_numel,), 3.0, device=DEV)
    counter = B.step_counter(bad)
    B.dopt_step_counted(L, B.AdamConfig(), counter, g[0], *s, p, main_grad_out=mg)
    torch.cuda.synchronize()
    _equal(before, s + p)
    assert torch.all(mg == 3.0)
    assert B.counter_state(counter) == (bad, B.DOPT_COUNTER_BAD_STEP)
    counter[0] = 1  # a good number again: the next launch steps and clears the status
    B.dopt_step_counted(L, B.AdamConfig(), counter, g[0], *s, p)
    torch.cuda.synchronize()
    assert B.counter_state(counter) == (2, 0)
    assert not torch.equal(before[0], s[0])


def test_counted_empty_layout_still_counts():
    L = B.dopt_build_range_map([0, 0], 2, 0, 1).to_device()
    z = torch.zeros(8, device=DEV)
    zb = torch.zeros(8, device=DEV, dtype=torch.bfloat16)
    counter = B.step_counter(5)
    B.dopt_step_counted(L, B.AdamConfig(), counter, [zb, zb.clone()], z, z.clone(), z.clone(),
                        [zb.clone(), zb.clone()])
    assert B.counter_state(counter) == (6, 0)


def test_step_plan_counted():
    L, s, p, g, _ = _case([9000] * 7, [1, 0] * 3 + [1], 7, 10000, 2, steps=1, seed=12)
    s2, p2 = _clone(s, p)
    adam = B.AdamConfig(grad_scale=1.0 / 7)
    c1, c2 = B.step_counter(1), B.step_counter(1)
    plan = B.StepPlan(L, adam, g[0], *s2, p2)
    for _ in range(3):
        B.dopt_step_counted(L, adam, c1, g[0], *s, p)
        plan.step_counted(c2)
    torch.cuda.synchronize()
    _equal(s + p, s2 + p2)
    assert B.counter_state(c1) == B.counter_state(c2) == (4, 0)
    with pytest.raises(B.DoptError):
        plan.step_counted(torch.zeros(8, dtype=torch.int32, device=DEV))


def test_counted_gpt2_small_every_element():
    """The GPT-2-small buffer, 3 counted steps replayed from one graph,
    against 3 host-numbered steps, every element bit for bit."""
    w = W.gpt2_small()
    L = B.dopt_build_range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit,
                               list(w.wd_mask)).to_device()
    N = L.padded_numel
    master, m, v = W.make_state(w, N, DEV)
    params = W.make_params(master, w.D)
    grads = W.make_grads(w, N, 1, DEV)
    adam = B.AdamConfig(**w.adam_kwargs())
    a = [master.clone(), m.clone(), v.clone()]
    pa = [x.clone() for x in params]
    counter = B.step_counter(1)
    graph = torch.cuda.CUDAGraph()
    B.dopt_step_counted(L, adam, B.step_counter(1), grads, *[x.clone() for x in a],
                        [x.clone() for x in pa])  # warm-up
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        B.dopt_step_counted(L, adam, counter, grads, master, m, v, params)
    for t in range(1, 4):
        graph.replay()
        B.dopt_step(L, adam, t, grads, *a, pa)
    torch.cuda.synchronize()
    _equal([master, m, v] + params, a + pa)
    assert B.counter_state(counter) == (4, 0)
    del graph
    assert np.isfinite(t2np_f32(master[:1000])).all()


FIRST_USE = r"""
import torch
from zero_distributed_optimizer_gb300 import binding as B
L = B.dopt_build_range_map([3000, 17, 2500], 2, 0, 8, [1, 0, 1]).to_device()
N = L.padded_numel
gen = torch.Generator(device="cuda").manual_seed(4)
grads = [(torch.randn(N, device="cuda", generator=gen) * 1e-3).bfloat16() for _ in range(2)]
state = [torch.randn(N, device="cuda", generator=gen) * 0.02, torch.zeros(N, device="cuda"),
         torch.zeros(N, device="cuda")]
params = [state[0].bfloat16() for _ in range(2)]
ref = [x.clone() for x in state], [p.clone() for p in params]
adam = B.AdamConfig(grad_scale=0.5)
counter = B.step_counter(1)
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g):  # the library's first launches happen inside the capture
    B.dopt_step_counted(L, adam, counter, grads, *state, params)
for _ in range(3):
    g.replay()
for t in range(1, 4):
    B.dopt_step(L, adam, t, grads, *ref[0], ref[1])
torch.cuda.synchronize()
for x, y in zip(state + params, ref[0] + ref[1]):
    assert torch.equal(x.view(torch.int16), y.view(torch.int16))
assert B.counter_state(counter) == (4, 0)
print("ok")
"""


def test_counted_capture_as_first_use():
    """In a fresh process the first launches of the library can be the
    captured ones (kernels are loaded on first use)."""
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "-c", FIRST_USE], capture_output=True, text=True,
                         timeout=300, cwd=root)
    assert out.returncode == 0 and out.stdout.strip().endswith("ok"), out.stdout + out.stderr


def test_several_counted_steps_in_one_graph():
    """Four counted steps captured in one graph (each counter kernel a
    programmatic dependent of the step kernel before it), replayed three
    times, with the counter moved by the caller between replays, equal host
    steps at the same step numbers."""
    L, s, p, g, _ = _case([65536, 1000, 65536, 3], [1, 0, 1, 0], 8, 0, 64, steps=1, seed=18)
    s2, p2 = _clone(s, p)
    adam = B.AdamConfig(grad_scale=1.0 / 8)
    ws, wp = _clone(s, p)
    B.dopt_step_counted(L, adam, B.step_counter(1), g[0], *ws, wp)  # kernels loaded
    torch.cuda.synchronize()
    counter = B.step_counter(1)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(4):
            B.dopt_step_counted(L, adam, counter, g[0], *s2, p2)
    numbers = []
    for start in (1, 100, 5):
        counter[0] = start
        graph.replay()
        numbers += list(range(start, start + 4))
    for t in numbers:
        B.dopt_step(L, adam, t, g[0], *s, p)
    torch.cuda.synchronize()
    _equal(s + p, s2 + p2)
    assert B.counter_state(counter) == (9, 0)


def test_counted_after_a_counter_write_on_the_stream():
    """A caller's kernel that rewrites the counter right before the counted
    step: the counter kernel, started early, must use the rewritten number."""
    L, s, p, g, _ = _case([3000, 17, 2500], [1, 0, 1], 2, 0, 8, steps=1, seed=21)
    s2, p2 = _clone(s, p)
    adam = B.AdamConfig(lr=2e-3, grad_scale=0.5)
    counter = B.step_counter(1)
    for t in (7, 8, 1234, 3):
        counter.fill_(t)  # the last 7 elements are scratch: zeroed or rewritten by the step
        counter[1:].zero_()
        B.dopt_step_counted(L, adam, counter, g[0], *s2, p2)
        B.dopt_step(L, adam, t, g[0], *s, p)
    torch.cuda.synchronize()
    _equal(s + p, s2 + p2)
    assert B.counter_state(counter) == (4, 0)


def _clip_case(seed=31, grad_dtype="bf16", instances=1):
    return _case([5000, 1, 7, 300, 20000, 3, 9999], [1, 0, 1, 0, 1, 1, 0], 8, 0, 1, grad_dtype,
                 steps=3, seed=seed, instances=instances)


@pytest.mark.parametrize("grad_dtype,instances", [("bf16", 1), ("fp16", 2), ("fp32", 4)])
def test_clipped_counted_equals_clipped_in_a_graph(grad_dtype, instances):
    """Three counted clipped steps replayed from one graph equal three
    clipped steps with host step numbers: state, params, main grads and
    the norm report, bit for bit."""
    L, s, p, g, _ = _clip_case(grad_dtype=grad_dtype, instances=instances)
    N = L.padded_numel
    s2, p2 = _clone(s, p)
    adam = B.AdamConfig(grad_scale=1.0 / 8)
    mg, mg2 = (torch.full((N,), -1.0, device=DEV) for _ in range(2))  # padding stays -1
    ws, ws2 = B.clip_workspace(DEV), B.clip_workspace(DEV)
    rep, rep2 = B.clip_report(DEV), B.clip_report(DEV)
    gsrc = [[x.clone() for x in gs] for gs in g]
    gbuf = [x.clone() for x in g[0]]
    # warm-up on copies
    ws_, wp_ = _clone(s, p)
    B.dopt_step_clipped_counted(L, adam, B.step_counter(1), 0.05, gbuf, *ws_, wp_,
                                torch.empty(N, device=DEV), B.clip_workspace(DEV))
    torch.cuda.synchronize()
    counter = B.step_counter(1)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        B.dopt_step_clipped_counted(L, adam, counter, 0.05, gbuf, *s2, p2, mg2, ws2,
                                    norm_out=rep2, skip_nonfinite=True)
    for t in range(1, 4):
        for x, y in zip(gbuf, gsrc[t - 1]):
            x.copy_(y)
        graph.replay()
        B.dopt_step_clipped(L, adam, t, 0.05, gsrc[t - 1], *s, p, mg, ws, norm_out=rep,
                            skip_nonfinite=True)
        torch.cuda.synchronize()
        assert torch.equal(rep, rep2)
    _equal(s + p + [mg], s2 + p2 + [mg2])
    assert B.counter_state(counter) == (4, 0)


def test_clipped_counted_bad_step_and_skip():
    """A bad step number stores nothing but the main grads and the report; a
    step that the non-finite check skips gives its number back."""
    L, s, p, g, _ = _clip_case(seed=32)
    N = L.padded_numel
    adam = B.AdamConfig(grad_scale=1.0 / 8)
    before = [x.clone() for x in s + p]
    mg = torch.full((N,), -1.0, device=DEV)
    counter = B.step_counter(0)
    B.dopt_step_clipped_counted(L, adam, counter, 0.05, g[0], *s, p, mg, B.clip_workspace(DEV))
    torch.cuda.synchronize()
    _equal(before, s + p)
    assert B.counter_state(counter) == (0, B.DOPT_COUNTER_BAD_STEP)
    assert not torch.all(mg == -1.0)  # the norm pass ran
    # a NaN grad: skipped, and the step number is given back
    counter[0] = 5
    bad = [x.clone() for x in g[0]]
    bad[3][1234] = float("nan")
    rep = B.clip_report(DEV)
    B.dopt_step_clipped_counted(L, adam, counter, 0.05, bad, *s, p, mg, B.clip_workspace(DEV),
                                norm_out=rep, skip_nonfinite=True)
    torch.cuda.synchronize()
    _equal(before, s + p)
    norm, coef, nonfinite = B.read_clip_report(rep)
    assert nonfinite == 1 and np.isnan(coef)
    assert B.counter_state(counter) == (5, 0)
    # the same number then steps with clean grads
    ref = [x.clone() for x in before]
    B.dopt_step_clipped_counted(L, adam, counter, 0.05, g[0], *s, p, mg, B.clip_workspace(DEV),
                                skip_nonfinite=True)
    B.dopt_step_clipped(L, adam, 5, 0.05, g[0], *ref[:3], ref[3:], torch.empty(N, device=DEV),
                        B.clip_workspace(DEV))
    torch.cuda.synchronize()
    _equal(ref, s + p)
    assert B.counter_state(counter) == (6, 0)
