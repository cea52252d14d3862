"""Parity of the CUDA step (through the C ABI) with the CPU oracle, element by
element, on small and ragged layouts that span several 2048-element tiles;
plus the gather kernel, edge cases and error paths on the device."""
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


def _oracle_adam(adam: B.AdamConfig):
    return oracle.make_adam(**asdict(adam))


class Case:
    """Device and host (oracle) copies of one small problem, stepped together."""

    def __init__(self, sizes, wd, D, bucket, pad, grad_dtype="bf16", steps=2, seed=0,
                 main_grad=True):
        self.sizes, self.wd, self.D, self.bucket, self.pad = list(sizes), wd, D, bucket, pad
        self.L = B.dopt_build_range_map(self.sizes, D, bucket, pad, wd).to_device()
        N = self.N = self.L.padded_numel
        master, m, v, params, grads = W.random_case(N, D, steps, grad_dtype, seed)
        self.grads = grads
        self.grad_dtype = grad_dtype
        self.h = [master.numpy().copy(), m.numpy().copy(), v.numpy().copy()]
        self.hp = [t2np_bf16(p).copy() for p in params]
        self.d = [master.to(DEV), m.to(DEV), v.to(DEV)]
        self.dp = [p.to(DEV) for p in params]
        self.init = ([a.copy() for a in self.h], [p.copy() for p in self.hp])
        self.hmg = np.full(N, -3.0, np.float32) if main_grad else None
        self.dmg = torch.full((N,), -3.0, device=DEV) if main_grad else None

    def step(self, i, t, adam, gather=True, device=True, host=True):
        if device:
            dg = [g.to(DEV) for g in self.grads[i]]
            B.dopt_step(self.L, adam, t, dg, *self.d, self.dp, gather=gather, main_grad_out=self.dmg)
        if host:
            hg = [t2np_bf16(g) if self.grad_dtype == "bf16" else g.numpy().copy()
                  for g in self.grads[i]]
            oracle.step(self.sizes, self.wd, self.D, self.bucket, self.pad, _oracle_adam(adam), t,
                        hg, *self.h, self.hp, gather=gather, main_grad_out=self.hmg)

    def compare(self):
        torch.cuda.synchronize()
        diffs = {}
        for name, d, h in zip(("master", "exp_avg", "exp_avg_sq"), self.d, self.h):
            diffs[name] = assert_f32_close(t2np_f32(d), h, name)
        for r in range(self.D):
            diffs[f"param{r}"] = assert_bf16_close(t2np_bf16(self.dp[r]), self.hp[r], f"param{r}")
        if self.hmg is not None:
            diffs["main_grad"] = assert_f32_close(t2np_f32(self.dmg), self.hmg, "main_grad")
        return diffs

    def padding_mask(self):
        owned = np.zeros(self.N, bool)
        for a, b in self.L.param_offsets():
            owned[a:b] = True
        return ~owned


def run_case(sizes, wd, D, bucket, pad, steps=2, grad_dtype="bf16", gather=True, adam=None,
             seed=0):
    c = Case(sizes, wd, D, bucket, pad, grad_dtype, steps, seed)
    adam = adam or B.AdamConfig(grad_scale=1.0 / D)
    for i in range(steps):
        c.step(i, i + 1, adam, gather=gather)
    diffs = c.compare()
    # padding is untouched on the device, in every buffer
    pad_mask = c.padding_mask()
    if pad_mask.any():
        for d, h0 in zip(c.d, c.init[0]):
            assert np.array_equal(t2np_f32(d)[pad_mask].view(np.uint32), h0[pad_mask].view(np.uint32))
        for dp, h0 in zip(c.dp, c.init[1]):
            assert np.array_equal(t2np_bf16(dp)[pad_mask], h0[pad_mask])
        assert np.all(t2np_f32(c.dmg)[pad_mask] == -3.0)
    return diffs


CASES = [
    # sizes, wd mask, D, bucket_elems, pad_unit
    ([130, 260, 90, 310, 210], None, 4, 0, 1),                      # the page's toy layout
    ([2], None, 3, 0, 1),                                            # AllReduce example shape
    ([5000, 1, 7, 300, 20000, 3, 9999], [1, 0, 1, 0, 1, 1, 0], 8, 0, 1),  # ragged, odd edges
    ([70001], None, 1, 0, 1),                                        # D=1, ragged tail
    ([4096, 333, 12345, 8, 77777], [0, 1, 1, 0, 1], 3, 20000, 1),     # odd D, buckets
    ([31000, 17, 64000, 5], [1, 0, 1, 0], 5, 30000, 3),
    ([9000] * 7, [1, 0] * 3 + [1], 7, 10000, 2),
    ([65536, 1000, 65536], [1, 0, 1], 16, 0, 64),
    ([40000, 12, 24000], [1, 0, 1], 17, 20000, 1),
    ([123457, 99], [1, 0], 64, 0, 1),
    ([64] * 300 + [5000], None, 2, 4096, 64),                         # many small params
    ([1, 2, 3, 4, 5, 6, 7, 8, 9, 10] * 20, [1, 0] * 100, 4, 64, 1),   # many tiny pieces per tile
    ([0, 500, 0, 0, 1200, 0], None, 4, 0, 1),                         # zero-size params
]


@pytest.mark.parametrize("grad_dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_parity_small(case, grad_dtype):
    sizes, wd, D, bucket, pad = CASES[case]
    run_case(sizes, wd, D, bucket, pad, steps=2, grad_dtype=grad_dtype, seed=case)


@pytest.mark.parametrize("D", [2, 4, 8, 16])
def test_parity_write_back_without_gather(D):
    sizes, wd = [3000, 7, 20000, 513], [1, 0, 1, 0]
    run_case(sizes, wd, D, 8000, 1, steps=2, gather=False, seed=D)


def test_toy_workload_three_steps():
    """The page's toy layout with the toy workload's own inputs."""
    w = W.toy_1000()
    L = B.dopt_build_range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit, w.wd_mask).to_device()
    N = L.padded_numel
    assert N == 1000
    master, m, v = W.make_state(w, N, DEV)
    params = W.make_params(master, w.D)
    h = [t2np_f32(master).copy(), t2np_f32(m).copy(), t2np_f32(v).copy()]
    hp = [t2np_bf16(p).copy() for p in params]
    adam = B.AdamConfig(**w.adam_kwargs())
    for t in range(1, w.steps + 1):
        grads = W.make_grads(w, N, t, DEV)
        B.dopt_step(L, adam, t, grads, master, m, v, params)
        oracle.step(list(w.sizes), list(w.wd_mask), w.D, w.bucket_elems, w.pad_unit,
                    _oracle_adam(adam), t, [t2np_bf16(g) for g in grads], *h, hp)
    torch.cuda.synchronize()
    assert_f32_close(t2np_f32(master), h[0], "master")
    assert_f32_close(t2np_f32(m), h[1], "m")
    assert_f32_close(t2np_f32(v), h[2], "v")
    for r in range(w.D):
        assert_bf16_close(t2np_bf16(params[r]), hp[r], f"param{r}")


def test_allreduce_example_on_device():
    """Tutorial AllReduce example: [1,2],[2,3],[3,3] -> main grads [6, 8]."""
    L = B.dopt_build_range_map([2], 3, 0, 1).to_device()
    grads = [torch.tensor(x + [0.0], device=DEV).bfloat16() for x in ([1, 2], [2, 3], [3, 3])]
    z = lambda: torch.zeros(4, device=DEV)  # noqa: E731  (16-byte alignment needs >= 4 floats)
    master, m, v = z(), z(), z()
    params = [torch.zeros(8, device=DEV, dtype=torch.bfloat16) for _ in range(3)]
    mg = torch.full((4,), -1.0, device=DEV)
    B.dopt_step(L, B.AdamConfig(grad_scale=1.0), 1, grads, master, m, v, params, main_grad_out=mg)
    torch.cuda.synchronize()
    assert mg.tolist() == [6.0, 8.0, -1.0, -1.0]


def test_gather_kernel_equals_fused_gather():
    sizes, wd = [10000, 3, 7777, 64, 20001], [1, 0, 1, 0, 1]
    for D in (2, 3, 8):
        a = Case(sizes, wd, D, 9000, 1, steps=1, seed=40 + D)
        b = Case(sizes, wd, D, 9000, 1, steps=1, seed=40 + D)
        adam = B.AdamConfig(grad_scale=1.0 / D)
        a.step(0, 1, adam, gather=True, host=False)
        b.step(0, 1, adam, gather=False, host=False)
        B.dopt_gather(b.L, b.dp)
        torch.cuda.synchronize()
        for r in range(D):
            assert torch.equal(a.dp[r].view(torch.int16), b.dp[r].view(torch.int16))


def test_gather_kernel_against_oracle_semantics():
    """dopt_gather copies each rank's owned elements from its replica to all
    others and leaves padding alone."""
    sizes, D = [1000, 37, 5000], 4
    L = B.dopt_build_range_map(sizes, D, 0, 3).to_device()
    N = L.padded_numel
    g = torch.Generator(device="cpu").manual_seed(1)
    reps = [torch.randn(N, generator=g).bfloat16() for _ in range(D)]
    dreps = [r.to(DEV) for r in reps]
    B.dopt_gather(L, dreps)
    torch.cuda.synchronize()
    want = [t2np_bf16(r).copy() for r in reps]
    for pc in L.pieces():
        a, b = pc["gbuf_world"]
        for r in range(D):
            want[r][a:b] = t2np_bf16(reps[pc["rank"]])[a:b]
    for r in range(D):
        assert np.array_equal(t2np_bf16(dreps[r]), want[r])


def test_nan_and_inf_grads_propagate_like_the_oracle():
    c = Case([3000, 5000], [1, 0], 4, 0, 1, steps=1, seed=3)
    g = c.grads[0]
    g[1][10] = float("nan")
    g[2][20] = float("inf")
    g[0][30] = float("-inf")
    g[3][30] = float("inf")  # inf + -inf = NaN
    c.step(0, 1, B.AdamConfig(grad_scale=0.25))
    c.compare()
    assert torch.isnan(c.d[0][10]).item() and torch.isnan(c.d[0][30]).item()


def test_checkpoint_resume_is_bitwise(tmp_path):
    """Three steps in a row equal one step, a save and load of all state
    (torch.save), and two more steps."""
    sizes, wd, D = [20000, 5, 3000], [1, 0, 1], 4
    a = Case(sizes, wd, D, 0, 8, steps=3, seed=9)
    b = Case(sizes, wd, D, 0, 8, steps=3, seed=9)
    adam = B.AdamConfig(grad_scale=0.25)
    for i in range(3):
        a.step(i, i + 1, adam, host=False)
    b.step(0, 1, adam, host=False)
    torch.cuda.synchronize()
    path = tmp_path / "ckpt.pt"
    torch.save({"state": b.d, "params": b.dp, "step": 1}, path)
    ck = torch.load(path)
    L2 = B.dopt_build_range_map(sizes, D, 0, 8, wd).to_device()
    for i in range(1, 3):
        dg = [g.to(DEV) for g in b.grads[i]]
        B.dopt_step(L2, adam, ck["step"] + i, dg, *ck["state"], ck["params"])
    torch.cuda.synchronize()
    for x, y in zip(a.d, ck["state"]):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    for x, y in zip(a.dp, ck["params"]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_step_on_a_side_stream():
    c = Case([50000, 77], [1, 0], 8, 0, 64, steps=1, seed=12)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dg = [g.to(DEV) for g in c.grads[0]]
        B.dopt_step(c.L, B.AdamConfig(grad_scale=0.125), 1, dg, *c.d, c.dp,
                    main_grad_out=c.dmg, stream=s)
    s.synchronize()
    c.step(0, 1, B.AdamConfig(grad_scale=0.125), device=False)
    c.compare()


def test_empty_layout_is_a_noop():
    L = B.dopt_build_range_map([], 2, 0, 1).to_device()
    t = torch.zeros(4, device=DEV)
    p = [torch.zeros(8, device=DEV, dtype=torch.bfloat16) for _ in range(2)]
    B.dopt_step(L, B.AdamConfig(), 1, [x.clone() for x in p], t, t.clone(), t.clone(), p)
    L = B.dopt_build_range_map([0, 0], 2, 0, 4)
    B.dopt_step(L, B.AdamConfig(), 1, [x.clone() for x in p], t, t.clone(), t.clone(), p)
    torch.cuda.synchronize()


def test_device_errors():
    sizes, D = [1000, 24], 2
    L = B.dopt_build_range_map(sizes, D, 0, 4)  # tables not on the device yet
    N = L.padded_numel
    st = [torch.zeros(N + 8, device=DEV) for _ in range(3)]
    p = [torch.zeros(N + 8, device=DEV, dtype=torch.bfloat16) for _ in range(D)]
    g = [torch.zeros(N + 8, device=DEV, dtype=torch.bfloat16) for _ in range(D)]
    with pytest.raises(B.DoptError) as e:
        B.dopt_step(L, B.AdamConfig(), 1, g, *st, p)
    assert e.value.code == B.DOPT_E_STATE
    L.to_device()
    with pytest.raises(B.DoptError) as e:  # 2-byte offset: not 16-byte aligned
        B.dopt_step(L, B.AdamConfig(), 1, [g[0][1:], g[1]], *st, p)
    assert e.value.code == B.DOPT_E_ALIGN
    with pytest.raises(B.DoptError) as e:  # too short: caught by the binding
        B.dopt_step(L, B.AdamConfig(), 1, g, st[0][: N - 1], st[1], st[2], p)
    assert e.value.code == B.DOPT_E_ARG
    with pytest.raises(B.DoptError) as e:
        B.dopt_gather(L, [p[0][1:], p[1]])
    assert e.value.code == B.DOPT_E_ALIGN
    B.dopt_step(L, B.AdamConfig(), 1, g, *st, p)  # the context is still usable
    torch.cuda.synchronize()


def test_step_plan_equals_per_call_binding():
    """A StepPlan (arguments checked once) gives the same results as the
    per-call binding, for whole steps and for bucket launches."""
    sizes, wd, D = [30000, 7, 20000, 513, 9000], [1, 0, 1, 0, 1], 4
    L = B.dopt_build_range_map(sizes, D, 15000, 8, wd).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, 2, "bf16", 33)
    a = [master.to(DEV), m.to(DEV), v.to(DEV)]
    b = [x.clone() for x in a]
    pa = [p.to(DEV) for p in params]
    pb = [p.clone() for p in pa]
    ga = [g.to(DEV) for g in grads[0]]
    gb = [g.clone() for g in ga]
    adam = B.AdamConfig(grad_scale=0.25)
    plan = B.StepPlan(L, adam, gb, *b, pb)
    B.dopt_step(L, adam, 1, ga, *a, pa)
    plan.step(1)
    for k in range(L.n_buckets):
        B.dopt_step_buckets(L, adam, 2, k, 1, ga, *a, pa)
        plan.step_buckets(2, k)
    torch.cuda.synchronize()
    for x, y in zip(a + pa, b + pb):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
