"""The all-reduce (force_all_reduce) paths and bucket-range launches on the
device, against the oracle and against the whole-buffer step."""
from dataclasses import asdict

import pytest
import torch

import oracle
from parity import assert_bf16_close, assert_f32_close, t2np_bf16, t2np_f32
from zero_distributed_optimizer_gb300 import binding as B
from zero_distributed_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [
    ([130, 260, 90, 310, 210], None, 4, 0, 1),
    ([5000, 1, 7, 300, 20000, 3, 9999], [1, 0, 1, 0, 1, 1, 0], 8, 0, 1),
    ([4096, 333, 12345, 8, 77777], [0, 1, 1, 0, 1], 3, 20000, 1),
    ([65536, 1000, 65536], [1, 0, 1], 16, 0, 64),
    ([123457, 99], [1, 0], 64, 0, 1),
    ([1000, 3, 2000, 5, 700], None, 1, 1000, 1),
]


def _host_grads(grads, dtype):
    return [t2np_bf16(g).copy() if dtype == "bf16" else g.numpy().copy() for g in grads]


def _compare_grads(dev, host, dtype, what):
    for r, (d, h) in enumerate(zip(dev, host)):
        if dtype == "bf16":
            assert_bf16_close(t2np_bf16(d), h, f"{what}[{r}]", ulps=0)
        else:
            assert_f32_close(t2np_f32(d), h, f"{what}[{r}]")


def test_allreduce_example_on_every_rank():
    """Tutorial "AllReduce": [1,2], [2,3], [3,3] -> [6,8] on every rank."""
    L = B.dopt_build_range_map([2], 3, 0, 1).to_device()
    for dtype in (torch.bfloat16, torch.float32):
        grads = [torch.tensor(x + [-2.0, 0, 0, 0, 0, 0], device=DEV).to(dtype)
                 for x in ([1, 2], [2, 3], [3, 3])]
        B.dopt_allreduce(L, grads, 1.0)
        torch.cuda.synchronize()
        for g in grads:
            assert g.float().tolist()[:3] == [6.0, 8.0, -2.0]


@pytest.mark.parametrize("grad_dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_allreduce_matches_oracle(case, grad_dtype):
    sizes, wd, D, bucket, pad = CASES[case]
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd).to_device()
    N = L.padded_numel
    _, _, _, _, grads = W.random_case(N, D, 1, grad_dtype, seed=200 + case)
    host = _host_grads(grads[0], grad_dtype)
    dev = [g.to(DEV) for g in grads[0]]
    B.dopt_allreduce(L, dev, 1.0 / D)
    oracle.allreduce(sizes, D, bucket, pad, 1.0 / D, host)
    torch.cuda.synchronize()
    _compare_grads(dev, host, grad_dtype, "grads")


@pytest.mark.parametrize("grad_dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_step_allreduce_matches_oracle(case, grad_dtype):
    """force_all_reduce step = the oracle's step followed by its all-reduce
    of the same (unmodified) grads."""
    sizes, wd, D, bucket, pad = CASES[case]
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, 2, grad_dtype, seed=300 + case)
    h = [master.numpy().copy(), m.numpy().copy(), v.numpy().copy()]
    hp = [t2np_bf16(p).copy() for p in params]
    d = [master.to(DEV), m.to(DEV), v.to(DEV)]
    dp = [p.to(DEV) for p in params]
    adam = B.AdamConfig(grad_scale=1.0 / D)
    oadam = oracle.make_adam(**asdict(adam))
    for i in range(2):
        hg = _host_grads(grads[i], grad_dtype)
        dg = [g.to(DEV) for g in grads[i]]
        B.dopt_step_allreduce(L, adam, i + 1, dg, *d, dp)
        oracle.step(sizes, wd, D, bucket, pad, oadam, i + 1, hg, *h, hp)
        oracle.allreduce(sizes, D, bucket, pad, adam.grad_scale, hg)
        torch.cuda.synchronize()
        _compare_grads(dg, hg, grad_dtype, f"grads step {i + 1}")
    for name, x, y in zip(("master", "exp_avg", "exp_avg_sq"), d, h):
        assert_f32_close(t2np_f32(x), y, name)
    for r in range(D):
        assert_bf16_close(t2np_bf16(dp[r]), hp[r], f"param{r}")


def _run_buckets(L, adam, grads, state, params, order, streams=1, gather=True, mg=None):
    ss = [torch.cuda.current_stream()] + [torch.cuda.Stream() for _ in range(streams - 1)]
    start = torch.cuda.Event()
    start.record()
    for s in ss[1:]:
        s.wait_event(start)
    for i, k in enumerate(order):
        s = ss[i % streams]
        with torch.cuda.stream(s):
            B.dopt_step_buckets(L, adam, 1, k, 1, grads, *state, params, gather=gather,
                                main_grad_out=mg, stream=s)
    for s in ss[1:]:
        ev = torch.cuda.Event()
        ev.record(s)
        torch.cuda.current_stream().wait_event(ev)
    torch.cuda.synchronize()


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("streams", [1, 3])
def test_bucket_launches_equal_whole_step(case, streams):
    """Per-bucket launches, in reverse order and over several streams, give
    the whole-buffer step bit for bit (every element belongs to one bucket)."""
    sizes, wd, D, bucket, pad = CASES[case]
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, 1, "bf16", seed=400 + case)
    g = [x.to(DEV) for x in grads[0]]
    a = [master.to(DEV), m.to(DEV), v.to(DEV)]
    b = [x.clone() for x in a]
    pa = [p.to(DEV) for p in params]
    pb = [p.clone() for p in pa]
    mga = torch.full((N,), -4.0, device=DEV)
    mgb = mga.clone()
    adam = B.AdamConfig(grad_scale=1.0 / D)
    B.dopt_step(L, adam, 1, g, *a, pa, main_grad_out=mga)
    _run_buckets(L, adam, g, b, pb, order=list(reversed(range(L.n_buckets))), streams=streams,
                 mg=mgb)
    for x, y in zip(a + pa + [mga], b + pb + [mgb]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_bucket_range_launch_covers_only_its_buckets():
    sizes, D = [5000, 7000, 3000, 9000, 4000], 4
    L = B.dopt_build_range_map(sizes, D, 6000, 8).to_device()
    assert L.n_buckets >= 3
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, 1, "bf16", seed=5)
    g = [x.to(DEV) for x in grads[0]]
    d = [master.to(DEV), m.to(DEV), v.to(DEV)]
    before = [x.clone() for x in d]
    dp = [p.to(DEV) for p in params]
    B.dopt_step_buckets(L, B.AdamConfig(grad_scale=0.25), 1, 1, L.n_buckets - 2, g, *d, dp)
    torch.cuda.synchronize()
    bk = L.buckets()
    lo, hi = bk[1][0], bk[-2][1]
    for x, x0 in zip(d, before):
        assert torch.equal(x[:lo], x0[:lo]) and torch.equal(x[hi:], x0[hi:])
        assert not torch.equal(x[lo:hi], x0[lo:hi])
    with pytest.raises(B.DoptError) as e:
        B.dopt_step_buckets(L, B.AdamConfig(), 1, L.n_buckets, 1, g, *d, dp)
    assert e.value.code == B.DOPT_E_ARG
    B.dopt_step_buckets(L, B.AdamConfig(), 1, 0, 0, g, *d, dp)
    torch.cuda.synchronize()


def test_bucket_launches_full_size_sweep_1mi():
    """The 256 Mi sweep layout with 1 Mi buckets (256 buckets), D=8: one
    launch per bucket over two streams equals the single launch."""
    w = W.sweep_256m(8, 1)
    L = B.dopt_build_range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit,
                               list(w.wd_mask)).to_device()
    N = L.padded_numel
    master, m, v = W.make_state(w, N, DEV)
    params = W.make_params(master, w.D)
    grads = W.make_grads(w, N, 1, DEV)
    a = [master, m, v]
    b = [x.clone() for x in a]
    pa = params
    pb = [p.clone() for p in pa]
    adam = B.AdamConfig(**w.adam_kwargs())
    B.dopt_step(L, adam, 1, grads, *a, pa)
    _run_buckets(L, adam, grads, b, pb, order=list(range(L.n_buckets)), streams=2)
    for x, y in zip(a + pa, b + pb):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
