"""Layouts where nearly every 8-element vector straddles a run edge (params of
1 to 7 elements, so decay flags and owner ranks change inside vectors, and
whole warps of such vectors), against the oracle element by element: the
plain step (with and without the gather), the counted step, the step with
the all-reduce and the clipped step."""
from dataclasses import asdict

import numpy as np
import pytest
import torch

import oracle
from parity import assert_bf16_close, assert_f32_close, t2np_bf16, t2np_f32, t2np_grad
from zero_distributed_optimizer_gb300 import binding as B
from zero_distributed_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"

# sizes seed, D, instances, bucket, pad, grad dtype
CASES = [
    (1, 4, 1, 0, 1, "bf16"),
    (2, 3, 1, 700, 1, "bf16"),
    (3, 8, 2, 0, 3, "fp32"),
    (4, 8, 1, 1500, 1, "fp16"),
    (5, 16, 4, 0, 1, "bf16"),
    (6, 6, 3, 900, 2, "fp32"),
]


def _layout(seed):
    rng = np.random.default_rng(4_000 + seed)
    n = 700
    sizes = [int(x) for x in rng.integers(1, 8, n)]
    wd = [int(x) for x in rng.integers(0, 2, n)]
    return sizes, wd


def _host_grads(grads):
    return [t2np_grad(g) for g in grads]


def _setup(case, steps=2):
    seed, D, inst, bucket, pad, dtype = case
    sizes, wd = _layout(seed)
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd, instances=inst).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, steps, dtype, seed)
    h = [master.numpy().copy(), m.numpy().copy(), v.numpy().copy()]
    hp = [t2np_bf16(p).copy() for p in params]
    d = [master.to(DEV), m.to(DEV), v.to(DEV)]
    dp = [p.to(DEV) for p in params]
    return sizes, wd, D, inst, bucket, pad, dtype, L, N, grads, h, hp, d, dp


def _compare(d, dp, h, hp, D):
    for name, x, y in zip(("master", "exp_avg", "exp_avg_sq"), d, h):
        assert_f32_close(t2np_f32(x), y, name)
    for r in range(D):
        assert_bf16_close(t2np_bf16(dp[r]), hp[r], f"param{r}")


@pytest.mark.parametrize("gather", [True, False])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_straddling_step(case, gather):
    sizes, wd, D, inst, bucket, pad, dtype, L, N, grads, h, hp, d, dp = _setup(CASES[case])
    adam = B.AdamConfig(grad_scale=1.0 / D)
    oadam = oracle.make_adam(**asdict(adam))
    dmg = torch.full((N,), -5.0, device=DEV)
    hmg = np.full(N, -5.0, np.float32)
    for t in (1, 2):
        B.dopt_step(L, adam, t, [g.to(DEV) for g in grads[t - 1]], *d, dp, gather=gather,
                    main_grad_out=dmg)
        oracle.step(sizes, wd, D, bucket, pad, oadam, t, _host_grads(grads[t - 1]), *h, hp,
                    gather=gather, main_grad_out=hmg, instances=inst)
    torch.cuda.synchronize()
    _compare(d, dp, h, hp, D)
    assert_f32_close(t2np_f32(dmg), hmg, "main_grad")


@pytest.mark.parametrize("case", range(len(CASES)))
def test_straddling_counted_and_allreduce_steps(case):
    sizes, wd, D, inst, bucket, pad, dtype, L, N, grads, h, hp, d, dp = _setup(CASES[case])
    adam = B.AdamConfig(grad_scale=1.0 / D)
    oadam = oracle.make_adam(**asdict(adam))
    counter = B.step_counter(1)
    # step 1 counted, step 2 with the all-reduce of the grads
    B.dopt_step_counted(L, adam, counter, [g.to(DEV) for g in grads[0]], *d, dp)
    oracle.step(sizes, wd, D, bucket, pad, oadam, 1, _host_grads(grads[0]), *h, hp,
                instances=inst)
    dg = [g.to(DEV) for g in grads[1]]
    hg = _host_grads(grads[1])
    B.dopt_step_allreduce(L, adam, 2, dg, *d, dp)
    oracle.step(sizes, wd, D, bucket, pad, oadam, 2, hg, *h, hp, instances=inst)
    oracle.allreduce(sizes, D, bucket, pad, adam.grad_scale, hg, instances=inst)
    torch.cuda.synchronize()
    _compare(d, dp, h, hp, D)
    for r in range(D):
        if dtype == "fp32":
            assert_f32_close(t2np_f32(dg[r]), hg[r], f"grads[{r}]")
        else:  # the rounded sums, bit for bit
            assert np.array_equal(t2np_grad(dg[r]).view(np.uint16), hg[r].view(np.uint16)), f"grads[{r}]"


@pytest.mark.parametrize("case", range(len(CASES)))
def test_straddling_clipped_step(case):
    sizes, wd, D, inst, bucket, pad, dtype, L, N, grads, h, hp, d, dp = _setup(CASES[case], steps=1)
    adam = B.AdamConfig(grad_scale=1.0 / D)
    hg = _host_grads(grads[0])
    nsq = oracle.grad_norm_sq(sizes, D, bucket, pad, adam.grad_scale, hg, instances=inst)
    max_norm = 0.5 * float(np.sqrt(nsq))
    coef = oracle.clip_coef(nsq, max_norm)
    norm_out = torch.zeros(2, device=DEV)
    B.dopt_step_clipped(L, adam, 1, max_norm, [g.to(DEV) for g in grads[0]], *d, dp,
                        torch.empty(N, device=DEV), B.clip_workspace(DEV), norm_out=norm_out)
    oracle.step(sizes, wd, D, bucket, pad, oracle.make_adam(**asdict(adam)), 1, hg, *h, hp,
                clip_coef=coef, instances=inst)
    torch.cuda.synchronize()
    assert abs(norm_out[0].item() - np.sqrt(nsq)) <= 1e-6 * np.sqrt(nsq)
    _compare(d, dp, h, hp, D)
