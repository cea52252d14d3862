"""Randomised parity: random layouts and options, each stepped on the device
and by the oracle and compared element by element (seeded, reproducible)."""
from dataclasses import asdict

import numpy as np
import pytest
import torch

import oracle
from parity import assert_f32_close, assert_param_close, t2np_f32, t2np_grad, t2np_param
from zero_distributed_optimizer_gb300 import binding as B
from zero_distributed_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def random_config(seed):
    rng = np.random.default_rng(10_000 + seed)
    n = int(rng.integers(1, 40))
    kind = rng.integers(0, 3)
    if kind == 0:
        sizes = [int(x) for x in rng.integers(0, 300, n)]          # tiny params
    elif kind == 1:
        sizes = [int(x) for x in rng.integers(1, 40000, n)]        # mixed
    else:
        sizes = [int(x) * 8 for x in rng.integers(1, 20000, n)]    # vector-aligned
    D = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8, 12, 16, 24, 32, 64]))
    divisors = [i for i in range(1, D + 1) if D % i == 0]
    instances = int(rng.choice(divisors))
    bucket = int(rng.choice([0, int(rng.integers(1, max(2, sum(sizes) // 2 + 2)))]))
    pad = int(rng.choice([1, 2, 3, 8, 64]))
    wd = [int(x) for x in rng.integers(0, 2, n)]
    dtype = str(rng.choice(["bf16", "fp32"]))
    gather = bool(rng.integers(0, 2))
    round_grad = bool(rng.integers(0, 2))
    steps = int(rng.integers(1, 4))
    scale = float(rng.choice([1.0, 1.0 / D, 0.3]))
    param_dtype = "bf16"
    if seed >= 40:  # later seeds draw the 16-bit types from all of them
        more = np.random.default_rng(20_000 + seed)
        dtype = str(more.choice(["bf16", "fp16", "fp32"]))
        param_dtype = str(more.choice(["bf16", "fp16"]))
    return sizes, wd, D, instances, bucket, pad, dtype, gather, round_grad, steps, scale, \
        param_dtype


@pytest.mark.parametrize("seed", range(70))
def test_random_parity(seed):
    sizes, wd, D, inst, bucket, pad, dtype, gather, rg, steps, scale, pdt = random_config(seed)
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd, instances=inst).to_device()
    N = L.padded_numel
    assert N == oracle.range_map(sizes, D // inst, bucket, pad).numel
    if N == 0:
        return
    master, m, v, params, grads = W.random_case(N, D, steps, dtype, seed)
    if pdt == "fp16":
        params = [p.float().half() for p in params]
    h = [master.numpy().copy(), m.numpy().copy(), v.numpy().copy()]
    hp = [t2np_param(p) for p in params]
    hmg = np.full(N, -3.0, np.float32)
    d = [master.to(DEV), m.to(DEV), v.to(DEV)]
    dp = [p.to(DEV) for p in params]
    dmg = torch.full((N,), -3.0, device=DEV)
    adam = B.AdamConfig(grad_scale=scale)
    oadam = oracle.make_adam(**asdict(adam))
    for i in range(steps):
        hg = [t2np_grad(g) for g in grads[i]]
        B.dopt_step(L, adam, i + 1, [g.to(DEV) for g in grads[i]], *d, dp, gather=gather,
                    main_grad_out=dmg, round_grad=rg)
        oracle.step(sizes, wd, D, bucket, pad, oadam, i + 1, hg, *h, hp, gather=gather,
                    main_grad_out=hmg, instances=inst, round_grad=rg)
    torch.cuda.synchronize()
    for name, x, y in zip(("master", "exp_avg", "exp_avg_sq"), d, h):
        assert_f32_close(t2np_f32(x), y, name)
    assert_f32_close(t2np_f32(dmg), hmg, "main_grad")
    for r in range(D):
        assert_param_close(dp[r], hp[r], f"param{r}")
