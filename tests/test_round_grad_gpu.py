"""DOPT_STEP_ROUND_GRAD on the device against the oracle: the reduced grad
is rounded to the grad type before clipping and Adam."""
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

CASES = [
    # sizes, wd, D, instances, bucket, pad
    ([5000, 1, 7, 300, 20000, 3, 9999], [1, 0, 1, 0, 1, 1, 0], 8, 1, 0, 1),
    ([4096, 333, 12345, 8, 77777], [0, 1, 1, 0, 1], 3, 1, 20000, 1),
    ([65536, 1000, 65536], [1, 0, 1], 8, 2, 0, 64),
]


def _host(grads, dtype):
    return [t2np_bf16(g).copy() if dtype == "bf16" else g.numpy().copy() for g in grads]


@pytest.mark.parametrize("mode", ["step", "step_allreduce", "clipped"])
@pytest.mark.parametrize("grad_dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_round_grad_matches_oracle(case, grad_dtype, mode):
    sizes, wd, D, inst, bucket, pad = CASES[case]
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd, instances=inst).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, 2, grad_dtype, seed=900 + case)
    h = [master.numpy().copy(), m.numpy().copy(), v.numpy().copy()]
    hp = [t2np_bf16(p).copy() for p in params]
    hmg = np.full(N, -3.0, np.float32)
    d = [master.to(DEV), m.to(DEV), v.to(DEV)]
    dp = [p.to(DEV) for p in params]
    dmg = torch.full((N,), -3.0, device=DEV)
    adam = B.AdamConfig(grad_scale=0.3)  # not a power of two: the sums need rounding
    oadam = oracle.make_adam(**asdict(adam))
    ws = B.clip_workspace(DEV)
    for i in range(2):
        hg = _host(grads[i], grad_dtype)
        dg = [g.to(DEV) for g in grads[i]]
        coef = 1.0
        if mode == "clipped":
            nsq = oracle.grad_norm_sq(sizes, D, bucket, pad, adam.grad_scale, hg, instances=inst,
                                      round_grad=True)
            max_norm = 0.3 * float(np.sqrt(nsq))
            coef = oracle.clip_coef(nsq, max_norm)
            B.dopt_step_clipped(L, adam, i + 1, max_norm, dg, *d, dp, dmg, ws, round_grad=True)
        elif mode == "step_allreduce":
            B.dopt_step_allreduce(L, adam, i + 1, dg, *d, dp, main_grad_out=dmg, round_grad=True)
        else:
            B.dopt_step(L, adam, i + 1, dg, *d, dp, main_grad_out=dmg, round_grad=True)
        oracle.step(sizes, wd, D, bucket, pad, oadam, i + 1, hg, *h, hp, main_grad_out=hmg,
                    clip_coef=coef, instances=inst, round_grad=True)
        if mode == "step_allreduce":
            oracle.allreduce(sizes, D, bucket, pad, adam.grad_scale, hg, instances=inst)
            torch.cuda.synchronize()
            for r in range(D):
                if grad_dtype == "bf16":
                    assert_bf16_close(t2np_bf16(dg[r]), hg[r], f"grads[{r}]", ulps=0)
                else:
                    assert_f32_close(t2np_f32(dg[r]), hg[r], f"grads[{r}]")
    torch.cuda.synchronize()
    for name, x, y in zip(("master", "exp_avg", "exp_avg_sq"), d, h):
        assert_f32_close(t2np_f32(x), y, name)
    assert_f32_close(t2np_f32(dmg), hmg, "main_grad")
    for r in range(D):
        assert_bf16_close(t2np_bf16(dp[r]), hp[r], f"param{r}")
