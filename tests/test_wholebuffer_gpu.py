"""Every element of full-size buffers against the oracle: the GPT-2-small
layout (D=8, 10 steps) and the 256 Mi sweep layout at its extremes (D=16
with 1 Mi buckets, D=1 with 64 Mi buckets), one dopt_step launch per step
as the benchmark times it.  The oracle steps the whole host copy of the
buffer (on host threads, in disjoint windows); master, m, v, the main
grads and all D param replicas are compared element by element."""
from dataclasses import asdict

import numpy as np
import pytest
import torch

import oracle
from parity import (assert_bf16_close, assert_f32_close, oracle_step_whole, t2np_bf16,
                    t2np_f32)
from zero_distributed_optimizer_gb300 import binding as B
from zero_distributed_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _whole_buffer(w: W.Workload):
    L = B.dopt_build_range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit,
                               list(w.wd_mask)).to_device()
    N = L.padded_numel
    master, m, v = W.make_state(w, N, DEV)
    params = W.make_params(master, w.D)
    host = [t2np_f32(master).copy(), t2np_f32(m).copy(), t2np_f32(v).copy(),
            [t2np_bf16(p).copy() for p in params]]
    mg = torch.full((N,), -5.0, device=DEV)
    hmg = np.full(N, -5.0, np.float32)
    adam = B.AdamConfig(**w.adam_kwargs())
    oadam = oracle.make_adam(**asdict(adam))
    for t in range(1, w.steps + 1):
        grads = W.make_grads(w, N, t, DEV)
        B.dopt_step(L, adam, t, grads, master, m, v, params, main_grad_out=mg)
        hg = [t2np_bf16(g) if w.grad_dtype == "bf16" else t2np_f32(g) for g in grads]
        del grads
        oracle_step_whole(list(w.sizes), list(w.wd_mask), w.D, w.bucket_elems, w.pad_unit,
                          oadam, t, hg, host[0], host[1], host[2], host[3], main_grad_out=hmg)
        del hg
    torch.cuda.synchronize()
    not_exact = 0
    for name, x, y in zip(("master", "exp_avg", "exp_avg_sq"), (master, m, v), host):
        not_exact += assert_f32_close(t2np_f32(x), y, name)
    not_exact += assert_f32_close(t2np_f32(mg), hmg, "main_grad")
    for r in range(w.D):
        not_exact += assert_bf16_close(t2np_bf16(params[r]), host[3][r], f"param{r}")
    del master, m, v, params, mg
    torch.cuda.empty_cache()
    return N, not_exact


def test_gpt2_small_every_element():
    N, not_exact = _whole_buffer(W.gpt2_small())
    assert N == 124_439_808 + 256
    assert not_exact == 0  # same operations, same order, one rounding each


@pytest.mark.parametrize("D,bucket_mi", [(16, 1), (1, 64)])
def test_sweep_256m_every_element(D, bucket_mi):
    N, not_exact = _whole_buffer(W.sweep_256m(D, bucket_mi))
    assert N >= 1 << 28
    assert not_exact == 0
