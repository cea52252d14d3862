"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (one dopt_step launch per step over the whole buffer).

The whole buffers live on the device; the oracle steps sampled windows of
them (both ends of every bucket with its padding, piece boundaries +-64
elements, and random 64 Ki stretches).  Elements are independent, so each
window is compared exactly against the full computation."""
from dataclasses import asdict

import numpy as np
import pytest
import torch

import oracle
from parity import assert_bf16_close, assert_f32_close, sample_windows, t2np_bf16, t2np_f32
from zero_distributed_optimizer_gb300 import binding as B
from zero_distributed_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_workload(w: W.Workload, seed: int = 0, steps=None, n_edges=48, n_random=12):
    steps = steps or w.steps
    L = B.dopt_build_range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit,
                               list(w.wd_mask)).to_device()
    O = oracle.range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit)
    assert L.padded_numel == O.numel and L.pieces() == O.pieces  # bit-exact range map
    N = L.padded_numel
    wins = sample_windows(L.buckets(), O.pieces, N, seed, n_edges=n_edges, n_random=n_random)
    if N > (1 << 31):  # both sides of the int32 element boundary
        from parity import merge_windows
        wins = merge_windows(wins + [((1 << 31) - 4096, (1 << 31) + 4096)], N)
    master, m, v = W.make_state(w, N, DEV)
    params = W.make_params(master, w.D)
    host = []
    for a, b in wins:
        host.append([t2np_f32(master[a:b]).copy(), t2np_f32(m[a:b]).copy(),
                     t2np_f32(v[a:b]).copy(), [t2np_bf16(p[a:b]).copy() for p in params],
                     np.full(b - a, -5.0, np.float32)])
    mg = torch.full((N,), -5.0, device=DEV)
    adam = B.AdamConfig(**w.adam_kwargs())
    oadam = oracle.make_adam(**asdict(adam))
    for t in range(1, steps + 1):
        grads = W.make_grads(w, N, t, DEV)
        B.dopt_step(L, adam, t, grads, master, m, v, params, main_grad_out=mg)
        for (a, b), hs in zip(wins, host):
            hg = [t2np_bf16(g[a:b]) if w.grad_dtype == "bf16" else t2np_f32(g[a:b]).copy()
                  for g in grads]
            oracle.step(list(w.sizes), list(w.wd_mask), w.D, w.bucket_elems, w.pad_unit, oadam,
                        t, hg, hs[0], hs[1], hs[2], hs[3], main_grad_out=hs[4], window=(a, b))
        del grads
    torch.cuda.synchronize()
    not_exact = 0
    for (a, b), hs in zip(wins, host):
        not_exact += assert_f32_close(t2np_f32(master[a:b]), hs[0], f"master[{a}:{b}]")
        not_exact += assert_f32_close(t2np_f32(m[a:b]), hs[1], f"m[{a}:{b}]")
        not_exact += assert_f32_close(t2np_f32(v[a:b]), hs[2], f"v[{a}:{b}]")
        not_exact += assert_f32_close(t2np_f32(mg[a:b]), hs[4], f"main_grad[{a}:{b}]")
        for r in range(w.D):
            not_exact += assert_bf16_close(t2np_bf16(params[r][a:b]), hs[3][r], f"param{r}[{a}:{b}]")
    compared = sum(b - a for a, b in wins)
    del master, m, v, params, mg
    torch.cuda.empty_cache()
    return compared, not_exact


def test_gpt2_small_full_size():
    compared, _ = run_workload(W.gpt2_small())
    assert compared > 500_000


def test_llama_1p3b_full_size():
    compared, _ = run_workload(W.llama_1p3b(), seed=1)
    assert compared > 500_000


@pytest.mark.parametrize("D", W.SWEEP_D)
@pytest.mark.parametrize("bucket_mi", W.SWEEP_BUCKET_MI)
def test_sweep_256m_full_size(D, bucket_mi):
    run_workload(W.sweep_256m(D, bucket_mi), seed=D * 100 + bucket_mi, n_edges=24, n_random=4)


def test_moe_many_small_fp32_grads_full_size():
    compared, _ = run_workload(W.moe_many_small(), seed=5)
    assert compared > 500_000


def test_beyond_two_billion_elements():
    """A buffer of more than 2^31 elements (element offsets beyond int32),
    D=1, bf16 grads, two buckets: sampled windows, including both sides of
    element 2^31, match the oracle."""
    big = (1 << 31) + 12345
    w = W.Workload("beyond_2g", (big // 2, 3, big - big // 2 - 3), (1, 0, 1), D=1,
                   bucket_elems=big // 2, pad_unit=64, grad_dtype="bf16",
                   grad_dist="normal1e-3", m_init="zero", v_init="zero", steps=2)
    compared, _ = run_workload(w, seed=9, n_edges=16, n_random=4)
    assert compared > 100_000
