"""The staged step (DOPT_STEP_STAGE: each tile's grads and state moved into
shared memory by bulk copies before the update) against the oracle, every
element, and against the default path bit for bit: small and ragged layouts
over several tiles, every D it takes, all three grad types, with and
without the gather, the main-grad output, the rounded grad and fp16
params; the counted form; a launch over a strict subset of buckets; and the
GPT-2-small buffer at full size on sampled windows.  No staged CTA may run
out of its copy wait."""
from dataclasses import asdict

import numpy as np
import pytest
import torch

import oracle
from parity import (assert_bf16_close, assert_f32_close, assert_param_close, sample_windows,
                    t2np_bf16, t2np_f32, t2np_grad, t2np_param)
from zero_distributed_optimizer_gb300 import binding as B
from zero_distributed_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [
    # sizes, wd mask, D, bucket_elems, pad_unit
    ([130, 260, 90, 310, 210], None, 4, 0, 1),
    ([5000, 1, 7, 300, 20000, 3, 9999], [1, 0, 1, 0, 1, 1, 0], 8, 0, 1),
    ([70001], None, 1, 0, 1),
    ([4096, 333, 12345, 8, 77777], [0, 1, 1, 0, 1], 2, 20000, 1),
    ([65536, 1000, 65536, 5], [1, 0, 1, 1], 16, 0, 64),
    ([64] * 300 + [5000], None, 2, 4096, 64),
    ([1, 2, 3, 4, 5, 6, 7, 8, 9, 10] * 20, [1, 0] * 100, 4, 64, 1),
    ([0, 500, 0, 0, 1200, 0], None, 8, 0, 1),
]


def _step_both(case, grad_dtype, gather, round_grad, param_dtype, steps=2):
    sizes, wd, D, bucket, pad = CASES[case]
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, steps, grad_dtype, seed=50 + case)
    if param_dtype == "fp16":
        params = [p.float().half() for p in params]
    hs = [master.numpy().copy(), m.numpy().copy(), v.numpy().copy()]
    hp = [t2np_param(p) for p in params]
    hmg = np.full(N, -3.0, np.float32)
    staged = [[master.to(DEV), m.to(DEV), v.to(DEV)], [p.to(DEV) for p in params],
              torch.full((N,), -3.0, device=DEV)]
    plain = [[x.clone() for x in staged[0]], [p.clone() for p in staged[1]], staged[2].clone()]
    adam = B.AdamConfig(grad_scale=1.0 / D)
    for i in range(steps):
        dg = [g.to(DEV) for g in grads[i]]
        B.dopt_step(L, adam, i + 1, dg, *staged[0], staged[1], gather=gather,
                    main_grad_out=staged[2], round_grad=round_grad, stage=True)
        B.dopt_step(L, adam, i + 1, dg, *plain[0], plain[1], gather=gather,
                    main_grad_out=plain[2], round_grad=round_grad)
        oracle.step(sizes, wd, D, bucket, pad, oracle.make_adam(**asdict(adam)), i + 1,
                    [t2np_grad(g) for g in grads[i]], *hs, hp, gather=gather,
                    main_grad_out=hmg, round_grad=round_grad)
    torch.cuda.synchronize()
    not_exact = 0
    for name, x, y in zip(("master", "exp_avg", "exp_avg_sq"), staged[0], hs):
        not_exact += assert_f32_close(t2np_f32(x), y, name)
    not_exact += assert_f32_close(t2np_f32(staged[2]), hmg, "main_grad")
    for r in range(D):
        not_exact += assert_param_close(staged[1][r], hp[r], f"param{r}")
    assert not_exact == 0
    for x, y in zip(staged[0] + staged[1] + [staged[2]], plain[0] + plain[1] + [plain[2]]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("grad_dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_staged_matches_oracle(case, grad_dtype):
    _step_both(case, grad_dtype, gather=True, round_grad=False, param_dtype="bf16")


@pytest.mark.parametrize("case", [0, 1, 3, 4])
def test_staged_options(case):
    """Without the gather, with the rounded reduced grad, with fp16 params."""
    _step_both(case, "bf16", gather=False, round_grad=False, param_dtype="bf16")
    _step_both(case, "fp16", gather=True, round_grad=True, param_dtype="fp16")
    _step_both(case, "fp32", gather=False, round_grad=True, param_dtype="bf16")


def test_staged_counted_equals_plain_step():
    """The counted staged step, replayed from a CUDA graph, equals dopt_step
    at the same step numbers bit for bit."""
    sizes, wd, D, bucket, pad = CASES[1]
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, 1, "bf16", seed=9)
    g = [x.to(DEV) for x in grads[0]]
    a = [master.to(DEV), m.to(DEV), v.to(DEV)]
    pa = [p.to(DEV) for p in params]
    b = [x.clone() for x in a]
    pb = [p.clone() for p in pa]
    adam = B.AdamConfig(grad_scale=1.0 / D)
    counter = B.step_counter(3, DEV)
    B.dopt_step_counted(L, adam, counter, g, *a, pa, stage=True)  # step 3, outside the graph
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        B.dopt_step_counted(L, adam, counter, g, *a, pa, stage=True)
    for _ in range(3):
        graph.replay()  # steps 4, 5, 6 (capturing did not run the step)
    for t in (3, 4, 5, 6):
        B.dopt_step(L, adam, t, g, *b, pb)
    torch.cuda.synchronize()
    assert B.counter_state(counter) == (7, 0)
    for x, y in zip(a + pa, b + pb):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_staged_bucket_subset_matches_oracle_and_leaves_the_rest():
    sizes, D = [5000, 7000, 3000, 9000, 4000, 11], 4
    L = B.dopt_build_range_map(sizes, D, 6000, 1).to_device()
    assert L.n_buckets >= 3
    N = L.padded_numel
    bk = L.buckets()
    lo, hi = bk[1][0], bk[-2][1]
    master, m, v, params, grads = W.random_case(N, D, 1, "bf16", seed=17)
    d = [master.to(DEV), m.to(DEV), v.to(DEV)]
    dp = [p.to(DEV) for p in params]
    before = [x.clone() for x in d + dp]
    adam = B.AdamConfig(grad_scale=0.25)
    B.dopt_step_buckets(L, adam, 1, 1, L.n_buckets - 2, [x.to(DEV) for x in grads[0]], *d, dp,
                        stage=True)
    w = slice(lo, hi)
    hs = [master.numpy()[w].copy(), m.numpy()[w].copy(), v.numpy()[w].copy()]
    hp = [t2np_bf16(p)[w].copy() for p in params]
    oracle.step(sizes, None, D, 6000, 1, oracle.make_adam(**asdict(adam)), 1,
                [t2np_grad(x)[w].copy() for x in grads[0]], *hs, hp, window=(lo, hi))
    torch.cuda.synchronize()
    for name, x, y in zip(("master", "exp_avg", "exp_avg_sq"), d, hs):
        assert assert_f32_close(t2np_f32(x[w]), y, name) == 0
    for r in range(D):
        assert assert_bf16_close(t2np_bf16(dp[r][w]), hp[r], f"param{r}") == 0
    for x, x0 in zip(d + dp, before):
        assert torch.equal(x[:lo].view(torch.int16), x0[:lo].view(torch.int16))
        assert torch.equal(x[hi:].view(torch.int16), x0[hi:].view(torch.int16))


def test_staged_refusals():
    L = B.dopt_build_range_map([100, 200], 8, 0, 1, instances=2).to_device()
    N = L.padded_numel
    st = [torch.zeros(N, device=DEV) for _ in range(3)]
    g = [torch.zeros(N, dtype=torch.bfloat16, device=DEV) for _ in range(8)]
    p = [torch.zeros(N, dtype=torch.bfloat16, device=DEV) for _ in range(8)]
    with pytest.raises(B.DoptError) as e:
        B.dopt_step(L, B.AdamConfig(), 1, g, *st, p, stage=True)
    assert e.value.code == B.DOPT_E_ARG
    L3 = B.dopt_build_range_map([100, 200], 3, 0, 1).to_device()
    with pytest.raises(B.DoptError) as e:
        B.dopt_step(L3, B.AdamConfig(), 1, g[:3], *st, p[:3], stage=True)
    assert e.value.code == B.DOPT_E_ARG


def test_staged_gpt2_small_full_size():
    """The GPT-2-small buffer (D = 8) at full size, three staged steps:
    sampled windows against the oracle, and no copy wait ran out."""
    B.stage_timeouts(reset=True)
    w = W.gpt2_small()
    L = B.dopt_build_range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit,
                               list(w.wd_mask)).to_device()
    O = oracle.range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit)
    N = L.padded_numel
    wins = sample_windows(L.buckets(), O.pieces, N, seed=21, n_edges=32, n_random=6)
    master, m, v = W.make_state(w, N, DEV)
    params = W.make_params(master, w.D)
    host = [[t2np_f32(master[a:b]).copy(), t2np_f32(m[a:b]).copy(), t2np_f32(v[a:b]).copy(),
             [t2np_bf16(p[a:b]).copy() for p in params]] for a, b in wins]
    adam = B.AdamConfig(**w.adam_kwargs())
    oadam = oracle.make_adam(**asdict(adam))
    for t in (1, 2, 3):
        grads = W.make_grads(w, N, t, DEV)
        B.dopt_step(L, adam, t, grads, master, m, v, params, stage=True)
        for (a, b), hs in zip(wins, host):
            oracle.step(list(w.sizes), list(w.wd_mask), w.D, w.bucket_elems, w.pad_unit, oadam,
                        t, [t2np_bf16(g[a:b]) for g in grads], *hs, window=(a, b))
        del grads
    torch.cuda.synchronize()
    not_exact = 0
    for (a, b), hs in zip(wins, host):
        for name, x, y in zip(("master", "exp_avg", "exp_avg_sq"), (master, m, v), hs[:3]):
            not_exact += assert_f32_close(t2np_f32(x[a:b]), y, f"{name}[{a}:{b}]")
        for r in range(w.D):
            not_exact += assert_bf16_close(t2np_bf16(params[r][a:b]), hs[3][r], f"param{r}")
    assert not_exact == 0
    assert B.stage_timeouts() == 0
