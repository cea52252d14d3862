"""FP16 grads (DOPT_FP16) and FP16 params (DOPT_STEP_PARAMS_FP16) on the
device against the oracle (reading R7b of the oracle: IEEE binary16, exact
widening, nearest-even narrowing with overflow to Inf), on every entry
point that reads or writes them."""
from dataclasses import asdict

import numpy as np
import pytest
import torch

import oracle
from parity import (assert_f16_close, assert_f32_close, assert_param_close, sample_windows,
                    t2np_f32, t2np_grad, t2np_param)
from zero_distributed_optimizer_gb300 import binding as B
from zero_distributed_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [
    # sizes, wd, D, instances, bucket, pad
    ([130, 260, 90, 310, 210], None, 4, 1, 0, 1),
    ([5000, 1, 7, 300, 20000, 3, 9999], [1, 0, 1, 0, 1, 1, 0], 8, 1, 0, 1),
    ([4096, 333, 12345, 8, 77777], [0, 1, 1, 0, 1], 3, 1, 20000, 1),
    ([65536, 1000, 65536], [1, 0, 1], 16, 4, 0, 64),
    ([123457, 99], [1, 0], 12, 3, 0, 1),
]


def _case(i, grad_dtype, param_dtype, steps, seed):
    sizes, wd, D, inst, bucket, pad = CASES[i]
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd, instances=inst).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, steps, grad_dtype, seed)
    if param_dtype == "fp16":
        params = [p.float().half() for p in params]
    return L, N, (sizes, wd, D, inst, bucket, pad), master, m, v, params, grads


@pytest.mark.parametrize("param_dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("grad_dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_step_parity(case, grad_dtype, param_dtype):
    L, N, (sizes, wd, D, inst, bucket, pad), master, m, v, params, grads = _case(
        case, grad_dtype, param_dtype, 2, 1100 + case)
    h = [master.numpy().copy(), m.numpy().copy(), v.numpy().copy()]
    hp = [t2np_param(p) for p in params]
    hmg = np.full(N, -3.0, np.float32)
    d = [master.to(DEV), m.to(DEV), v.to(DEV)]
    dp = [p.to(DEV) for p in params]
    dmg = torch.full((N,), -3.0, device=DEV)
    adam = B.AdamConfig(grad_scale=1.0 / D)
    oadam = oracle.make_adam(**asdict(adam))
    for i in range(2):
        gather = i == 0
        B.dopt_step(L, adam, i + 1, [g.to(DEV) for g in grads[i]], *d, dp, gather=gather,
                    main_grad_out=dmg)
        oracle.step(sizes, wd, D, bucket, pad, oadam, i + 1, [t2np_grad(g) for g in grads[i]],
                    *h, hp, gather=gather, main_grad_out=hmg, instances=inst)
    torch.cuda.synchronize()
    for name, x, y in zip(("master", "exp_avg", "exp_avg_sq"), d, h):
        assert_f32_close(t2np_f32(x), y, name)
    assert_f32_close(t2np_f32(dmg), hmg, "main_grad")
    for r in range(D):
        assert_param_close(dp[r], hp[r], f"param{r}")


@pytest.mark.parametrize("case", range(len(CASES)))
def test_allreduce_and_step_allreduce_fp16(case):
    L, N, (sizes, wd, D, inst, bucket, pad), master, m, v, params, grads = _case(
        case, "fp16", "fp16", 1, 1200 + case)
    hg = [t2np_grad(g) for g in grads[0]]
    dg = [g.to(DEV) for g in grads[0]]
    B.dopt_allreduce(L, dg, 1.0 / D)
    oracle.allreduce(sizes, D, bucket, pad, 1.0 / D, hg, instances=inst)
    torch.cuda.synchronize()
    for r in range(D):
        assert_f16_close(dg[r].cpu().numpy(), hg[r], f"allreduce[{r}]", ulps=0)
    # fused with the step
    hg = [t2np_grad(g) for g in grads[0]]
    dg = [g.to(DEV) for g in grads[0]]
    h = [master.numpy().copy(), m.numpy().copy(), v.numpy().copy()]
    hp = [t2np_param(p) for p in params]
    d = [master.to(DEV), m.to(DEV), v.to(DEV)]
    dp = [p.to(DEV) for p in params]
    adam = B.AdamConfig(grad_scale=1.0 / D)
    B.dopt_step_allreduce(L, adam, 1, dg, *d, dp)
    oracle.step(sizes, wd, D, bucket, pad, oracle.make_adam(**asdict(adam)), 1, hg, *h, hp,
                instances=inst)
    oracle.allreduce(sizes, D, bucket, pad, adam.grad_scale, hg, instances=inst)
    torch.cuda.synchronize()
    for r in range(D):
        assert_f16_close(dg[r].cpu().numpy(), hg[r], f"grads[{r}]", ulps=0)
        assert_param_close(dp[r], hp[r], f"param{r}")
    for name, x, y in zip(("master", "exp_avg", "exp_avg_sq"), d, h):
        assert_f32_close(t2np_f32(x), y, name)


@pytest.mark.parametrize("case", [0, 1, 3])
def test_clipped_fp16_with_rounding(case):
    L, N, (sizes, wd, D, inst, bucket, pad), master, m, v, params, grads = _case(
        case, "fp16", "fp16", 1, 1300 + case)
    hg = [t2np_grad(g) for g in grads[0]]
    adam = B.AdamConfig(grad_scale=1.0 / D)
    nsq = oracle.grad_norm_sq(sizes, D, bucket, pad, adam.grad_scale, hg, instances=inst,
                              round_grad=True)
    max_norm = 0.25 * float(np.sqrt(nsq))
    coef = oracle.clip_coef(nsq, max_norm)
    h = [master.numpy().copy(), m.numpy().copy(), v.numpy().copy()]
    hp = [t2np_param(p) for p in params]
    hmg = np.zeros(N, np.float32)
    d = [master.to(DEV), m.to(DEV), v.to(DEV)]
    dp = [p.to(DEV) for p in params]
    mg = torch.zeros(N, device=DEV)
    rep = B.clip_report(DEV)
    B.dopt_step_clipped(L, adam, 1, max_norm, [g.to(DEV) for g in grads[0]], *d, dp, mg,
                        B.clip_workspace(DEV), norm_out=rep, round_grad=True, skip_nonfinite=True)
    oracle.step(sizes, wd, D, bucket, pad, oracle.make_adam(**asdict(adam)), 1, hg, *h, hp,
                main_grad_out=hmg, clip_coef=coef, instances=inst, round_grad=True)
    norm, c, bad = B.read_clip_report(rep)
    assert bad == 0 and abs(norm - np.sqrt(nsq)) <= 1e-6 * np.sqrt(nsq)
    assert abs(c - coef) <= 1e-6 * coef
    assert_f32_close(t2np_f32(mg), hmg, "main_grad")
    for name, x, y in zip(("master", "exp_avg", "exp_avg_sq"), d, h):
        assert_f32_close(t2np_f32(x), y, name)
    for r in range(D):
        assert_param_close(dp[r], hp[r], f"param{r}")


def test_fp16_overflow_counts_once_rounded():
    """60000 + 60000 is finite in fp32 and beyond fp16: with the rounding to
    the grad type it is non-finite and the checked step is skipped."""
    sizes, D = [64, 64], 2
    L = B.dopt_build_range_map(sizes, D, 0, 1).to_device()
    N = L.padded_numel
    g = [torch.zeros(N, dtype=torch.float16, device=DEV) for _ in range(D)]
    g[0][7] = g[1][7] = 60000.0
    st = [torch.full((N,), 0.5, device=DEV), torch.zeros(N, device=DEV), torch.zeros(N, device=DEV)]
    p = [torch.zeros(N, dtype=torch.float16, device=DEV) for _ in range(D)]
    for rg, want in ((False, 0), (True, 1)):
        assert oracle.count_nonfinite(sizes, D, 0, 1, 1.0, [x.cpu().numpy() for x in g],
                                      round_grad=rg) == want
        rep = B.clip_report(DEV)
        before = st[0].clone()
        B.dopt_step_clipped(L, B.AdamConfig(grad_scale=1.0), 1, 1e9, g, *st, p,
                            torch.empty(N, device=DEV), B.clip_workspace(DEV), norm_out=rep,
                            round_grad=rg, skip_nonfinite=True)
        assert B.read_clip_report(rep)[2] == want
        assert torch.equal(before, st[0]) == bool(want)


def test_counted_host_grads_and_gather_fp16():
    """The counted step with fp16 params, the zero-copy host grads in fp16,
    and the standalone gather of fp16 params give dopt_step's results."""
    L, N, cfg, master, m, v, params, grads = _case(1, "fp16", "fp16", 1, 1400)
    D = cfg[2]
    adam = B.AdamConfig(grad_scale=1.0 / D)
    base = [master.to(DEV), m.to(DEV), v.to(DEV)]
    pbase = [p.to(DEV) for p in params]
    B.dopt_step(L, adam, 1, [g.to(DEV) for g in grads[0]], *base, pbase)
    runs = []
    # counted
    a = [master.to(DEV), m.to(DEV), v.to(DEV)]
    pa = [p.to(DEV) for p in params]
    B.dopt_step_counted(L, adam, B.step_counter(1), [g.to(DEV) for g in grads[0]], *a, pa)
    runs.append(a + pa)
    # zero-copy host grads
    b = [master.to(DEV), m.to(DEV), v.to(DEV)]
    pb = [p.to(DEV) for p in params]
    host = [g.contiguous().pin_memory() for g in grads[0]]
    B.dopt_step(L, adam, 1, host, *b, pb, host_grads=True)
    runs.append(b + pb)
    # step without the gather, then the gather kernel
    c = [master.to(DEV), m.to(DEV), v.to(DEV)]
    pc = [p.to(DEV) for p in params]
    B.dopt_step(L, adam, 1, [g.to(DEV) for g in grads[0]], *c, pc, gather=False)
    B.dopt_gather(L, pc)
    runs.append(c + pc)
    torch.cuda.synchronize()
    for run in runs:
        for x, y in zip(base + pbase, run):
            assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_gpt2_small_fp16_full_size_windows():
    """The GPT-2-small layout with fp16 grads and fp16 params at full size,
    3 steps, sampled windows against the oracle."""
    w = W.gpt2_small().with_(grad_dtype="fp16")
    L = B.dopt_build_range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit,
                               list(w.wd_mask)).to_device()
    O = oracle.range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit)
    N = L.padded_numel
    wins = sample_windows(L.buckets(), O.pieces, N, seed=123, n_edges=24, n_random=6)
    master, m, v = W.make_state(w, N, DEV)
    params = [master.half() for _ in range(w.D)]
    host = [[t2np_f32(master[a:b]).copy(), t2np_f32(m[a:b]).copy(), t2np_f32(v[a:b]).copy(),
             [params[r][a:b].cpu().numpy().copy() for r in range(w.D)]] for a, b in wins]
    adam = B.AdamConfig(**w.adam_kwargs())
    oadam = oracle.make_adam(**asdict(adam))
    for t in range(1, 4):
        grads = W.make_grads(w, N, t, DEV)
        assert grads[0].dtype == torch.float16
        B.dopt_step(L, adam, t, grads, master, m, v, params)
        for (a, b), hs in zip(wins, host):
            oracle.step(list(w.sizes), list(w.wd_mask), w.D, w.bucket_elems, w.pad_unit, oadam, t,
                        [g[a:b].cpu().numpy() for g in grads], hs[0], hs[1], hs[2], hs[3],
                        window=(a, b))
        del grads
    torch.cuda.synchronize()
    for (a, b), hs in zip(wins, host):
        assert_f32_close(t2np_f32(master[a:b]), hs[0], f"master[{a}:{b}]")
        assert_f32_close(t2np_f32(m[a:b]), hs[1], f"m[{a}:{b}]")
        assert_f32_close(t2np_f32(v[a:b]), hs[2], f"v[{a}:{b}]")
        for r in range(w.D):
            assert_f16_close(params[r][a:b].cpu().numpy(), hs[3][r], f"param{r}[{a}:{b}]")
