"""Several distributed-optimizer instances (distributed-optimizer page, §5) on the device, against
the oracle: reduce-scatter inside each instance of R = D/I ranks, sums across
instances in instance order, write-back and gather inside each instance."""
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

# Every group size the compile-time grouped kernels take (D = 4 in 2; 8 in
# 2, 4; 16 in 2, 4, 8, where fp32 grads take the run-time form), the
# run-time form (D = 6 in 3), and groups of one rank (D = 8 in 8, D = 4 in
# 4), which take the one-instance kernels.
CASES = [
    # sizes, wd, D, instances, bucket, pad
    ([130, 260, 90, 310, 210], None, 4, 2, 0, 1),
    ([5000, 1, 7, 300, 20000, 3, 9999], [1, 0, 1, 0, 1, 1, 0], 8, 2, 0, 1),
    ([4096, 333, 12345, 8, 77777], [0, 1, 1, 0, 1], 6, 3, 20000, 1),
    ([65536, 1000, 65536], [1, 0, 1], 16, 4, 0, 64),
    ([123457, 99], [1, 0], 8, 8, 0, 1),
    ([31000, 17, 64000, 5], [1, 0, 1, 0], 8, 4, 30000, 3),
    ([40000, 3, 24000, 77], [1, 0, 1, 1], 16, 2, 0, 1),
    ([40000, 3, 24000, 77], [0, 1, 1, 0], 16, 8, 30000, 2),
    ([999, 1001, 64], None, 4, 4, 0, 1),
]


def _host(grads, dtype):
    return [t2np_bf16(g).copy() if dtype == "bf16" else g.numpy().copy() for g in grads]


def _run(case, grad_dtype, gather=True, steps=2, seed=0):
    sizes, wd, D, inst, bucket, pad = case
    R = D // inst
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd, instances=inst).to_device()
    N = L.padded_numel
    assert N == oracle.range_map(sizes, R, bucket, pad).numel
    master, m, v, params, grads = W.random_case(N, D, steps, grad_dtype, seed)
    h = [master.numpy().copy(), m.numpy().copy(), v.numpy().copy()]
    hp = [t2np_bf16(p).copy() for p in params]
    hmg = np.full(N, -3.0, np.float32)
    d = [master.to(DEV), m.to(DEV), v.to(DEV)]
    dp = [p.to(DEV) for p in params]
    dmg = torch.full((N,), -3.0, device=DEV)
    adam = B.AdamConfig(grad_scale=1.0 / D)
    oadam = oracle.make_adam(**asdict(adam))
    for i in range(steps):
        B.dopt_step(L, adam, i + 1, [g.to(DEV) for g in grads[i]], *d, dp, gather=gather,
                    main_grad_out=dmg)
        oracle.step(sizes, wd, D, bucket, pad, oadam, i + 1, _host(grads[i], grad_dtype), *h, hp,
                    gather=gather, main_grad_out=hmg, instances=inst)
    torch.cuda.synchronize()
    for name, x, y in zip(("master", "exp_avg", "exp_avg_sq"), d, h):
        assert_f32_close(t2np_f32(x), y, name)
    assert_f32_close(t2np_f32(dmg), hmg, "main_grad")
    for r in range(D):
        assert_bf16_close(t2np_bf16(dp[r]), hp[r], f"param{r}")
    return L, d, dp


@pytest.mark.parametrize("grad_dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_instances_parity(case, grad_dtype):
    _run(CASES[case], grad_dtype, gather=True, seed=500 + case)


@pytest.mark.parametrize("case", range(len(CASES)))
def test_instances_write_back_without_gather(case):
    _run(CASES[case], "bf16", gather=False, seed=600 + case)


def test_instances_rank_order_on_device():
    """D=4 as 2 instances, fp32 grads 2^24, 1 | 1, -2^24: the device's
    reduced grad is 1 (instance sums 2^24 and 1 - 2^24); one instance gives 0."""
    vals = [2.0 ** 24, 1.0, 1.0, -(2.0 ** 24)]
    for inst, want in ((2, 1.0), (1, 0.0)):
        L = B.dopt_build_range_map([1], 4, 0, 1, instances=inst).to_device()
        N = max(L.padded_numel, 8)
        grads = [torch.tensor([x] + [0.0] * (N - 1), device=DEV) for x in vals]
        st = [torch.zeros(N, device=DEV) for _ in range(3)]
        p = [torch.zeros(N, device=DEV, dtype=torch.bfloat16) for _ in range(4)]
        mg = torch.full((N,), 9.0, device=DEV)
        B.dopt_step(L, B.AdamConfig(grad_scale=1.0), 1, grads, *st, p, main_grad_out=mg)
        torch.cuda.synchronize()
        assert mg[0].item() == want


@pytest.mark.parametrize("case", range(len(CASES)))
def test_instances_gather_kernel(case):
    """Step without gather, then dopt_gather = step with gather."""
    sizes, wd, D, inst, bucket, pad = CASES[case]
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd, instances=inst).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, 1, "bf16", seed=700 + case)
    g = [x.to(DEV) for x in grads[0]]
    a = [master.to(DEV), m.to(DEV), v.to(DEV)]
    b = [x.clone() for x in a]
    pa = [p.to(DEV) for p in params]
    pb = [p.clone() for p in pa]
    adam = B.AdamConfig(grad_scale=1.0 / D)
    B.dopt_step(L, adam, 1, g, *a, pa, gather=True)
    B.dopt_step(L, adam, 1, g, *b, pb, gather=False)
    B.dopt_gather(L, pb)
    torch.cuda.synchronize()
    for x, y in zip(pa, pb):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("case", range(len(CASES)))
def test_instances_allreduce_and_clipped(case):
    sizes, wd, D, inst, bucket, pad = CASES[case]
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd, instances=inst).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, 1, "bf16", seed=800 + case)
    # all-reduce
    hg = _host(grads[0], "bf16")
    dg = [x.to(DEV) for x in grads[0]]
    B.dopt_allreduce(L, dg, 1.0 / D)
    oracle.allreduce(sizes, D, bucket, pad, 1.0 / D, hg, instances=inst)
    torch.cuda.synchronize()
    for r in range(D):
        assert_bf16_close(t2np_bf16(dg[r]), hg[r], f"allreduce[{r}]", ulps=0)
    # clipped step
    hg = _host(grads[0], "bf16")
    adam = B.AdamConfig(grad_scale=1.0 / D)
    nsq = oracle.grad_norm_sq(sizes, D, bucket, pad, adam.grad_scale, hg, instances=inst)
    max_norm = 0.3 * float(np.sqrt(nsq))
    coef = oracle.clip_coef(nsq, max_norm)
    h = [master.numpy().copy(), m.numpy().copy(), v.numpy().copy()]
    hp = [t2np_bf16(p).copy() for p in params]
    d = [master.to(DEV), m.to(DEV), v.to(DEV)]
    dp = [p.to(DEV) for p in params]
    norm_out = torch.zeros(2, device=DEV)
    B.dopt_step_clipped(L, adam, 1, max_norm, [x.to(DEV) for x in grads[0]], *d, dp,
                        torch.empty(N, device=DEV), B.clip_workspace(DEV), norm_out=norm_out)
    oracle.step(sizes, wd, D, bucket, pad, oracle.make_adam(**asdict(adam)), 1, hg, *h, hp,
                clip_coef=coef, instances=inst)
    torch.cuda.synchronize()
    assert abs(norm_out[0].item() - np.sqrt(nsq)) <= 1e-6 * np.sqrt(nsq)
    for name, x, y in zip(("master", "exp_avg", "exp_avg_sq"), d, h):
        assert_f32_close(t2np_f32(x), y, name)
    for r in range(D):
        assert_bf16_close(t2np_bf16(dp[r]), hp[r], f"param{r}")


def test_instances_gpt2_small_full_size():
    """The GPT-2-small layout at full size with D=8 as 2 instances of 4
    ranks (buckets sharded 4 ways), 3 steps, sampled windows."""
    w = W.gpt2_small()
    inst, R, steps = 2, 4, 3
    L = B.dopt_build_range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit, list(w.wd_mask),
                               instances=inst).to_device()
    O = oracle.range_map(list(w.sizes), R, w.bucket_elems, w.pad_unit)
    assert L.padded_numel == O.numel and L.pieces() == O.pieces
    N = L.padded_numel
    wins = sample_windows(L.buckets(), O.pieces, N, seed=91, n_edges=24, n_random=6)
    master, m, v = W.make_state(w, N, DEV)
    params = W.make_params(master, w.D)
    host = [[t2np_f32(master[a:b]).copy(), t2np_f32(m[a:b]).copy(), t2np_f32(v[a:b]).copy(),
             [t2np_bf16(p[a:b]).copy() for p in params]] for a, b in wins]
    adam = B.AdamConfig(**w.adam_kwargs())
    oadam = oracle.make_adam(**asdict(adam))
    for t in range(1, steps + 1):
        grads = W.make_grads(w, N, t, DEV)
        B.dopt_step(L, adam, t, grads, master, m, v, params)
        for (a, b), hs in zip(wins, host):
            oracle.step(list(w.sizes), list(w.wd_mask), w.D, w.bucket_elems, w.pad_unit, oadam, t,
                        [t2np_bf16(g[a:b]) for g in grads], hs[0], hs[1], hs[2], hs[3],
                        window=(a, b), instances=inst)
        del grads
    torch.cuda.synchronize()
    for (a, b), hs in zip(wins, host):
        assert_f32_close(t2np_f32(master[a:b]), hs[0], f"master[{a}:{b}]")
        assert_f32_close(t2np_f32(m[a:b]), hs[1], f"m[{a}:{b}]")
        assert_f32_close(t2np_f32(v[a:b]), hs[2], f"v[{a}:{b}]")
        for r in range(w.D):
            assert_bf16_close(t2np_bf16(params[r][a:b]), hs[3][r], f"param{r}[{a}:{b}]")
