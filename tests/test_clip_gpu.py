"""Parity of the clipped step (global grad-norm clipping before AdamW) with
the oracle.

The oracle's norm^2 is an fp64 sum in piece order; the device sums fp32
squares pairwise per 8 elements and then in fp64, so the two norms differ by
at most a few units in the 24th bit (relative error <= 4 * 2^-24 from the
square and the three pairwise additions).  The coefficient therefore agrees
to ~2e-7 relative, a clipped grad to an ulp or two, which keeps master/m/v
inside the 1e-6 relative (+1e-7) tolerance and params inside 1 bf16 ulp."""
from dataclasses import asdict

import math

import numpy as np
import pytest
import torch

import oracle
from parity import assert_bf16_close, assert_f32_close, sample_windows, t2np_bf16, t2np_f32
from zero_distributed_optimizer_gb300 import binding as B
from zero_distributed_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
NORM_RTOL = 1e-6


def _run_small(sizes, wd, D, bucket, pad, grad_dtype, steps, clip_frac, seed):
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, steps, grad_dtype, seed)
    h = [master.numpy().copy(), m.numpy().copy(), v.numpy().copy()]
    hp = [t2np_bf16(p).copy() for p in params]
    d = [master.to(DEV), m.to(DEV), v.to(DEV)]
    dp = [p.to(DEV) for p in params]
    mg = torch.full((N,), -9.0, device=DEV)
    hmg = np.full(N, -9.0, np.float32)
    ws = B.clip_workspace(DEV)
    norm_out = torch.zeros(2, device=DEV)
    adam = B.AdamConfig(grad_scale=1.0 / D)
    oadam = oracle.make_adam(**asdict(adam))
    for i in range(steps):
        t = i + 1
        hg = [t2np_bf16(g) if grad_dtype == "bf16" else g.numpy().copy() for g in grads[i]]
        nsq = oracle.grad_norm_sq(sizes, D, bucket, pad, adam.grad_scale, hg)
        max_norm = clip_frac * float(np.sqrt(nsq)) if nsq > 0 else 1.0
        coef = oracle.clip_coef(nsq, max_norm)
        B.dopt_step_clipped(L, adam, t, max_norm, [g.to(DEV) for g in grads[i]], *d, dp, mg, ws,
                            norm_out=norm_out)
        oracle.step(sizes, wd, D, bucket, pad, oadam, t, hg, *h, hp, main_grad_out=hmg,
                    clip_coef=coef)
        torch.cuda.synchronize()
        got_norm, got_coef = norm_out.tolist()
        assert abs(got_norm - np.sqrt(nsq)) <= NORM_RTOL * np.sqrt(nsq) + 1e-30
        assert abs(got_coef - coef) <= NORM_RTOL * coef
        if clip_frac >= 1.0:
            assert got_coef == 1.0 and coef == 1.0
    assert_f32_close(t2np_f32(d[0]), h[0], "master")
    assert_f32_close(t2np_f32(d[1]), h[1], "exp_avg")
    assert_f32_close(t2np_f32(d[2]), h[2], "exp_avg_sq")
    assert_f32_close(t2np_f32(mg), hmg, "main_grad")
    for r in range(D):
        assert_bf16_close(t2np_bf16(dp[r]), hp[r], f"param{r}")


CLIP_CASES = [
    ([130, 260, 90, 310, 210], None, 4, 0, 1),
    ([5000, 1, 7, 300, 20000, 3, 9999], [1, 0, 1, 0, 1, 1, 0], 8, 0, 1),
    ([4096, 333, 12345, 8, 77777], [0, 1, 1, 0, 1], 3, 20000, 1),
    ([65536, 1000, 65536], [1, 0, 1], 16, 0, 64),
    ([123457, 99], [1, 0], 64, 0, 1),
    ([64] * 300 + [5000], None, 2, 4096, 64),
    ([600000, 17, 300001], [1, 0, 1], 8, 400000, 64),  # many CTAs' partials
]


@pytest.mark.parametrize("grad_dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("case", range(len(CLIP_CASES)))
def test_clipped_parity_small(case, grad_dtype):
    sizes, wd, D, bucket, pad = CLIP_CASES[case]
    _run_small(sizes, wd, D, bucket, pad, grad_dtype, steps=2, clip_frac=0.3, seed=100 + case)


def test_no_clipping_when_norm_is_small():
    sizes, wd, D = [20000, 7, 3000], [1, 0, 1], 4
    _run_small(sizes, wd, D, 0, 8, "bf16", steps=2, clip_frac=4.0, seed=7)


def test_clipped_with_large_max_norm_equals_plain_step():
    """A coefficient of exactly 1 gives the plain step bit for bit."""
    sizes, wd, D = [50000, 13, 7001], [1, 0, 1], 8
    L = B.dopt_build_range_map(sizes, D, 0, 64, wd).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, 1, "bf16", 3)
    a = [master.to(DEV), m.to(DEV), v.to(DEV)]
    b = [x.clone() for x in a]
    pa = [p.to(DEV) for p in params]
    pb = [p.clone() for p in pa]
    g = [x.to(DEV) for x in grads[0]]
    adam = B.AdamConfig(grad_scale=0.125)
    B.dopt_step(L, adam, 1, g, *a, pa)
    B.dopt_step_clipped(L, adam, 1, 1e30, g, *b, pb, torch.empty(N, device=DEV),
                        B.clip_workspace(DEV))
    torch.cuda.synchronize()
    for x, y in zip(a + pa, b + pb):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_clipped_workspace_reuse_and_side_stream():
    """The workspace is reset by every call: repeated calls on one workspace,
    on a side stream, give the same result as fresh workspaces."""
    sizes, wd, D = [300000, 5, 70000], [1, 0, 1], 4
    L = B.dopt_build_range_map(sizes, D, 0, 8, wd).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, 3, "bf16", 4)
    a = [master.to(DEV), m.to(DEV), v.to(DEV)]
    b = [x.clone() for x in a]
    pa = [p.to(DEV) for p in params]
    pb = [p.clone() for p in pa]
    mg = torch.empty(N, device=DEV)
    ws = B.clip_workspace(DEV)
    s = torch.cuda.Stream()
    adam = B.AdamConfig(grad_scale=0.25)
    for i in range(3):
        g = [x.to(DEV) for x in grads[i]]
        B.dopt_step_clipped(L, adam, i + 1, 0.01, g, *a, pa, mg, B.clip_workspace(DEV))
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            B.dopt_step_clipped(L, adam, i + 1, 0.01, g, *b, pb, mg, ws, stream=s)
        s.synchronize()
    for x, y in zip(a + pa, b + pb):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_clipped_gpt2_small_full_size():
    """The GPT-2-small layout at full size, 3 steps with clipping engaged:
    the oracle computes the global norm over the whole buffer and steps
    sampled windows."""
    w = W.gpt2_small()
    steps = 3
    L = B.dopt_build_range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit,
                               list(w.wd_mask)).to_device()
    O = oracle.range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit)
    N = L.padded_numel
    wins = sample_windows(L.buckets(), O.pieces, N, seed=77, n_edges=24, n_random=6)
    master, m, v = W.make_state(w, N, DEV)
    params = W.make_params(master, w.D)
    host = [[t2np_f32(master[a:b]).copy(), t2np_f32(m[a:b]).copy(), t2np_f32(v[a:b]).copy(),
             [t2np_bf16(p[a:b]).copy() for p in params]] for a, b in wins]
    mg = torch.empty(N, device=DEV)
    ws = B.clip_workspace(DEV)
    norm_out = torch.zeros(2, device=DEV)
    adam = B.AdamConfig(**w.adam_kwargs())
    oadam = oracle.make_adam(**asdict(adam))
    for t in range(1, steps + 1):
        grads = W.make_grads(w, N, t, DEV)
        hg_full = [t2np_bf16(g) for g in grads]
        nsq = oracle.grad_norm_sq(list(w.sizes), w.D, w.bucket_elems, w.pad_unit, w.grad_scale,
                                  hg_full)
        max_norm = 0.5 * float(np.sqrt(nsq))
        coef = oracle.clip_coef(nsq, max_norm)
        B.dopt_step_clipped(L, adam, t, max_norm, grads, master, m, v, params, mg, ws,
                            norm_out=norm_out)
        for (a, b), hs in zip(wins, host):
            oracle.step(list(w.sizes), list(w.wd_mask), w.D, w.bucket_elems, w.pad_unit, oadam, t,
                        [x[a:b].copy() for x in hg_full], hs[0], hs[1], hs[2], hs[3],
                        window=(a, b), clip_coef=coef)
        torch.cuda.synchronize()
        got_norm, got_coef = norm_out.tolist()
        assert abs(got_norm - np.sqrt(nsq)) <= NORM_RTOL * np.sqrt(nsq)
        assert abs(got_coef - coef) <= NORM_RTOL * coef
        del grads, hg_full
    for (a, b), hs in zip(wins, host):
        assert_f32_close(t2np_f32(master[a:b]), hs[0], f"master[{a}:{b}]")
        assert_f32_close(t2np_f32(m[a:b]), hs[1], f"m[{a}:{b}]")
        assert_f32_close(t2np_f32(v[a:b]), hs[2], f"v[{a}:{b}]")
        for r in range(w.D):
            assert_bf16_close(t2np_bf16(params[r][a:b]), hs[3][r], f"param{r}[{a}:{b}]")


def test_clipped_step_is_deterministic():
    """Each CTA adds its partial sum in a fixed order and the CTAs' partials
    are summed exactly, so two runs from the same inputs are bitwise
    equal."""
    sizes, wd, D = [700000, 5, 300001], [1, 0, 1], 8
    L = B.dopt_build_range_map(sizes, D, 0, 64, wd).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, 2, "bf16", 12)
    runs = []
    for _ in range(2):
        d = [master.to(DEV), m.to(DEV), v.to(DEV)]
        dp = [p.to(DEV) for p in params]
        norm_out = torch.zeros(2, device=DEV)
        ws = B.clip_workspace(DEV)
        mg = torch.empty(N, device=DEV)
        for i in range(2):
            B.dopt_step_clipped(L, B.AdamConfig(grad_scale=0.125), i + 1, 0.01,
                                [g.to(DEV) for g in grads[i]], *d, dp, mg, ws, norm_out=norm_out)
        torch.cuda.synchronize()
        runs.append(d + dp + [norm_out])
    for x, y in zip(*runs):
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32),
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y.view(torch.int32))


@pytest.mark.parametrize("D", [8, 2])  # 4 tiles per CTA; the persistent grid
@pytest.mark.parametrize("log2_scale", [0, -60, 40])
def test_norm_sum_is_exact(D, log2_scale):
    """With grads k * 2^s (k integer below 256, in replica 0 only, the other
    replicas zero, scaling 1) every square, every CTA's fp64 partial and the
    total are exact, so the norm^2 the kernel leaves in the workspace (a
    double at byte 16) must equal the integer sum of k^2, times 4^s, bit for
    bit: thousands of CTAs' partials added through the digits and carries
    of the exact accumulator, at scales that put them low, in the middle
    and high in its range."""
    sizes, wd = [700000, 5, 300001, 4096], [1, 0, 1, 1]
    L = B.dopt_build_range_map(sizes, D, 0, 64, wd).to_device()
    N = L.padded_numel
    rng = np.random.default_rng(31 + D)
    k = rng.integers(0, 256, size=N, dtype=np.int64)
    g0 = torch.from_numpy(k.astype(np.float32) * np.float32(2.0 ** log2_scale)).to(torch.bfloat16)
    assert torch.equal(g0.float(), torch.from_numpy(k.astype(np.float32) * np.float32(2.0 ** log2_scale)))
    grads = [g0.to(DEV)] + [torch.zeros(N, dtype=torch.bfloat16, device=DEV) for _ in range(D - 1)]
    master = torch.zeros(N, device=DEV)
    m, v = torch.zeros(N, device=DEV), torch.zeros(N, device=DEV)
    params = [torch.zeros(N, dtype=torch.bfloat16, device=DEV) for _ in range(D)]
    ws = B.clip_workspace(DEV)
    mg = torch.empty(N, device=DEV)
    B.dopt_step_clipped(L, B.AdamConfig(grad_scale=1.0), 1, 3.0e38, grads, master, m, v, params,
                        mg, ws)
    torch.cuda.synchronize()
    owned = np.zeros(N, dtype=bool)
    for a, b in L.param_offsets():
        owned[a:b] = True
    exact = int((k[owned] ** 2).sum())
    want = math.ldexp(float(exact), 2 * log2_scale)  # exact: the sum has < 53 bits
    assert exact < 2 ** 53
    got = ws[16:24].cpu().view(torch.float64).item()
    assert got == want, (got, want)


@pytest.mark.parametrize("D", [8, 2])  # 4 tiles per CTA; the persistent grid
def test_norm_sum_is_rounded_once(D):
    """Three CTAs' partials: 2^91 (tile 0, every grad 2^40) and twice
    3 * 2^36 (tiles 1 and 2, three grads 2^18 each), each exact.  Their exact
    sum, 2^91 + 0.75 ulp, rounds once to 2^91 + 2^39; added one after the
    other in fp64 each small partial (0.375 ulp) would vanish and leave
    2^91.  Tiles 0, 1 and 2 fall in three different CTAs both with 4 tiles
    per CTA (12 tiles: 3 CTAs taking every third tile) and with the
    persistent grid (one tile each)."""
    tiles = 12
    L = B.dopt_build_range_map([tiles * 2048], D, 0, 64).to_device()
    N = L.padded_numel
    assert N == tiles * 2048
    g0 = torch.zeros(N, dtype=torch.bfloat16)
    g0[:2048] = 2.0 ** 40
    g0[2048:2048 + 3] = 2.0 ** 18
    g0[4096:4096 + 3] = 2.0 ** 18
    grads = [g0.to(DEV)] + [torch.zeros(N, dtype=torch.bfloat16, device=DEV) for _ in range(D - 1)]
    master = torch.zeros(N, device=DEV)
    m, v = torch.zeros(N, device=DEV), torch.zeros(N, device=DEV)
    params = [torch.zeros(N, dtype=torch.bfloat16, device=DEV) for _ in range(D)]
    ws = B.clip_workspace(DEV)
    mg = torch.empty(N, device=DEV)
    B.dopt_step_clipped(L, B.AdamConfig(grad_scale=1.0), 1, 3.0e38, grads, master, m, v, params,
                        mg, ws)
    torch.cuda.synchronize()
    got = ws[16:24].cpu().view(torch.float64).item()
    assert got == float(2 ** 91 + 6 * 2 ** 36) == 2.0 ** 91 + 2.0 ** 39, got


@pytest.mark.parametrize("D", [8, 2])
def test_clipped_parity_huge_grads(D):
    """Grads far beyond fp32's square root of its largest value (some
    elements 2^70 and 2^100 times larger, bf16 still holds them): the norm is
    a finite sum of fp64 squares, as in the oracle, not Inf from an fp32
    square, and the clipped step matches the oracle, run edges included."""
    sizes, wd, bucket, pad = [5000, 1, 7, 300, 20000, 3, 9999], [1, 0, 1, 0, 1, 1, 0], 0, 1
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, 1, "bf16", 77)
    rng = np.random.default_rng(5)
    g = [x.float() for x in grads[0]]
    for r in range(D):
        big = rng.random(N) < 0.01
        huge = (rng.random(N) < 0.001) & ~big  # at most 2^100 times larger
        g[r][torch.from_numpy(big)] *= 2.0 ** 70
        g[r][torch.from_numpy(huge)] *= 2.0 ** 100
    g = [x.to(torch.bfloat16) for x in g]
    assert all(torch.isfinite(x.float()).all() for x in g)
    hg = [t2np_bf16(x) for x in g]
    adam = B.AdamConfig(grad_scale=1.0 / D)
    oadam = oracle.make_adam(**asdict(adam))
    nsq = oracle.grad_norm_sq(sizes, D, bucket, pad, adam.grad_scale, hg)
    assert np.isfinite(nsq) and nsq > 2.0 ** 140  # some fp32 squares would overflow
    max_norm = 0.5 * float(np.sqrt(nsq))
    coef = oracle.clip_coef(nsq, max_norm)
    h = [master.numpy().copy(), m.numpy().copy(), v.numpy().copy()]
    hp = [t2np_bf16(p).copy() for p in params]
    hmg = np.full(N, -9.0, np.float32)
    d = [master.to(DEV), m.to(DEV), v.to(DEV)]
    dp = [p.to(DEV) for p in params]
    mg = torch.full((N,), -9.0, device=DEV)
    ws = B.clip_workspace(DEV)
    norm_out = torch.zeros(2, device=DEV)
    B.dopt_step_clipped(L, adam, 1, max_norm, [x.to(DEV) for x in g], *d, dp, mg, ws,
                        norm_out=norm_out)
    oracle.step(sizes, wd, D, bucket, pad, oadam, 1, hg, *h, hp, main_grad_out=hmg, clip_coef=coef)
    torch.cuda.synchronize()
    got_norm, got_coef = norm_out.tolist()
    assert np.isfinite(got_norm)
    assert abs(got_norm - np.sqrt(nsq)) <= NORM_RTOL * np.sqrt(nsq)
    assert abs(got_coef - coef) <= NORM_RTOL * coef
    assert_f32_close(t2np_f32(d[0]), h[0], "master")
    assert_f32_close(t2np_f32(d[1]), h[1], "exp_avg")
    assert_f32_close(t2np_f32(d[2]), h[2], "exp_avg_sq")
    assert_f32_close(t2np_f32(mg), hmg, "main_grad")
    for r in range(D):
        assert_bf16_close(t2np_bf16(dp[r]), hp[r], f"param{r}")
