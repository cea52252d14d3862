"""The non-finite check of the clipped step (DOPT_STEP_SKIP_NONFINITE)
against the oracle's count (reading R13 of the oracle): the device counts
the owned elements whose reduced grad is Inf or NaN, and with the flag a
step with a non-zero count stores nothing but the main grads and the
report.  Without the flag, Inf/NaN grads propagate as the oracle's clipped
step says."""
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
    # sizes, wd, D, instances, bucket, pad, grad dtype
    ([5000, 1, 7, 300, 20000, 3, 9999], [1, 0, 1, 0, 1, 1, 0], 8, 1, 0, 1, "bf16"),
    ([4096, 333, 12345, 8, 77777], [0, 1, 1, 0, 1], 3, 1, 20000, 1, "fp32"),
    ([31000, 17, 64000, 5], [1, 0, 1, 0], 8, 2, 30000, 3, "bf16"),
]
INF_BF16, NINF_BF16, NAN_BF16 = 0x7F80, 0xFF80, 0x7FC0


def _owned(L):
    mask = np.zeros(L.padded_numel, bool)
    for a, b in L.param_offsets():
        mask[a:b] = True
    return mask


def _poison(grads, grad_dtype, where, rng):
    """Write Inf/-Inf/NaN into the given (replica, element) positions."""
    for r, i in where:
        kind = int(rng.integers(0, 3))
        if grad_dtype == "bf16":
            grads[r].view(torch.int16)[i] = [INF_BF16, NINF_BF16 - 0x10000, NAN_BF16][kind]
        else:
            grads[r][i] = [float("inf"), float("-inf"), float("nan")][kind]


def _host(grads, grad_dtype):
    return [t2np_bf16(g).copy() if grad_dtype == "bf16" else g.numpy().copy() for g in grads]


def _setup(case, seed):
    sizes, wd, D, inst, bucket, pad, gdt = case
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd, instances=inst).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, 1, gdt, seed)
    return L, N, [master, m, v], params, grads[0]


def _clipped(L, adam, grads, state, params, max_norm, skip, report=None):
    d = [x.to(DEV) for x in state]
    dp = [p.to(DEV) for p in params]
    mg = torch.full((L.padded_numel,), -7.0, device=DEV)
    rep = report if report is not None else B.clip_report(DEV)
    B.dopt_step_clipped(L, adam, 1, max_norm, [g.to(DEV) for g in grads], *d, dp, mg,
                        B.clip_workspace(DEV), norm_out=rep, skip_nonfinite=skip)
    torch.cuda.synchronize()
    return d, dp, mg, rep


@pytest.mark.parametrize("case", range(len(CASES)))
def test_clean_grads_step_as_without_the_check(case):
    L, N, state, params, grads = _setup(CASES[case], 900 + case)
    adam = B.AdamConfig(grad_scale=1.0 / L.D)
    a = _clipped(L, adam, grads, state, params, 0.05, skip=False)
    b = _clipped(L, adam, grads, state, params, 0.05, skip=True)
    for x, y in zip(a[0] + a[1] + [a[2]], b[0] + b[1] + [b[2]]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    norm, coef, bad = B.read_clip_report(b[3])
    assert bad == 0 and np.isfinite(coef) and 0 < coef < 1
    assert a[3][:2].tolist() == [norm, coef]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("n_bad", [1, 7])
def test_nonfinite_grads_skip_the_step(case, n_bad):
    sizes, wd, D, inst, bucket, pad, gdt = CASES[case]
    L, N, state, params, grads = _setup(CASES[case], 950 + case)
    rng = np.random.default_rng(case * 10 + n_bad)
    owned = np.flatnonzero(_owned(L))
    where = [(int(rng.integers(0, D)), int(owned[int(rng.integers(0, len(owned)))]))
             for _ in range(n_bad)]
    where.append((0, int(N - 1)) if not _owned(L)[N - 1] else where[0])  # padding too
    _poison(grads, gdt, where, rng)
    hg = _host(grads, gdt)
    want = oracle.count_nonfinite(sizes, D, bucket, pad, 1.0 / D, hg, instances=inst)
    assert 1 <= want <= n_bad
    adam = B.AdamConfig(grad_scale=1.0 / D)
    d, dp, mg, rep = _clipped(L, adam, grads, state, params, 0.05, skip=True)
    for x, x0 in zip(d, state):
        assert torch.equal(x.cpu().view(torch.int32), x0.view(torch.int32))
    for p, p0 in zip(dp, params):
        assert torch.equal(p.cpu().view(torch.int16), p0.view(torch.int16))
    norm, coef, bad = B.read_clip_report(rep)
    assert bad == want and np.isnan(coef) and not np.isfinite(norm)
    # the main grads are still reported, as the oracle's reduce-scatter gives them
    hmg = np.full(N, -7.0, np.float32)
    h = [x.numpy().copy() for x in state]
    oracle.step(sizes, wd, D, bucket, pad, oracle.make_adam(**asdict(adam)), 1, hg, *h,
                [t2np_bf16(p).copy() for p in params], main_grad_out=hmg, instances=inst)
    assert_f32_close(t2np_f32(mg), hmg, "main_grad")


def test_nonfinite_at_padding_is_not_counted():
    sizes, wd, D, bucket, pad = [100, 3, 29], None, 4, 0, 64
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd).to_device()
    N = L.padded_numel
    assert N > sum(sizes)
    master, m, v, params, grads = W.random_case(N, D, 1, "bf16", 3)
    g = grads[0]
    pad_pos = [i for i in range(N) if not _owned(L)[i]]
    for r in range(D):
        g[r].view(torch.int16)[pad_pos[r % len(pad_pos)]] = NAN_BF16
    adam = B.AdamConfig(grad_scale=0.25)
    a = _clipped(L, adam, g, [master, m, v], params, 0.05, skip=False)
    b = _clipped(L, adam, g, [master, m, v], params, 0.05, skip=True)
    for x, y in zip(a[0] + a[1], b[0] + b[1]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    assert B.read_clip_report(b[3])[2] == 0


def test_rounding_to_bf16_overflow_counts_only_when_rounded():
    """Max bf16 + 2^119 is finite in fp32 and a tie that bf16 rounds to Inf."""
    sizes, D = [40, 24], 2
    L = B.dopt_build_range_map(sizes, D, 0, 1).to_device()
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, 1, "bf16", 4)
    g = grads[0]
    g[0].view(torch.int16)[5] = 0x7F7F
    g[1].view(torch.int16)[5] = 0x7B00
    adam = B.AdamConfig(grad_scale=1.0)
    hg = _host(g, "bf16")
    for rg in (False, True):
        want = oracle.count_nonfinite(sizes, D, 0, 1, 1.0, hg, round_grad=rg)
        assert want == int(rg)
        d = [x.to(DEV) for x in (master, m, v)]
        dp = [p.to(DEV) for p in params]
        rep = B.clip_report(DEV)
        B.dopt_step_clipped(L, adam, 1, 1e30, [x.to(DEV) for x in g], *d, dp,
                            torch.empty(N, device=DEV), B.clip_workspace(DEV), norm_out=rep,
                            round_grad=rg, skip_nonfinite=True)
        assert B.read_clip_report(rep)[2] == want
        assert torch.equal(d[0].cpu(), master) == rg  # skipped only when rounded


def test_without_the_check_nonfinite_propagates_like_the_oracle():
    sizes, wd, D, inst, bucket, pad, gdt = CASES[0]
    L, N, state, params, grads = _setup(CASES[0], 77)
    owned = np.flatnonzero(_owned(L))
    grads[2][int(owned[1000])] = float("inf")  # bf16 tensor: +Inf
    hg = _host(grads, gdt)
    adam = B.AdamConfig(grad_scale=1.0 / D)
    nsq = oracle.grad_norm_sq(sizes, D, bucket, pad, adam.grad_scale, hg)
    coef = oracle.clip_coef(nsq, 0.5)
    assert np.isinf(nsq) and coef == 0.0
    d, dp, mg, rep = _clipped(L, adam, grads, state, params, 0.5, skip=False)
    h = [x.numpy().copy() for x in state]
    hp = [t2np_bf16(p).copy() for p in params]
    oracle.step(sizes, wd, D, bucket, pad, oracle.make_adam(**asdict(adam)), 1, hg, *h, hp,
                clip_coef=coef)
    for name, x, y in zip(("master", "exp_avg", "exp_avg_sq"), d, h):
        assert_f32_close(t2np_f32(x), y, name)  # NaN positions must agree
    for r in range(D):
        assert_bf16_close(t2np_bf16(dp[r]), hp[r], f"param{r}")
    assert np.isnan(t2np_f32(d[0])).sum() == 1


def test_workspace_reuse_resets_the_count():
    sizes, wd, D, inst, bucket, pad, gdt = CASES[1]
    L, N, state, params, grads = _setup(CASES[1], 5)
    clean = [g.clone() for g in grads]
    grads[1][int(np.flatnonzero(_owned(L))[10])] = float("nan")
    adam = B.AdamConfig(grad_scale=1.0 / D)
    ws, rep = B.clip_workspace(DEV), B.clip_report(DEV)
    d = [x.to(DEV) for x in state]
    dp = [p.to(DEV) for p in params]
    mg = torch.empty(N, device=DEV)
    for g, want_bad in ((grads, 1), (clean, 0), (grads, 1), (clean, 0)):
        before = d[0].clone()
        B.dopt_step_clipped(L, adam, 1, 0.05, [x.to(DEV) for x in g], *d, dp, mg, ws,
                            norm_out=rep, skip_nonfinite=True)
        assert B.read_clip_report(rep)[2] == want_bad
        assert torch.equal(before, d[0]) == bool(want_bad)


def test_gpt2_small_one_inf_skips_the_step():
    w = W.gpt2_small()
    L = B.dopt_build_range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit,
                               list(w.wd_mask)).to_device()
    N = L.padded_numel
    master, m, v = W.make_state(w, N, DEV)
    params = W.make_params(master, w.D)
    grads = W.make_grads(w, N, 1, DEV)
    grads[5].view(torch.int16)[N // 2 + 12345] = INF_BF16
    before = [master.clone(), params[3].clone()]
    rep = B.clip_report(DEV)
    B.dopt_step_clipped(L, B.AdamConfig(**w.adam_kwargs()), 1, 1.0, grads, master, m, v, params,
                        torch.empty(N, device=DEV), B.clip_workspace(DEV), norm_out=rep,
                        skip_nonfinite=True)
    norm, coef, bad = B.read_clip_report(rep)
    assert bad == 1 and np.isnan(coef) and np.isinf(norm)
    assert torch.equal(before[0], master) and torch.equal(before[1], params[3])
