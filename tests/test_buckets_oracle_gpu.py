"""Bucket-range launches (dopt_step_buckets) against the oracle.

The distributed-optimizer page (§2: the flat buffer is cut into buckets;
§4.2: a bucket's reduce-scatter starts as soon as all of its grads are
ready) lets each bucket be stepped on its own.  These tests launch the step
bucket by bucket, in reverse order (the order in which backward fills the
buckets), on one or three streams, with and without the fused all-gather,
and compare every element of every output with the oracle's step of the
same buckets; a launch over a strict subset of the buckets must match the
oracle inside that subset and leave every element outside it untouched,
bit for bit.  The last case is the 256 Mi-element sweep layout with 1 Mi
buckets at full size, compared on sampled windows."""
from dataclasses import asdict

import numpy as np
import pytest
import torch

import oracle
from parity import (assert_bf16_close, assert_f32_close, sample_windows, t2np_bf16, t2np_f32,
                    t2np_grad)
from zero_distributed_optimizer_gb300 import binding as B
from zero_distributed_optimizer_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"

# (sizes, wd_mask, D, bucket_elems, pad_unit, instances): several buckets
# each, params cut by shard edges, padding at every bucket end
CASES = [
    ([5000, 7000, 3000, 9000, 4000], None, 4, 6000, 8, 1),
    ([4096, 333, 12345, 8, 77777, 5, 20001], [0, 1, 1, 0, 1, 0, 1], 3, 12000, 1, 1),
    ([1000, 3, 2000, 5, 700, 4444], None, 1, 1000, 1, 1),
    ([130, 260, 90, 310, 210] * 6, [1, 1, 0, 1, 0] * 6, 8, 600, 2, 1),
    ([65536, 1000, 65536, 17, 3000, 70000], [1, 0, 1, 0, 1, 1], 16, 60000, 64, 1),
    ([9000, 1, 7, 300, 20000, 3, 9999, 12000], [1, 0, 1, 0, 1, 1, 0, 1], 8, 9000, 4, 2),
]


def _layout(case):
    sizes, wd, D, bucket, pad, inst = CASES[case]
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd, instances=inst).to_device()
    assert L.n_buckets >= 3
    return L


def _run_buckets(L, adam, t, grads, state, params, order, streams, gather, mg):
    """Launch buckets in `order`, one launch each, round-robin over
    `streams` streams forked from and joined back to the current one."""
    ss = [torch.cuda.current_stream()] + [torch.cuda.Stream() for _ in range(streams - 1)]
    fork = torch.cuda.Event()
    fork.record()
    for s in ss[1:]:
        s.wait_event(fork)
    for i, k in enumerate(order):
        s = ss[i % streams]
        with torch.cuda.stream(s):
            B.dopt_step_buckets(L, adam, t, k, 1, grads, *state, params, gather=gather,
                                main_grad_out=mg, stream=s)
    for s in ss[1:]:
        ev = torch.cuda.Event()
        ev.record(s)
        torch.cuda.current_stream().wait_event(ev)


def _compare(dev_state, dev_params, dev_mg, host_state, host_params, host_mg, sl=slice(None)):
    not_exact = 0
    for name, x, y in zip(("master", "exp_avg", "exp_avg_sq"), dev_state, host_state):
        not_exact += assert_f32_close(t2np_f32(x[sl]), y[sl], name)
    not_exact += assert_f32_close(t2np_f32(dev_mg[sl]), host_mg[sl], "main_grad")
    for r, (x, y) in enumerate(zip(dev_params, host_params)):
        not_exact += assert_bf16_close(t2np_bf16(x[sl]), y[sl], f"param{r}")
    return not_exact


@pytest.mark.parametrize("gather", [True, False])
@pytest.mark.parametrize("streams", [1, 3])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_bucket_launches_match_oracle(case, streams, gather):
    """Two steps, each as one launch per bucket in reverse bucket order,
    against the oracle's step over the whole buffer, every element."""
    sizes, wd, D, bucket, pad, inst = CASES[case]
    L = _layout(case)
    N = L.padded_numel
    master, m, v, params, grads = W.random_case(N, D, 2, "bf16", seed=700 + case)
    host_state = [master.numpy().copy(), m.numpy().copy(), v.numpy().copy()]
    host_params = [t2np_bf16(p).copy() for p in params]
    host_mg = np.full(N, -3.0, np.float32)
    dev_state = [master.to(DEV), m.to(DEV), v.to(DEV)]
    dev_params = [p.to(DEV) for p in params]
    dev_mg = torch.full((N,), -3.0, device=DEV)
    adam = B.AdamConfig(grad_scale=1.0 / D, weight_decay=0.05)
    oadam = oracle.make_adam(**asdict(adam))
    order = list(reversed(range(L.n_buckets)))
    not_exact = 0
    for t in (1, 2):
        dg = [g.to(DEV) for g in grads[t - 1]]
        _run_buckets(L, adam, t, dg, dev_state, dev_params, order, streams, gather, dev_mg)
        oracle.step(sizes, wd, D, bucket, pad, oadam, t, [t2np_grad(g) for g in grads[t - 1]],
                    *host_state, host_params, gather=gather, main_grad_out=host_mg,
                    instances=inst)
        torch.cuda.synchronize()
        not_exact += _compare(dev_state, dev_params, dev_mg, host_state, host_params, host_mg)
    assert not_exact == 0  # same operations in the same order: bit for bit


@pytest.mark.parametrize("case", range(len(CASES)))
def test_bucket_subset_launch_matches_oracle_and_leaves_the_rest(case):
    """One launch over buckets [1, n_buckets - 1): inside their span the
    oracle's step of that window; outside it nothing changes."""
    sizes, wd, D, bucket, pad, inst = CASES[case]
    L = _layout(case)
    N = L.padded_numel
    bk = L.buckets()
    first, count = 1, L.n_buckets - 2
    lo, hi = bk[first][0], bk[first + count - 1][1]
    master, m, v, params, grads = W.random_case(N, D, 1, "bf16", seed=800 + case)
    dev_state = [master.to(DEV), m.to(DEV), v.to(DEV)]
    dev_params = [p.to(DEV) for p in params]
    before = [x.clone() for x in dev_state + dev_params]
    dev_mg = torch.full((N,), -3.0, device=DEV)
    adam = B.AdamConfig(grad_scale=1.0 / D)
    dg = [g.to(DEV) for g in grads[0]]
    B.dopt_step_buckets(L, adam, 1, first, count, dg, *dev_state, dev_params, gather=True,
                        main_grad_out=dev_mg)
    w = slice(lo, hi)
    host_state = [master.numpy()[w].copy(), m.numpy()[w].copy(), v.numpy()[w].copy()]
    host_params = [t2np_bf16(p)[w].copy() for p in params]
    host_mg = np.full(hi - lo, -3.0, np.float32)
    oracle.step(sizes, wd, D, bucket, pad, oracle.make_adam(**asdict(adam)), 1,
                [t2np_grad(g)[w].copy() for g in grads[0]], *host_state, host_params,
                main_grad_out=host_mg, window=(lo, hi), instances=inst)
    torch.cuda.synchronize()
    assert _compare([x[w] for x in dev_state], [p[w] for p in dev_params], dev_mg[w],
                    host_state, host_params, host_mg) == 0
    for x, x0 in zip(dev_state + dev_params, before):
        assert torch.equal(x[:lo].view(torch.int16), x0[:lo].view(torch.int16))
        assert torch.equal(x[hi:].view(torch.int16), x0[hi:].view(torch.int16))
    assert torch.all(dev_mg[:lo] == -3.0) and torch.all(dev_mg[hi:] == -3.0)


def test_bucket_launches_full_size_sweep_1mi_match_oracle():
    """The 256 Mi sweep layout with 1 Mi buckets (D = 8), two steps, each as
    one launch per bucket in reverse order over two streams: sampled windows
    (both ends of every bucket with its padding, piece edges, random
    stretches) against the oracle."""
    w = W.sweep_256m(8, 1)
    L = B.dopt_build_range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit,
                               list(w.wd_mask)).to_device()
    O = oracle.range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit)
    assert L.n_buckets > 200 and L.pieces() == O.pieces
    N = L.padded_numel
    wins = sample_windows(L.buckets(), O.pieces, N, seed=11, n_edges=32, n_random=6)
    master, m, v = W.make_state(w, N, DEV)
    params = W.make_params(master, w.D)
    mg = torch.full((N,), -5.0, device=DEV)
    host = [[t2np_f32(master[a:b]).copy(), t2np_f32(m[a:b]).copy(), t2np_f32(v[a:b]).copy(),
             [t2np_bf16(p[a:b]).copy() for p in params], np.full(b - a, -5.0, np.float32)]
            for a, b in wins]
    adam = B.AdamConfig(**w.adam_kwargs())
    oadam = oracle.make_adam(**asdict(adam))
    order = list(reversed(range(L.n_buckets)))
    for t in (1, 2):
        grads = W.make_grads(w, N, t, DEV)
        _run_buckets(L, adam, t, grads, [master, m, v], params, order, 2, True, mg)
        for (a, b), hs in zip(wins, host):
            oracle.step(list(w.sizes), list(w.wd_mask), w.D, w.bucket_elems, w.pad_unit, oadam,
                        t, [t2np_bf16(g[a:b]) for g in grads], hs[0], hs[1], hs[2], hs[3],
                        main_grad_out=hs[4], window=(a, b))
        del grads
    torch.cuda.synchronize()
    not_exact = 0
    for (a, b), hs in zip(wins, host):
        not_exact += _compare([x[a:b] for x in (master, m, v)], [p[a:b] for p in params],
                              mg[a:b], hs[:3], hs[3], hs[4])
    assert not_exact == 0
    assert sum(b - a for a, b in wins) > 300_000
