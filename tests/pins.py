"""Pins for the CPU oracle: checks against facts fixed by the pages and by
mathematics, not against the oracle itself.

Every pin takes the oracle's ctypes library as an argument, so the same pins
run against the real oracle (tests/test_oracle_pins.py) and against copies of
it with a mistake planted in the source (tests/test_oracle_mutants.py), which
must each fail at least one pin.

Sources: the Megatron-LM distributed-optimizer page ("04 · 分布式优化器", §3
ownership demo, §4.1 ranges, §4.2-§4.4 step, §5 scaling before the
communication) and the distributed-training tutorial ("AllReduce" worked
example; ring all-reduce = reduce-scatter then all-gather; ZeRO-1 changes
only where the optimizer state lives).
"""
from __future__ import annotations

import json
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16_bits_of(values):
    """bf16 bits of values that are exactly representable in bf16."""
    f = np.asarray(values, dtype=np.float32)
    bits = f.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (bits >> 16).astype(np.uint16)


def _bits_to_f32(h):
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _state(numel, seed, m_scale=0.0, v_scale=0.0):
    rng = np.random.default_rng(seed)
    master = rng.normal(0, 0.02, numel).astype(np.float32)
    m = (rng.normal(0, m_scale, numel) if m_scale else np.zeros(numel)).astype(np.float32)
    v = (np.abs(rng.normal(0, v_scale, numel)) if v_scale else np.zeros(numel)).astype(np.float32)
    return master, m, v


def _params_from(master, D):
    bits = master.view(np.uint32)
    # truncation is fine for an initial value: any bf16 pattern is a valid start
    p = (bits >> 16).astype(np.uint16)
    return [p.copy() for _ in range(D)]


# ---------------------------------------------------------------------------
# Layout and range-map pins
# ---------------------------------------------------------------------------

def pin_page1_ownership(lib):
    """Page 1 §3: 1000 elements, DP 4, shard 250, rank 1 owns [250, 500);
    pieces per the four-range definitions of §4.1 (hand-derived fixture)."""
    g = _golden("page1_ownership.json")
    L = oracle.range_map(g["param_sizes"], g["dp_size"], 0, 1, lib=lib)
    assert L.numel == g["buffer_elems"]
    assert L.n_buckets == 1
    assert (int(L.bucket_start[0]), int(L.bucket_end[0])) == (0, 1000)
    shard = (L.bucket_end[0] - L.bucket_start[0]) // g["dp_size"]
    assert shard == g["shard"]
    assert [list(r) for r in zip(L.param_start.tolist(), L.param_end.tolist())] == g["param_ranges"]
    got = [{k: (list(v) if isinstance(v, tuple) else v) for k, v in pc.items()
            if k in ("rank", "param_id", "gbuf_world", "gbuf_world_in_bucket", "gbuf_local", "param")}
           for pc in L.pieces]
    assert got == g["pieces"], got
    # rank 1's pieces exactly cover its range [250, 500)
    r1 = [pc for pc in L.pieces if pc["rank"] == 1]
    assert r1[0]["gbuf_world"][0] == 250 and r1[-1]["gbuf_world"][1] == 500


def check_layout_invariants(L, sizes, D, bucket_elems, pad_unit):
    """The greedy bucket rule with padding, stated as properties that fix the
    layout uniquely (params in order and contiguous inside a bucket, each
    bucket a minimal multiple of D*pad_unit, closed as soon as it reaches
    bucket_elems, params never split across buckets)."""
    n = len(sizes)
    unit = D * pad_unit
    if n == 0:
        assert L.numel == 0 and L.n_buckets == 0 and not L.pieces
        return
    assert L.n_buckets >= 1
    assert L.bucket_start[0] == 0
    for k in range(L.n_buckets - 1):
        assert L.bucket_end[k] == L.bucket_start[k + 1]
    assert L.bucket_end[-1] == L.numel
    pb = L.param_bucket.tolist()
    assert pb[0] == 0 and all(b - a in (0, 1) for a, b in zip(pb, pb[1:]))
    assert pb[-1] == L.n_buckets - 1
    for k in range(L.n_buckets):
        members = [p for p in range(n) if pb[p] == k]
        assert members, "empty bucket"
        assert L.param_start[members[0]] == L.bucket_start[k]
        for a, b in zip(members, members[1:]):
            assert L.param_end[a] == L.param_start[b]
        for p in members:
            assert L.param_end[p] - L.param_start[p] == sizes[p]
        unpadded = sum(sizes[p] for p in members)
        size = L.bucket_end[k] - L.bucket_start[k]
        assert size % unit == 0 and 0 <= size - unpadded < unit
        if bucket_elems == 0:
            assert L.n_buckets == 1
        else:
            assert unpadded - sizes[members[-1]] < bucket_elems
            if k < L.n_buckets - 1:
                assert unpadded >= bucket_elems


def brute_force_pieces(L, D):
    """Element-by-element enumeration of ownership: for every buffer element
    find its bucket, its rank (by the equal split of §4.1) and its param, and
    group the elements of each (bucket, rank, param) into one piece."""
    groups = {}
    owners = {}
    for p in range(len(L.param_start)):
        for i in range(int(L.param_start[p]), int(L.param_end[p])):
            owners[i] = p
    for k in range(L.n_buckets):
        bs, be = int(L.bucket_start[k]), int(L.bucket_end[k])
        S = (be - bs) // D
        for i in range(bs, be):
            r = (i - bs) // S
            p = owners.get(i)
            if p is None:
                continue
            lo = bs + r * S
            rec = groups.setdefault((k, r, p), [])
            rec.append((i, i - bs, i - lo, i - int(L.param_start[p])))
    out = []
    for (k, r, p) in sorted(groups, key=lambda key: (key[0], key[1], groups[key][0][0])):
        els = groups[(k, r, p)]
        cols = list(zip(*els))
        for c in cols:  # each coordinate runs over consecutive integers
            assert list(c) == list(range(c[0], c[0] + len(c)))
        out.append({"gbuf_world": (cols[0][0], cols[0][-1] + 1),
                    "gbuf_world_in_bucket": (cols[1][0], cols[1][-1] + 1),
                    "gbuf_local": (cols[2][0], cols[2][-1] + 1),
                    "param": (cols[3][0], cols[3][-1] + 1),
                    "param_id": p, "bucket_id": k, "rank": r})
    return out


def random_tiny_layouts(count, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(count):
        n = int(rng.integers(0, 9))
        sizes = [int(x) for x in rng.integers(0, 21, n)]
        D = int(rng.integers(1, 9))
        bucket = int(rng.choice([0, int(rng.integers(1, 65))]))
        pad = int(rng.integers(1, 5))
        cases.append((sizes, D, bucket, pad))
    return cases


def pin_brute_force_range_maps(lib, count=300, seed=11):
    """Brute force on tiny layouts: the interval arithmetic of the range map
    equals element-by-element ownership, and the layout obeys the greedy
    bucket rule."""
    for sizes, D, bucket, pad in random_tiny_layouts(count, seed):
        L = oracle.range_map(sizes, D, bucket, pad, lib=lib)
        check_layout_invariants(L, sizes, D, bucket, pad)
        assert L.pieces == brute_force_pieces(L, D), (sizes, D, bucket, pad)


def pin_error_paths(lib):
    """Invalid layouts are refused."""
    assert oracle.range_map_rc([4, 4], 0, 0, 1, lib=lib) == oracle.ORC_E_ARG
    assert oracle.range_map_rc([4, -1], 2, 0, 1, lib=lib) == oracle.ORC_E_ARG
    assert oracle.range_map_rc([4, 4], 2, 0, 0, lib=lib) == oracle.ORC_E_ARG
    assert oracle.range_map_rc([4, 4], 2, -5, 1, lib=lib) == oracle.ORC_E_ARG


# ---------------------------------------------------------------------------
# Reduce-scatter pins
# ---------------------------------------------------------------------------

def _run_step(lib, sizes, wd, D, bucket, pad, adam, grads_per_step, master, m, v, params,
              gather=True, main_grad_out=None, t0=1):
    for i, grads in enumerate(grads_per_step):
        oracle.step(sizes, wd, D, bucket, pad, adam, t0 + i, grads, master, m, v, params,
                    gather=gather, main_grad_out=main_grad_out, lib=lib)


def pin_allreduce_example(lib):
    """Tutorial "AllReduce": [1,2], [2,3], [3,3] -> [6,8].  With D=3 and one
    2-element param the bucket pads to 3 (S=1): rank 0 keeps [6], rank 1
    keeps [8], rank 2 owns only padding; the concatenated shards equal the
    all-reduce."""
    g = _golden("allreduce_example.json")
    D = len(g["ranks_in"])
    L = oracle.range_map([2], D, 0, 1, lib=lib)
    assert L.numel == 3
    assert [(pc["rank"], pc["gbuf_world"]) for pc in L.pieces] == [(0, (0, 1)), (1, (1, 2))]
    for dtype in ("bf16", "fp32"):
        pad_val = 0.0
        vals = [np.array(list(r) + [pad_val], np.float32) for r in g["ranks_in"]]
        grads = [(_bf16_bits_of(x) if dtype == "bf16" else x.copy()) for x in vals]
        master, m, v = _state(3, 0)
        params = _params_from(master, D)
        out = np.full(3, -7.0, np.float32)
        oracle.step([2], None, D, 0, 1, oracle.make_adam(grad_scale=1.0), 1, grads, master, m, v,
                    params, main_grad_out=out, lib=lib)
        assert out[:2].tolist() == [float(x) for x in g["every_rank_out"]], out
        assert out[2] == -7.0  # padding untouched


def pin_rs_concat_equals_allreduce(lib, cases=40, seed=5):
    """Ring all-reduce is reduce-scatter followed by all-gather: the
    concatenation of every rank's reduced shard equals the element-wise sum
    over all replicas (inputs are small integers times powers of two, so
    every fp32 sum is exact and order-free)."""
    rng = np.random.default_rng(seed)
    for sizes, D, bucket, pad in random_tiny_layouts(cases, seed):
        if not sizes:
            continue
        L = oracle.range_map(sizes, D, bucket, pad, lib=lib)
        N = L.numel
        s = 0.5 if D % 2 else 1.0 / (1 << int(rng.integers(0, 3)))
        ints = [rng.integers(-64, 65, N) for _ in range(D)]
        grads = [_bf16_bits_of(x.astype(np.float32) / 8) for x in ints]
        master, m, v = _state(N, 1)
        params = _params_from(master, D)
        out = np.full(N, np.float32(12345.0), np.float32)
        oracle.step(sizes, None, D, bucket, pad, oracle.make_adam(grad_scale=s), 1, grads, master,
                    m, v, params, main_grad_out=out, lib=lib)
        want = s * (np.sum(np.stack(ints), axis=0).astype(np.float64) / 8)
        owned = np.zeros(N, bool)
        for p in range(len(sizes)):
            owned[L.param_start[p]:L.param_end[p]] = True
        assert np.array_equal(out[owned].astype(np.float64), want[owned]), (sizes, D)
        assert np.all(out[~owned] == np.float32(12345.0))


def pin_rank_order_accumulation(lib):
    """fp32 accumulation in rank order: 1 + 2^24 rounds to 2^24 (a tie, to
    even), then - 2^24 gives 0; any other order gives 1."""
    D = 3
    grads = [np.array([1.0, 0, 0], np.float32), np.array([2.0 ** 24, 0, 0], np.float32),
             np.array([-(2.0 ** 24), 0, 0], np.float32)]
    master, m, v = _state(3, 2)
    params = _params_from(master, D)
    out = np.full(3, 99.0, np.float32)
    oracle.step([1], None, D, 0, 1, oracle.make_adam(grad_scale=1.0), 1, grads, master, m, v,
                params, main_grad_out=out, lib=lib)
    assert out[0] == 0.0, out


def pin_scale_before_reduce(lib):
    """Page 1 §5: the scaling factor multiplies the grads before the
    communication.  1.5*2^127 + 1.5*2^127 overflows fp32, but with a factor
    of 1/2 applied first the sum is the finite 1.5*2^127."""
    big = np.float32(1.5 * 2.0 ** 127)
    D = 2
    grads = [np.array([big, 0], np.float32), np.array([big, 0], np.float32)]
    master, m, v = _state(2, 3)
    params = _params_from(master, D)
    out = np.zeros(2, np.float32)
    oracle.step([1], None, D, 0, 1, oracle.make_adam(grad_scale=0.5), 1, grads, master, m, v,
                params, main_grad_out=out, lib=lib)
    assert out[0] == big, out


# ---------------------------------------------------------------------------
# Adam pins
# ---------------------------------------------------------------------------

def _f32(x):
    return float(np.float32(x))


def pin_d1_is_adamw(lib, steps=5):
    """With D=1 and no scaling the step is plain AdamW (the tutorial's ZeRO-1
    only moves where the optimizer state lives).  Compared with PyTorch's
    AdamW run in float64 on the same bf16 gradients, with a weight-decay
    mask done as two param groups."""
    import torch

    sizes = [37, 100, 5, 64, 19]
    wd_mask = [1, 0, 1, 0, 1]
    n = sum(sizes)
    adam_f = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    master, m, v = _state(n, 4, m_scale=1e-4, v_scale=1e-6)
    params = _params_from(master, 1)
    rng = np.random.default_rng(9)
    grads_steps = []
    for _ in range(steps):
        g = rng.normal(0, 1e-3, n)
        g[::7] = rng.normal(0, 1.0, len(g[::7]))       # large
        g[3::11] = rng.normal(0, 1e-9, len(g[3::11]))  # below eps: eps matters
        g[5::13] = 0.0
        bits = (g.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        grads_steps.append([bits])

    t_params, groups = [], {0: [], 1: []}
    off = 0
    for size, w in zip(sizes, wd_mask):
        p = torch.tensor(master[off:off + size].astype(np.float64), requires_grad=True)
        t_params.append((p, off, size))
        groups[w].append(p)
        off += size
    opt = torch.optim.AdamW(
        [{"params": groups[1], "weight_decay": _f32(adam_f["weight_decay"])},
         {"params": groups[0], "weight_decay": 0.0}],
        lr=_f32(adam_f["lr"]), betas=(_f32(adam_f["beta1"]), _f32(adam_f["beta2"])),
        eps=_f32(adam_f["eps"]), foreach=False)
    for p, o, size in t_params:
        opt.state[p] = {"step": torch.tensor(0.0),
                        "exp_avg": torch.tensor(m[o:o + size].astype(np.float64)),
                        "exp_avg_sq": torch.tensor(v[o:o + size].astype(np.float64))}

    adam = oracle.make_adam(grad_scale=1.0, **adam_f)
    # fp32 rounding bound for m: b1*m and (1-b1)*g can cancel, so the error
    # scales with the magnitudes of the terms summed so far, not with |m|.
    u = 2.0 ** -24
    b1 = _f32(adam_f["beta1"])
    mag_m = np.abs(m.astype(np.float64))
    for t, grads in enumerate(grads_steps, start=1):
        oracle.step(sizes, wd_mask, 1, 0, 1, adam, t, grads, master, m, v, params, lib=lib)
        gf = _bits_to_f32(grads[0]).astype(np.float64)
        for p, o, size in t_params:
            p.grad = torch.tensor(gf[o:o + size])
        opt.step()
        mag_m = b1 * mag_m + (1 - b1) * np.abs(gf)

    ref_w = np.concatenate([p.detach().numpy() for p, _, _ in t_params])
    ref_m = np.concatenate([opt.state[p]["exp_avg"].numpy() for p, _, _ in t_params])
    ref_v = np.concatenate([opt.state[p]["exp_avg_sq"].numpy() for p, _, _ in t_params])
    np.testing.assert_allclose(master, ref_w, rtol=2e-6, atol=1e-9)
    assert np.all(np.abs(m - ref_m) <= 2e-6 * np.abs(ref_m) + 8 * u * steps * mag_m)
    np.testing.assert_allclose(v, ref_v, rtol=2e-6, atol=1e-18)
    # the bf16 params are the round-to-nearest-even of the fp32 master
    want_p = torch.tensor(master).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(params[0], want_p)


def _d_independent_run(lib, D, sizes, wd, pad, bucket, G, K, steps):
    L = oracle.range_map(sizes, D, bucket, pad, lib=lib)
    N = L.numel
    n = sum(sizes)
    # buffer-indexed copies of the per-param initial state
    master0, m0, v0 = _state(n, 21, m_scale=1e-4, v_scale=1e-6)
    master = np.zeros(N, np.float32)
    m = np.zeros(N, np.float32)
    v = np.zeros(N, np.float32)
    off = 0
    for p, size in enumerate(sizes):
        s0, s1 = int(L.param_start[p]), int(L.param_end[p])
        master[s0:s1] = master0[off:off + size]
        m[s0:s1] = m0[off:off + size]
        v[s0:s1] = v0[off:off + size]
        off += size
    params = _params_from(master, D)
    adam = oracle.make_adam(grad_scale=1.0 / D)
    for t in range(1, steps + 1):
        grads = []
        for r in range(D):
            g = np.zeros(N, np.float32)
            off = 0
            for p, size in enumerate(sizes):
                s0 = int(L.param_start[p])
                g[s0:s0 + size] = (G[t - 1][off:off + size] + (2 * r - (D - 1)) * K) / 1024.0
                off += size
            grads.append(_bf16_bits_of(g))
        oracle.step(sizes, wd, D, bucket, pad, adam, t, grads, master, m, v, params, lib=lib)
    per_param = []
    for p in range(len(sizes)):
        s0, s1 = int(L.param_start[p]), int(L.param_end[p])
        per_param.append((master[s0:s1].copy(), m[s0:s1].copy(), v[s0:s1].copy(),
                          params[0][s0:s1].copy(), [x[s0:s1].copy() for x in params]))
    return per_param


def pin_d_independence(lib, steps=3):
    """Params are independent of D for integer-valued grads: with
    g_r = (G + (2r - D + 1) K) / 1024 and scaling 1/D, every fp32 partial sum
    is exact and the reduced grad is G/1024 for every D in {1,2,4,8,16}, so
    master, m, v and all D bf16 replicas must be bitwise the same."""
    rng = np.random.default_rng(17)
    sizes = [33, 7, 129, 64, 1, 90]
    wd = [1, 0, 1, 1, 0, 1]
    n = sum(sizes)
    G = [rng.integers(-64, 65, n).astype(np.float32) for _ in range(steps)]
    base = None
    for D, pad, bucket in ((1, 1, 0), (2, 3, 100), (4, 1, 50), (8, 2, 0), (16, 1, 64)):
        res = _d_independent_run(lib, D, sizes, wd, pad, bucket, G, K=2, steps=steps)
        for p in range(len(sizes)):
            for rep in res[p][4]:
                assert np.array_equal(rep, res[p][3]), (D, p)
        if base is None:
            base = res
            continue
        for p in range(len(sizes)):
            for a, b in zip(res[p][:4], base[p][:4]):
                assert np.array_equal(a.view(np.uint32) if a.dtype == np.float32 else a,
                                      b.view(np.uint32) if b.dtype == np.float32 else b), (D, p)


def pin_bf16_rounding(lib):
    """fp32 -> bf16 is round-to-nearest-even (checked against PyTorch's own
    conversion on ties, carries into the exponent, overflow, subnormals,
    infinities and NaN)."""
    import torch

    specials = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 3.4028235e38, -3.4028235e38,
                         1e-40, -1e-40, 1.17549435e-38, 65504.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8,
                         1.0 + 2 ** -8 + 2 ** -20, 1.0 - 2 ** -9, 255.5, 256.5],
                        np.float32)
    ties = ((np.arange(0, 64, dtype=np.uint32) << 16) | 0x3F808000).view(np.float32)
    rng = np.random.default_rng(3)
    rnd = rng.integers(0, 2 ** 32, 4000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    rnd = rnd[np.isfinite(rnd)]
    x = np.concatenate([specials, ties, rnd]).astype(np.float32)
    got = oracle.f32_to_bf16(x, lib=lib)
    want = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    nan = oracle.f32_to_bf16(np.array([np.nan], np.float32), lib=lib)[0]
    assert (nan & 0x7F80) == 0x7F80 and (nan & 0x7F) != 0 and (nan & 0x40)
    back = oracle.bf16_to_f32(want, lib=lib)
    assert np.array_equal(back.view(np.uint32), want.astype(np.uint32) << 16)


# ---------------------------------------------------------------------------
# Step structure pins
# ---------------------------------------------------------------------------

def pin_gather_and_padding(lib):
    """All-gather (distributed-optimizer page, §4.4): with the gather every replica holds the new
    params; without it only the owning rank's replica changes on its range.
    Padding is never written."""
    sizes = [10, 27, 3]
    D, pad = 4, 3
    L = oracle.range_map(sizes, D, 0, pad, lib=lib)
    N = L.numel
    owned = np.zeros(N, bool)
    for p in range(len(sizes)):
        owned[L.param_start[p]:L.param_end[p]] = True
    assert N == 48 and owned.sum() == 40
    rng = np.random.default_rng(1)
    grads = [_bf16_bits_of(rng.integers(-8, 9, N).astype(np.float32)) for _ in range(D)]
    for gather in (True, False):
        master, m, v = _state(N, 6)
        params = [(np.arange(N, dtype=np.uint16) * 7 + r) for r in range(D)]
        before = [p.copy() for p in params]
        mb, mmb, vb = master.copy(), m.copy(), v.copy()
        oracle.step(sizes, None, D, 0, pad, oracle.make_adam(grad_scale=0.25), 1, grads, master,
                    m, v, params, gather=gather, lib=lib)
        want = oracle.f32_to_bf16(master, lib=lib)
        for arr, arr0 in ((master, mb), (m, mmb), (v, vb)):
            assert np.array_equal(arr[~owned].view(np.uint32), arr0[~owned].view(np.uint32))
            assert not np.array_equal(arr[owned], arr0[owned])
        S = N // D
        for r in range(D):
            assert np.array_equal(params[r][~owned], before[r][~owned])
            mine = np.zeros(N, bool)
            mine[r * S:(r + 1) * S] = True
            if gather:
                assert np.array_equal(params[r][owned], want[owned])
            else:
                assert np.array_equal(params[r][owned & mine], want[owned & mine])
                assert np.array_equal(params[r][owned & ~mine], before[r][owned & ~mine])


def pin_window_equals_full(lib):
    """Elements are independent: a window of the buffer stepped alone gives
    the same values as the full step."""
    sizes = [100, 250, 77, 300]
    wd = [1, 0, 1, 0]
    D, pad, bucket = 4, 2, 200
    L = oracle.range_map(sizes, D, bucket, pad, lib=lib)
    N = L.numel
    rng = np.random.default_rng(8)
    grads = [_bf16_bits_of((rng.integers(-100, 100, N) / 64).astype(np.float32)) for _ in range(D)]
    master, m, v = _state(N, 10, 1e-4, 1e-6)
    params = _params_from(master, D)
    full = [master.copy(), m.copy(), v.copy(), [p.copy() for p in params]]
    oracle.step(sizes, wd, D, bucket, pad, oracle.make_adam(grad_scale=0.25), 2, grads, full[0],
                full[1], full[2], full[3], lib=lib)
    for w0, w1 in ((0, N), (13, 411), (200, 208), (N - 5, N)):
        sub = [master[w0:w1].copy(), m[w0:w1].copy(), v[w0:w1].copy(),
               [p[w0:w1].copy() for p in params]]
        oracle.step(sizes, wd, D, bucket, pad, oracle.make_adam(grad_scale=0.25), 2,
                    [g[w0:w1].copy() for g in grads], sub[0], sub[1], sub[2], sub[3],
                    window=(w0, w1), lib=lib)
        for a, b in zip(sub[:3], full[:3]):
            assert np.array_equal(a.view(np.uint32), b[w0:w1].view(np.uint32))
        for a, b in zip(sub[3], full[3]):
            assert np.array_equal(a, b[w0:w1])


# ---------------------------------------------------------------------------
# Global-norm clipping pins (tutorial §8.3)
# ---------------------------------------------------------------------------

def pin_clip_norm_closed_form(lib):
    """norm^2 of four reduced grads of 1.5 (D=2, two halves of 0.75) is 9;
    with max_norm at least the norm the coefficient is exactly 1."""
    D = 2
    grads = [_bf16_bits_of(np.array([0.75] * 4, np.float32)) for _ in range(D)]
    nsq = oracle.grad_norm_sq([4], D, 0, 1, 1.0, grads, lib=lib)
    assert nsq == 9.0, nsq
    assert oracle.clip_coef(nsq, 3.5, lib=lib) == 1.0
    assert oracle.clip_coef(nsq, 1e9, lib=lib) == 1.0
    assert 0.0 < oracle.clip_coef(nsq, 1.5, lib=lib) < 0.5
    # padding is not part of the norm
    grads_p = [_bf16_bits_of(np.array([0.75] * 4 + [100.0] * 2, np.float32)) for _ in range(D)]
    assert oracle.grad_norm_sq([4], D, 0, 3, 1.0, grads_p, lib=lib) == 9.0


def _clip_vs_torch(lib, grad_std, steps=3, seed=13):
    import torch

    sizes = [50, 13, 200, 7]
    wd_mask = [1, 0, 1, 1]
    n = sum(sizes)
    adam_f = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    master, m, v = _state(n, seed, m_scale=1e-4, v_scale=1e-6)
    params = _params_from(master, 1)
    rng = np.random.default_rng(seed)
    t_params, groups = [], {0: [], 1: []}
    off = 0
    for size, w in zip(sizes, wd_mask):
        p = torch.tensor(master[off:off + size].astype(np.float64), requires_grad=True)
        t_params.append((p, off, size))
        groups[w].append(p)
        off += size
    opt = torch.optim.AdamW(
        [{"params": groups[1], "weight_decay": _f32(adam_f["weight_decay"])},
         {"params": groups[0], "weight_decay": 0.0}],
        lr=_f32(adam_f["lr"]), betas=(_f32(adam_f["beta1"]), _f32(adam_f["beta2"])),
        eps=_f32(adam_f["eps"]), foreach=False)
    for p, o, size in t_params:
        opt.state[p] = {"step": torch.tensor(0.0),
                        "exp_avg": torch.tensor(m[o:o + size].astype(np.float64)),
                        "exp_avg_sq": torch.tensor(v[o:o + size].astype(np.float64))}
    adam = oracle.make_adam(grad_scale=1.0, **adam_f)
    u = 2.0 ** -24
    b1 = _f32(adam_f["beta1"])
    mag_m = np.abs(m.astype(np.float64))
    for t in range(1, steps + 1):
        g = rng.normal(0, grad_std, n).astype(np.float32)
        bits = (g.view(np.uint32) >> 16).astype(np.uint16)
        gf = _bits_to_f32(bits).astype(np.float64)
        max_norm = 0.5 * float(np.sqrt(np.sum(gf * gf)))
        nsq = oracle.grad_norm_sq(sizes, 1, 0, 1, 1.0, [bits], lib=lib)
        coef = oracle.clip_coef(nsq, max_norm, lib=lib)
        oracle.step(sizes, wd_mask, 1, 0, 1, adam, t, [bits], master, m, v, params,
                    clip_coef=coef, lib=lib)
        for p, o, size in t_params:
            p.grad = torch.tensor(gf[o:o + size])
        total = torch.nn.utils.clip_grad_norm_([p for p, _, _ in t_params], max_norm)
        assert abs(np.sqrt(nsq) - float(total)) <= 1e-12 * float(total)
        opt.step()
        gclip = np.concatenate([p.grad.numpy() for p, _, _ in t_params])
        mag_m = b1 * mag_m + (1 - b1) * np.abs(gclip)
    ref_w = np.concatenate([p.detach().numpy() for p, _, _ in t_params])
    ref_m = np.concatenate([opt.state[p]["exp_avg"].numpy() for p, _, _ in t_params])
    ref_v = np.concatenate([opt.state[p]["exp_avg_sq"].numpy() for p, _, _ in t_params])
    np.testing.assert_allclose(master, ref_w, rtol=2e-6, atol=1e-9)
    assert np.all(np.abs(m - ref_m) <= 2e-6 * np.abs(ref_m) + 8 * u * steps * mag_m)
    np.testing.assert_allclose(v, ref_v, rtol=4e-6, atol=1e-20)


def pin_clip_d1_matches_torch(lib):
    """D=1 with clipping equals PyTorch's clip_grad_norm_ followed by AdamW
    (float64), for a large norm and for a norm small enough that the 1e-6
    in the coefficient's denominator matters."""
    _clip_vs_torch(lib, grad_std=1.0, seed=13)
    _clip_vs_torch(lib, grad_std=1e-5, seed=14)


def pin_clip_off_equals_plain_step(lib):
    """A coefficient of 1 (norm below max_norm) leaves the step bitwise equal
    to the step without clipping."""
    sizes, wd = [100, 27, 300], [1, 0, 1]
    D, pad = 4, 2
    L = oracle.range_map(sizes, D, 0, pad, lib=lib)
    N = L.numel
    rng = np.random.default_rng(2)
    grads = [_bf16_bits_of((rng.integers(-50, 50, N) / 256).astype(np.float32)) for _ in range(D)]
    nsq = oracle.grad_norm_sq(sizes, D, 0, pad, 0.25, grads, lib=lib)
    coef = oracle.clip_coef(nsq, 2.0 * float(np.sqrt(nsq)) + 1.0, lib=lib)
    assert coef == 1.0
    a = list(_state(N, 3, 1e-4, 1e-6)) + [_params_from(_state(N, 3)[0], D)]
    b = [x.copy() for x in a[:3]] + [[p.copy() for p in a[3]]]
    adam = oracle.make_adam(grad_scale=0.25)
    oracle.step(sizes, wd, D, 0, pad, adam, 1, grads, a[0], a[1], a[2], a[3], lib=lib)
    oracle.step(sizes, wd, D, 0, pad, adam, 1, grads, b[0], b[1], b[2], b[3], clip_coef=coef,
                lib=lib)
    for x, y in zip(a[:3], b[:3]):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))


def pin_clip_d_independence(lib):
    """With clipping engaged, integer-valued grads still give results that
    are bitwise independent of D: the reduced grads are the same, their
    squares are exact in double and so is their sum, in any order."""
    rng = np.random.default_rng(23)
    sizes = [33, 7, 129, 64]
    wd = [1, 0, 1, 1]
    n = sum(sizes)
    G = rng.integers(-64, 65, n).astype(np.float32)
    base = None
    for D, pad in ((1, 1), (2, 3), (4, 1), (8, 2), (16, 1)):
        L = oracle.range_map(sizes, D, 0, pad, lib=lib)
        N = L.numel
        master, m, v = np.zeros(N, np.float32), np.zeros(N, np.float32), np.zeros(N, np.float32)
        m0, _, _ = _state(n, 31)
        grads = []
        for r in range(D):
            g = np.zeros(N, np.float32)
            off = 0
            for p, size in enumerate(sizes):
                s0 = int(L.param_start[p])
                g[s0:s0 + size] = (G[off:off + size] + (2 * r - (D - 1)) * 2) / 1024.0
                master[s0:s0 + size] = m0[off:off + size]
                off += size
            grads.append(_bf16_bits_of(g))
        params = _params_from(master, D)
        nsq = oracle.grad_norm_sq(sizes, D, 0, pad, 1.0 / D, grads, lib=lib)
        coef = oracle.clip_coef(nsq, 0.25 * float(np.sqrt(nsq)), lib=lib)
        assert coef < 1.0
        oracle.step(sizes, wd, D, 0, pad, oracle.make_adam(grad_scale=1.0 / D), 1, grads, master,
                    m, v, params, clip_coef=coef, lib=lib)
        res = [(master[int(L.param_start[p]):int(L.param_end[p])].copy(),
                m[int(L.param_start[p]):int(L.param_end[p])].copy()) for p in range(len(sizes))]
        if base is None:
            base = (nsq, coef, res)
            continue
        assert nsq == base[0] and coef == base[1], D
        for (a, b), (c, d) in zip(res, base[2]):
            assert np.array_equal(a.view(np.uint32), c.view(np.uint32))
            assert np.array_equal(b.view(np.uint32), d.view(np.uint32))


# ---------------------------------------------------------------------------
# All-reduce pins (distributed-optimizer page, §5 force_all_reduce; tutorial "AllReduce")
# ---------------------------------------------------------------------------

def pin_allreduce_every_rank(lib):
    """Tutorial "AllReduce": [1,2], [2,3], [3,3] -> [6,8] on every rank, in
    bf16 and in fp32 grad buffers; padding untouched."""
    g = _golden("allreduce_example.json")
    D = len(g["ranks_in"])
    for dtype in ("bf16", "fp32"):
        vals = [np.array(list(r) + [-2.0], np.float32) for r in g["ranks_in"]]
        grads = [(_bf16_bits_of(x) if dtype == "bf16" else x.copy()) for x in vals]
        oracle.allreduce([2], D, 0, 1, 1.0, grads, lib=lib)
        for x in grads:
            f = _bits_to_f32(x) if dtype == "bf16" else x
            assert f[:2].tolist() == [float(v) for v in g["every_rank_out"]], f
            assert f[2] == -2.0


def pin_allreduce_is_rs_then_gather(lib, cases=30, seed=41):
    """All-reduce equals the concatenated reduce-scatter shards copied to
    every rank: each replica's buffer becomes the main grads the step
    reports (exact integer inputs), and the step is unchanged by it."""
    rng = np.random.default_rng(seed)
    for sizes, D, bucket, pad in random_tiny_layouts(cases, seed):
        if not sizes or sum(sizes) == 0:
            continue
        L = oracle.range_map(sizes, D, bucket, pad, lib=lib)
        N = L.numel
        ints = [rng.integers(-30, 31, N) for _ in range(D)]
        grads = [_bf16_bits_of(x.astype(np.float32) / 4) for x in ints]
        before = [x.copy() for x in grads]
        master, m, v = _state(N, 5)
        params = _params_from(master, D)
        mg = np.full(N, 7.0, np.float32)
        oracle.step(sizes, None, D, bucket, pad, oracle.make_adam(grad_scale=0.5), 1, grads,
                    master, m, v, params, main_grad_out=mg, lib=lib)
        oracle.allreduce(sizes, D, bucket, pad, 0.5, grads, lib=lib)
        owned = np.zeros(N, bool)
        for p in range(len(sizes)):
            owned[L.param_start[p]:L.param_end[p]] = True
        for x, x0 in zip(grads, before):
            assert np.array_equal(_bits_to_f32(x)[owned], mg[owned])
            assert np.array_equal(x[~owned], x0[~owned])


def pin_allreduce_rounds_to_nearest_even(lib):
    """The all-reduced bf16 buffer is the round-to-nearest-even of the fp32
    reduced grads (PyTorch's conversion of the step's main grads), with sums
    that need rounding."""
    import torch

    rng = np.random.default_rng(8)
    sizes, D, pad = [500, 333], 3, 1
    L = oracle.range_map(sizes, D, 0, pad, lib=lib)
    N = L.numel
    grads = [(rng.normal(0, 1, N).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
             for _ in range(D)]
    master, m, v = _state(N, 9)
    mg = np.zeros(N, np.float32)
    oracle.step(sizes, None, D, 0, pad, oracle.make_adam(grad_scale=1.0), 1, grads, master, m, v,
                _params_from(master, D), main_grad_out=mg, lib=lib)
    oracle.allreduce(sizes, D, 0, pad, 1.0, grads, lib=lib)
    want = torch.tensor(mg).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    n = sum(sizes)  # one bucket: the owned elements come first, then padding
    assert np.count_nonzero(_bits_to_f32(want[:n]) != mg[:n]) > n // 4  # rounding happens
    for x in grads:
        assert np.array_equal(x[:n], want[:n])


# ---------------------------------------------------------------------------
# Optimizer instances (distributed-optimizer page, §5, num_distributed_optimizer_instances > 1)
# ---------------------------------------------------------------------------

def pin_instances_hierarchical_order(lib):
    """Page 1 §5: with several optimizer instances the reduce-scatter stays
    inside an instance and an all-reduce across instances follows.  D=4 in 2
    instances, fp32 grads 2^24, 1 | 1, -2^24 at one element: the instance
    sums are 2^24 (1 + 2^24 is a tie, to even) and 1 - 2^24, their sum is 1;
    one instance (the flat rank-order sum) gives 0."""
    vals = [2.0 ** 24, 1.0, 1.0, -(2.0 ** 24)]
    for instances, R, want in ((2, 2, 1.0), (1, 4, 0.0)):
        grads = [np.array([x] + [0.0] * (R - 1), np.float32) for x in vals]
        master, m, v = _state(R, 2)
        out = np.full(R, 99.0, np.float32)
        oracle.step([1], None, 4, 0, 1, oracle.make_adam(grad_scale=1.0), 1, grads, master, m,
                    v, _params_from(master, 4), main_grad_out=out, instances=instances, lib=lib)
        assert out[0] == want, (instances, out)
        assert oracle.grad_norm_sq([1], 4, 0, 1, 1.0, grads, instances=instances,
                                   lib=lib) == want * want


def pin_instances_factorizations(lib):
    """Integer-valued grads make every grouping exact: D=8 as 1, 2, 4 or 8
    instances gives bitwise the same master, m, v and params per param."""
    rng = np.random.default_rng(29)
    sizes = [33, 7, 129, 64, 1, 90]
    wd = [1, 0, 1, 1, 0, 1]
    n = sum(sizes)
    G = rng.integers(-64, 65, n).astype(np.float32)
    D = 8
    base = None
    for instances in (1, 2, 4, 8):
        R = D // instances
        L = oracle.range_map(sizes, R, 0, 1, lib=lib)
        N = L.numel
        m0, _, _ = _state(n, 31)
        master = np.zeros(N, np.float32)
        m = np.zeros(N, np.float32)
        v = np.zeros(N, np.float32)
        grads = []
        for r in range(D):
            g = np.zeros(N, np.float32)
            off = 0
            for p, size in enumerate(sizes):
                s0 = int(L.param_start[p])
                g[s0:s0 + size] = (G[off:off + size] + (2 * r - (D - 1)) * 2) / 1024.0
                master[s0:s0 + size] = m0[off:off + size]
                off += size
            grads.append(_bf16_bits_of(g))
        params = _params_from(master, D)
        oracle.step(sizes, wd, D, 0, 1, oracle.make_adam(grad_scale=1.0 / D), 1, grads, master,
                    m, v, params, instances=instances, lib=lib)
        res = []
        for p in range(len(sizes)):
            a, b = int(L.param_start[p]), int(L.param_end[p])
            res.append([master[a:b].view(np.uint32).copy(), m[a:b].view(np.uint32).copy(),
                        v[a:b].view(np.uint32).copy()] + [x[a:b].copy() for x in params])
        if base is None:
            base = res
            continue
        for x, y in zip(res, base):
            for a, b in zip(x, y):
                assert np.array_equal(a, b), instances


def pin_instances_write_back_and_gather(lib):
    """Without the gather only rank r of every instance holds the update of
    the elements rank r owns; the gather spreads it inside each instance."""
    sizes, D, instances = [37, 50], 6, 2
    R = D // instances
    L = oracle.range_map(sizes, R, 0, 1, lib=lib)
    N = L.numel
    rng = np.random.default_rng(4)
    grads = [_bf16_bits_of(rng.integers(-8, 9, N).astype(np.float32)) for _ in range(D)]
    for gather in (False, True):
        master, m, v = _state(N, 6)
        params = [(np.arange(N, dtype=np.uint16) * 3 + r) for r in range(D)]
        before = [p.copy() for p in params]
        oracle.step(sizes, None, D, 0, 1, oracle.make_adam(grad_scale=1.0 / D), 1, grads, master,
                    m, v, params, gather=gather, instances=instances, lib=lib)
        want = oracle.f32_to_bf16(master, lib=lib)
        S = N // R
        for rep in range(D):
            r = rep % R
            mine = np.zeros(N, bool)
            mine[r * S:(r + 1) * S] = True
            owned = np.zeros(N, bool)
            owned[:sum(sizes)] = True
            if gather:
                assert np.array_equal(params[rep][owned], want[owned])
            else:
                assert np.array_equal(params[rep][owned & mine], want[owned & mine])
                assert np.array_equal(params[rep][owned & ~mine], before[rep][owned & ~mine])


# ---------------------------------------------------------------------------
# Reduced grad rounded to the grad type (optional reading)
# ---------------------------------------------------------------------------

def pin_round_grad(lib):
    """With round_grad the reduced grads are rounded to the grad type: the
    reported main grads are PyTorch's bf16 rounding of the unrounded ones;
    the step equals a D=1 step fed those rounded values with scaling 1; the
    norm is the sum of their squares; fp32 grads are left as they are."""
    import torch

    sizes, wd, D, pad = [300, 41, 129], [1, 0, 1], 3, 2
    L = oracle.range_map(sizes, D, 0, pad, lib=lib)
    N = L.numel
    rng = np.random.default_rng(77)
    grads = [(rng.normal(0, 1, N).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
             for _ in range(D)]
    adam = oracle.make_adam(grad_scale=0.3)  # not a power of two: sums need rounding
    master0, m0, v0 = _state(N, 13, 1e-4, 1e-6)
    runs = {}
    for rg in (False, True):
        master, m, v = master0.copy(), m0.copy(), v0.copy()
        params = _params_from(master0, D)
        mg = np.zeros(N, np.float32)
        oracle.step(sizes, wd, D, 0, pad, adam, 1, grads, master, m, v, params, main_grad_out=mg,
                    round_grad=rg, lib=lib)
        runs[rg] = (master, m, v, params, mg)
    owned = np.zeros(N, bool)
    for p in range(len(sizes)):
        owned[L.param_start[p]:L.param_end[p]] = True
    want = torch.tensor(runs[False][4]).to(torch.bfloat16).float().numpy()
    assert np.array_equal(runs[True][4][owned], want[owned])
    assert np.count_nonzero(want[owned] != runs[False][4][owned]) > owned.sum() // 2
    # a D=1 step on the rounded values (exact in bf16, scaling 1) is the same step
    bits = (want.view(np.uint32) >> 16).astype(np.uint16)
    master, m, v = master0.copy(), m0.copy(), v0.copy()
    params = _params_from(master0, 1)
    L1 = oracle.range_map(sizes, 1, 0, 1, lib=lib)
    assert L1.numel == sum(sizes)
    idx = np.flatnonzero(owned)
    sub = [a[idx].copy() for a in (master, m, v)]
    oracle.step(sizes, wd, 1, 0, 1, oracle.make_adam(grad_scale=1.0), 1, [bits[idx].copy()],
                *sub, [params[0][idx].copy()], lib=lib)
    for a, b in zip(sub, runs[True][:3]):
        assert np.array_equal(a.view(np.uint32), b[idx].view(np.uint32))
    nsq = oracle.grad_norm_sq(sizes, D, 0, pad, 0.3, grads, round_grad=True, lib=lib)
    ref = float(np.sum(want[owned].astype(np.float64) ** 2))
    assert abs(nsq - ref) <= 1e-12 * ref
    # fp32 grads: the grad type is fp32, nothing to round
    g32 = [rng.normal(0, 1, N).astype(np.float32) for _ in range(D)]
    a = oracle.grad_norm_sq(sizes, D, 0, pad, 0.3, g32, lib=lib)
    b = oracle.grad_norm_sq(sizes, D, 0, pad, 0.3, g32, round_grad=True, lib=lib)
    assert a == b


def pin_nonfinite_count(lib):
    """Reading R13 of the oracle: the count is over owned elements of the
    reduced grad.  Closed cases: one Inf counts 1; +Inf and -Inf in two
    replicas (a NaN sum) count 1, not 2; NaN at padding counts 0; scaling
    comes first (distributed-optimizer page, §5), so 1.5*2^127 in two replicas counts 0 with a
    factor of 1/2 and 1 with a factor of 1; a reduced grad that is finite in
    fp32 but rounds to bf16 Inf (max bf16 + 2^119, a tie rounded to even)
    counts only with the rounding of R12; across two instances the
    instance sums Inf and -Inf give a NaN that counts 1.  Random layouts:
    the count equals the number of non-finite owned main grads a step
    reports."""
    sizes, D = [5, 6], 4  # 11 owned elements, padded to 12
    N = oracle.range_map(sizes, D, 0, 1, lib=lib).numel
    assert N == 12

    def f32(entries):
        g = [np.zeros(N, np.float32) for _ in range(D)]
        for r, i, x in entries:
            g[r][i] = x
        return g

    def count(g, scale=1.0, **kw):
        return oracle.count_nonfinite(sizes, D, 0, 1, scale, g, lib=lib, **kw)

    inf, nan = np.float32(np.inf), np.float32(np.nan)
    assert count(f32([])) == 0
    assert count(f32([(1, 3, inf)])) == 1
    assert count(f32([(0, 7, inf), (2, 7, -inf)])) == 1
    assert count(f32([(3, 11, nan)])) == 0
    assert count(f32([(3, 11, nan), (1, 10, nan), (0, 0, -inf)])) == 2
    big = np.float32(1.5 * 2.0 ** 127)
    assert count(f32([(0, 4, big), (1, 4, big)]), scale=0.5) == 0
    assert count(f32([(0, 4, big), (1, 4, big)]), scale=1.0) == 1
    # bf16 grads: max bf16 (0x7F7F) + 2^119 (0x7B00) is finite in fp32 and
    # a tie between max bf16 and Inf in bf16, which goes to the even Inf
    g = [np.zeros(N, np.uint16) for _ in range(D)]
    g[0][2], g[1][2] = 0x7F7F, 0x7B00
    assert count(g) == 0
    assert count(g, round_grad=True) == 1
    # two instances of two ranks: Inf + 0 | -Inf + 0 -> NaN
    gi = f32([(0, 5, inf), (3, 5, -inf)])
    assert oracle.count_nonfinite(sizes, D, 0, 1, 1.0, gi, instances=2, lib=lib) == 1
    # random layouts with scattered Inf/NaN, against the step's main grads
    rng = np.random.default_rng(17)
    for _ in range(20):
        n = int(rng.integers(1, 6))
        sz = [int(x) for x in rng.integers(0, 40, n)]
        Dr = int(rng.integers(1, 6))
        pad = int(rng.integers(1, 5))
        Nr = oracle.range_map(sz, Dr, 0, pad, lib=lib).numel
        if Nr == 0:
            continue
        gr = [rng.normal(0, 1, Nr).astype(np.float32) for _ in range(Dr)]
        for _ in range(int(rng.integers(0, 6))):
            gr[int(rng.integers(0, Dr))][int(rng.integers(0, Nr))] = rng.choice([inf, -inf, nan])
        master, m, v = _state(Nr, 3)
        params = _params_from(master, Dr)
        mg = np.zeros(Nr, np.float32)
        oracle.step(sz, None, Dr, 0, pad, oracle.make_adam(grad_scale=0.5), 1, gr, master, m, v,
                    params, main_grad_out=mg, lib=lib)
        L = oracle.range_map(sz, Dr, 0, pad, lib=lib)
        owned = np.zeros(Nr, bool)
        for p in range(n):
            owned[L.param_start[p]:L.param_end[p]] = True
        want = int(np.count_nonzero(~np.isfinite(mg[owned])))
        assert oracle.count_nonfinite(sz, Dr, 0, pad, 0.5, gr, lib=lib) == want


def pin_f16_conversions(lib):
    """IEEE binary16 (reading R7b), against numpy's float16, which
    implements the standard's conversions: widening every one of the 65536
    bit patterns; narrowing every finite half, every midpoint between
    neighbouring halves (ties go to the even one), the floats just beside
    those midpoints, the overflow edge, subnormals and random floats."""
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = allbits.view(np.float16).astype(np.float32)
    got = np.array([lib.orc_f16_to_f32(int(b)) for b in allbits], np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))

    finite = want[np.isfinite(want)]
    pos = np.unique(np.abs(finite.astype(np.float64)))
    mids = (pos[:-1] + pos[1:]) / 2  # exact in fp32 for binary16 neighbours
    mids32 = mids.astype(np.float32)
    assert np.array_equal(mids32.astype(np.float64), mids)
    rng = np.random.default_rng(23)
    rand = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 12, 20000))).astype(np.float32)
    edge = np.array([0.0, -0.0, 65504.0, 65519.996, 65520.0, 65536.0, 1e30, 2.0 ** -24,
                     2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -26, 2.0 ** -14, 6.1e-5, 1e-8,
                     np.inf, -np.inf, np.nan], np.float32)
    xs = np.concatenate([finite, -finite, mids32, -mids32,
                         np.nextafter(mids32, np.float32(np.inf)),
                         np.nextafter(mids32, np.float32(0)), rand, edge])
    with np.errstate(over="ignore"):
        want16 = xs.astype(np.float16).view(np.uint16)
    got16 = np.array([lib.orc_f32_to_f16(float(x)) for x in xs], np.uint16)
    wnan = np.isnan(want16.view(np.float16))
    assert np.array_equal(np.isnan(got16.view(np.float16)), wnan)
    bad = np.flatnonzero(got16[~wnan] != want16[~wnan])
    assert bad.size == 0, (xs[~wnan][bad[:5]], got16[~wnan][bad[:5]], want16[~wnan][bad[:5]])


def pin_f16_grads_and_params(lib):
    """FP16 grads whose values are exact in both fp16 and bf16 give the bf16
    path's step, main grads and all-reduce bit for bit; fp16 params are
    numpy's float16 rounding of the updated master; with the rounding of
    R12 the main grads are numpy's float16 of the unrounded ones; and
    60000 + 60000 (finite in fp32, beyond fp16's 65504) is non-finite only
    once rounded to fp16."""
    sizes, wd, D, pad = [300, 41, 129], [1, 0, 1], 4, 2
    L = oracle.range_map(sizes, D, 0, pad, lib=lib)
    N = L.numel
    owned = np.zeros(N, bool)
    for p in range(len(sizes)):
        owned[L.param_start[p]:L.param_end[p]] = True
    rng = np.random.default_rng(29)
    vals = [(rng.integers(-64, 65, N) * 2.0 ** -10).astype(np.float32) for _ in range(D)]
    g16 = [v.astype(np.float16) for v in vals]
    gbf = [(v.view(np.uint32) >> 16).astype(np.uint16) for v in vals]  # exact
    adam = oracle.make_adam(grad_scale=0.25)
    master0, m0, v0 = _state(N, 31, 1e-4, 1e-6)
    out = {}
    for name, g in (("f16", g16), ("bf16", gbf)):
        master, m, v = master0.copy(), m0.copy(), v0.copy()
        params = _params_from(master0, D)
        mg = np.zeros(N, np.float32)
        oracle.step(sizes, wd, D, 0, pad, adam, 1, [x.copy() for x in g], master, m, v, params,
                    main_grad_out=mg, lib=lib)
        ar = [x.copy() for x in g]
        oracle.allreduce(sizes, D, 0, pad, 0.25, ar, lib=lib)
        arf = [x.astype(np.float32) if name == "f16" else
               (x.astype(np.uint32) << 16).view(np.float32) for x in ar]
        out[name] = (master, m, v, params, mg, arf)
    for a, b in zip(out["f16"][:3] + (out["f16"][4],), out["bf16"][:3] + (out["bf16"][4],)):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    for a, b in zip(out["f16"][5], out["bf16"][5]):
        assert np.array_equal(a[owned], b[owned])
    # fp16 params
    master, m, v = master0.copy(), m0.copy(), v0.copy()
    p16 = [master0.astype(np.float16) for _ in range(D)]
    p_before = [p.copy() for p in p16]
    oracle.step(sizes, wd, D, 0, pad, adam, 1, [x.copy() for x in g16], master, m, v, p16,
                lib=lib)
    assert np.array_equal(master.view(np.uint32), out["f16"][0].view(np.uint32))
    for p, p0 in zip(p16, p_before):
        assert np.array_equal(p[owned].view(np.uint16), master[owned].astype(np.float16).view(np.uint16))
        assert np.array_equal(p[~owned].view(np.uint16), p0[~owned].view(np.uint16))
    # the rounding of R12 in fp16
    gr = [rng.normal(0, 1, N).astype(np.float16) for _ in range(D)]
    runs = {}
    for rg in (False, True):
        mg = np.zeros(N, np.float32)
        master, m, v = master0.copy(), m0.copy(), v0.copy()
        oracle.step(sizes, wd, D, 0, pad, oracle.make_adam(grad_scale=0.3), 1, gr, master, m, v,
                    _params_from(master0, D), main_grad_out=mg, round_grad=rg, lib=lib)
        runs[rg] = mg
    want = runs[False].astype(np.float16).astype(np.float32)
    assert np.array_equal(runs[True][owned], want[owned])
    assert np.count_nonzero(want[owned] != runs[False][owned]) > owned.sum() // 2
    # overflow only once rounded to fp16
    go = [np.zeros(N, np.float16) for _ in range(D)]
    go[0][3] = go[1][3] = np.float16(60000.0)
    assert oracle.count_nonfinite(sizes, D, 0, pad, 1.0, go, lib=lib) == 0
    assert oracle.count_nonfinite(sizes, D, 0, pad, 1.0, go, round_grad=True, lib=lib) == 1


ALL_PINS = [
    pin_page1_ownership,
    pin_brute_force_range_maps,
    pin_error_paths,
    pin_allreduce_example,
    pin_rs_concat_equals_allreduce,
    pin_rank_order_accumulation,
    pin_scale_before_reduce,
    pin_d1_is_adamw,
    pin_d_independence,
    pin_bf16_rounding,
    pin_gather_and_padding,
    pin_window_equals_full,
    pin_clip_norm_closed_form,
    pin_clip_d1_matches_torch,
    pin_clip_off_equals_plain_step,
    pin_clip_d_independence,
    pin_allreduce_every_rank,
    pin_allreduce_is_rs_then_gather,
    pin_allreduce_rounds_to_nearest_even,
    pin_instances_hierarchical_order,
    pin_instances_factorizations,
    pin_instances_write_back_and_gather,
    pin_round_grad,
    pin_nonfinite_count,
    pin_f16_conversions,
    pin_f16_grads_and_params,
]
