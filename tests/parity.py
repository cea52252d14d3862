"""Comparison helpers for the CUDA path against the oracle.

Tolerances: fp32 master/m/v within 1e-6 relative + 1e-7 absolute; bf16
params within 1 bf16 ulp; NaN where the other side has NaN.  Both sides use
the same rank-order fp32 arithmetic with one rounding per operation, so the
expected outcome is bit-for-bit equality; the counts of elements that are
not bit-identical are returned for reporting.
"""
from __future__ import annotations

import numpy as np

RTOL = 1e-6
ATOL = 1e-7


def t2np_bf16(t):
    import torch

    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def t2np_f32(t):
    return t.detach().cpu().numpy()


def np_bf16_from_torch(t):
    return t2np_bf16(t)


def bf16_is_nan(bits):
    bits = np.asarray(bits, np.uint16)
    return ((bits & 0x7F80) == 0x7F80) & ((bits & 0x7F) != 0)


def bf16_order_key(bits):
    b = np.asarray(bits, np.uint16).astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def assert_f32_close(gpu, orc, what, rtol=RTOL, atol=ATOL) -> int:
    gpu = np.asarray(gpu, np.float32)
    orc = np.asarray(orc, np.float32)
    assert gpu.shape == orc.shape, what
    nan_g, nan_o = np.isnan(gpu), np.isnan(orc)
    assert np.array_equal(nan_g, nan_o), f"{what}: NaN positions differ"
    ok = ~nan_o
    g = gpu[ok].astype(np.float64)
    o = orc[ok].astype(np.float64)
    inf = np.isinf(o)
    assert np.array_equal(g[inf], o[inf]), f"{what}: infinities differ"
    fin = ~inf
    err = np.abs(g[fin] - o[fin])
    bad = err > atol + rtol * np.abs(o[fin])
    if bad.any():
        idx = np.flatnonzero(ok)[np.flatnonzero(fin)[bad]][:5]
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside tolerance, e.g. "
                             f"index {idx.tolist()} gpu {gpu[idx].tolist()} oracle {orc[idx].tolist()}")
    return int(np.count_nonzero(gpu[ok].view(np.uint32) != orc[ok].view(np.uint32)))


def assert_bf16_close(gpu_bits, orc_bits, what, ulps=1) -> int:
    gpu_bits = np.asarray(gpu_bits, np.uint16)
    orc_bits = np.asarray(orc_bits, np.uint16)
    assert gpu_bits.shape == orc_bits.shape, what
    ng, no = bf16_is_nan(gpu_bits), bf16_is_nan(orc_bits)
    assert np.array_equal(ng, no), f"{what}: NaN positions differ"
    ok = ~no
    d = np.abs(bf16_order_key(gpu_bits[ok]) - bf16_order_key(orc_bits[ok]))
    if (d > ulps).any():
        idx = np.flatnonzero(ok)[d > ulps][:5]
        raise AssertionError(f"{what}: {int((d > ulps).sum())} elements beyond {ulps} ulp, e.g. "
                             f"index {idx.tolist()} gpu {gpu_bits[idx].tolist()} "
                             f"oracle {orc_bits[idx].tolist()}")
    return int(np.count_nonzero(gpu_bits[ok] != orc_bits[ok]))


def f16_is_nan(bits):
    bits = np.asarray(bits, np.uint16)
    return ((bits & 0x7C00) == 0x7C00) & ((bits & 0x3FF) != 0)


def assert_f16_close(gpu, orc, what, ulps=1) -> int:
    """IEEE fp16 arrays (float16 or their uint16 bits) within `ulps` units
    in the last place; NaN where the other side has NaN."""
    gpu_bits = np.asarray(gpu).view(np.uint16) if np.asarray(gpu).dtype == np.float16 \
        else np.asarray(gpu, np.uint16)
    orc_bits = np.asarray(orc).view(np.uint16) if np.asarray(orc).dtype == np.float16 \
        else np.asarray(orc, np.uint16)
    assert gpu_bits.shape == orc_bits.shape, what
    ng, no = f16_is_nan(gpu_bits), f16_is_nan(orc_bits)
    assert np.array_equal(ng, no), f"{what}: NaN positions differ"
    ok = ~no
    d = np.abs(bf16_order_key(gpu_bits[ok]) - bf16_order_key(orc_bits[ok]))  # same sign layout
    if (d > ulps).any():
        idx = np.flatnonzero(ok)[d > ulps][:5]
        raise AssertionError(f"{what}: {int((d > ulps).sum())} elements beyond {ulps} ulp, e.g. "
                             f"index {idx.tolist()} gpu {gpu_bits[idx].tolist()} "
                             f"oracle {orc_bits[idx].tolist()}")
    return int(np.count_nonzero(gpu_bits[ok] != orc_bits[ok]))


def t2np_grad(t):
    """A grad tensor as the oracle takes it: bf16 as uint16 bits, fp16 as
    float16, fp32 as float32 (copies)."""
    import torch

    if t.dtype == torch.bfloat16:
        return t2np_bf16(t).copy()
    return t.detach().cpu().numpy().copy()


def t2np_param(t):
    """A param replica as the oracle takes it: bf16 bits or float16."""
    return t2np_grad(t)


def assert_param_close(gpu_t, orc, what) -> int:
    """A device param replica (bf16 or fp16) against the oracle's, 1 ulp."""
    import torch

    if gpu_t.dtype == torch.float16:
        return assert_f16_close(gpu_t.detach().cpu().numpy(), orc, what)
    return assert_bf16_close(t2np_bf16(gpu_t), orc, what)


def merge_windows(wins, numel):
    wins = sorted((max(0, a), min(numel, b)) for a, b in wins if min(numel, b) > max(0, a))
    out = []
    for a, b in wins:
        if out and a <= out[-1][1]:
            out[-1] = (out[-1][0], max(out[-1][1], b))
        else:
            out.append((a, b))
    return out


def sample_windows(buckets, pieces, numel, seed, n_edges=48, n_random=12, rand_len=1 << 16,
                   edge=64):
    """Exact-comparison windows for a large buffer: both ends of every
    bucket (with its padding), `n_edges` piece boundaries +-edge elements
    (rank and param edges), and `n_random` random stretches."""
    rng = np.random.default_rng(seed)
    wins = []
    for a, b in buckets:
        wins.append((a, a + 4 * edge))
        wins.append((b - 4 * edge, b))
    bounds = sorted({pc["gbuf_world"][0] for pc in pieces} | {pc["gbuf_world"][1] for pc in pieces})
    if len(bounds) > n_edges:
        pick = rng.choice(len(bounds), n_edges, replace=False)
        bounds = [bounds[i] for i in sorted(pick)]
    wins += [(x - edge, x + edge) for x in bounds]
    for _ in range(n_random):
        a = int(rng.integers(0, max(1, numel - rand_len)))
        wins.append((a, a + rand_len))
    return merge_windows(wins, numel)


def oracle_step_whole(sizes, wd_mask, D, bucket_elems, pad_unit, adam, t, grads, master,
                      exp_avg, exp_avg_sq, params, main_grad_out=None, threads=None, **kw):
    """The oracle's step over a whole buffer, cut into disjoint windows that
    host threads step at the same time.  Every output element depends on
    its own inputs alone and the ctypes call releases the GIL, so the
    result equals one call over the whole buffer bit for bit (a CPU test
    checks that)."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    n = len(master)
    k = max(1, min(threads or os.cpu_count() or 1, 32))
    cuts = [n * i // k for i in range(k + 1)]

    def one(i):
        a, b = cuts[i], cuts[i + 1]
        if a == b:
            return
        oracle.step(sizes, wd_mask, D, bucket_elems, pad_unit, adam, t, [g[a:b] for g in grads],
                    master[a:b], exp_avg[a:b], exp_avg_sq[a:b], [p[a:b] for p in params],
                    main_grad_out=None if main_grad_out is None else main_grad_out[a:b],
                    window=(a, b), **kw)

    with ThreadPoolExecutor(k) as ex:
        list(ex.map(one, range(k)))
