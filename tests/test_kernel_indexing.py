"""CPU model of the kernels' work split, checked before any GPU run.

The model follows the kernels' decomposition: a launch covers a run view
(runs [run_begin, run_limit) and the tiles from tile0 that span them),
2048-element tiles, a per-tile first-run index, a per-warp ballot over 32 run
ends, a per-thread walk, the 8-element vector path inside one run and the
element path at run edges, in both of its forms: the warp's straddling
vectors shared out over its lanes (four per round, one element per lane:
the step, all-reduce and gather kernels) and one lane per straddling vector
(the norm pass).  It checks that every owned element of the view is
visited exactly once, that nothing outside it is visited, and that every
8-element vector access lies inside the buffer.  The run table is rebuilt
here from the pieces with the library's rule (touching pieces of one bucket
with the same owner rank and decay flag merge)."""
import numpy as np
import pytest

import pins
from zero_distributed_optimizer_gb300 import binding as B

TILE, THREADS, VEC = 2048, 256, 8


def runs_from_pieces(pieces, decays, n_buckets):
    runs, bucket_run, last_bucket = [], [0] * (n_buckets + 1), -1
    for pc in pieces:
        meta = (1 if decays[pc["param_id"]] else 0) | (pc["rank"] << 8)
        a, b = pc["gbuf_world"]
        if runs and runs[-1][1] == a and runs[-1][2] == meta and last_bucket == pc["bucket_id"]:
            runs[-1][1] = b
        else:
            for k in range(last_bucket + 1, pc["bucket_id"] + 1):
                bucket_run[k] = len(runs)
            last_bucket = pc["bucket_id"]
            runs.append([a, b, meta])
    for k in range(last_bucket + 1, n_buckets + 1):
        bucket_run[k] = len(runs)
    return runs, bucket_run


def tile_index(numel, runs):
    n_tiles = (numel + TILE - 1) // TILE
    out, j = [], 0
    for t in range(n_tiles + 1):
        while j < len(runs) and runs[j][1] <= t * TILE:
            j += 1
        out.append(j)
    return out


def view(runs, bucket_run, first, count):
    lo_run, hi_run = bucket_run[first], bucket_run[first + count]
    if lo_run >= hi_run:
        return lo_run, hi_run, 0, 0
    tile0 = runs[lo_run][0] // TILE
    tiles = (runs[hi_run - 1][1] + TILE - 1) // TILE - tile0
    return lo_run, hi_run, tile0, tiles


def owned_at(e, j, numel, start, end, run_limit):
    """The element path's lookup: (owned, run index) walking from run j."""
    if e >= numel:
        return False, j
    while j < run_limit and end[j] <= e:
        j += 1
    return j < run_limit and start[j] <= e, j


def simulate(numel, runs, tile_run, run_begin, run_limit, tile0, tiles, visits, shared=True):
    start = [r[0] for r in runs]
    end = [r[1] for r in runs]
    vector_accesses = 0
    for b in range(tiles):
        tile = tile0 + b
        assert tile < len(tile_run) - 1
        for warp in range(THREADS // 32):
            wb = tile * TILE + warp * 32 * VEC
            j = max(tile_run[tile], run_begin)
            while True:  # the ballot over 32 run ends
                c = sum(1 for lane in range(32)
                        if j + lane < run_limit and end[j + lane] <= wb)
                j += c
                if c < 32:
                    break
            mixed = []  # lanes whose vector straddles a run edge (the ballot)
            for lane in range(32):
                e0 = wb + lane * VEC
                if e0 >= numel:
                    continue
                jj = j
                while jj < run_limit and end[jj] <= e0:
                    jj += 1
                if jj >= run_limit or start[jj] >= e0 + VEC:
                    continue
                if start[jj] <= e0 and e0 + VEC <= end[jj]:
                    assert e0 % VEC == 0 and e0 + VEC <= numel
                    visits[e0:e0 + VEC] += 1
                    vector_accesses += 1
                    continue
                if not shared:  # one lane per vector, element after element
                    for k in range(VEC):
                        owned, jj = owned_at(e0 + k, jj, numel, start, end, run_limit)
                        if owned:
                            visits[e0 + k] += 1
                    continue
                mixed.append(lane)
            # rounds of 4 straddling vectors, octet o taking the o-th one left,
            # lane k of the octet element k, each walking from the warp's run j
            for r0 in range(0, len(mixed), 4):
                for octet in range(4):
                    if r0 + octet >= len(mixed):
                        continue
                    src = mixed[r0 + octet]
                    for k in range(VEC):
                        e = wb + src * VEC + k
                        assert wb <= e < wb + 32 * VEC
                        owned, _ = owned_at(e, j, numel, start, end, run_limit)
                        if owned:
                            visits[e] += 1
    return vector_accesses


def check_layout(sizes, D, bucket, pad, wd=None, instances=1):
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd, instances=instances)
    decays = wd if wd is not None else [1] * len(sizes)
    runs, bucket_run = runs_from_pieces(L.pieces(), decays, L.n_buckets)
    for (a, b, _), (c, d, _) in zip(runs, runs[1:]):
        assert a < b <= c < d  # sorted, disjoint, non-empty
    N = L.padded_numel
    tr = tile_index(N, runs)
    owned = np.zeros(N, np.int32)
    for a, b in L.param_offsets():
        owned[a:b] = 1
    # one launch over every bucket, with either element path
    for shared in (True, False):
        visits = np.zeros(N, np.int32)
        nvec = simulate(N, runs, tr, *view(runs, bucket_run, 0, L.n_buckets), visits, shared)
        assert np.array_equal(visits, owned)
    # one launch per bucket, and one over a middle range of buckets
    visits = np.zeros(N, np.int32)
    for k in range(L.n_buckets):
        simulate(N, runs, tr, *view(runs, bucket_run, k, 1), visits)
    assert np.array_equal(visits, owned)
    if L.n_buckets >= 3:
        visits = np.zeros(N, np.int32)
        simulate(N, runs, tr, *view(runs, bucket_run, 1, L.n_buckets - 2), visits)
        mid = np.zeros(N, np.int32)
        buckets = L.buckets()
        mid[buckets[1][0]:buckets[-2][1]] = owned[buckets[1][0]:buckets[-2][1]]
        assert np.array_equal(visits, mid)
    return nvec


def test_tiny_layouts():
    for sizes, D, bucket, pad in pins.random_tiny_layouts(200, seed=7):
        check_layout(sizes, D, bucket, pad)


@pytest.mark.parametrize("case", [
    ([130, 260, 90, 310, 210], 4, 0, 1, None),
    ([2], 3, 0, 1, None),
    ([5000, 1, 7, 300, 20000, 3, 9999], 8, 0, 1, [1, 0, 1, 0, 1, 1, 0]),
    ([70001], 1, 0, 1, None),
    ([4096, 333, 12345, 8, 77777], 3, 20000, 1, [0, 1, 1, 0, 1]),
    ([31000, 17, 64000, 5], 5, 30000, 3, [1, 0, 1, 0]),
    ([64] * 300 + [5000], 2, 4096, 64, None),
    ([1, 2, 3, 4, 5, 6, 7, 8, 9, 10] * 20, 4, 64, 1, [1, 0] * 100),
    ([123457, 99], 64, 0, 1, [1, 0]),
    ([0, 500, 0, 0, 1200, 0], 4, 0, 1, None),
    ([3] * 2000, 16, 0, 1, [1, 0] * 1000),  # more than 32 runs per warp
    ([1000, 3, 2000, 5, 700], 1, 1000, 1, None),  # D=1: buckets touch, runs must not merge
    ([300000, 5, 70001, 4096, 123], 8, 100000, 64, [1, 0, 1, 1, 0]),
    ([5000, 7000, 3000, 9000, 4000], 4, 6000, 8, None),
])
def test_parity_layouts(case):
    sizes, D, bucket, pad, wd = case
    check_layout(sizes, D, bucket, pad, wd)


def test_vector_path_dominates_on_aligned_layouts():
    """With sizes that are multiples of 8 every vector lies inside one run."""
    sizes = [8 * 1000, 8 * 333, 8 * 2049]
    nvec = check_layout(sizes, 4, 0, 8)
    assert nvec == sum(sizes) // 8


@pytest.mark.parametrize("D,instances", [(8, 2), (6, 3), (16, 4), (8, 8)])
def test_instance_layouts(D, instances):
    """Layouts sharded R = D / instances ways (runs carry the rank inside the
    instance)."""
    check_layout([5000, 1, 7, 300, 20000, 3, 9999], D, 0, 1, [1, 0, 1, 0, 1, 1, 0], instances)
    check_layout([31000, 17, 64000, 5], D, 30000, 3, [1, 0, 1, 0], instances)
