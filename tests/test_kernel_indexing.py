"""CPU model of the step kernel's work split, checked before any GPU run.

The model follows the kernel's decomposition: 2048-element tiles, a per-tile
first-run index, a per-warp ballot over 32 run ends, a per-thread walk, the
8-element vector path inside one run and the element path at run edges.  It
checks that every owned element is visited exactly once, that no padding
element is visited, and that every 8-element vector access lies inside the
buffer.  The run table is rebuilt here from the pieces with the kernel's
merge rule (touching pieces with the same owner rank and decay flag)."""
import numpy as np
import pytest

import pins
from zero_distributed_optimizer_gb300 import binding as B

TILE, THREADS, VEC = 2048, 256, 8


def runs_from_pieces(pieces, decays):
    runs = []
    for pc in pieces:
        meta = (1 if decays[pc["param_id"]] else 0) | (pc["rank"] << 8)
        a, b = pc["gbuf_world"]
        if runs and runs[-1][1] == a and runs[-1][2] == meta:
            runs[-1][1] = b
        else:
            runs.append([a, b, meta])
    return runs


def simulate(numel, runs):
    nr = len(runs)
    start = [r[0] for r in runs]
    end = [r[1] for r in runs]
    visits = np.zeros(numel, np.int32)
    vector_accesses = 0
    n_tiles = (numel + TILE - 1) // TILE
    tile_run = []
    j = 0
    for t in range(n_tiles + 1):
        while j < nr and end[j] <= t * TILE:
            j += 1
        tile_run.append(j)
    for tile in range(n_tiles):
        for warp in range(THREADS // 32):
            wb = tile * TILE + warp * 32 * VEC
            j = tile_run[tile]
            while True:
                c = 0
                for lane in range(32):
                    idx = j + lane
                    if idx < nr and end[idx] <= wb:
                        c += 1
                j += c
                if c < 32:
                    break
            for lane in range(32):
                e0 = wb + lane * VEC
                if e0 >= numel:
                    continue
                jj = j
                while jj < nr and end[jj] <= e0:
                    jj += 1
                if jj >= nr or start[jj] >= e0 + VEC:
                    continue
                if start[jj] <= e0 and e0 + VEC <= end[jj]:
                    assert e0 % VEC == 0 and e0 + VEC <= numel
                    visits[e0:e0 + VEC] += 1
                    vector_accesses += 1
                    continue
                for k in range(VEC):
                    e = e0 + k
                    if e >= numel:
                        break
                    while jj < nr and end[jj] <= e:
                        jj += 1
                    if jj >= nr:
                        break
                    if start[jj] > e:
                        continue
                    visits[e] += 1
    return visits, vector_accesses


def check_layout(sizes, D, bucket, pad, wd=None):
    L = B.dopt_build_range_map(sizes, D, bucket, pad, wd)
    decays = wd if wd is not None else [1] * len(sizes)
    runs = runs_from_pieces(L.pieces(), decays)
    for (a, b, _), (c, d, _) in zip(runs, runs[1:]):
        assert a < b <= c < d  # sorted, disjoint, non-empty
    visits, nvec = simulate(L.padded_numel, runs)
    owned = np.zeros(L.padded_numel, np.int32)
    for a, b in L.param_ranges():
        owned[a:b] = 1
    assert np.array_equal(visits, owned)
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
])
def test_parity_layouts(case):
    sizes, D, bucket, pad, wd = case
    check_layout(sizes, D, bucket, pad, wd)


def test_vector_path_dominates_on_aligned_layouts():
    """With sizes that are multiples of 8 every vector lies inside one run."""
    sizes = [8 * 1000, 8 * 333, 8 * 2049]
    nvec = check_layout(sizes, 4, 0, 8)
    assert nvec == sum(sizes) // 8
