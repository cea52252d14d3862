"""The CPU oracle against what the pages and mathematics fix (see pins.py)."""
import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, lib):
    pin(lib)


def test_configs_layout_invariants(lib):
    """The five workloads' layouts obey the greedy bucket rule; the GPT-2
    small layout has 3 buckets of 40 Mi and 256 padding elements."""
    from zero_distributed_optimizer_gb300 import workloads as W

    cfgs = W.all_configs() + [W.sweep_256m(D, b) for D in W.SWEEP_D for b in W.SWEEP_BUCKET_MI]
    for w in cfgs:
        L = oracle.range_map(w.sizes, w.D, w.bucket_elems, w.pad_unit, lib=lib)
        pins.check_layout_invariants(L, list(w.sizes), w.D, w.bucket_elems, w.pad_unit)
        # every non-padding element is owned by exactly one piece
        covered = sum(pc["gbuf_world"][1] - pc["gbuf_world"][0] for pc in L.pieces)
        assert covered == w.numel
    g = W.gpt2_small()
    L = oracle.range_map(g.sizes, g.D, g.bucket_elems, g.pad_unit, lib=lib)
    assert g.numel == 124_439_808 and L.n_buckets == 3 and L.numel - g.numel == 256
