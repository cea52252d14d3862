"""The test-side helpers that run the oracle, checked on the CPU."""
import numpy as np
import pytest

import oracle
from parity import oracle_step_whole


@pytest.mark.parametrize("grad_f32", [False, True])
@pytest.mark.parametrize("threads", [1, 3, 7])
def test_threaded_whole_buffer_step_equals_single_call(grad_f32, threads):
    """oracle_step_whole (disjoint windows on host threads) gives the single
    whole-buffer call's outputs bit for bit, over windows cutting through
    pieces, rank shards and buckets."""
    sizes, wd, D, bucket, pad = [5000, 1, 7, 300, 20000, 3, 9999], [1, 0, 1, 0, 1, 1, 0], 4, 6000, 8
    N = oracle.range_map(sizes, D, bucket, pad).numel
    rng = np.random.default_rng(11)
    if grad_f32:
        grads = [rng.normal(0, 1e-2, N).astype(np.float32) for _ in range(D)]
    else:
        grads = [(rng.normal(0, 1e-2, N).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
                 for _ in range(D)]
    state = [rng.normal(0, 0.02, N).astype(np.float32), np.zeros(N, np.float32),
             np.zeros(N, np.float32)]
    params = [(state[0].view(np.uint32) >> 16).astype(np.uint16) for _ in range(D)]
    adam = oracle.make_adam(grad_scale=1.0 / D)
    a = [x.copy() for x in state] + [[p.copy() for p in params], np.full(N, -1.0, np.float32)]
    b = [x.copy() for x in state] + [[p.copy() for p in params], np.full(N, -1.0, np.float32)]
    for t in (1, 2):
        oracle.step(sizes, wd, D, bucket, pad, adam, t, grads, a[0], a[1], a[2], a[3],
                    main_grad_out=a[4])
        oracle_step_whole(sizes, wd, D, bucket, pad, adam, t, grads, b[0], b[1], b[2], b[3],
                          main_grad_out=b[4], threads=threads)
    for x, y in zip(a[:3] + [a[4]], b[:3] + [b[4]]):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    for x, y in zip(a[3], b[3]):
        assert np.array_equal(x, y)
    assert not np.array_equal(a[0], state[0])
