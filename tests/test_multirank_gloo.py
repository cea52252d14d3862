"""The benchmark's N>1 path on CPU: two gloo ranks, each stepping its own
replica of a workload (no collective on the data path), meeting only for the
barrier and the max-over-ranks timing reduction."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import numpy as np
    import torch.distributed as dist

    import bench
    import oracle
    from zero_distributed_optimizer_gb300 import workloads as W

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (world, rank, rank)
    # each rank steps its own replica of the toy workload with the oracle
    w = W.toy_1000()
    L = oracle.range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit)
    master, m, v = (t.numpy().copy() for t in W.make_state(w, L.numel, "cpu"))
    params = [np.zeros(L.numel, np.uint16) for _ in range(w.D)]
    grads = [g.view(__import__("torch").int16).numpy().view(np.uint16).copy()
             for g in W.make_grads(w, L.numel, 1, "cpu")]
    oracle.step(list(w.sizes), list(w.wd_mask), w.D, 0, 1, oracle.make_adam(**w.adam_kwargs()),
                1, grads, master, m, v, params)
    dist.barrier()
    # per-rank "times" differ; every rank must see the maximum
    got = bench.max_over_ranks(10.0 + rank, world)
    out[rank] = (got, float(master.sum()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_and_max_over_ranks():
    world = 2
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    assert out[0][0] == out[1][0] == 11.0
    # independent replicas of the same workload compute the same values
    assert out[0][1] == out[1][1]


def test_single_rank_max_is_identity():
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
