"""Multi-rank host logic of bench.py on CPU: a world-size-2 gloo group reduces the
per-rank timed-region lengths to their maximum and aggregates whole-job
throughput over all ranks, and splits a global batch into per-rank shards that
cover it exactly once (data parallel over the batch, weak scaling: every rank
keeps N images; there is no collective on the data path).  The shards are a
valid partition of the method: the oracle's input gradient of the whole batch
is the concatenation of the ranks' results on their shards."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [12.5, 20.0][rank]
    max_ms = bench.reduce_max(local_ms, True)
    flops = bench.useful_flops(__import__("conv2d_backward_implicit_gb300.workloads",
                                          fromlist=["x"]).RESNET)
    value = bench.aggregate_throughput(flops, 100, world, max_ms)
    # Each rank's shard of a global batch of 5 images, gathered on every rank.
    lo, hi = bench.shard_bounds(5, world, rank)
    spans = [None] * world
    dist.all_gather_object(spans, (lo, hi))
    out[rank] = (max_ms, value, spans)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    import bench
    from conv2d_backward_implicit_gb300 import workloads
    flops = bench.useful_flops(workloads.RESNET)
    for rank in (0, 1):
        max_ms, value, spans = out[rank]
        assert max_ms == 20.0
        assert value == pytest.approx(flops * 100 * 2 / 0.020 / 1e12)
        assert spans == [(0, 3), (3, 5)]
    # The shards partition the method: grad_in of the batch = the shards' grad_in.
    import numpy as np
    import oracle
    wl = workloads.STRIDED
    rng = np.random.default_rng(0)
    g = rng.standard_normal((5, 6, 4, 4))
    w = rng.standard_normal((6, 3, 3, 3))
    whole = oracle.dgrad(g, w, 8, 8, wl.stride, wl.padding_h, wl.padding_w)
    parts = [oracle.dgrad(g[lo:hi], w, 8, 8, wl.stride, wl.padding_h, wl.padding_w)
             for lo, hi in out[0][2]]
    assert np.array_equal(np.concatenate(parts), whole)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.5, False) == 3.5
    assert bench.aggregate_throughput(1e12, 10, 1, 1000.0) == pytest.approx(10.0)
