"""Layer-partitioned sharding over ranks (gloo, world size 2 and 3, on the CPU).

The per-rank reduction here is the fp64 oracle (test-only, passed in as reduce_fn), so
these tests check the partitioning and the gather; the CUDA reduction itself is covered
by the GPU parity tests.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from adaptive_gradient_summation_gb300.sharding import partition_segments, sharded_reduce


def test_partitions_are_whole_balanced_runs():
    offs = np.cumsum([0, 10, 1, 1, 50, 3, 3, 30, 2])
    for world in (1, 2, 3, 4, 8, 20):
        b = partition_segments(offs, world)
        assert len(b) == world + 1 and b[0] == 0 and b[-1] == len(offs) - 1
        assert all(x <= y for x, y in zip(b, b[1:]))          # contiguous, whole segments
    b = partition_segments(np.cumsum([0] + [100] * 8), 4)
    assert b == [0, 2, 4, 6, 8]                                # equal segments, equal runs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_reduce(grads, offs, out):
    import oracle
    r = oracle.adasum_reduce([g.numpy() for g in grads], offs)
    out.copy_(torch.from_numpy(r["out"]))


def _worker(rank, world, port, K, lengths, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rs = np.random.default_rng(7)
        offs = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
        grads = [torch.from_numpy(rs.standard_normal(int(offs[-1])).astype(np.float32))
                 for _ in range(K)]
        out = sharded_reduce(grads, offs, reduce_fn=_oracle_reduce)
        q.put((rank, out.numpy().copy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_reduce_equals_unsharded_gloo(world):
    import oracle
    oracle.build()
    K, lengths = 4, [5, 0, 17, 3, 40, 1, 9]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, K, lengths, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    rs = np.random.default_rng(7)
    offs = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    grads = [rs.standard_normal(int(offs[-1])).astype(np.float32) for _ in range(K)]
    ref = oracle.adasum_reduce(grads, offs)["out"]
    for r in range(world):
        assert np.array_equal(results[r], ref)
