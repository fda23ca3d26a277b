"""Layer-partitioned sharding with the CUDA library (gloo ranks as processes on one GPU).

Two ranks each hold the same K gradients on the GPU; rank r combines the segments of its
partition with the library's default entry point, and the partitions are all-gathered
(through host copies, which is what gloo gathers), so every rank ends with the whole
result.  The ranks' kernels never wait on one another; they share the device only.
Every rank's result is compared with the fp64 oracle segment by segment.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, name, shrink, q):
    import torch.distributed as dist
    import adaptive_gradient_summation_gb300 as ags
    from adaptive_gradient_summation_gb300 import workloads
    from adaptive_gradient_summation_gb300.sharding import sharded_reduce
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ags.load_library()
        wl = workloads.make(name, device="cuda:0", shrink=shrink)   # same seed on every rank
        before = ags.launch_count()
        out = sharded_reduce(wl.grads, wl.seg_offsets)
        torch.cuda.synchronize()
        launched = ags.launch_count() - before
        q.put((rank, out.cpu(), launched))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("name,shrink", [("bert_large_k16", 64), ("resnet50_k8", 16)])
def test_sharded_reduce_with_the_cuda_library(native, world, name, shrink):
    from adaptive_gradient_summation_gb300 import workloads
    from parity import check_against_oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, name, shrink, q))
             for r in range(world)]
    for p in procs:
        p.start()
    results = {}
    for _ in range(world):
        rank, out, launched = q.get(timeout=300)
        results[rank] = (out, launched)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    wl = workloads.make(name, device="cuda:0", shrink=shrink)   # the ranks' inputs
    for r in range(world):
        out, launched = results[r]
        assert launched > 0, "the rank's partition did not run on the CUDA library"
        check_against_oracle(wl.grads, wl.seg_offsets, out)
    # every rank holds the same bits
    for r in range(1, world):
        assert torch.equal(results[r][0], results[0][0])
