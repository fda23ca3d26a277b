"""Layer-partitioned sharding of the Adasum combine over several ranks.

The paper partitions optimizer state (and the effective gradient) across GPUs so that
every layer falls in one partition, each GPU runs the Adasum reduction only for the
layers of its partition, and the partitions are then broadcast to every GPU ("Scaling
Distributed Training with Adaptive Summation", Section 4).  On one box the same idea
shards one Adasum call: segments are independent, so whole segments are dealt to ranks
in contiguous, byte-balanced runs; each rank reduces its run with the library; an
all-gather assembles the full result on every rank.  No partition ever splits a segment.

This module is host-side orchestration over torch.distributed; the arithmetic runs in
the CUDA library (or in whatever `reduce_fn` the caller passes).
"""
from __future__ import annotations

import numpy as np
import torch


def partition_segments(seg_offsets, world_size: int, bytes_per_position: int = 1):
    """Split segments [0, L) into `world_size` contiguous runs of whole segments with
    about equal bytes.  Returns world_size + 1 segment indices (run r = [b[r], b[r+1])).

    Greedy on the running byte count: run r ends at the first segment boundary at or
    past r+1 equal shares, so every run gets whole segments and no segment is split.
    """
    offs = np.asarray(seg_offsets, dtype=np.int64)
    L = offs.shape[0] - 1
    if world_size < 1:
        raise ValueError("world_size must be >= 1")
    total = int(offs[-1]) * bytes_per_position
    bounds = [0]
    for r in range(1, world_size):
        target = total * r / world_size
        s = int(np.searchsorted(offs * bytes_per_position, target, side="left"))
        s = min(max(s, bounds[-1]), L)
        bounds.append(s)
    bounds.append(L)
    return bounds


def _default_reduce(grads, offs, out):
    import adaptive_gradient_summation_gb300 as ags
    return ags.reduce(grads, offs, out=out)


def sharded_reduce(grads, seg_offsets, *, group=None, out: torch.Tensor | None = None,
                   reduce_fn=None) -> torch.Tensor:
    """Adasum of the same K worker gradients on every rank of `group`, sharded by layer.

    Every rank holds all K gradients (the usual data-parallel layout after a gather of the
    per-worker effective gradients, or K local microbatches); rank r reduces the
    segments of partition r only, then the partitions are all-gathered so every rank ends
    with the full result.  `reduce_fn(grads, offsets, out)` runs one partition (default:
    the CUDA library); the result equals a single unsharded call segment by segment.
    """
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    offs = np.asarray(seg_offsets, dtype=np.int64)
    n = int(offs[-1])
    es = grads[0].element_size()
    bounds = partition_segments(offs, world, es * len(grads))
    lo_s, hi_s = bounds[rank], bounds[rank + 1]
    lo, hi = int(offs[lo_s]), int(offs[hi_s])
    if out is None:
        out = torch.empty(n, dtype=grads[0].dtype, device=grads[0].device)
    reduce_fn = reduce_fn or _default_reduce
    if hi > lo:
        part = [g[lo:hi] for g in grads]
        sub = offs[lo_s:hi_s + 1] - lo
        reduce_fn(part, sub, out[lo:hi])
    # all-gather the partitions: pad every rank's piece to the longest, gather, trim.
    # gloo gathers host tensors, so device results travel through host copies there.
    sizes = [int(offs[bounds[r + 1]] - offs[bounds[r]]) for r in range(world)]
    width = max(max(sizes), 1)
    via_host = out.device.type == "cuda" and dist.get_backend(group) == "gloo"
    gdev = torch.device("cpu") if via_host else out.device
    piece = torch.zeros(width, dtype=out.dtype, device=gdev)
    piece[: hi - lo] = out[lo:hi].to(gdev)
    gathered = [torch.empty_like(piece) for _ in range(world)]
    dist.all_gather(gathered, piece, group=group)
    for r in range(world):
        a, b = int(offs[bounds[r]]), int(offs[bounds[r + 1]])
        out[a:b] = gathered[r][: b - a].to(out.device)
    return out
