"""Parity at full size, in the launch configuration bench.py times, on EVERY segment.

Every workload runs at its full size through the same entry points as the benchmark,
and every one of its segments is compared with the fp64 oracle (the paper combines each
layer on its own, so the oracle runs segment by segment): ResNet-50 K=8 (161 segments,
25.6M positions), BERT-Large K=16 (391 segments, 335M positions, bf16), the GPT set
K=8 with the fused Momentum-SGD step (195 segments, 1.31B positions, bf16; zero and
seeded momentum) and the 10,000-segment K=64 set.

The oracle is plain single-threaded C called through ctypes, which releases the GIL, so
segments are spread over a pool of host threads (no process is forked after the GPU is
initialised).  A byte budget bounds how much oracle scratch is live at once.
"""
import concurrent.futures
import os
import threading

import numpy as np
import pytest
import torch

import adaptive_gradient_summation_gb300 as ags
import oracle
from adaptive_gradient_summation_gb300 import workloads
from parity import (FP32_RTOL, check_bf16_elements, check_fp32_segments, to_f64,
                    to_oracle_input)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _mem_available_bytes() -> int:
    try:
        with open("/proc/meminfo") as fh:
            for line in fh:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def _need_host_memory(nbytes: int):
    avail = _mem_available_bytes()
    if avail and avail < nbytes:
        pytest.skip(f"needs about {nbytes / 2**30:.0f} GiB of host memory, "
                    f"{avail / 2**30:.0f} GiB available")


class _ByteGate:
    """At most `budget` bytes of oracle scratch in flight (a task larger than the budget
    runs alone)."""

    def __init__(self, budget: int):
        self.budget, self.used = budget, 0
        self.cv = threading.Condition()

    def take(self, n: int):
        with self.cv:
            while self.used > 0 and self.used + n > self.budget:
                self.cv.wait()
            self.used += n

    def give(self, n: int):
        with self.cv:
            self.used -= n
            self.cv.notify_all()


def for_every_segment(offs, K, fn, bytes_per_pos):
    """Runs fn(s, lo, hi) for every nonempty segment on a thread pool (largest first);
    returns the results by segment."""
    lens = np.diff(offs)
    segs = sorted((int(s) for s in np.nonzero(lens)[0]), key=lambda s: -int(lens[s]))
    gate = _ByteGate(max(4 << 30, min(_mem_available_bytes() // 3, 64 << 30)))
    workers = max(1, min(32, os.cpu_count() or 1))

    def task(s):
        lo, hi = int(offs[s]), int(offs[s + 1])
        need = (hi - lo) * bytes_per_pos
        gate.take(need)
        try:
            return s, fn(s, lo, hi)
        finally:
            gate.give(need)

    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        return dict(ex.map(task, segs))


def _host(t: torch.Tensor) -> np.ndarray:
    return to_oracle_input(t)


def _values(host: np.ndarray) -> np.ndarray:
    """fp64 values of host data: float32, or bf16 bits (exact widening)."""
    if host.dtype == np.uint16:
        return (host.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return host.astype(np.float64)


@pytest.mark.parametrize("name", ["resnet50_k8", "bert_large_k16"])
def test_full_size_every_segment(native, name):
    wl = workloads.make(name, device=DEV)
    _need_host_memory(wl.K * wl.N * wl.grads[0].element_size() + 8 * wl.N + (8 << 30))
    out = torch.empty_like(wl.grads[0])
    ags.reduce(wl.grads, wl.seg_offsets, out=out)
    torch.cuda.synchronize()
    assert ags.recomputed_segments() == 0
    bf16 = wl.dtype == torch.bfloat16
    grads = [_host(g) for g in wl.grads]
    got = _host(out)
    del wl.grads

    def check(s, lo, hi):
        ref = oracle.adasum_reduce([g[lo:hi] for g in grads], [0, hi - lo], want_mag=bf16)
        if bf16:
            return check_bf16_elements(_values(got[lo:hi]), ref["out64"], ref["mag"], wl.K,
                                       what=f"{name} segment {s}")
        return check_fp32_segments(_values(got[lo:hi]), ref["out64"], [0, hi - lo],
                                   what=f"{name} segment {s}")

    worst = for_every_segment(wl.seg_offsets, wl.K, check, 24 * wl.K)
    assert len(worst) == wl.L


def test_full_size_small_segments_everything(native):
    wl = workloads.make("small_segments_k64", device=DEV)
    out = ags.reduce(wl.grads, wl.seg_offsets)
    torch.cuda.synchronize()
    ref = oracle.adasum_reduce([to_oracle_input(g) for g in wl.grads], wl.seg_offsets)
    check_fp32_segments(to_f64(out), ref["out64"], wl.seg_offsets)
    # the categories that must be exact: all-zero segments and disjoint supports
    got = to_f64(out)
    for s in np.nonzero(wl.seg_kind == workloads.KIND_ORTHOGONAL)[0]:
        lo, hi = int(wl.seg_offsets[s]), int(wl.seg_offsets[s + 1])
        exact = sum(to_f64(g[lo:hi]) for g in wl.grads)
        assert np.array_equal(got[lo:hi], exact), s


@pytest.mark.parametrize("init", ["zero", "random"])
def test_full_size_momentum_every_segment(native, init):
    wl = workloads.make("gpt_k8_momentum", device=DEV, momentum_init=init)
    _need_host_memory(wl.K * wl.N * 2 + 18 * wl.N + (8 << 30))
    w0 = wl.master_w.cpu().numpy()
    v0 = wl.momentum.cpu().numpy()
    out = torch.empty_like(wl.grads[0])
    ags.reduce_momentum_sgd(wl.grads, wl.seg_offsets, wl.master_w, wl.momentum,
                            lr=wl.lr, mu=wl.mu, out=out)
    torch.cuda.synchronize()
    grads = [_host(g) for g in wl.grads]
    del wl.grads
    got = _host(out)
    w1 = wl.master_w.cpu().numpy()
    v1 = wl.momentum.cpu().numpy()
    lr32, mu32 = float(np.float32(wl.lr)), float(np.float32(wl.mu))

    def check(s, lo, hi):
        ref = oracle.adasum_reduce([g[lo:hi] for g in grads], [0, hi - lo], want_mag=True)
        r = check_bf16_elements(_values(got[lo:hi]), ref["out64"], ref["mag"], wl.K,
                                what=f"gpt segment {s}")
        w_ref, v_ref = oracle.momentum_sgd(ref["out64"], w0[lo:hi], v0[lo:hi], lr32, mu32)
        nv = np.linalg.norm(v_ref.astype(np.float64))
        ev = np.linalg.norm(v1[lo:hi].astype(np.float64) - v_ref)
        assert ev <= FP32_RTOL * nv + 1e-30, f"momentum segment {s}: {ev:.3e} vs {nv:.3e}"
        ew = np.linalg.norm(w1[lo:hi].astype(np.float64) - w_ref)
        tol = (FP32_RTOL * wl.lr * nv + 2.0**-23 * np.linalg.norm(w_ref.astype(np.float64))
               + 1e-30)
        assert ew <= tol, f"weights segment {s}: {ew:.3e} > {tol:.3e}"
        return r

    worst = for_every_segment(wl.seg_offsets, wl.K, check, 24 * wl.K + 40)
    assert len(worst) == wl.L
