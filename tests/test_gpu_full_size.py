"""Parity at full size, in the launch configuration bench.py times.

Every workload runs at its full size through the same entry points as the benchmark.
Segments are combined independently, so the oracle checks a sample of whole segments
(the smallest, the largest, the first, the last and a few seeded random ones) on its
own; the small-segment set (10,000 segments, K = 64) is checked in full.
"""
import numpy as np
import pytest
import torch

import adaptive_gradient_summation_gb300 as ags
import oracle
from adaptive_gradient_summation_gb300 import workloads
from parity import (check_bf16_elements, check_fp32_segments, check_momentum, to_f64,
                    to_oracle_input)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def sample_segments(offs, n_random=3, seed=0):
    lens = np.diff(offs)
    nz = np.nonzero(lens)[0]
    picks = {int(nz[np.argmin(lens[nz])]), int(np.argmax(lens)), int(nz[0]), int(nz[-1])}
    rs = np.random.default_rng(seed)
    picks |= set(int(x) for x in rs.choice(nz, size=min(n_random, nz.size), replace=False))
    return sorted(picks)


def oracle_on_segment(grads, lo, hi, want_mag):
    sub = [to_oracle_input(g[lo:hi]) for g in grads]
    return oracle.adasum_reduce(sub, [0, hi - lo], want_mag=want_mag)


@pytest.mark.parametrize("name", ["resnet50_k8", "bert_large_k16"])
def test_full_size_sampled_segments(native, name):
    wl = workloads.make(name, device=DEV)
    out = torch.empty_like(wl.grads[0])
    ags.reduce(wl.grads, wl.seg_offsets, out=out)
    torch.cuda.synchronize()
    bf16 = wl.dtype == torch.bfloat16
    for s in sample_segments(wl.seg_offsets):
        lo, hi = int(wl.seg_offsets[s]), int(wl.seg_offsets[s + 1])
        ref = oracle_on_segment(wl.grads, lo, hi, want_mag=bf16)
        got = to_f64(out[lo:hi])
        if bf16:
            check_bf16_elements(got, ref["out64"], ref["mag"], wl.K, what=f"segment {s}")
        else:
            check_fp32_segments(got, ref["out64"], [0, hi - lo], what=f"segment {s}")


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
def test_full_size_momentum_sampled_segments(native, init):
    wl = workloads.make("gpt_k8_momentum", device=DEV, momentum_init=init)
    segs = sample_segments(wl.seg_offsets, n_random=2)
    keep_w = {s: wl.master_w[int(wl.seg_offsets[s]):int(wl.seg_offsets[s + 1])].cpu().numpy()
              for s in segs}
    keep_v = {s: wl.momentum[int(wl.seg_offsets[s]):int(wl.seg_offsets[s + 1])].cpu().numpy()
              for s in segs}
    out = torch.empty_like(wl.grads[0])
    ags.reduce_momentum_sgd(wl.grads, wl.seg_offsets, wl.master_w, wl.momentum,
                            lr=wl.lr, mu=wl.mu, out=out)
    torch.cuda.synchronize()
    lr32, mu32 = float(np.float32(wl.lr)), float(np.float32(wl.mu))
    for s in segs:
        lo, hi = int(wl.seg_offsets[s]), int(wl.seg_offsets[s + 1])
        ref = oracle_on_segment(wl.grads, lo, hi, want_mag=True)
        check_bf16_elements(to_f64(out[lo:hi]), ref["out64"], ref["mag"], wl.K,
                            what=f"segment {s}")
        w_ref, v_ref = oracle.momentum_sgd(ref["out64"], keep_w[s], keep_v[s], lr32, mu32)
        check_momentum(wl.master_w[lo:hi], wl.momentum[lo:hi], w_ref, v_ref, [0, hi - lo], wl.lr)
