"""CPU checks of the seeded input generators (adaptive_gradient_summation_gb300/workloads.py):
the model-shaped sets have the architectures' tensor counts and sizes, and the
10,000-segment set has the structure its special segments claim (no GPU)."""
import numpy as np
import torch

from adaptive_gradient_summation_gb300 import workloads


def test_model_shapes():
    for numels, count, total in ((workloads.resnet50_numels(), 161, 25_557_032),
                                 (workloads.bert_large_numels(), 391, 335_141_888),
                                 (workloads.gpt_numels(), 195, 1_311_182_848)):
        assert len(numels) == count
        assert sum(numels) == total
        offs = workloads.offsets_from_numels(numels)
        assert offs[0] == 0 and offs[-1] == total and np.all(np.diff(offs) >= 0)


def test_generators_are_seeded():
    a = workloads.make("resnet50_k8", shrink=512)
    b = workloads.make("resnet50_k8", shrink=512)
    assert all(torch.equal(x, y) for x, y in zip(a.grads, b.grads))


def test_small_segment_set_structure():
    wl = workloads.make("small_segments_k64", shrink=8)
    offs, kind = wl.seg_offsets, wl.seg_kind
    lens = np.diff(offs)
    assert wl.K == 64 and wl.L == 1250
    assert lens.min() >= 1 and lens.max() <= 4096
    g = torch.stack(wl.grads).numpy()  # [K, N]
    zero_everywhere = 0
    for s in range(wl.L):
        x = g[:, offs[s]:offs[s + 1]]
        if kind[s] == workloads.KIND_ORTHOGONAL:
            # every position is nonzero on at most one worker: disjoint supports
            assert np.all((x != 0).sum(axis=0) <= 1), s
        elif kind[s] == workloads.KIND_PARALLEL:
            # every worker is a positive power-of-two multiple of the first
            r = x / x[0]
            ratios = r[:, 0]
            assert np.all(np.isin(ratios, [2.0 ** j for j in range(-4, 5)])), s
            assert np.array_equal(r, np.broadcast_to(ratios[:, None], r.shape)), s
        elif kind[s] == workloads.KIND_ZERO_SOME:
            zero_rows = np.all(x == 0, axis=1)
            assert zero_rows.any(), s
            zero_everywhere += int(zero_rows.all())
    assert zero_everywhere == 1
    frac = {k: float(np.mean(kind == k)) for k in (workloads.KIND_ZERO_SOME, workloads.KIND_PARALLEL,
                                                    workloads.KIND_ORTHOGONAL)}
    assert all(0.02 < f < 0.09 for f in frac.values()), frac
