"""The L2-reuse route (one persistent kernel; the combine re-reads each unit in reverse a
few tens of MB after its Gram, so the second read comes from L2), on the test build
with the route switched on (ADASUM_REUSE=1), against the fp64 oracle.

Layouts: BERT-Large-shaped sets (shrunk and at a quarter size), random mixes of long and
short segments (segments that span many steps and CTAs, units of many small segments,
empty segments, segments taken by the small-segment kernels), unaligned pointers,
8 and 16 workers; results deterministic across calls; nearly cancelling segments are
flagged and recomputed.
"""
import numpy as np
import pytest
import torch

import adaptive_gradient_summation_gb300 as ags
from adaptive_gradient_summation_gb300 import workloads
from parity import check_against_oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _reuse_on(hooks, monkeypatch):
    monkeypatch.setenv("ADASUM_REUSE", "1")


def _launched(name_prefix):
    stats = ags.profile_collect()
    return any(k.startswith(name_prefix) for k in stats)


def _grads(K, n, seed, shift=0):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    s = torch.randn(n + shift, generator=gen, device=DEV)
    out = []
    for k in range(K):
        rho = 0.3 + 0.05 * (k % 8)
        z = torch.randn(n + shift, generator=gen, device=DEV)
        out.append((rho * s + (1 - rho * rho) ** 0.5 * z).to(torch.bfloat16)[shift:])
    return out


@pytest.mark.parametrize("shrink", [64, 16, 4])
def test_reuse_bert_shapes(native, shrink):
    wl = workloads.make("bert_large_k16", device=DEV, shrink=shrink)
    ags.profile_enable(True)
    out = ags.reduce(wl.grads, wl.seg_offsets)
    torch.cuda.synchronize()
    assert _launched("reuse<bf16,16>")
    ags.profile_enable(False)
    assert ags.get_last_error() == ags.Status.OK
    check_against_oracle(wl.grads, wl.seg_offsets, out)
    again = ags.reduce(wl.grads, wl.seg_offsets)
    torch.cuda.synchronize()
    assert torch.equal(out, again)


@pytest.mark.parametrize("K", [8, 16])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_reuse_random_layouts(native, K, seed):
    rs = np.random.default_rng(seed)
    lengths = []
    for _ in range(40):
        kind = rs.integers(0, 4)
        if kind == 0:
            lengths.append(int(rs.integers(0, 40)))          # empty / tiny (warp kernel)
        elif kind == 1:
            lengths.append(int(rs.integers(40, 5000)))       # short
        elif kind == 2:
            lengths.append(int(rs.integers(5000, 300_000)))  # medium
        else:
            lengths.append(int(rs.integers(300_000, 3_000_000)))  # spans several steps
    offs = workloads.offsets_from_numels(lengths)
    grads = _grads(K, int(offs[-1]), seed=100 + seed, shift=seed % 2)
    out = ags.reduce(grads, offs)
    torch.cuda.synchronize()
    assert ags.get_last_error() == ags.Status.OK
    check_against_oracle(grads, offs, out)
    assert torch.equal(out, ags.reduce(grads, offs))


def test_reuse_small_units_and_steps(native, monkeypatch):
    """Tiny units, steps and lag: many steps per segment, combines soon after the Gram."""
    monkeypatch.setenv("ADASUM_REUSE_UNIT_MB", "1")
    monkeypatch.setenv("ADASUM_REUSE_STEP_MB", "1")
    monkeypatch.setenv("ADASUM_REUSE_LAG_MB", "1")
    monkeypatch.setenv("ADASUM_REUSE_KEEP_MB", "1")
    lengths = [1_000_003, 7, 0, 65_536, 300_001, 33, 2_000_000]
    offs = workloads.offsets_from_numels(lengths)
    grads = _grads(16, int(offs[-1]), seed=7)
    out = ags.reduce(grads, offs)
    torch.cuda.synchronize()
    assert ags.get_last_error() == ags.Status.OK
    check_against_oracle(grads, offs, out)


def test_reuse_flagged_segments_are_recomputed(native):
    """Nearly opposite pairs: the finisher flags every segment, the combine skips them,
    and the recompute path (on chip and fp64) writes them."""
    gen = torch.Generator(device=DEV).manual_seed(5)
    lengths = [400_001, 5_000, 70_000]
    offs = workloads.offsets_from_numels(lengths)
    n = int(offs[-1])
    grads = []
    for _ in range(8):
        a = torch.randn(n, generator=gen, device=DEV)
        grads += [a.to(torch.bfloat16),
                  (-(1 - 1e-2) * a + 1e-3 * torch.randn(n, generator=gen, device=DEV)).to(torch.bfloat16)]
    out = ags.reduce(grads, offs)
    torch.cuda.synchronize()
    check_against_oracle(grads, offs, out)
    assert ags.recomputed_segments() == len(lengths)


def test_reuse_and_default_route_both_match_the_oracle(native, monkeypatch):
    wl = workloads.make("bert_large_k16", device=DEV, shrink=32)
    reuse = ags.reduce(wl.grads, wl.seg_offsets).clone()
    monkeypatch.setenv("ADASUM_REUSE", "0")
    tiled = ags.reduce(wl.grads, wl.seg_offsets)
    torch.cuda.synchronize()
    check_against_oracle(wl.grads, wl.seg_offsets, reuse)
    check_against_oracle(wl.grads, wl.seg_offsets, tiled)
