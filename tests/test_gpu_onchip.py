"""The small-segment kernels (adasum_onchip.cuh): one segment per CTA or thread-block
cluster, held in shared memory, the whole tree on chip; and segments of at most 32
positions one warp each, the tree on the values in double-float arithmetic.

Plain reductions send every segment of at most 32 positions to the warp kernel and, for
up to 64 workers and when small segments are numerous, every segment that fits in a
cluster's shared memory to the on-chip kernel; the rest take the tiled route.  (The
tests here force the on-chip kernel for every small segment and allow clusters of 16.)  These tests pick segment lengths around each
cluster-size boundary (1, 2, 4, 8, 16 CTAs), unaligned starts, padded worker counts,
nearly cancelling sets (the on-chip recompute), segments mixed with tiled ones, and
compare with the fp64 oracle at the stated tolerances.
"""
import numpy as np
import pytest
import torch

import adaptive_gradient_summation_gb300 as ags
from adaptive_gradient_summation_gb300 import workloads
from parity import check_against_oracle, oracle_reduce, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DATA_BYTES = 80 * 1024  # shared memory per CTA for the K x P block (fp32-sized slots)
TINY = 32               # segments up to this length: one warp each, double-float


@pytest.fixture(autouse=True)
def _onchip_for_every_small_segment(monkeypatch, hooks):
    """By default the library uses the on-chip kernel only when small segments are
    numerous (thousands); these tests use it for every small segment, with clusters of
    up to 16 CTAs (switches honoured by the test build of the library)."""
    monkeypatch.setenv("ADASUM_ONCHIP", "force")
    monkeypatch.setenv("ADASUM_ONCHIP_MAX_CLUSTER", "16")


def positions_per_cta(K):
    return DATA_BYTES // (4 * K)


def rand_grads(K, n, dtype, seed, corr=0.6):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    s = torch.randn(n, generator=gen, device=DEV)
    return [(corr * s + (1 - corr * corr) ** 0.5 * torch.randn(n, generator=gen, device=DEV)).to(dtype)
            for _ in range(K)]


def boundary_lengths(K, vw):
    """Lengths just below and above the capacity of 1, 2, 4, 8 and 16 CTAs."""
    cap = positions_per_cta(K)
    out = [1, 2, 3, vw - 1, vw + 1, 37]
    for c in (1, 2, 4, 8, 16):
        out += [c * cap - 2 * vw - 3, c * cap - vw + 1]
    out += [c * cap + 5 for c in (1, 2, 4, 8)]
    return [n for n in out if n > 0]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K", [2, 4, 8, 16, 32, 64])
def test_cluster_size_boundaries(native, K, dtype):
    vw = 4 if dtype == torch.float32 else 8
    lengths = boundary_lengths(K, vw)
    offs = workloads.offsets_from_numels(lengths)
    grads = rand_grads(K, int(offs[-1]), dtype, seed=700 + K)
    out = ags.reduce(grads, offs)
    torch.cuda.synchronize()
    check_against_oracle(grads, offs, out)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K", [3, 5, 12, 24, 48])
def test_padded_worker_counts(native, K, dtype):
    lengths = [1, 9, 333, 2049, 7000]
    offs = workloads.offsets_from_numels(lengths)
    grads = rand_grads(K, int(offs[-1]), dtype, seed=720 + K)
    out = ags.reduce(grads, offs)
    torch.cuda.synchronize()
    check_against_oracle(grads, offs, out)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_unaligned_buffers(native, dtype):
    """Gradients at an odd element offset: no bulk copies, every element loaded alone."""
    K, lengths = 16, [5, 300, 1281, 4000]
    offs = workloads.offsets_from_numels(lengths)
    n = int(offs[-1])
    base = rand_grads(K, n + 1, dtype, seed=731)
    grads = [g[1:] for g in base]
    out_buf = torch.empty(n + 1, dtype=dtype, device=DEV)
    out = out_buf[1:]
    ags.reduce(grads, offs, out=out)
    torch.cuda.synchronize()
    check_against_oracle(grads, offs, out)


@pytest.mark.parametrize("K", [16, 64])
def test_mixed_with_tiled_segments(native, monkeypatch, K):
    """A segment too long for 16 CTAs between small ones: all three routes in one call,
    and the same answers (within tolerance) with the small-segment kernels switched off."""
    cap = positions_per_cta(K)
    lengths = [7, 16 * cap + 1000, 300, cap * 3, 1]
    offs = workloads.offsets_from_numels(lengths)
    grads = rand_grads(K, int(offs[-1]), torch.float32, seed=740 + K)
    on = ags.reduce(grads, offs)
    torch.cuda.synchronize()
    ref = oracle_reduce(grads, offs)
    check_against_oracle(grads, offs, on, ref=ref)
    monkeypatch.setenv("ADASUM_ONCHIP", "0")
    monkeypatch.setenv("ADASUM_TINY", "0")
    off = ags.reduce(grads, offs)
    torch.cuda.synchronize()
    check_against_oracle(grads, offs, off, ref=ref)
    assert not torch.equal(on, off)  # the switch really changes the route


def _cancelling_set(K, n, dtype, seed, eps=1e-3):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    out = []
    for _ in range(K // 2):
        a = torch.randn(n, generator=gen, device=DEV)
        b = -(1 - eps) * a + eps * 0.1 * torch.randn(n, generator=gen, device=DEV)
        out += [a.to(dtype), b.to(dtype)]
    return out


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K", [4, 16, 64])
def test_cancelling_segments_recomputed_on_chip(native, K, dtype):
    """Every segment nearly cancels at level 0, so every one above 32 positions is
    recomputed; the lengths span one CTA and clusters of several."""
    cap = positions_per_cta(K)
    lengths = [1, 3, 40, cap - 5, 2 * cap + 7, 5 * cap]
    offs = workloads.offsets_from_numels(lengths)
    grads = _cancelling_set(K, int(offs[-1]), dtype, seed=760 + K)
    out = ags.reduce(grads, offs)
    torch.cuda.synchronize()
    check_against_oracle(grads, offs, out)
    # segments of at most 32 positions take the warp kernel, which has no fast pass
    assert ags.recomputed_segments() == sum(n > TINY for n in lengths)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_segments_flagged_at_the_top_tree(native, dtype):
    """More one-CTA segments than CTAs fit at once (each CTA then loads its next segment
    while it finishes the current one), some of them cancelling only at the last level:
    workers 0-31 near +s, workers 32-63 near -(1 - 1e-3) s.  Those are flagged by the
    top tree, after the next segment's rows were issued, and recomputed from reloaded
    rows; every segment must match the oracle."""
    K = 64
    rs = np.random.default_rng(781)
    lengths = [int(n) for n in rs.integers(33, positions_per_cta(K) + 1, size=700)]
    offs = workloads.offsets_from_numels(lengths)
    n = int(offs[-1])
    gen = torch.Generator(device=DEV).manual_seed(782)
    s_ = torch.randn(n, generator=gen, device=DEV)
    top = torch.zeros(n, dtype=torch.bool, device=DEV)
    cancelling = [i for i in range(len(lengths)) if i % 7 == 3]
    for i in cancelling:
        top[offs[i]:offs[i + 1]] = True
    grads = []
    for k in range(K):
        z = torch.randn(n, generator=gen, device=DEV)
        sign = 1.0 if k < K // 2 else -(1 - 1e-3)
        grads.append(torch.where(top, sign * s_ + 0.01 * z, 0.6 * s_ + 0.8 * z).to(dtype))
    out = ags.reduce(grads, offs)
    torch.cuda.synchronize()
    check_against_oracle(grads, offs, out)
    assert ags.recomputed_segments() >= len(cancelling)
    assert ags.get_last_error() == ags.Status.OK


def test_recompute_pair_is_bitwise_symmetric(native):
    """The on-chip recompute keeps the pair operator's exact commutativity."""
    a, b = _cancelling_set(2, 3000, torch.float32, seed=771)
    offs = [0, 1000, 3000]
    ab = ags.reduce([a, b], offs)
    ba = ags.reduce([b, a], offs)
    torch.cuda.synchronize()
    assert torch.equal(ab, ba)


def test_small_segment_set_subset(native):
    """A 1/8 slice of the 10,000-segment K = 64 set: orthogonal segments exact, the rest
    within tolerance."""
    wl = workloads.make("small_segments_k64", device=DEV, shrink=8)
    out = ags.reduce(wl.grads, wl.seg_offsets)
    torch.cuda.synchronize()
    check_against_oracle(wl.grads, wl.seg_offsets, out)
    got = to_f64(out)
    for s in np.nonzero(wl.seg_kind == workloads.KIND_ORTHOGONAL)[0]:
        lo, hi = int(wl.seg_offsets[s]), int(wl.seg_offsets[s + 1])
        exact = sum(to_f64(g[lo:hi]) for g in wl.grads)
        assert np.array_equal(got[lo:hi], exact), s


def test_bulk_copy_wait_reports_timeout(native, monkeypatch):
    """16 bulk-copy bytes that never arrive (injected on the host) end the wait after its
    clock budget with a status, and the context stays usable."""
    grads = rand_grads(8, 5000, torch.float32, seed=780)
    offs = [0, 1000, 5000]
    assert ags.get_last_error() == ags.Status.OK
    monkeypatch.setenv("ADASUM_FAULT_INJECT", "timeout")
    ags.reduce(grads, offs)
    torch.cuda.synchronize()
    assert ags.get_last_error() == ags.Status.ERR_TIMEOUT
    monkeypatch.delenv("ADASUM_FAULT_INJECT")
    out = ags.reduce(grads, offs)
    torch.cuda.synchronize()
    assert ags.get_last_error() == ags.Status.OK
    check_against_oracle(grads, offs, out)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K", [2, 4, 7, 16, 32, 64, 128, 256])
def test_tiny_segments_one_warp_each(native, K, dtype):
    """Lengths 1..32 (and 33, just past the warp kernel) at every worker count, including
    those above the on-chip kernel's 64."""
    lengths = list(range(1, 34)) * 3
    offs = workloads.offsets_from_numels(lengths)
    grads = rand_grads(K, int(offs[-1]), dtype, seed=790 + K, corr=0.3)
    out = ags.reduce(grads, offs)
    torch.cuda.synchronize()
    check_against_oracle(grads, offs, out)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_tiny_kernels_agree_bitwise(native, dtype):
    """Up to 64 workers the warp kernel holds every value in registers; above, it reads
    the leaves in turn.  64 more zero workers add a zero right subtree, and Adasum(x, 0) =
    x exactly, so 128 workers must reproduce the 64-worker bits."""
    lengths = list(range(1, 33)) * 4
    offs = workloads.offsets_from_numels(lengths)
    grads = rand_grads(64, int(offs[-1]), dtype, seed=797, corr=0.5)
    zeros = [torch.zeros_like(grads[0]) for _ in range(64)]
    a = ags.reduce(grads, offs)
    b = ags.reduce(grads + zeros, offs)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    check_against_oracle(grads, offs, a)


def test_tiny_segments_pair_symmetry_and_special_cases(native):
    """Adasum(a, b) == Adasum(b, a) bitwise, Adasum(g, g) == g, Adasum(g, 0) == g and
    disjoint supports give the exact sum, on segments of the warp kernel."""
    n = 20 * 16
    offs = np.arange(0, n + 1, 16, dtype=np.int64)
    a, b = rand_grads(2, n, torch.float32, seed=795, corr=0.2)
    assert torch.equal(ags.reduce([a, b], offs), ags.reduce([b, a], offs))
    assert torch.equal(ags.reduce([a, a.clone()], offs), a)
    assert torch.equal(ags.reduce([a, torch.zeros_like(a)], offs), a)
    mask = (torch.arange(n, device=DEV) % 3 == 0)
    x, y = torch.where(mask, a, 0.0), torch.where(mask, 0.0, b)
    assert torch.equal(ags.reduce([x, y], offs), x + y)


@pytest.mark.parametrize("scale", [1e-20, 1e15])
def test_tiny_segments_extreme_magnitudes(native, scale):
    """The warp kernel scales each segment by a power of two before squaring, so values
    whose squares fall outside fp32's range still combine correctly."""
    lengths = [1, 5, 17, 32]
    offs = workloads.offsets_from_numels(lengths)
    grads = [g * scale for g in rand_grads(8, int(offs[-1]), torch.float32, seed=797, corr=0.4)]
    out = ags.reduce(grads, offs)
    torch.cuda.synchronize()
    check_against_oracle(grads, offs, out)


@pytest.mark.parametrize("scale", [1e-22, 1e25])
@pytest.mark.parametrize("K", [4, 16, 64])
def test_onchip_fast_pass_extreme_magnitudes(native, K, scale):
    """Small segments held on chip whose squares leave fp32's range: the fast pass's
    range check (a worker with a nonzero value and a squared norm below n 2^-96 or above
    2^80, over the cluster) sends them to the
    recompute, which scales them by a power of two first."""
    lengths = [40, 300, 1000, 2 * positions_per_cta(K) + 7]
    offs = workloads.offsets_from_numels(lengths)
    grads = [g * scale for g in rand_grads(K, int(offs[-1]), torch.float32, seed=960 + K, corr=0.4)]
    out = ags.reduce(grads, offs)
    torch.cuda.synchronize()
    check_against_oracle(grads, offs, out)
    assert ags.recomputed_segments() == len(lengths)


@pytest.mark.parametrize("K", [2, 16])
def test_flagged_tiled_segments(native, monkeypatch, K):
    """Segments that take the tiled route and get flagged: those that fit 16 CTAs are
    recomputed by the on-chip kernel, a longer one by the fp64 path; both within
    tolerance."""
    monkeypatch.setenv("ADASUM_ONCHIP", "1")     # the default routing (few segments: tiled)
    cap16 = 16 * positions_per_cta(K)
    lengths = [cap16 + 999, 5000, 700]
    offs = workloads.offsets_from_numels(lengths)
    grads = _cancelling_set(K, int(offs[-1]), torch.float32, seed=800 + K)
    out = ags.reduce(grads, offs)
    torch.cuda.synchronize()
    check_against_oracle(grads, offs, out)
    assert ags.recomputed_segments() == len(lengths)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K", [4, 16, 64])
def test_flagged_segments_share_the_recompute_clusters(native, monkeypatch, K, dtype):
    """With the fast pass off every segment is tiled; nearly cancelling ones are all
    recomputed in one launch of the largest clusters.  Short segments leave some CTAs of
    their cluster without a vector, and there are more flagged segments than clusters fit
    on the device, so each cluster works through several list entries in turn."""
    monkeypatch.setenv("ADASUM_ONCHIP", "1")
    monkeypatch.setenv("ADASUM_ONCHIP_FAST", "0")
    rs = np.random.default_rng(900 + K)
    cap16 = 16 * positions_per_cta(K)
    lengths = [33, 40, 47, 61, 100, 257, cap16 - 9, cap16] + list(rs.integers(33, 3 * TINY * 16, size=300))
    offs = workloads.offsets_from_numels(lengths)
    grads = _cancelling_set(K, int(offs[-1]), dtype, seed=910 + K)
    out = ags.reduce(grads, offs)
    torch.cuda.synchronize()
    check_against_oracle(grads, offs, out)
    assert ags.recomputed_segments() == len(lengths)
    again = ags.reduce(grads, offs)
    torch.cuda.synchronize()
    assert torch.equal(out, again)  # the order clusters take the entries in is not visible


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_in_place_output(native, dtype):
    """out may be one of the gradients: every kernel reads a segment's inputs before it
    writes that segment's output (the recompute rereads level-0 inputs, which the fast
    pass left untouched)."""
    K = 16
    cap = positions_per_cta(K)
    lengths = [5, 32, 300, cap + 9, 3 * cap]
    offs = workloads.offsets_from_numels(lengths)
    n = int(offs[-1])
    for grads in (rand_grads(K, n, dtype, seed=810), _cancelling_set(K, n, dtype, seed=811)):
        keep = [g.clone() for g in grads]
        ags.reduce(grads, offs, out=grads[5])
        torch.cuda.synchronize()
        check_against_oracle(keep, offs, grads[5])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K", [8, 64, 256])
def test_wide_tiny_segments(native, K, dtype):
    """Hundreds of segments of 33..128 positions next to tiny and larger ones."""
    rs = np.random.default_rng(830 + K)
    lengths = list(rs.integers(33, 129, size=400)) + [1, 32, 64, 65, 128, 129, 2000]
    offs = workloads.offsets_from_numels(lengths)
    grads = rand_grads(K, int(offs[-1]), dtype, seed=831 + K, corr=0.4)
    out = ags.reduce(grads, offs)
    torch.cuda.synchronize()
    check_against_oracle(grads, offs, out)


def test_wide_tiny_segments_cancelling_and_symmetric(native):
    rs = np.random.default_rng(840)
    lengths = list(rs.integers(33, 129, size=400))
    offs = workloads.offsets_from_numels(lengths)
    n = int(offs[-1])
    grads = _cancelling_set(16, n, torch.float32, seed=841)
    out = ags.reduce(grads, offs)
    torch.cuda.synchronize()
    check_against_oracle(grads, offs, out)
    a, b = grads[0], grads[1]
    assert torch.equal(ags.reduce([a, b], offs), ags.reduce([b, a], offs))
    assert torch.equal(ags.reduce(grads[8:] + grads[:8], offs), out)   # sibling swap
