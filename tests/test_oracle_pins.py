"""Pins for the fp64 CPU oracle, against what the paper and mathematics fix.

Nothing here compares the oracle with itself.  The pins are:
  * hand-worked pair and tree values (exact rationals, derivation in the comments);
  * an independent exact-rational derivation of the operator from the two emulated
    sequential SGD paths ("Scaling Distributed Training with Adaptive Summation",
    Section 3, Equations 1-2, Appendix A.1-A.2), applied as a recursive binary tree;
  * the paper's stated special cases (tests/golden/paper_claims.txt): orthogonal inputs
    sum, parallel inputs average, the orthogonality metric is 1 for orthogonal sets and
    1/64 for 64 parallel equal-norm gradients, layers are combined independently;
  * algebraic identities: Adasum(g, g) = g, a zero operand gives a plain sum,
    commutativity, scale equivariance;
  * library routines: torch's fp32 -> bf16 rounding, torch.optim.SGD's momentum step.
"""
from fractions import Fraction
import os

import numpy as np
import pytest
import torch

from exact_adasum import (adasum_chain_exact, adasum_pair_exact, adasum_tree_exact,
                          adasum_tree_exact_padded, adasum_tree_exact_segments)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def f32(*vs):
    return [np.asarray(v, dtype=np.float32) for v in vs]


def claims():
    rows = {}
    with open(os.path.join(GOLDEN, "paper_claims.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            cid, cite, stmt = [x.strip() for x in line.split("|", 2)]
            rows[cid] = (cite, stmt)
    return rows


# --------------------------------------------------------------------- hand-worked values

HAND = [
    # a=(1,0), b=(1,1): a.b=1, |a|^2=1, |b|^2=2 -> alpha=1-1/2=1/2, beta=1-1/4=3/4
    #   -> (1/2)(1,0) + (3/4)(1,1) = (5/4, 3/4)
    ([[1, 0], [1, 1]], [Fraction(5, 4), Fraction(3, 4)]),
    # a=(3,-1,2), b=(1,2,0): a.b=1, |a|^2=14, |b|^2=5 -> alpha=27/28, beta=9/10
    #   -> (531/140, 117/140, 27/14)
    ([[3, -1, 2], [1, 2, 0]], [Fraction(531, 140), Fraction(117, 140), Fraction(27, 14)]),
    # tree over (1,0),(0,1),(1,1),(2,-1):
    #   level 0: (1,0),(0,1) orthogonal -> (1,1);  (1,1),(2,-1): a.b=1, alpha=3/4,
    #            beta=9/10 -> (51/20, -3/20)
    #   level 1: (1,1),(51/20,-3/20): a.b=12/5, |a|^2=2, |b|^2=261/40 -> alpha=2/5,
    #            beta=71/87 -> (1439/580, 161/580)
    ([[1, 0], [0, 1], [1, 1], [2, -1]], [Fraction(1439, 580), Fraction(161, 580)]),
]


@pytest.mark.parametrize("vectors,expected", HAND)
def test_hand_worked_values(oracle_mod, vectors, expected):
    # the independent derivation agrees with the hand calculation exactly ...
    assert adasum_tree_exact(vectors) == expected
    # ... and the oracle agrees with both to fp64 rounding
    r = oracle_mod.adasum_reduce(f32(*vectors), [0, len(vectors[0])])
    exp = np.array([float(x) for x in expected])
    np.testing.assert_allclose(r["out64"], exp, rtol=4e-16, atol=0)


# --------------------------------------------------- independent exact derivation (brute)

@pytest.mark.parametrize("K", [1, 2, 4, 8])
def test_matches_sequential_emulation_exactly(oracle_mod, K):
    rs = np.random.default_rng(1000 + K)
    for n in range(1, 18):
        for _ in range(3):
            vecs = [rs.integers(-3, 4, size=n).astype(np.float32) for _ in range(K)]
            if rs.random() < 0.3:                        # zero operands now and then
                vecs[int(rs.integers(0, K))][:] = 0
            exact = np.array([float(x) for x in adasum_tree_exact(vecs)])
            got = oracle_mod.adasum_reduce(vecs, [0, n])["out64"]
            nrm = np.linalg.norm(exact)
            if nrm == 0:
                assert np.all(got == 0)
            else:
                assert np.linalg.norm(got - exact) <= 1e-13 * nrm, (K, n, vecs)


def test_multi_segment_exact(oracle_mod):
    rs = np.random.default_rng(7)
    offs = [0, 3, 3, 10, 11, 20]                     # includes an empty segment
    vecs = [rs.integers(-4, 5, size=20).astype(np.float32) for _ in range(4)]
    exact = np.array([float(x) for x in adasum_tree_exact_segments(vecs, offs)])
    got = oracle_mod.adasum_reduce(vecs, offs)["out64"]
    np.testing.assert_allclose(got, exact, rtol=1e-14, atol=1e-14)


def test_tree_pairs_neighbours_not_halves(oracle_mod):
    """The tree pairs (2i, 2i+1).  Adasum is not associative, so pairing (i, i+K/2)
    gives another result -- the pin can tell the two apart."""
    vecs = [[1, 0, 0], [1, 2, 0], [0, 1, 3], [2, -1, 1]]
    neighbours = adasum_tree_exact(vecs)
    other = adasum_pair_exact(adasum_pair_exact(vecs[0], vecs[2]),
                              adasum_pair_exact(vecs[1], vecs[3]))
    assert neighbours != other
    got = oracle_mod.adasum_reduce(f32(*vecs), [0, 3])["out64"]
    np.testing.assert_allclose(got, [float(x) for x in neighbours], rtol=1e-15)
    assert not np.allclose(got, [float(x) for x in other], rtol=1e-6)


# ------------------------------------------------------------ the paper's special cases

def test_claims_file_lists_every_checked_claim():
    assert set(claims()) == {"orthogonal_sum", "parallel_average",
                             "orthogonality_orthogonal", "orthogonality_parallel_64",
                             "per_layer"}


def test_orthogonal_inputs_sum_bit_exact(oracle_mod):
    """claim orthogonal_sum: disjoint supports -> every dot is exactly 0 -> plain sum."""
    rs = np.random.default_rng(3)
    n, K = 257, 8
    owner = rs.integers(0, K, size=n)
    vals = rs.standard_normal(n).astype(np.float32)
    vecs = [np.where(owner == k, vals, 0).astype(np.float32) for k in range(K)]
    got = oracle_mod.adasum_reduce(vecs, [0, n])
    assert np.array_equal(got["out64"], vals.astype(np.float64))
    assert np.array_equal(got["out"], vals)


def test_orthogonal_nonaxis_pair(oracle_mod):
    """claim orthogonal_sum with overlapping supports: a.b = 0 exactly."""
    a, b = f32([1, 2, 3, 0], [2, -1, 0, 5])
    got = oracle_mod.adasum_reduce([a, b], [0, 4])["out64"]
    assert np.array_equal(got, (a.astype(np.float64) + b))


@pytest.mark.parametrize("c", [0.25, 0.5, 2.0, 4.0, -1.0, -0.5, 3.0])
def test_parallel_pair_averages(oracle_mod, c):
    """claim parallel_average: b = c a gives (a + b) / 2 (for c < 0 as well)."""
    rs = np.random.default_rng(11)
    a = rs.integers(-1000, 1001, size=33).astype(np.float32)   # c * a is exact in fp32
    b = (np.float32(c) * a).astype(np.float32)
    got = oracle_mod.adasum_reduce([a, b], [0, 33])["out64"]
    exp = (a.astype(np.float64) + b.astype(np.float64)) / 2
    np.testing.assert_allclose(got, exp, rtol=1e-15, atol=1e-300)


def test_parallel_tree_is_mean(oracle_mod):
    """Pairwise averages up a power-of-two tree give the plain mean of the scales."""
    rs = np.random.default_rng(5)
    s = rs.standard_normal(19).astype(np.float32)
    scales = np.ldexp(1.0, rs.integers(-2, 3, size=16))
    vecs = [(np.float32(c) * s).astype(np.float32) for c in scales]
    got = oracle_mod.adasum_reduce(vecs, [0, 19])["out64"]
    np.testing.assert_allclose(got, scales.mean() * s.astype(np.float64), rtol=1e-14)


def test_orthogonality_metric_claims(oracle_mod):
    """claims orthogonality_orthogonal (=1) and orthogonality_parallel_64 (=1/64)."""
    rs = np.random.default_rng(9)
    n, K = 640, 64
    owner = rs.integers(0, K, size=n)
    vals = rs.standard_normal(n).astype(np.float32)
    orth = [np.where(owner == k, vals, 0).astype(np.float32) for k in range(K)]
    r = oracle_mod.adasum_reduce(orth, [0, n], want_ortho=True)["ortho"]
    assert r[0] == pytest.approx(1.0, rel=1e-14)
    s = rs.standard_normal(n).astype(np.float32)
    par = [s.copy() for _ in range(K)]
    r = oracle_mod.adasum_reduce(par, [0, n], want_ortho=True)["ortho"]
    assert r[0] == pytest.approx(1.0 / 64, rel=1e-14)


def test_per_layer_independence(oracle_mod):
    """claim per_layer: one call over L segments equals L one-segment calls, bitwise."""
    rs = np.random.default_rng(13)
    offs = [0, 5, 17, 17, 64, 65]
    vecs = [rs.standard_normal(65).astype(np.float32) for _ in range(4)]
    whole = oracle_mod.adasum_reduce(vecs, offs)["out64"]
    parts = []
    for s in range(len(offs) - 1):
        lo, hi = offs[s], offs[s + 1]
        if hi > lo:
            parts.append(oracle_mod.adasum_reduce([v[lo:hi] for v in vecs],
                                                  [0, hi - lo])["out64"])
    assert np.array_equal(whole, np.concatenate(parts))


# ------------------------------------------------------------------ algebraic identities

def test_idempotent(oracle_mod):
    g = np.random.default_rng(1).standard_normal(100).astype(np.float32)
    got = oracle_mod.adasum_reduce([g, g.copy()], [0, 100])
    assert np.array_equal(got["out"], g)
    got = oracle_mod.adasum_reduce([g] * 8, [0, 100])
    assert np.array_equal(got["out"], g)


def test_zero_operand(oracle_mod):
    b = np.random.default_rng(2).standard_normal(50).astype(np.float32)
    z = np.zeros(50, np.float32)
    assert np.array_equal(oracle_mod.adasum_reduce([z, b], [0, 50])["out"], b)
    assert np.array_equal(oracle_mod.adasum_reduce([b, z], [0, 50])["out"], b)
    zz = oracle_mod.adasum_reduce([z, z, z, z], [0, 50])
    assert np.array_equal(zz["out64"], np.zeros(50)) and not np.any(np.isnan(zz["out64"]))


def test_commutative_bitwise(oracle_mod):
    rs = np.random.default_rng(4)
    a, b = (rs.standard_normal(77).astype(np.float32) for _ in range(2))
    ab = oracle_mod.adasum_reduce([a, b], [0, 77])["out64"]
    ba = oracle_mod.adasum_reduce([b, a], [0, 77])["out64"]
    assert np.array_equal(ab, ba)


@pytest.mark.parametrize("c", [0.125, 2.0, 1024.0])
def test_scale_equivariance(oracle_mod, c):
    rs = np.random.default_rng(6)
    vecs = [rs.standard_normal(40).astype(np.float32) for _ in range(4)]
    base = oracle_mod.adasum_reduce(vecs, [0, 40])["out64"]
    scaled = oracle_mod.adasum_reduce([(np.float32(c) * v).astype(np.float32) for v in vecs],
                                      [0, 40])["out64"]
    assert np.array_equal(scaled, c * base)


def test_magnitude_bound_dominates(oracle_mod):
    rs = np.random.default_rng(8)
    vecs = [rs.standard_normal(60).astype(np.float32) for _ in range(8)]
    r = oracle_mod.adasum_reduce(vecs, [0, 60], want_mag=True)
    assert np.all(r["mag"] >= np.abs(r["out64"]) * (1 - 1e-15))


# The magnitude bound m sizes the fp32 floor of every bf16 tolerance, so it is pinned
# exactly: at a pair, m = |alpha| m_a + |beta| m_b with m = |g| at the leaves.
MAG_HAND = [
    # a=(1,0), b=(1,1): alpha=1/2, beta=3/4 -> m = (1/2)(1,0) + (3/4)(1,1) = (5/4, 3/4)
    ([[1, 0], [1, 1]], [Fraction(5, 4), Fraction(3, 4)]),
    # a=(1,0), b=(3,1): a.b=3, |a|^2=1, |b|^2=10 -> alpha = 1 - 3/2 = -1/2 (negative),
    #   beta = 1 - 3/20 = 17/20.  out = -(1/2)(1,0) + (17/20)(3,1) = (41/20, 17/20), but
    #   m = (1/2)(1,0) + (17/20)(3,1) = (61/20, 17/20)
    ([[1, 0], [3, 1]], [Fraction(61, 20), Fraction(17, 20)]),
    # the same with every entry negated: the same coefficients, m from |g|: (61/20, 17/20)
    ([[-1, 0], [-3, -1]], [Fraction(61, 20), Fraction(17, 20)]),
    # tree over (1,0),(0,1),(1,1),(2,-1) (values in HAND above):
    #   level 0: m = (1,1) for the orthogonal pair; (3/4)(1,1) + (9/10)(2,1) = (51/20, 33/20)
    #   level 1: (2/5)(1,1) + (71/87)(51/20, 33/20) = (4317/1740, 3039/1740)
    #          = (1439/580, 1013/580)   (out is (1439/580, 161/580))
    ([[1, 0], [0, 1], [1, 1], [2, -1]], [Fraction(1439, 580), Fraction(1013, 580)]),
]


@pytest.mark.parametrize("vecs,expected", MAG_HAND)
def test_magnitude_bound_hand_worked(oracle_mod, vecs, expected):
    r = oracle_mod.adasum_reduce(f32(*vecs), [0, len(vecs[0])], want_mag=True)
    assert np.allclose(r["mag"], [float(x) for x in expected], rtol=1e-15, atol=0)


def test_magnitude_bound_closed_form(oracle_mod):
    """m = sum_k |c_k| |g_k|, with the leaf coefficients c_k of out = sum_k c_k g_k taken
    from the exact sequential-emulation derivation (not from the oracle).  Includes
    near-parallel pairs of unequal length, where a coefficient is negative."""
    from exact_adasum import adasum_tree_exact_coefficients
    rs = np.random.default_rng(31)
    seen_negative = False
    for K in (2, 4, 8):
        for trial in range(4):
            n = 5
            vecs = [rs.integers(-3, 4, size=n).astype(np.float32) for _ in range(K)]
            if trial % 2:  # a longer near-parallel partner: a.b > 2|a|^2
                vecs[1] = (3 * vecs[0] + rs.integers(-1, 2, size=n)).astype(np.float32)
            c = adasum_tree_exact_coefficients(vecs)
            seen_negative |= any(x < 0 for x in c)
            m = [sum(abs(ck) * abs(Fraction(float(v[j]))) for ck, v in zip(c, vecs))
                 for j in range(n)]
            got = oracle_mod.adasum_reduce(vecs, [0, n], want_mag=True)["mag"]
            assert np.allclose(got, [float(x) for x in m], rtol=1e-12, atol=1e-12), (K, trial)
    assert seen_negative


# ------------------------------------------------------------------- library-routine pins

def test_bf16_encoder_matches_torch(oracle_mod):
    rs = np.random.default_rng(21)
    bits = rs.integers(0, 2**32, size=4000, dtype=np.uint64).astype(np.uint32)
    special = np.array([0x00000000, 0x80000000, 0x3F808000, 0x3F818000, 0x3F80C000,
                        0x00008000, 0x00018000, 0x00000001, 0x007FFFFF, 0x7F7FFFFF,
                        0x7F7F8000, 0x7F7F7FFF, 0xFF7F8000, 0x7F800000, 0xFF800000,
                        0x00800000, 0x3F7FFFFF], dtype=np.uint32)
    bits = np.concatenate([bits, special])
    f = bits.view(np.float32)
    f = f[~np.isnan(f)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle_mod.bf16_encode(f.astype(np.float64))
    assert np.array_equal(got, ref)
    assert np.isnan(oracle_mod.bf16_decode(oracle_mod.bf16_encode([np.nan]))[0])
    # decode is exact
    back = oracle_mod.bf16_decode(ref)
    exp = torch.from_numpy(ref.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    assert np.array_equal(back, exp)


def test_bf16_single_rounding_from_fp64(oracle_mod):
    """fp64 -> bf16 rounds once: 1 + 2^-8 + 2^-40 is just above a tie and must round up,
    whereas rounding through fp32 first would land on the tie and round to even (down)."""
    x = 1.0 + 2.0**-8 + 2.0**-40
    got = oracle_mod.bf16_decode(oracle_mod.bf16_encode([x]))[0]
    assert got == 1.0 + 2.0**-7


@pytest.mark.parametrize("init", ["zero", "random"])
def test_momentum_matches_torch_sgd(oracle_mod, init):
    rs = np.random.default_rng(31)
    n = 301
    A = rs.standard_normal(n) * 1e-2
    w = (rs.standard_normal(n) * 0.02).astype(np.float32)
    v = np.zeros(n, np.float32) if init == "zero" else \
        (rs.standard_normal(n) * 0.01).astype(np.float32)
    lr, mu = float(np.float32(0.1)), float(np.float32(0.9))
    p = torch.nn.Parameter(torch.from_numpy(w.astype(np.float64)))
    opt = torch.optim.SGD([p], lr=lr, momentum=mu, dampening=0, nesterov=False,
                          weight_decay=0)
    if init == "random":
        opt.state[p]["momentum_buffer"] = torch.from_numpy(v.astype(np.float64))
    p.grad = torch.from_numpy(A.copy())
    opt.step()
    w_ref = p.detach().numpy().astype(np.float32)
    v_ref = opt.state[p]["momentum_buffer"].numpy().astype(np.float32)
    w_got, v_got = oracle_mod.momentum_sgd(A, w, v, lr, mu)
    assert np.array_equal(v_got, v_ref)
    assert np.array_equal(w_got, w_ref)


# ------------------------------------------------------------------------- bad arguments

def test_rejects_no_workers(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.adasum_reduce([], [0, 2])


# ------------------------------------------------ any worker count, and the linear chain

@pytest.mark.parametrize("K", [3, 5, 6, 7, 9, 12, 13])
def test_odd_counts_carry_the_last_node(oracle_mod, K):
    """Reading for worker counts that are not powers of two: pairs (2i, 2i+1) at every
    level, an unpaired last node moves on unchanged.  Pinned two ways: exactly against
    the power-of-two tree with zero vectors appended (Adasum(x, 0) = x), and bit for bit
    against the oracle's own power-of-two path on the zero-padded input."""
    rs = np.random.default_rng(100 + K)
    n = 9
    vecs = [rs.integers(-3, 4, size=n).astype(np.float32) for _ in range(K)]
    exact = np.array([float(x) for x in adasum_tree_exact_padded(vecs)])
    got = oracle_mod.adasum_reduce(vecs, [0, n])["out64"]
    nrm = np.linalg.norm(exact)
    assert np.linalg.norm(got - exact) <= 1e-13 * max(nrm, 1e-300)
    p2 = 1 << (K - 1).bit_length()
    padded = vecs + [np.zeros(n, np.float32)] * (p2 - K)
    assert np.array_equal(got, oracle_mod.adasum_reduce(padded, [0, n])["out64"])


@pytest.mark.parametrize("K", [2, 3, 4, 5, 8])
def test_chain_matches_sequential_emulation_exactly(oracle_mod, K):
    """The linear recursion g[0,n+1] = Adasum(g[0,n], g_{n+1}), pinned to the exact
    sequential-emulation derivation applied left to right."""
    rs = np.random.default_rng(200 + K)
    for n in (1, 4, 11):
        vecs = [rs.integers(-3, 4, size=n).astype(np.float32) for _ in range(K)]
        exact = np.array([float(x) for x in adasum_chain_exact(vecs)])
        got = oracle_mod.adasum_reduce(vecs, [0, n], chain=True)["out64"]
        nrm = np.linalg.norm(exact)
        if nrm == 0:
            assert np.all(got == 0)
        else:
            assert np.linalg.norm(got - exact) <= 1e-13 * nrm


def test_chain_and_tree_differ_from_four_workers(oracle_mod):
    """Two and three workers give the same result either way; from four on the chain
    and the tree pair different nodes."""
    vecs = f32([1, 0, 0], [1, 2, 0], [0, 1, 3], [2, -1, 1])
    for k in (2, 3):
        assert np.array_equal(oracle_mod.adasum_reduce(vecs[:k], [0, 3])["out64"],
                              oracle_mod.adasum_reduce(vecs[:k], [0, 3], chain=True)["out64"])
    tree = oracle_mod.adasum_reduce(vecs, [0, 3])["out64"]
    chain = oracle_mod.adasum_reduce(vecs, [0, 3], chain=True)["out64"]
    assert not np.allclose(tree, chain, rtol=1e-6)


def test_rejects_decreasing_offsets(oracle_mod):
    vecs = f32([1, 2, 3], [3, 4, 5])
    with pytest.raises(ValueError):
        oracle_mod.adasum_reduce(vecs, [0, 2, 1, 3])


# ----------------------------------------------------- Adasum after the optimizer (Fig. 3)

def test_local_momentum_updates_match_torch_sgd_per_worker(oracle_mod):
    """Each worker's state update is torch.optim.SGD's momentum buffer update; with one
    worker the whole step is torch's SGD step."""
    rs = np.random.default_rng(300)
    n, K = 57, 4
    grads = [rs.standard_normal(n).astype(np.float32) for _ in range(K)]
    v = [(rs.standard_normal(n) * 0.01).astype(np.float32) for _ in range(K)]
    w = (rs.standard_normal(n) * 0.02).astype(np.float32)
    lr, mu = float(np.float32(0.1)), float(np.float32(0.9))
    v_new, _ = oracle_mod.local_momentum_adasum(grads, [0, n], v, w, lr, mu)
    for k in range(K):
        p = torch.nn.Parameter(torch.zeros(n, dtype=torch.float64))
        opt = torch.optim.SGD([p], lr=lr, momentum=mu)
        opt.state[p]["momentum_buffer"] = torch.from_numpy(v[k].astype(np.float64))
        p.grad = torch.from_numpy(grads[k].astype(np.float64))
        opt.step()
        assert np.array_equal(v_new[k], opt.state[p]["momentum_buffer"].numpy().astype(np.float32))
    # one worker: exactly SGD
    _, w1 = oracle_mod.local_momentum_adasum(grads[:1], [0, n], v[:1], w, lr, mu)
    p = torch.nn.Parameter(torch.from_numpy(w.astype(np.float64)))
    opt = torch.optim.SGD([p], lr=lr, momentum=mu)
    opt.state[p]["momentum_buffer"] = torch.from_numpy(v[0].astype(np.float64))
    p.grad = torch.from_numpy(grads[0].astype(np.float64))
    opt.step()
    np.testing.assert_allclose(w1, p.detach().numpy().astype(np.float32), rtol=0, atol=1e-7)


def test_local_momentum_first_step_equals_allreduce_then_step(oracle_mod):
    """With zero momentum, Adasum after the optimizer and Adasum-then-heavy-ball agree
    (scale equivariance: Adasum(-lr g) = -lr Adasum(g))."""
    rs = np.random.default_rng(301)
    n, K = 40, 8
    grads = [rs.standard_normal(n).astype(np.float32) for _ in range(K)]
    offs = [0, 13, 40]
    w = (rs.standard_normal(n) * 0.02).astype(np.float32)
    zeros = [np.zeros(n, np.float32) for _ in range(K)]
    lr, mu = float(np.float32(0.1)), float(np.float32(0.9))
    _, w_local = oracle_mod.local_momentum_adasum(grads, offs, zeros, w, lr, mu)
    A = oracle_mod.adasum_reduce(grads, offs)["out64"]
    w_r1, _ = oracle_mod.momentum_sgd(A, w, np.zeros(n, np.float32), lr, mu)
    np.testing.assert_allclose(w_local, w_r1, rtol=0, atol=2e-8)
