"""Exact rational Adasum, derived independently of the oracle's formula.

"Scaling Distributed Training with Adaptive Summation", Section 3, reaches the Adasum
operator by emulating two sequential SGD steps and averaging the two processing orders.
This module follows those steps literally, in exact rational arithmetic:

  1. Process b1 then b2 from w0 with step alpha:  w1 = w0 - alpha g1.
  2. The second gradient, taken at w1 instead of w0, is corrected to first order
     (Equation 2): g2(w1) = g2 + H2 (w1 - w0) = g2 - alpha H2 g1.
  3. The Hessian is estimated from the gradient itself, H2 = g2 g2^T (Appendix A.1), built
     here as an explicit outer-product matrix.
  4. The step is the optimal one for that estimate, alpha = 1 / |g2|^2 (Appendix A.2).
  5. The effective gradient of the two steps is g1 + g2(w1), i.e. w2 = w0 - alpha (...).
  6. The opposite order (b2 first) gives the mirror expression; Adasum is their average.

The 0/0 case (a zero gradient, so H = 0 and alpha undefined) contributes no correction:
the correction term H g is the zero vector whatever alpha is.

For more than two gradients the operator is applied as a binary tree, pairing (2i, 2i+1)
at every level (Section 3's recursive application), written here as a recursive nesting
rather than the oracle's level loop.

The result is exact, so it pins the fp64 oracle up to its own rounding.  Nothing here is
shared with the oracle or with the CUDA library.
"""
from __future__ import annotations

from fractions import Fraction


def _frac(x):
    if isinstance(x, (int, Fraction)):
        return Fraction(x)
    return Fraction(float(x))          # exact: every binary float is a rational


def _vec(v):
    return [_frac(x) for x in v]


def _dot(u, v):
    return sum((a * b for a, b in zip(u, v)), Fraction(0))


def _outer(u, v):
    return [[a * b for b in v] for a in u]


def _matvec(M, v):
    return [sum((m * x for m, x in zip(row, v)), Fraction(0)) for row in M]


def _sequential_effective_gradient(first, second):
    """Effective gradient of processing `first` then `second` (steps 1-5 above)."""
    H = _outer(second, second)                       # Hessian estimate of the 2nd loss
    norm2 = _dot(second, second)
    Hg = _matvec(H, first)                           # H2 g1
    if norm2 == 0:
        corr = [Fraction(0)] * len(first)            # H2 = 0: nothing to correct
    else:
        alpha = Fraction(1) / norm2                  # optimal step for the estimate
        corr = [alpha * x for x in Hg]
    second_at_w1 = [s - c for s, c in zip(second, corr)]
    return [f + s for f, s in zip(first, second_at_w1)]


def adasum_pair_exact(a, b):
    """Average of the two sequential-emulation orders (step 6)."""
    a, b = _vec(a), _vec(b)
    ab = _sequential_effective_gradient(a, b)
    ba = _sequential_effective_gradient(b, a)
    return [(x + y) / 2 for x, y in zip(ab, ba)]


def adasum_tree_exact(vectors):
    """Binary tree over a power-of-two number of vectors: pairs (2i, 2i+1), recursively."""
    k = len(vectors)
    if k == 0 or (k & (k - 1)):
        raise ValueError("need a power-of-two number of vectors")
    if k == 1:
        return _vec(vectors[0])
    left = adasum_tree_exact(vectors[: k // 2])
    right = adasum_tree_exact(vectors[k // 2:])
    return adasum_pair_exact(left, right)


def adasum_chain_exact(vectors):
    """The linear recursion of the same section: g[0,n+1] = Adasum(g[0,n], g_{n+1})."""
    acc = _vec(vectors[0])
    for v in vectors[1:]:
        acc = adasum_pair_exact(acc, v)
    return acc


def adasum_tree_exact_padded(vectors):
    """A tree over any number of vectors, taken as the power-of-two tree over the
    vectors followed by zero vectors (an unpaired node then meets a zero node, and
    Adasum(x, 0) = x)."""
    k = len(vectors)
    p = 1
    while p < k:
        p *= 2
    n = len(vectors[0])
    return adasum_tree_exact(list(vectors) + [[0] * n] * (p - k))


def adasum_tree_exact_segments(vectors, offsets):
    """Per-layer application: every segment [offs[s], offs[s+1]) on its own."""
    out = []
    for s in range(len(offsets) - 1):
        lo, hi = int(offsets[s]), int(offsets[s + 1])
        if hi == lo:
            continue
        out += adasum_tree_exact([v[lo:hi] for v in vectors])
    return out


def _sequential_coefficients(first, second):
    """Steps 1-5 on nodes carried as (vector, leaf coefficients): the corrected second
    gradient subtracts alpha (second . first) second, so the effective gradient of the
    two steps is  first + second - ((second . first) / |second|^2) second."""
    (fv, fc), (sv, sc) = first, second
    norm2 = _dot(sv, sv)
    t = Fraction(0) if norm2 == 0 else _dot(sv, fv) / norm2
    vec = [f + s - t * s for f, s in zip(fv, sv)]
    coef = [f + s - t * s for f, s in zip(fc, sc)]
    return vec, coef


def adasum_tree_exact_coefficients(vectors):
    """The binary tree of adasum_tree_exact, returning the leaf coefficients c_k of
    out = sum_k c_k g_k (every node is a linear combination of the leaves; its
    coefficients follow the same two averaged orders as its vector)."""
    k = len(vectors)
    if k == 0 or (k & (k - 1)):
        raise ValueError("need a power-of-two number of vectors")

    def node(lo, hi):
        if hi - lo == 1:
            c = [Fraction(0)] * k
            c[lo] = Fraction(1)
            return _vec(vectors[lo]), c
        mid = (lo + hi) // 2
        a, b = node(lo, mid), node(mid, hi)
        ab, ba = _sequential_coefficients(a, b), _sequential_coefficients(b, a)
        return ([(x + y) / 2 for x, y in zip(ab[0], ba[0])],
                [(x + y) / 2 for x, y in zip(ab[1], ba[1])])

    return node(0, k)[1]
