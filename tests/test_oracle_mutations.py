"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a temporary copy of oracle/adasum_oracle.c (the committed
file is never touched), compiles it on the CPU, and checks that the pins of
test_oracle_pins.py's kind reject it: hand-worked values, the exact sequential-emulation
derivation, the zero-operand rule, torch's bf16 rounding and torch's SGD step.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from exact_adasum import adasum_tree_exact

SRC = os.path.join(os.path.dirname(oracle.__file__), "adasum_oracle.c")

MUTANTS = {
    "dropped_half": ("d / (2.0 * p)", "d / p"),
    "wrong_sign": ("double alpha = 1.0 - ", "double alpha = 1.0 + "),
    "beta_uses_p": ("d / (2.0 * q)", "d / (2.0 * p)"),
    "dot_is_norm": ("d += a[j] * b[j];", "d += a[j] * a[j];"),
    "pairs_halves": ("const double *a = level + (size_t)(2 * i) * (size_t)n;\n"
                     "        const double *b = level + (size_t)(2 * i + 1) * (size_t)n;",
                     "const double *a = level + (size_t)(i) * (size_t)n;\n"
                     "        const double *b = level + (size_t)(i + width / 2) * (size_t)n;"),
    "no_zero_guard": ("1.0 - (p == 0.0 ? 0.0 : d / (2.0 * p))", "1.0 - d / (2.0 * p)"),
    "bf16_truncates": ("double r = nearbyint(ldexp(ax, -q));", "double r = floor(ldexp(ax, -q));"),
    "momentum_no_mu": ("double vn = mu * (double)v[j] + A[j];", "double vn = (double)v[j] + A[j];"),
    "momentum_sign": ("double wn = (double)w[j] - lr * vn;", "double wn = (double)w[j] + lr * vn;"),
    "carry_dropped": ("memmove(level + to, level + from, (size_t)n * sizeof(double));",
                      "(void)from; (void)to;"),
    "chain_skips_one": ("for (int k = 1; k < K; ++k) {", "for (int k = 2; k < K; ++k) {"),
    "mag_signed": ("fabs(alpha) * ma[j] + fabs(beta) * mb[j]", "alpha * ma[j] + beta * mb[j]"),
    "mag_unweighted": ("fabs(alpha) * ma[j] + fabs(beta) * mb[j]", "ma[j] + mb[j]"),
    "mag_coefficients_only": ("fabs(alpha) * ma[j] + fabs(beta) * mb[j]", "fabs(alpha) + fabs(beta)"),
    "mag_inflated": ("fabs(alpha) * ma[j] + fabs(beta) * mb[j]",
                     "2.0 * (fabs(alpha) * ma[j] + fabs(beta) * mb[j])"),
    "mag_leaf_signed": ("mlevel[(size_t)k * (size_t)n + j] = fabs(v[j]);",
                        "mlevel[(size_t)k * (size_t)n + j] = v[j];"),
}

# Magnitude bound m = |alpha| m_a + |beta| m_b, hand-worked (one case has alpha < 0 and
# one negative inputs; see test_oracle_pins.py).
MAG_PINS = [
    ([[1, 0], [1, 1]], [1.25, 0.75]),
    ([[1, 0], [3, 1]], [61 / 20, 17 / 20]),
    ([[-1, 0], [-3, -1]], [61 / 20, 17 / 20]),
    ([[1, 0], [0, 1], [1, 1], [2, -1]], [1439 / 580, 1013 / 580]),
]


def _pins_pass(lib) -> bool:
    f32 = lambda v: np.asarray(v, np.float32)  # noqa: E731
    # hand-worked values
    for vecs in ([[1, 0], [1, 1]], [[3, -1, 2], [1, 2, 0]], [[1, 0], [0, 1], [1, 1], [2, -1]]):
        exp = np.array([float(x) for x in adasum_tree_exact(vecs)])
        got = oracle.adasum_reduce([f32(v) for v in vecs], [0, len(vecs[0])], lib=lib)["out64"]
        if not np.allclose(got, exp, rtol=1e-14, atol=0):
            return False
    # exact sequential-emulation derivation, random integer vectors
    rs = np.random.default_rng(77)
    for K in (2, 4, 8):
        for n in (1, 3, 8):
            vecs = [rs.integers(-3, 4, size=n).astype(np.float32) for _ in range(K)]
            exp = np.array([float(x) for x in adasum_tree_exact(vecs)])
            got = oracle.adasum_reduce(vecs, [0, n], lib=lib)["out64"]
            if not np.allclose(got, exp, rtol=1e-12, atol=1e-12):
                return False
    # odd worker counts: against the zero-padded exact tree
    from exact_adasum import adasum_chain_exact, adasum_tree_exact_padded
    for K in (3, 5, 7):
        vecs = [rs.integers(-3, 4, size=5).astype(np.float32) for _ in range(K)]
        exp = np.array([float(x) for x in adasum_tree_exact_padded(vecs)])
        got = oracle.adasum_reduce(vecs, [0, 5], lib=lib)["out64"]
        if not np.allclose(got, exp, rtol=1e-12, atol=1e-12):
            return False
        exp = np.array([float(x) for x in adasum_chain_exact(vecs)])
        got = oracle.adasum_reduce(vecs, [0, 5], lib=lib, chain=True)["out64"]
        if not np.allclose(got, exp, rtol=1e-12, atol=1e-12):
            return False
    # magnitude bound
    for vecs, exp in MAG_PINS:
        got = oracle.adasum_reduce([f32(v) for v in vecs], [0, 2], lib=lib, want_mag=True)["mag"]
        if not np.allclose(got, exp, rtol=1e-14, atol=0):
            return False
    # zero operand
    b = f32([1.5, -2.0, 0.25])
    z = np.zeros(3, np.float32)
    got = oracle.adasum_reduce([z, b], [0, 3], lib=lib)["out64"]
    if not np.array_equal(got, b.astype(np.float64)):
        return False
    # bf16 rounding against torch
    vals = np.random.default_rng(5).standard_normal(2000).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    if not np.array_equal(oracle.bf16_encode(vals.astype(np.float64), lib=lib), ref):
        return False
    # momentum step against torch.optim.SGD
    A = np.linspace(-1, 1, 17)
    w = np.linspace(0.5, -0.5, 17).astype(np.float32)
    v = np.linspace(-0.1, 0.1, 17).astype(np.float32)
    p = torch.nn.Parameter(torch.from_numpy(w.astype(np.float64)))
    opt = torch.optim.SGD([p], lr=0.1, momentum=0.9)
    opt.state[p]["momentum_buffer"] = torch.from_numpy(v.astype(np.float64))
    p.grad = torch.from_numpy(A.copy())
    opt.step()
    w_got, v_got = oracle.momentum_sgd(A, w, v, 0.1, 0.9, lib=lib)
    if not (np.array_equal(w_got, p.detach().numpy().astype(np.float32)) and
            np.array_equal(v_got, opt.state[p]["momentum_buffer"].numpy().astype(np.float32))):
        return False
    return True


def test_unmutated_oracle_passes_the_pins(oracle_mod):
    assert _pins_pass(oracle.open_library(oracle.build()))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant_src = tmp_path / f"mutant_{name}.c"
    mutant_src.write_text(src.replace(old, new))
    lib_path = oracle.build(force=True, src=str(mutant_src),
                            out=str(tmp_path / f"mutant_{name}.so"))
    with np.errstate(all="ignore"):
        assert not _pins_pass(oracle.open_library(lib_path)), f"pins missed mutant {name}"
