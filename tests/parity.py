"""Comparison of GPU results with the fp64 oracle, at the stated tolerances.

fp32 storage: per segment, |out - ref|_2 <= 1e-5 |ref|_2, and a segment whose oracle
result is exactly zero must come out exactly zero.

bf16 storage: per element, |out - ref| <= 2 ulp_bf16(ref) + K 2^-23 m, where ref is the
unrounded fp64 oracle value and m the oracle's magnitude bound (m = sum_k |c_k| |g_k|,
carried through the tree).  The second term is the size of the fp32 arithmetic error
of the GPU (Gram sums, coefficients and the K-term combine are all fp32): without it,
elements whose value cancels far below m would be held to an error far below the fp32
rounding of the terms they are built from.

Momentum (fp32 state): per segment, |v' - v'_ref| <= 1e-5 |v'_ref| and
|w' - w'_ref| <= 1e-5 lr |v'_ref| + 2^-23 |w'_ref| (one fp32 rounding of w).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

FP32_RTOL = 1e-5


def to_oracle_input(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    if t.dtype == torch.float32:
        return t.numpy().copy()
    raise TypeError(t.dtype)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    e = np.floor(np.log2(np.maximum(ax, 2.0**-126)))
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def oracle_reduce(grads, offsets, **kw):
    return oracle.adasum_reduce([to_oracle_input(g) for g in grads], offsets, **kw)


def check_fp32_segments(got: np.ndarray, ref: np.ndarray, offsets, rtol=FP32_RTOL,
                        what="out"):
    worst = 0.0
    for s in range(len(offsets) - 1):
        lo, hi = int(offsets[s]), int(offsets[s + 1])
        if hi == lo:
            continue
        r, g = ref[lo:hi], got[lo:hi]
        nr = np.linalg.norm(r)
        if nr == 0:
            assert np.all(g == 0), f"{what}: segment {s} should be exactly zero"
            continue
        err = np.linalg.norm(g - r) / nr
        worst = max(worst, err)
        assert err <= rtol, f"{what}: segment {s} [{lo},{hi}) rel err {err:.3e} > {rtol:.1e}"
    return worst


def check_bf16_elements(got: np.ndarray, ref: np.ndarray, mag: np.ndarray, K: int,
                        what="out"):
    tol = 2 * ulp_bf16(ref) + K * 2.0**-23 * mag
    err = np.abs(got - ref)
    bad = err > tol
    if bad.any():
        i = int(np.argmax(err / np.maximum(tol, 1e-300)))
        raise AssertionError(f"{what}: {int(bad.sum())} of {got.size} bf16 elements outside "
                             f"tolerance; worst at {i}: got {got[i]!r} ref {ref[i]!r} "
                             f"tol {tol[i]!r} mag {mag[i]!r}")
    return float(np.max(err / np.maximum(tol, 1e-300))) if got.size else 0.0


def check_against_oracle(grads, offsets, out: torch.Tensor, ref=None):
    """Compare a GPU adasum_reduce result with the oracle; returns the worst ratio."""
    if ref is None:
        ref = oracle_reduce(grads, offsets, want_mag=out.dtype == torch.bfloat16)
    got = to_f64(out)
    if out.dtype == torch.float32:
        return check_fp32_segments(got, ref["out64"], offsets)
    return check_bf16_elements(got, ref["out64"], ref["mag"], len(grads))


def check_momentum(w_new, v_new, w_ref, v_ref, offsets, lr):
    w_new, v_new = to_f64(w_new), to_f64(v_new)
    w_ref, v_ref = w_ref.astype(np.float64), v_ref.astype(np.float64)
    for s in range(len(offsets) - 1):
        lo, hi = int(offsets[s]), int(offsets[s + 1])
        if hi == lo:
            continue
        nv = np.linalg.norm(v_ref[lo:hi])
        ev = np.linalg.norm(v_new[lo:hi] - v_ref[lo:hi])
        assert ev <= FP32_RTOL * nv + 1e-30, f"momentum segment {s}: {ev:.3e} vs {nv:.3e}"
        ew = np.linalg.norm(w_new[lo:hi] - w_ref[lo:hi])
        tol = FP32_RTOL * lr * nv + 2.0**-23 * np.linalg.norm(w_ref[lo:hi]) + 1e-30
        assert ew <= tol, f"weights segment {s}: {ew:.3e} > {tol:.3e}"
