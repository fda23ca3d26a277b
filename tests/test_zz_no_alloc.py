"""adasum_pair_noalloc, the allocation-free two-worker entry point.

Some callers cannot call cudaMalloc when they reduce (their framework's allocator holds
the GPU's memory, or they cannot afford the synchronisation an allocation implies); for
them the library offers a variant whose scratch is a fixed device array inside the
library.  Its results are checked against the fp64 CPU oracle at the tests' tolerances
and against the allocating entry point adasum_pair, on calls in a row that reuse the
scratch.  This file is named to be collected last, so a run that stops at the first
failure has run every other test before it; every test here also passes in a fresh
process on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

import adaptive_gradient_summation_gb300 as ags
from parity import (check_fp32_segments, oracle_reduce, to_f64, ulp_bf16)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
MAX_N = 33_554_432
CODE = {torch.float32: 0, torch.bfloat16: 1}


def _noalloc_raw(a_ptr, b_ptr, n, code, out_ptr):
    lib = ags.load_library()
    return lib.adasum_pair_noalloc(ctypes.c_void_p(a_ptr), ctypes.c_void_p(b_ptr), n, code,
                                   ctypes.c_void_p(out_ptr),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _noalloc(a, b, out):
    return _noalloc_raw(a.data_ptr(), b.data_ptr(), a.numel(), CODE[a.dtype], out.data_ptr())


def _inputs(n, dtype, seed):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    a = torch.randn(n, generator=gen, device=DEV)
    b = 0.5 * a + 0.8 * torch.randn(n, generator=gen, device=DEV)
    return a.to(dtype), b.to(dtype)


def _check_oracle(got, a, b):
    """fp32: |out - ref| <= 1e-5 |ref| (normwise); bf16: per element within 2 bf16 ulps
    of the unrounded reference plus the fp32-arithmetic floor 2 * 2^-23 * m."""
    ref = oracle_reduce([a, b], [0, a.numel()], want_mag=got.dtype == torch.bfloat16)
    g = to_f64(got)
    if got.dtype == torch.float32:
        check_fp32_segments(g, ref["out64"], [0, got.numel()], what="noalloc")
    else:
        tol = 2 * ulp_bf16(ref["out64"]) + 2 * 2.0**-23 * ref["mag"]
        assert np.all(np.abs(g - ref["out64"]) <= tol), "noalloc bf16 outside tolerance"


def _check_against_pair(got, ref, a, b):
    if got.dtype == torch.float32:
        check_fp32_segments(to_f64(got), to_f64(ref), [0, got.numel()], what="noalloc vs pair")
    else:
        # two fp32 evaluations, each rounded once to bf16
        g, r = to_f64(got), to_f64(ref)
        mag = np.abs(to_f64(a)) + np.abs(to_f64(b))
        assert np.all(np.abs(g - r) <= 2 * ulp_bf16(r) + 2 * 2.0**-23 * mag)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_noalloc_matches_oracle_and_pair_on_two_calls_in_a_row(native, dtype):
    # first call: a large pair spanning many tiles and a ragged tail
    a, b = _inputs(5_000_003, dtype, seed=1)
    out = torch.empty_like(a)
    assert _noalloc(a, b, out) == 0
    ref = ags.pair(a, b)
    torch.cuda.synchronize()
    _check_oracle(out, a, b)
    _check_against_pair(out, ref, a, b)
    # second call, right after: a smaller pair reusing the same scratch
    a2, b2 = _inputs(70_001, dtype, seed=2)
    out2 = torch.empty_like(a2)
    assert _noalloc(a2, b2, out2) == 0
    ref2 = ags.pair(a2, b2)
    torch.cuda.synchronize()
    _check_oracle(out2, a2, b2)
    _check_against_pair(out2, ref2, a2, b2)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_noalloc_at_the_maximum_size(native, dtype):
    """n = ADASUM_NOALLOC_MAX_N: all 4,096 tile slots of the scratch and the coefficient
    slots after them in use (through the Python wrapper)."""
    a, b = _inputs(MAX_N, dtype, seed=3)
    out = torch.empty_like(a)
    ags.pair_noalloc(a, b, out)
    torch.cuda.synchronize()
    _check_oracle(out, a, b)
    # and a one-tile call right after must not see the big call's slots
    a1, b1 = _inputs(1000, dtype, seed=4)
    out1 = torch.empty_like(a1)
    ags.pair_noalloc(a1, b1, out1)
    torch.cuda.synchronize()
    _check_oracle(out1, a1, b1)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_noalloc_in_place(native, dtype):
    a, b = _inputs(300_007, dtype, seed=5)
    expect = torch.empty_like(a)
    assert _noalloc(a, b, expect) == 0
    x, y = a.clone(), b.clone()
    assert _noalloc(x, y, x) == 0          # out == a
    torch.cuda.synchronize()
    assert torch.equal(x, expect)
    x, y = a.clone(), b.clone()
    assert _noalloc(x, y, y) == 0          # out == b
    torch.cuda.synchronize()
    assert torch.equal(y, expect)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_noalloc_unaligned_pointers(native, dtype):
    n = 100_003
    base_a, base_b = _inputs(n + 8, dtype, seed=6)
    a, b = base_a[1:1 + n], base_b[3:3 + n]
    out_base = torch.empty(n + 8, dtype=dtype, device=DEV)
    out = out_base[5:5 + n]
    assert _noalloc(a, b, out) == 0
    torch.cuda.synchronize()
    _check_oracle(out, a.contiguous(), b.contiguous())


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_noalloc_zero_operand_gives_the_other(native, dtype):
    """Adasum(0, b) = b: the zero operand's 0/0 quotient is 0, so both coefficients are
    1 and the output is b bit for bit."""
    _, b = _inputs(65_537, dtype, seed=7)
    z = torch.zeros_like(b)
    out = torch.empty_like(b)
    assert _noalloc(z, b, out) == 0
    torch.cuda.synchronize()
    assert torch.equal(out, b)
    assert _noalloc(b, z, out) == 0
    torch.cuda.synchronize()
    assert torch.equal(out, b)


def test_noalloc_rejects_bad_arguments(native):
    n = 4096
    buf = torch.zeros(2 * n, device=DEV)
    a, b = buf[:n], torch.ones(n, device=DEV)
    # output overlapping an input other than exactly: ERR_ALIAS, nothing launched
    assert _noalloc_raw(a.data_ptr(), b.data_ptr(), n, 0, buf[7:].data_ptr()) == ags.Status.ERR_ALIAS
    assert _noalloc_raw(a.data_ptr(), b.data_ptr(), n, 0, b.data_ptr() + 4) == ags.Status.ERR_ALIAS
    # sizes beyond the scratch, negative sizes, bad dtypes, null pointers
    assert _noalloc_raw(a.data_ptr(), a.data_ptr(), MAX_N + 1, 0, a.data_ptr()) == ags.Status.ERR_UNSUPPORTED
    assert _noalloc_raw(a.data_ptr(), b.data_ptr(), -1, 0, a.data_ptr()) == ags.Status.ERR_INVALID_ARG
    assert _noalloc_raw(a.data_ptr(), b.data_ptr(), n, 7, a.data_ptr()) == ags.Status.ERR_INVALID_ARG
    assert _noalloc_raw(0, b.data_ptr(), n, 0, a.data_ptr()) == ags.Status.ERR_INVALID_ARG
    assert _noalloc_raw(a.data_ptr(), b.data_ptr(), 0, 0, a.data_ptr()) == ags.Status.OK
    torch.cuda.synchronize()
    assert torch.equal(buf, torch.zeros_like(buf))  # nothing was written
