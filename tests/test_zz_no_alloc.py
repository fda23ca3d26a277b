"""adasum_pair_noalloc, the allocation-free two-worker entry point, against adasum_pair.

Some callers cannot call cudaMalloc when they reduce (their framework's allocator holds
the GPU's memory, or they cannot afford the synchronisation an allocation implies); for
them the library offers a variant whose scratch is a fixed device array inside the
library.  This file is named to be collected last, so a run that stops at the first
failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import adaptive_gradient_summation_gb300 as ags
from parity import check_fp32_segments, to_f64, ulp_bf16

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
MAX_N = 33_554_432


def _noalloc(lib, a, b, out, dtype_code):
    return lib.adasum_pair_noalloc(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()),
                                   a.numel(), dtype_code, ctypes.c_void_p(out.data_ptr()),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _inputs(n, dtype, seed):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    a = torch.randn(n, generator=gen, device=DEV)
    b = 0.5 * a + 0.8 * torch.randn(n, generator=gen, device=DEV)
    return a.to(dtype), b.to(dtype)


def _same_within_tolerance(got, ref, a, b, dtype):
    if dtype == torch.float32:
        check_fp32_segments(to_f64(got), to_f64(ref), [0, got.numel()])
    else:
        # two fp32 evaluations each rounded once to bf16: at most 2 bf16 ulps apart, plus
        # the fp32 floor of the tests (K 2^-23 times the magnitude of the terms).
        g, r = to_f64(got), to_f64(ref)
        mag = np.abs(to_f64(a)) + np.abs(to_f64(b))
        tol = 2 * ulp_bf16(r) + 2 * 2.0**-23 * mag
        assert np.all(np.abs(g - r) <= tol)


@pytest.mark.parametrize("dtype,code", [(torch.float32, 0), (torch.bfloat16, 1)])
def test_noalloc_matches_pair_on_two_calls_in_a_row(native, dtype, code):
    lib = ags.load_library()
    # first call: a large pair spanning many tiles and a ragged tail
    a, b = _inputs(5_000_003, dtype, seed=1)
    out = torch.empty_like(a)
    assert _noalloc(lib, a, b, out, code) == 0
    ref = ags.pair(a, b)
    torch.cuda.synchronize()
    _same_within_tolerance(out, ref, a, b, dtype)
    # second call, right after: a smaller pair reusing the same scratch
    a2, b2 = _inputs(70_001, dtype, seed=2)
    out2 = torch.empty_like(a2)
    assert _noalloc(lib, a2, b2, out2, code) == 0
    ref2 = ags.pair(a2, b2)
    torch.cuda.synchronize()
    _same_within_tolerance(out2, ref2, a2, b2, dtype)


def test_noalloc_rejects_sizes_beyond_the_maximum(native):
    lib = ags.load_library()
    a = torch.zeros(16, device=DEV)
    st = lib.adasum_pair_noalloc(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(a.data_ptr()),
                                 MAX_N + 1, 0, ctypes.c_void_p(a.data_ptr()), None)
    assert st == ags.Status.ERR_UNSUPPORTED
