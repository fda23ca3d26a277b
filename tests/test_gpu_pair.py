"""The two-worker, one-segment path (adasum_pair.cuh): one cooperative kernel with one grid
barrier, double-float Gram sums and a double-float combine rounded once.  Taken by
adasum_pair and by adasum_reduce with two workers and one segment that the kernel's CTAs
hold in registers (about 1.2M fp32 or 5M bf16 elements on a GB300); longer ones take the
tiled route.  Compared with the fp64 oracle; the fp32 result is the exact value rounded
once, so it is held to 1e-7 normwise, not the 1e-5 tolerance.
"""
import numpy as np
import pytest
import torch

import adaptive_gradient_summation_gb300 as ags
from parity import check_against_oracle, oracle_reduce, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _pair(n, dtype, seed, corr=0.5, scale=1.0):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    a = torch.randn(n, generator=gen, device=DEV)
    b = corr * a + (1 - corr * corr) ** 0.5 * torch.randn(n, generator=gen, device=DEV)
    return (a * scale).to(dtype), (b * scale).to(dtype)


def _ulp_bf16(x):
    ax = np.maximum(np.abs(x), 2.0**-133)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def _check_rounded_once(a, b, out):
    """fp32: normwise within 1e-7 of the oracle; bf16: within one bf16 ulp per element."""
    ref = oracle_reduce([a, b], [0, a.numel()])["out64"]
    got = to_f64(out)
    if out.dtype == torch.float32:
        nr = np.linalg.norm(ref)
        assert np.linalg.norm(got - ref) <= 1e-7 * nr + 1e-300
    else:
        assert np.all(np.abs(got - ref) <= _ulp_bf16(ref) + 1e-12 * np.abs(ref))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("n", [1, 3, 8, 9, 31, 1000, 65_537, 1_048_576])
def test_fused_pair_matches_oracle(native, dtype, n):
    a, b = _pair(n, dtype, seed=n % 1000 + 7)
    out = ags.pair(a, b)
    torch.cuda.synchronize()
    _check_rounded_once(a, b, out)
    assert ags.recomputed_segments() == 0


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("n", [2_000_001, 9_000_000])
def test_large_pairs(native, dtype, n):
    """Past what the fused kernel's CTAs hold in registers: the tiled route."""
    a, b = _pair(n, dtype, seed=11)
    out = ags.pair(a, b)
    torch.cuda.synchronize()
    check_against_oracle([a, b], [0, n], out)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_fused_pair_unaligned_and_in_place(native, dtype):
    a, b = _pair(100_003, dtype, seed=12)
    a1, b1 = a[1:], b[1:]
    out = ags.pair(a1, b1)
    torch.cuda.synchronize()
    _check_rounded_once(a1, b1, out)
    expect = ags.pair(a, b)
    x = a.clone()
    ags.reduce([x, b], [0, a.numel()], out=x)
    torch.cuda.synchronize()
    assert torch.equal(x, expect)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("eps", [1e-3, 1e-6])
def test_fused_pair_cancelling(native, dtype, eps):
    """b nearly cancels a: the coefficients are about 1.5 and the result is tiny next to
    the inputs.  The double-float Gram and combine keep it accurate without a recompute."""
    gen = torch.Generator(device=DEV).manual_seed(13)
    a = torch.randn(50_000, generator=gen, device=DEV)
    b = -(1 - eps) * a + eps * 0.1 * torch.randn(50_000, generator=gen, device=DEV)
    a, b = a.to(dtype), b.to(dtype)
    out = ags.pair(a, b)
    torch.cuda.synchronize()
    check_against_oracle([a, b], [0, a.numel()], out)


@pytest.mark.parametrize("scale", [1e-30, 1e-20, 1e20, 1e30])
def test_fused_pair_extreme_magnitudes(native, scale):
    """Squares outside fp32's range: each thread scales its values by a power of two."""
    a, b = _pair(300_000, torch.float32, seed=14, scale=scale)
    out = ags.pair(a, b)
    torch.cuda.synchronize()
    _check_rounded_once(a, b, out)


def test_fused_pair_mixed_magnitudes_across_ctas(native):
    """Parts of the vectors 1e40 apart: the CTAs' partial sums have different exponents
    and are brought to the largest exactly; the tiny part still gets its coefficient."""
    a, b = _pair(400_000, torch.float32, seed=15)
    scale = torch.ones(400_000, device=DEV)
    scale[:200_000] = 1e-20
    scale[200_000:] = 1e20
    a, b = a * scale, b * scale
    out = ags.pair(a, b)
    torch.cuda.synchronize()
    _check_rounded_once(a, b, out)
    small = slice(0, 200_000)
    ref = oracle_reduce([a, b], [0, 400_000])["out64"]
    got = to_f64(out)
    assert np.linalg.norm(got[small] - ref[small]) <= 1e-6 * np.linalg.norm(ref[small])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_fused_pair_symmetric_and_special_cases(native, dtype):
    a, b = _pair(123_457, dtype, seed=16)
    assert torch.equal(ags.pair(a, b), ags.pair(b, a))
    assert torch.equal(ags.pair(a, a.clone()), a)
    z = torch.zeros_like(a)
    assert torch.equal(ags.pair(a, z), a)
    assert torch.equal(ags.pair(z, z), z)
    mask = torch.arange(a.numel(), device=DEV) % 3 == 0
    x, y = torch.where(mask, a, 0), torch.where(mask, 0, b)
    assert torch.equal(ags.pair(x, y), x + y)
    first = ags.pair(a, b).clone()
    assert torch.equal(ags.pair(a, b), first)  # deterministic


def test_fused_pair_agrees_with_tiled_route(native, hooks, monkeypatch):
    a, b = _pair(777_777, torch.float32, seed=17)
    fused = ags.pair(a, b).clone()
    monkeypatch.setenv("ADASUM_PAIR_FUSED", "0")
    tiled = ags.pair(a, b)
    torch.cuda.synchronize()
    ref = oracle_reduce([a, b], [0, a.numel()])["out64"]
    nr = np.linalg.norm(ref)
    assert np.linalg.norm(to_f64(fused) - ref) <= 1e-7 * nr
    assert np.linalg.norm(to_f64(tiled) - ref) <= 1e-5 * nr


def test_fused_pair_barrier_timeout_is_reported(native, hooks, monkeypatch):
    """Every CTA waits at the grid barrier without arriving (injected on the host): the
    waits run out after their clock budget, the status word says so, and the next call
    (no injection) is correct -- the barrier's state was not disturbed."""
    a, b = _pair(200_000, torch.float32, seed=18)
    assert ags.get_last_error() == ags.Status.OK
    monkeypatch.setenv("ADASUM_FAULT_INJECT", "timeout")
    ags.pair(a, b)
    torch.cuda.synchronize()
    monkeypatch.delenv("ADASUM_FAULT_INJECT")
    assert ags.get_last_error() == ags.Status.ERR_TIMEOUT
    assert ags.get_last_error() == ags.Status.OK  # reading clears it
    out = ags.pair(a, b)
    torch.cuda.synchronize()
    _check_rounded_once(a, b, out)


def test_fused_pair_graph_replays(native):
    """Captured after a warm-up call and replayed several times: the grid barrier resets
    itself at every crossing, so every replay gives the direct call's result."""
    a, b = _pair(500_001, torch.float32, seed=19)
    out = torch.empty_like(a)
    expect = ags.pair(a, b).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ags.pair(a, b, out=out, stream=s)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ags.pair(a, b, out=out, stream=s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, expect)


def test_fused_pair_dtypes_alternate(native):
    """fp32 and bf16 calls in turn (their kernels fit different numbers of CTAs) share
    one grid barrier: every crossing completes, none runs out of its budget."""
    assert ags.get_last_error() == ags.Status.OK
    for dtype in (torch.float32, torch.bfloat16, torch.float32, torch.bfloat16):
        a, b = _pair(1_000_000, dtype, seed=20)
        out = ags.pair(a, b)
        torch.cuda.synchronize()
        _check_rounded_once(a, b, out)
    assert ags.get_last_error() == ags.Status.OK


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_fused_pair_through_reduce_and_in_place_on_b(native, dtype):
    """adasum_reduce with two workers and one segment is the same kernel as adasum_pair
    (bitwise), and the output may also be the second operand."""
    a, b = _pair(250_007, dtype, seed=21)
    expect = ags.pair(a, b).clone()
    via_reduce = ags.reduce([a, b], [0, a.numel()])
    y = b.clone()
    ags.reduce([a, y], [0, a.numel()], out=y)
    torch.cuda.synchronize()
    assert torch.equal(via_reduce, expect)
    assert torch.equal(y, expect)
