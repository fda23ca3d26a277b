"""Memory-safety stand-ins on the GPU (compute-sanitizer is closed on this machine).

1. Canary words around the output, and the inputs compared before and after: odd and
   unaligned sizes, every dtype, tree depths from one stage to two, on the product
   library.  Nothing outside `out` may change and the inputs must be untouched.
2. The test build (device-side index checks on every tile, chunk and segment descriptor,
   guard bands after every workspace region): the same sweep plus the small-segment and
   recompute paths must report no failed check and no touched guard byte.
Every result is also compared with the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import adaptive_gradient_summation_gb300 as ags
from adaptive_gradient_summation_gb300 import workloads
from parity import check_against_oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
GUARD = 4096          # elements of canary before and after the output
CANARY = 0x5A5A       # 16-bit pattern (as bits of every element)

SIZES = [[1], [7], [31], [33], [4097], [1, 7, 0, 31, 33, 4097], [70_001, 3, 65_536]]


def _canary_buffer(n, dtype, shift):
    """A buffer of GUARD + shift + n + GUARD elements filled with the canary; returns
    (buffer, out view of n elements starting `shift` elements after the front guard)."""
    nb = GUARD + shift + n + GUARD
    if dtype == torch.bfloat16:
        buf = torch.full((nb,), CANARY, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    else:
        buf = torch.full((nb,), (CANARY << 16) | CANARY, dtype=torch.int32, device=DEV).view(torch.float32)
    return buf, buf[GUARD + shift: GUARD + shift + n]


def _guards_intact(buf, n, shift):
    bits = buf.view(torch.int16) if buf.dtype == torch.bfloat16 else buf.view(torch.int32)
    want = CANARY if buf.dtype == torch.bfloat16 else (CANARY << 16) | CANARY
    front, back = bits[: GUARD + shift], bits[GUARD + shift + n:]
    return bool((front == want).all()) and bool((back == want).all())


def _inputs(K, n, dtype, seed, shift):
    """K inputs as views starting `shift` elements into larger buffers (unaligned when
    shift is not a multiple of the 16-byte vector)."""
    gen = torch.Generator(device=DEV).manual_seed(seed)
    s = torch.randn(n + shift, generator=gen, device=DEV)
    out = []
    for _ in range(K):
        z = torch.randn(n + shift, generator=gen, device=DEV)
        out.append((0.6 * s + 0.8 * z).to(dtype)[shift:])
    return out


def _sweep(K, dtype, shift, seed):
    for lengths in SIZES:
        offs = workloads.offsets_from_numels(lengths)
        n = int(offs[-1])
        grads = _inputs(K, n, dtype, seed, shift)
        before = [g.clone() for g in grads]
        buf, out = _canary_buffer(n, dtype, shift)
        ags.reduce(grads, offs, out=out)
        torch.cuda.synchronize()
        assert _guards_intact(buf, n, shift), (K, dtype, shift, lengths)
        assert all(torch.equal(a, b) for a, b in zip(grads, before)), "an input changed"
        check_against_oracle(grads, offs, out)
        seed += 1


@pytest.mark.parametrize("shift", [0, 1, 3])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K", [2, 5, 16, 64])
def test_output_canaries_and_inputs_untouched(native, K, dtype, shift):
    _sweep(K, dtype, shift, seed=1000 + K)


@pytest.mark.parametrize("shift", [0, 3])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K", [2, 16, 64])
def test_bounds_checked_build(native, hooks, K, dtype, shift):
    """On the test build: no index check fails and no workspace guard byte changes,
    for the tiled route and then with every small segment forced on chip."""
    assert ags.get_last_error() == ags.Status.OK
    _sweep(K, dtype, shift, seed=2000 + K)
    assert ags.get_last_error() == ags.Status.OK
    assert hooks.adasum_debug_workspace_guards() == 0


def test_bounds_checked_build_small_segment_and_recompute_paths(native, hooks, monkeypatch):
    """The on-chip fast pass (forced), the warp kernel for tiny segments, and the
    recompute paths (nearly cancelling pairs: on-chip recompute and the fp64 path), all
    under the index checks."""
    monkeypatch.setenv("ADASUM_ONCHIP", "force")
    monkeypatch.setenv("ADASUM_ONCHIP_MAX_CLUSTER", "16")
    for K in (4, 16, 64):
        wl = workloads.make("small_segments_k64", device=DEV, shrink=50)
        grads = wl.grads[:K]
        out = ags.reduce(grads, wl.seg_offsets)
        torch.cuda.synchronize()
        check_against_oracle(grads, wl.seg_offsets, out)
        assert ags.get_last_error() == ags.Status.OK
        assert hooks.adasum_debug_workspace_guards() == 0
    monkeypatch.delenv("ADASUM_ONCHIP")
    # nearly opposite pairs: every segment is flagged; 5,000 positions go to the on-chip
    # recompute, 70,001 to the fp64 path
    gen = torch.Generator(device=DEV).manual_seed(77)
    lengths = [70_001, 5_000, 17]
    offs = workloads.offsets_from_numels(lengths)
    n = int(offs[-1])
    grads = []
    for _ in range(8):
        a = torch.randn(n, generator=gen, device=DEV)
        grads += [a, -(1 - 1e-3) * a + 1e-4 * torch.randn(n, generator=gen, device=DEV)]
    out = ags.reduce(grads, offs)
    torch.cuda.synchronize()
    check_against_oracle(grads, offs, out)
    assert ags.recomputed_segments() >= 2
    assert ags.get_last_error() == ags.Status.OK
    assert hooks.adasum_debug_workspace_guards() == 0


def test_guard_query_is_unsupported_in_the_product_library(native):
    assert ags.load_library().adasum_debug_workspace_guards() == -1
