"""GB300-native Adasum: the data-parallel gradient combine of "Scaling Distributed
Training with Adaptive Summation" (Maleki et al., arXiv 2006.02924), on one GPU.

K worker gradients, each a flat vector split into layer segments, are combined per
segment by a binary tree of the Adasum pair operator (Section 3):

    Adasum(a, b) = (1 - a.b/(2|a|^2)) a + (1 - a.b/(2|b|^2)) b

All arithmetic runs in hand-written sm_103a kernels behind the C ABI of
include/adasum.h (libadasum_gb300.so).  This module only marshals torch tensors into
that ABI: it checks dtypes, devices, lengths and contiguity, passes pointers and the
current CUDA stream, and raises AdasumError on a non-OK status.  There is no CPU or
PyTorch fallback: if the library is not built, every call raises.
"""
from __future__ import annotations

import ctypes
from typing import Sequence

import numpy as np
import torch

from ._native import AdasumError, KernelStat, Status, check, library_path, load_library

__all__ = ["reduce", "pair", "pair_noalloc", "reduce_momentum_sgd", "local_momentum_reduce", "reduce_from_host", "AdasumError",
           "Status", "load_library", "library_path", "get_last_error", "release_workspace",
           "launch_count", "recomputed_segments", "profile_enable", "profile_collect", "version"]

_DTYPE_CODE = {torch.float32: 0, torch.bfloat16: 1}


def _as_list(grads) -> list:
    if isinstance(grads, torch.Tensor):
        if grads.dim() != 2:
            raise ValueError("a tensor of gradients must be 2-D (K x N)")
        return list(grads.unbind(0))
    return list(grads)


def _check_grads(grads: list):
    if len(grads) == 0:
        raise ValueError("need at least one gradient")
    g0 = grads[0]
    if g0.dtype not in _DTYPE_CODE:
        raise TypeError(f"gradients must be float32 or bfloat16, got {g0.dtype}")
    if g0.device.type != "cuda":
        raise ValueError("gradients must be CUDA tensors (use reduce_from_host for host data)")
    n = g0.numel()
    for g in grads:
        if g.dtype != g0.dtype or g.device != g0.device:
            raise ValueError("all gradients must share dtype and device")
        if g.dim() != 1 or g.numel() != n:
            raise ValueError("all gradients must be 1-D with the same length")
        if not g.is_contiguous():
            raise ValueError("gradients must be contiguous")
    return g0.dtype, g0.device, n


def _offsets(seg_offsets, n: int) -> np.ndarray:
    if seg_offsets is None:
        return np.array([0, n], dtype=np.int64)
    if isinstance(seg_offsets, torch.Tensor):
        seg_offsets = seg_offsets.detach().cpu().numpy()
    offs = np.ascontiguousarray(np.asarray(seg_offsets, dtype=np.int64))
    if offs.ndim != 1 or offs.shape[0] < 1:
        raise ValueError("seg_offsets must be a 1-D sequence of L+1 offsets")
    if offs[-1] != n:
        raise ValueError(f"seg_offsets must end at the gradient length {n}, got {offs[-1]}")
    return offs


def _stream_handle(device, stream):
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def reduce(grads, seg_offsets=None, *, out: torch.Tensor | None = None,
           stream: torch.cuda.Stream | None = None, chain: bool = False,
           orthogonality: bool = False):
    """Adasum of K worker gradients per segment (``adasum_reduce``; with ``chain=True``
    the left-to-right recursion of ``adasum_reduce_chain``, K <= 16; with
    ``orthogonality=True`` also the per-segment metric |A|^2 / sum_k |g_k|^2 of
    ``adasum_reduce_orthogonality``, returned as ``(out, ortho)``).

    grads: K 1-D CUDA tensors (float32 or bfloat16, equal length), or a K x N tensor.
    seg_offsets: L+1 offsets (segment s = [offs[s], offs[s+1])); None = one segment.
    out: optional output (same dtype/device/length); may be one of the gradients.
    Returns ``out``.  Asynchronous on the current (or given) stream.
    """
    grads = _as_list(grads)
    dtype, device, n = _check_grads(grads)
    offs = _offsets(seg_offsets, n)
    if out is None:
        out = torch.empty(n, dtype=dtype, device=device)
    elif out.dtype != dtype or out.device != device or out.numel() != n or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor like the gradients")
    lib = load_library()
    K = len(grads)
    ptrs = (ctypes.c_void_p * K)(*[g.data_ptr() for g in grads])
    L = offs.shape[0] - 1
    offs_p = offs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    with torch.cuda.device(device):
        if orthogonality:
            if chain:
                raise ValueError("the orthogonality metric is defined for the tree")
            ortho = torch.empty(max(L, 0), dtype=torch.float32, device=device)
            st = lib.adasum_reduce_orthogonality(ptrs, K, offs_p, L, _DTYPE_CODE[dtype],
                                                 ctypes.c_void_p(out.data_ptr()),
                                                 ctypes.c_void_p(ortho.data_ptr()),
                                                 _stream_handle(device, stream))
            check(st, "adasum_reduce_orthogonality")
            return out, ortho
        fn = lib.adasum_reduce_chain if chain else lib.adasum_reduce
        st = fn(ptrs, K, offs_p, L, _DTYPE_CODE[dtype], ctypes.c_void_p(out.data_ptr()),
                _stream_handle(device, stream))
    check(st, "adasum_reduce_chain" if chain else "adasum_reduce")
    return out


def pair(a: torch.Tensor, b: torch.Tensor, *, out: torch.Tensor | None = None,
         stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Adasum(a, b) of two equal-length CUDA vectors (``adasum_pair``)."""
    dtype, device, n = _check_grads([a, b])
    if out is None:
        out = torch.empty(n, dtype=dtype, device=device)
    elif out.dtype != dtype or out.device != device or out.numel() != n or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor like the inputs")
    lib = load_library()
    with torch.cuda.device(device):
        st = lib.adasum_pair(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()), n,
                             _DTYPE_CODE[dtype], ctypes.c_void_p(out.data_ptr()),
                             _stream_handle(device, stream))
    check(st, "adasum_pair")
    return out


def pair_noalloc(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor, *,
                 stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Adasum(a, b) without any device allocation (``adasum_pair_noalloc``), for callers
    that cannot allocate device memory.  ``out`` must be provided; n is limited to
    ADASUM_NOALLOC_MAX_N (33,554,432) elements."""
    dtype, device, n = _check_grads([a, b])
    if out.dtype != dtype or out.device != device or out.numel() != n or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor like the inputs")
    lib = load_library()
    with torch.cuda.device(device):
        st = lib.adasum_pair_noalloc(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()),
                                     n, _DTYPE_CODE[dtype], ctypes.c_void_p(out.data_ptr()),
                                     _stream_handle(device, stream))
    check(st, "adasum_pair_noalloc")
    return out


def reduce_momentum_sgd(grads, seg_offsets, master_w: torch.Tensor, momentum: torch.Tensor, *,
                        lr: float, mu: float, out: torch.Tensor | None = None,
                        stream: torch.cuda.Stream | None = None):
    """Adasum then one heavy-ball step, fused (``adasum_reduce_momentum_sgd``):
    v <- mu v + Adasum(g),  w <- w - lr v, updating ``master_w`` and ``momentum`` (fp32)
    in place.  ``out`` (optional) receives the Adasum result in the gradient dtype."""
    grads = _as_list(grads)
    dtype, device, n = _check_grads(grads)
    offs = _offsets(seg_offsets, n)
    for name, t in (("master_w", master_w), ("momentum", momentum)):
        if t.dtype != torch.float32 or t.device != device or t.numel() != n or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float32 tensor of {n} elements on {device}")
    if out is not None and (out.dtype != dtype or out.device != device or out.numel() != n
                            or not out.is_contiguous()):
        raise ValueError("out must be a contiguous tensor like the gradients")
    lib = load_library()
    K = len(grads)
    ptrs = (ctypes.c_void_p * K)(*[g.data_ptr() for g in grads])
    with torch.cuda.device(device):
        st = lib.adasum_reduce_momentum_sgd(
            ptrs, K, offs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), offs.shape[0] - 1,
            _DTYPE_CODE[dtype], ctypes.c_void_p(master_w.data_ptr()),
            ctypes.c_void_p(momentum.data_ptr()), float(lr), float(mu),
            ctypes.c_void_p(0 if out is None else out.data_ptr()), _stream_handle(device, stream))
    check(st, "adasum_reduce_momentum_sgd")
    return master_w, momentum, out


def local_momentum_reduce(grads, seg_offsets, momenta, master_w: torch.Tensor, *, lr: float,
                          mu: float, stream: torch.cuda.Stream | None = None):
    """Adasum after the optimizer (``adasum_local_momentum_reduce``): every worker k takes
    its own heavy-ball step v_k <- mu v_k + g_k (``momenta[k]``, fp32, in place), then
    w <- w - lr Adasum(v_0, ..., v_{K-1}) updates ``master_w`` in place."""
    grads = _as_list(grads)
    dtype, device, n = _check_grads(grads)
    offs = _offsets(seg_offsets, n)
    momenta = list(momenta)
    if len(momenta) != len(grads):
        raise ValueError("one momentum buffer per worker")
    for t in momenta + [master_w]:
        if t.dtype != torch.float32 or t.device != device or t.numel() != n or not t.is_contiguous():
            raise ValueError(f"states must be contiguous float32 tensors of {n} elements on {device}")
    lib = load_library()
    K = len(grads)
    gp = (ctypes.c_void_p * K)(*[g.data_ptr() for g in grads])
    vp = (ctypes.c_void_p * K)(*[v.data_ptr() for v in momenta])
    with torch.cuda.device(device):
        st = lib.adasum_local_momentum_reduce(
            gp, K, offs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), offs.shape[0] - 1,
            _DTYPE_CODE[dtype], vp, ctypes.c_void_p(master_w.data_ptr()), float(lr), float(mu),
            _stream_handle(device, stream))
    check(st, "adasum_local_momentum_reduce")
    return master_w, momenta


def reduce_from_host(grads_host: Sequence[torch.Tensor], seg_offsets=None, *,
                     out_host: torch.Tensor | None = None,
                     stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """End-to-end Adasum of gradients held in host memory (``adasum_reduce_host``): the
    library copies them to the current device, combines them and copies the result back,
    pipelining groups of whole segments so that transfers and compute overlap, and
    returns once ``out_host`` holds the result.

    grads_host: K 1-D CPU tensors (float32 or bfloat16, equal length; pinned memory is
    copied asynchronously at full speed).  out_host: optional CPU tensor for the result
    (pinned by default); it may be one of the inputs.
    """
    grads_host = list(grads_host)
    if not grads_host:
        raise ValueError("need at least one gradient")
    g0 = grads_host[0]
    if g0.dtype not in _DTYPE_CODE:
        raise TypeError(f"gradients must be float32 or bfloat16, got {g0.dtype}")
    n = g0.numel()
    for g in grads_host:
        if g.device.type != "cpu" or g.dtype != g0.dtype or g.dim() != 1 or g.numel() != n \
                or not g.is_contiguous():
            raise ValueError("host gradients must be contiguous 1-D CPU tensors of one dtype and length")
    offs = _offsets(seg_offsets, n)
    if out_host is None:
        out_host = torch.empty(n, dtype=g0.dtype, pin_memory=True)
    elif (out_host.device.type != "cpu" or out_host.dtype != g0.dtype or out_host.numel() != n
          or not out_host.is_contiguous()):
        raise ValueError("out_host must be a contiguous CPU tensor like the gradients")
    lib = load_library()
    K = len(grads_host)
    ptrs = (ctypes.c_void_p * K)(*[g.data_ptr() for g in grads_host])
    device = torch.device("cuda", torch.cuda.current_device())
    st = lib.adasum_reduce_host(ptrs, K, offs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                offs.shape[0] - 1, _DTYPE_CODE[g0.dtype],
                                ctypes.c_void_p(out_host.data_ptr()), _stream_handle(device, stream))
    check(st, "adasum_reduce_host")
    return out_host


def get_last_error() -> int:
    """Device-side status after a synchronisation (``adasum_get_last_error``)."""
    return Status(load_library().adasum_get_last_error())


def release_workspace() -> None:
    check(load_library().adasum_release_workspace(), "adasum_release_workspace")


def launch_count() -> int:
    return int(load_library().adasum_launch_count())


def recomputed_segments() -> int:
    """Segments the last call recomputed in fp64 (synchronises the device)."""
    return int(load_library().adasum_recomputed_segments())


def profile_enable(on: bool = True) -> None:
    check(load_library().adasum_profile_enable(1 if on else 0), "adasum_profile_enable")


def profile_collect() -> dict:
    """{kernel name: (launches, total device ms, total algorithmic bytes)} since the last
    collect (bytes 0 for kernels the library does not rate)."""
    lib = load_library()
    cap = 64
    arr = (KernelStat * cap)()
    n = lib.adasum_profile_collect(arr, cap)
    return {arr[i].name.decode(): (int(arr[i].launches), float(arr[i].total_ms),
                                   float(arr[i].total_bytes))
            for i in range(min(n, cap))}


def version() -> str:
    v = int(load_library().adasum_version())
    return f"{v // 10000}.{(v // 100) % 100}.{v % 100}"
