"""Plain fp64 CPU oracle for the Adasum combine (ctypes loader for adasum_oracle.c).

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package; the product path (the CUDA library and its
Python binding) never does, and shares no code with it.

What the oracle computes, and the passages it follows, are stated in the header of
``adasum_oracle.c``: the pair operator of "Scaling Distributed Training with Adaptive
Summation" (Section 3, Equations 1-2, Appendix A.1-A.2), its binary-tree application over
workers (Section 3), per-layer segments (Section 3, after Figure 1) and the orthogonality
metric of Figure 1.  Every function here is pinned by tests against values fixed by the
paper and by mathematics (closed forms, exact rational arithmetic on an independent
derivation, library routines), not against itself.

Arrays are numpy: fp32 data as ``np.float32``; bf16 data as its raw bits in
``np.uint16`` (numpy has no bfloat16 type).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "adasum_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libadasum_oracle.so")

F32 = 0
BF16 = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle C source into a shared library (gcc, no FMA contraction)."""
    stale = (not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src))
    if force or stale:
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, src, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def open_library(path: str):
    """Load a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    vp, i64, dp = ctypes.c_void_p, ctypes.c_int64, ctypes.POINTER(ctypes.c_double)
    lib.oracle_adasum_reduce.argtypes = [ctypes.POINTER(vp), ctypes.c_int,
                                         ctypes.POINTER(i64), ctypes.c_int,
                                         ctypes.c_int, vp, dp, dp, dp]
    lib.oracle_adasum_reduce.restype = ctypes.c_int
    lib.oracle_adasum_chain.argtypes = lib.oracle_adasum_reduce.argtypes
    lib.oracle_adasum_chain.restype = ctypes.c_int
    lib.oracle_adasum_pair.argtypes = [vp, vp, i64, ctypes.c_int, vp, dp]
    lib.oracle_adasum_pair.restype = ctypes.c_int
    lib.oracle_momentum_sgd.argtypes = [dp, i64, vp, vp, ctypes.c_double,
                                        ctypes.c_double, vp, vp]
    lib.oracle_momentum_sgd.restype = ctypes.c_int
    lib.oracle_local_momentum_adasum.argtypes = [ctypes.POINTER(vp), ctypes.c_int,
                                                 ctypes.POINTER(i64), ctypes.c_int, ctypes.c_int,
                                                 ctypes.POINTER(vp), vp, ctypes.c_double,
                                                 ctypes.c_double]
    lib.oracle_local_momentum_adasum.restype = ctypes.c_int
    lib.oracle_bf16_encode.argtypes = [ctypes.c_double]
    lib.oracle_bf16_encode.restype = ctypes.c_uint16
    lib.oracle_bf16_decode.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_decode.restype = ctypes.c_double
    return lib


def _load(lib=None):
    global _lib
    if lib is not None:
        return lib
    with _lock:
        if _lib is None:
            _lib = open_library(build())
    return _lib


def _dtype_code(arr: np.ndarray) -> int:
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle inputs are float32 or bf16 bits (uint16), got {arr.dtype}")


def _dptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def adasum_reduce(grads, seg_offsets, *, want_out=True, want_mag=False, want_ortho=False,
                  lib=None, chain=False):
    """Adasum of K worker gradients, per segment, as a binary tree (fp64).

    grads: sequence of K 1-D arrays (all float32, or all uint16 bf16 bits) of equal length.
    seg_offsets: L+1 non-decreasing int64 offsets; segment s is [offs[s], offs[s+1]).
    Returns a dict with ``out64`` (fp64 result), ``out`` (rounded to the input dtype),
    and optionally ``mag`` (magnitude bound per element) and ``ortho`` (per segment).
    ``lib`` selects another compiled copy of the oracle (default: the one built here).
    ``chain=True`` uses the linear recursion g[0,n+1] = Adasum(g[0,n], g_{n+1}) instead of
    the binary tree.
    """
    lib = _load(lib)
    grads = [np.ascontiguousarray(g) for g in grads]
    K = len(grads)
    if K == 0:
        raise ValueError("need at least one gradient")
    code = _dtype_code(grads[0])
    n = grads[0].shape[0]
    for g in grads:
        if g.ndim != 1 or g.shape[0] != n or _dtype_code(g) != code:
            raise ValueError("all gradients must be 1-D, the same length and dtype")
    offs = np.ascontiguousarray(seg_offsets, dtype=np.int64)
    L = offs.shape[0] - 1
    if L < 0 or (L >= 0 and offs[-1] != n):
        raise ValueError("seg_offsets must end at the gradient length")
    ptrs = (ctypes.c_void_p * K)(*[g.ctypes.data for g in grads])
    out64 = np.empty(n, dtype=np.float64)
    out = np.empty(n, dtype=grads[0].dtype) if want_out else None
    mag = np.empty(n, dtype=np.float64) if want_mag else None
    ortho = np.empty(max(L, 0), dtype=np.float64) if want_ortho else None
    fn = lib.oracle_adasum_chain if chain else lib.oracle_adasum_reduce
    rc = fn(ptrs, K, offs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                  L, code, None if out is None else out.ctypes.data,
                                  _dptr(out64), _dptr(mag), _dptr(ortho))
    if rc != 0:
        raise ValueError(f"oracle_adasum_reduce failed with code {rc}")
    res = {"out64": out64}
    if want_out:
        res["out"] = out
    if want_mag:
        res["mag"] = mag
    if want_ortho:
        res["ortho"] = ortho
    return res


def adasum_pair(a, b, lib=None):
    """Adasum(a, b) for two equal-length vectors; returns (rounded, fp64)."""
    r = adasum_reduce([a, b], [0, np.asarray(a).shape[0]], lib=lib)
    return r["out"], r["out64"]


def momentum_sgd(A64, w, v, lr, mu, lib=None):
    """Heavy-ball step from the fp64 Adasum result: returns (w', v') as float32."""
    lib = _load(lib)
    A64 = np.ascontiguousarray(A64, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    n = A64.shape[0]
    if w.shape[0] != n or v.shape[0] != n:
        raise ValueError("A, w and v must have the same length")
    w_out = np.empty(n, dtype=np.float32)
    v_out = np.empty(n, dtype=np.float32)
    rc = lib.oracle_momentum_sgd(_dptr(A64), n, w.ctypes.data, v.ctypes.data,
                                 float(lr), float(mu), w_out.ctypes.data, v_out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_momentum_sgd failed with code {rc}")
    return w_out, v_out


def local_momentum_adasum(grads, seg_offsets, v, w, lr, mu, lib=None):
    """Adasum after the optimizer: per-worker heavy-ball steps v_k' = mu v_k + g_k, then
    w' = w + Adasum(-lr v_k').  Returns (v' list, w') as float32 arrays (copies)."""
    lib = _load(lib)
    grads = [np.ascontiguousarray(g) for g in grads]
    K = len(grads)
    code = _dtype_code(grads[0])
    offs = np.ascontiguousarray(seg_offsets, dtype=np.int64)
    vs = [np.array(x, dtype=np.float32, copy=True) for x in v]
    w_out = np.array(w, dtype=np.float32, copy=True)
    gp = (ctypes.c_void_p * K)(*[g.ctypes.data for g in grads])
    vp = (ctypes.c_void_p * K)(*[x.ctypes.data for x in vs])
    rc = lib.oracle_local_momentum_adasum(gp, K, offs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                          offs.shape[0] - 1, code, vp, w_out.ctypes.data,
                                          float(lr), float(mu))
    if rc != 0:
        raise ValueError(f"oracle_local_momentum_adasum failed with code {rc}")
    return vs, w_out


def bf16_encode(x, lib=None) -> np.ndarray:
    """fp64 values -> bf16 bits (uint16), one rounding to nearest even."""
    lib = _load(lib)
    x = np.asarray(x, dtype=np.float64).ravel()
    return np.fromiter((lib.oracle_bf16_encode(float(v)) for v in x), dtype=np.uint16,
                       count=x.shape[0])


def bf16_decode(h, lib=None) -> np.ndarray:
    """bf16 bits (uint16) -> exact fp64 values."""
    lib = _load(lib)
    h = np.asarray(h, dtype=np.uint16).ravel()
    return np.fromiter((lib.oracle_bf16_decode(int(v)) for v in h), dtype=np.float64,
                       count=h.shape[0])
