"""ctypes declarations for libadasum_gb300.so (the C ABI of include/adasum.h).

Argument marshalling only: no arithmetic of the method happens in Python.  Loading
fails loudly when the library has not been built; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import enum
import os
import threading

from . import _build

_lock = threading.Lock()


class Status(enum.IntEnum):
    OK = 0
    ERR_INVALID_ARG = 1
    ERR_UNSUPPORTED = 2
    ERR_ALIAS = 3
    ERR_NO_MEMORY = 4
    ERR_CUDA = 5
    ERR_TIMEOUT = 6
    ERR_BOUNDS = 7


class AdasumError(RuntimeError):
    """A non-OK status returned by the native library."""

    def __init__(self, status: int, where: str):
        self.status = Status(status) if status in Status._value2member_map_ else status
        super().__init__(f"{where}: {getattr(self.status, 'name', status)}")


class KernelStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 64), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double), ("total_bytes", ctypes.c_double)]


#: Every symbol include/adasum.h declares, with (restype, argtypes).
SIGNATURES = {
    "adasum_reduce": (ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int,
                                     ctypes.POINTER(ctypes.c_int64), ctypes.c_int,
                                     ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "adasum_reduce_host": (ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int,
                                          ctypes.POINTER(ctypes.c_int64), ctypes.c_int,
                                          ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "adasum_reduce_orthogonality": (ctypes.c_int, [
        ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, ctypes.POINTER(ctypes.c_int64),
        ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "adasum_reduce_chain": (ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int,
                                           ctypes.POINTER(ctypes.c_int64), ctypes.c_int,
                                           ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "adasum_pair": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                   ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "adasum_reduce_momentum_sgd": (ctypes.c_int, [
        ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, ctypes.POINTER(ctypes.c_int64),
        ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
        ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]),
    "adasum_pair_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                           ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "adasum_local_momentum_reduce": (ctypes.c_int, [
        ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, ctypes.POINTER(ctypes.c_int64),
        ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p,
        ctypes.c_float, ctypes.c_float, ctypes.c_void_p]),
    "adasum_get_last_error": (ctypes.c_int, []),
    "adasum_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "adasum_release_workspace": (ctypes.c_int, []),
    "adasum_version": (ctypes.c_int, []),
    "adasum_launch_count": (ctypes.c_int64, []),
    "adasum_debug_workspace_guards": (ctypes.c_int64, []),
    "adasum_recomputed_segments": (ctypes.c_int64, []),
    "adasum_profile_enable": (ctypes.c_int, [ctypes.c_int]),
    "adasum_profile_collect": (ctypes.c_int, [ctypes.POINTER(KernelStat), ctypes.c_int]),
}


def library_path() -> str:
    return _build.LIB_PATH


_libs = {}
_active = None


def _open(path: str, build_if_missing: bool, test_hooks: bool):
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(
                f"{os.path.basename(path)} is not built; run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        _build.build(test_hooks=test_hooks)
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load_library(build_if_missing: bool = False, test_hooks: bool = False):
    """The library the binding calls: the product build, unless a test has made the test
    build active (use_library).  ``test_hooks=True`` returns the test build itself.
    Raises if the requested library is not built."""
    with _lock:
        if not test_hooks and _active is not None:
            return _active
        path = _build.TEST_LIB_PATH if test_hooks else _build.LIB_PATH
        if path not in _libs:
            _libs[path] = _open(path, build_if_missing, test_hooks)
        return _libs[path]


def use_library(lib):
    """Make `lib` the library every binding call goes to (None: the product build);
    returns the previous choice.  Tests use it to run on the test build."""
    global _active
    with _lock:
        prev, _active = _active, lib
    return prev


def check(status: int, where: str) -> None:
    if status != 0:
        raise AdasumError(status, where)
