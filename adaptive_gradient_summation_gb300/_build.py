"""Build libadasum_gb300.so in-tree with nvcc for sm_103a (no torch involvement).

Translation units compile in parallel, then link into one shared library next to this
file, with the CUDA runtime linked statically so the library needs only the driver.
Only the C ABI symbols of include/adasum.h are exported.

Two variants are built from the same sources:
  libadasum_gb300.so       the product: reads no environment variable
  libadasum_gb300_test.so  the test build (-DADASUM_TEST_HOOKS -DADASUM_BOUNDS_CHECK):
                           device-side index checks on every tile, chunk and segment
                           descriptor (a failure sets a status bit, adasum_get_last_error
                           reports ADASUM_ERR_BOUNDS; nothing traps), and it also honours the
                           switches the tests use to force a route, switch a kernel off
                           or inject a fault on the host (ADASUM_ONCHIP, ADASUM_TINY,
                           ADASUM_WARP_GRAM, ADASUM_ONCHIP_FAST, ADASUM_ONCHIP_MAX_CLUSTER,
                           ADASUM_PAIR_FUSED, ADASUM_PDL, ADASUM_FAULT_INJECT)
"""
from __future__ import annotations

import concurrent.futures
import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_NAME = "libadasum_gb300.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
TEST_LIB_NAME = "libadasum_gb300_test.so"
TEST_LIB_PATH = os.path.join(PKG, TEST_LIB_NAME)
TEST_FLAGS = ["-DADASUM_TEST_HOOKS", "-DADASUM_BOUNDS_CHECK"]

SOURCES = ["adasum_api.cu", "launch_f32.cu", "launch_bf16.cu", "launch_f64.cu",
           "launch_onchip.cu", "adasum_noalloc.cu"]
HEADERS = ["adasum_internal.h", "adasum_kernels.cuh", "adasum_ptx.cuh",
           "adasum_onchip.cuh", "adasum_launch.h", "adasum_pair.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", f"-I{INCLUDE}"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return cand


def _fingerprint(extra_flags) -> str:
    h = hashlib.sha256()
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as fh:
            h.update(fh.read())
    with open(os.path.join(INCLUDE, "adasum.h"), "rb") as fh:
        h.update(fh.read())
    h.update(" ".join(ARCH + NVCC_FLAGS + list(extra_flags)).encode())
    h.update(os.uname().machine.encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra_flags=(), test_hooks: bool = False) -> str:
    """Compile and link one variant if its sources (or flags, or host arch) changed."""
    extra_flags = list(extra_flags) + (TEST_FLAGS if test_hooks else [])
    lib_path = TEST_LIB_PATH if test_hooks else LIB_PATH
    fp = _fingerprint(extra_flags)
    stamp = lib_path + ".stamp"
    if (not force and os.path.exists(lib_path) and os.path.exists(stamp)
            and open(stamp).read().strip() == fp):
        return lib_path
    build_dir = os.path.join(BUILD_DIR, "test" if test_hooks else "product")
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    with open(stamp, "w") as fh:
        fh.write(fp + "\n")
    return lib_path


def build_all(force: bool = False, verbose: bool = False) -> list:
    """Both variants, concurrently."""
    with concurrent.futures.ThreadPoolExecutor(max_workers=2) as ex:
        futs = [ex.submit(build, force, verbose, (), th) for th in (False, True)]
        return [f.result() for f in futs]


if __name__ == "__main__":
    print(build_all(force=True, verbose=True))
