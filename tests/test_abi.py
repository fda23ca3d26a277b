"""CPU checks of the C ABI: the library builds, loads without a GPU, and exports every
symbol include/adasum.h declares (no compute calls here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "adasum.h")


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"ADASUM_API\s+[\w\s\*]+?\b(adasum_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("adasum_reduce", "adasum_pair", "adasum_reduce_momentum_sgd",
                     "adasum_get_last_error", "adasum_status_string"):
        assert required in names


@pytest.mark.parametrize("test_hooks", [False, True])
def test_library_builds_and_exports_every_declared_symbol(test_hooks):
    from adaptive_gradient_summation_gb300 import _build
    path = _build.build(test_hooks=test_hooks)
    lib = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in adasum.h but not exported"


def test_product_library_reads_no_environment():
    """Every environment read in the native sources sits inside an
    `#ifdef ADASUM_TEST_HOOKS` block, so only the test build honours the switches."""
    csrc = os.path.join(ROOT, "adaptive_gradient_summation_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        guarded = []
        for no, line in enumerate(open(os.path.join(csrc, f)), 1):
            t = line.strip()
            if t.startswith("#if"):
                guarded.append("ADASUM_TEST_HOOKS" in t and t.startswith("#ifdef"))
            elif t.startswith("#else") and guarded:
                guarded[-1] = False
            elif t.startswith("#endif") and guarded:
                guarded.pop()
            if "getenv" in line and not t.startswith("//"):
                assert any(guarded), f"{f}:{no} reads the environment outside the test build"


def test_binding_declares_every_symbol():
    from adaptive_gradient_summation_gb300 import _native
    assert sorted(_native.SIGNATURES) == declared_functions()


def test_status_strings_without_gpu():
    import adaptive_gradient_summation_gb300 as ags
    lib = ags.load_library(build_if_missing=True)
    for st in ags.Status:
        assert lib.adasum_status_string(int(st)).decode() == "ADASUM_" + st.name
    assert ags.version() == "0.1.0"


def test_no_oracle_on_the_product_path():
    """The package and its native sources never reference the CPU oracle."""
    pkg = os.path.join(ROOT, "adaptive_gradient_summation_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "adasum_oracle" not in text, f


def test_binding_refuses_cpu_tensors():
    import torch
    import adaptive_gradient_summation_gb300 as ags
    with pytest.raises(ValueError):
        ags.reduce([torch.zeros(4), torch.zeros(4)])


def test_kernel_stat_layout_matches_the_header(tmp_path):
    """The binding's ctypes mirror of adasum_kernel_stat_t has the header's size and
    field offsets (compiled with the host C compiler; no GPU)."""
    import shutil
    import subprocess
    from adaptive_gradient_summation_gb300 import _native
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stddef.h>\n#include <stdio.h>\n#include "adasum.h"\n'
        "int main(void) {\n"
        '  printf("%zu %zu %zu %zu %zu\\n", sizeof(adasum_kernel_stat_t),\n'
        "         offsetof(adasum_kernel_stat_t, name), offsetof(adasum_kernel_stat_t, launches),\n"
        "         offsetof(adasum_kernel_stat_t, total_ms), offsetof(adasum_kernel_stat_t, total_bytes));\n"
        "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    ks = _native.KernelStat
    want = [ctypes.sizeof(ks), ks.name.offset, ks.launches.offset, ks.total_ms.offset,
            ks.total_bytes.offset]
    assert got == want
