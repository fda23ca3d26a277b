import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def native():
    """The CUDA library's Python binding; GPU tests only."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    import adaptive_gradient_summation_gb300 as ags
    ags.load_library()
    return ags


@pytest.fixture
def hooks(native):
    """Run the test on the test build of the library (built with -DADASUM_TEST_HOOKS),
    which honours the ADASUM_* environment switches (forced routes, kernels switched off,
    host-side fault injection); the product library reads no environment."""
    from adaptive_gradient_summation_gb300 import _native
    lib = _native.load_library(test_hooks=True)
    prev = _native.use_library(lib)
    try:
        yield lib
    finally:
        _native.use_library(prev)
