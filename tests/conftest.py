"""Shared test setup: repo root on sys.path, markers, GPU skip logic."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a kernels via the C ABI)")
    config.addinivalue_line("markers", "slow: full-size workloads")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def zlib():
    """The built C-ABI library (compiled in-tree for sm_103a if stale), or the
    prebuilt variant library named by ZGB_TEST_LIB: a test that checks an
    opt-in build runs this suite's cases against it in a child process."""
    from zero_sharded_mixed_gb300 import binding, build
    variant = os.environ.get("ZGB_TEST_LIB")
    if variant:
        binding.lib_path = variant
        binding._lib = None
    else:
        build.build()
    binding.load()
    return binding


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    torch.cuda.init()
    return torch.device("cuda", 0)
