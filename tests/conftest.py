import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libkda.so")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()


@pytest.fixture(scope="session")
def kda_lib():
    """libkda.so, built here if missing or stale (nvcc cross-compiles without a GPU)."""
    from kda_linear_attention_chunk_gb300 import build as kbuild
    import kda_linear_attention_chunk_gb300 as kda
    if kbuild.stale():
        kbuild.build()
    return kda.load()


@pytest.fixture(autouse=True)
def _no_device_timeouts(request):
    """Every GPU test must leave no bounded-wait timeout (bit 1 of the device
    error word) behind: a kernel that gave up on a wait wound down early, and
    its outputs must not be mistaken for results."""
    if request.node.get_closest_marker("gpu") is None:
        yield
        return
    import torch
    import kda_linear_attention_chunk_gb300 as kda
    if not torch.cuda.is_available():
        yield
        return
    request.getfixturevalue("kda_lib")   # builds libkda.so when missing or stale
    kda.device_error(reset=True)
    yield
    torch.cuda.synchronize()
    word = kda.device_error(reset=True)
    assert not (word & 1), f"a kernel wait timed out during the test (device error word {word:#x})"
