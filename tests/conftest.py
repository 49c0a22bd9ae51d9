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
