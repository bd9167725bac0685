import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle

    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def fa():
    """The product binding, with its CUDA library loaded (GPU tests only)."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_kv_cache_sm_gb300 as fa_mod

    fa_mod.load()
    return fa_mod


@pytest.fixture(scope="session")
def built():
    """The product binding with its library built and loaded; no device needed (host queries and
    argument checks only)."""
    import quantized_kv_cache_sm_gb300 as fa_mod
    from quantized_kv_cache_sm_gb300 import build as fa_build

    fa_build.build()
    fa_mod.load()
    return fa_mod
