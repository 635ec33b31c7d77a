import os
import sys

import pytest

TESTS = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(TESTS)
for p in (ROOT, TESTS):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle

    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def exattn_lib():
    """The built C library (compiled here if stale); no GPU needed to load it."""
    from exact_attention_65_gb300 import build

    build.build()
    import exact_attention_65_gb300 as ea

    return ea.load_library()


@pytest.fixture(scope="session")
def gpu(exattn_lib):
    """The CUDA path: the library plus a visible device. Fails (never skips)
    when no GPU is present, so a GPU run cannot pass vacuously."""
    import torch

    if not torch.cuda.is_available():
        raise RuntimeError("GPU tests need a CUDA device")
    import exact_attention_65_gb300 as ea

    torch.cuda.init()
    return ea
