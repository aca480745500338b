import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


@pytest.fixture(scope="session")
def gpu_lib():
    """The CUDA library, built in-tree if needed; the tests that use it are
    marked gpu and fail (not skip) when it cannot be built or loaded."""
    import draft_token_markov_gb300.build as b
    b.build()
    from draft_token_markov_gb300 import api
    return api
