import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size parity cases (minutes of CPU oracle time)")


@pytest.fixture(scope="session")
def lib():
    """The CUDA library through its C ABI (GPU tests only)."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gptq_post_weight_gb300 import _lib

    return _lib.load()


@pytest.fixture(scope="session")
def oracle_folds():
    """oracle.fold(hp, n, lam), computed once per `key` for the whole session
    (the f64 fold of a full-size group takes minutes on the host)."""
    import oracle

    cache = {}

    def get(hp, n, lam, key):
        k = (key, n, float(lam))
        if k not in cache:
            cache[k] = oracle.fold(hp, n, lam)
        return cache[k]

    return get
