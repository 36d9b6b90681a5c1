import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libnq.so")
    config.addinivalue_line("markers", "slow: statistical tests that take tens of seconds")


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="session")
def nq():
    """The CUDA binding, with libnq.so built for sm_103a (fails loudly if it cannot be)."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    from quantized_self_speculative_gb300 import build, nq as binding
    build.build()
    binding.lib()
    return binding
