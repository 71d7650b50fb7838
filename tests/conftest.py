import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture
def tuning():
    """Set launch-plan overrides through the C ABI (ssm_set_tuning) for one test; each knob
    set is put back to automatic (0) afterwards."""
    from speculative_decoding_mamba2_gb300 import ssm_set_tuning
    names = []

    def set_(name, value):
        ssm_set_tuning(name, int(value))
        names.append(name)

    yield set_
    for name in names:
        ssm_set_tuning(name, 0)
