import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


@pytest.fixture(scope="session")
def cuda_dev():
    """The CUDA device for -m gpu tests.  A GPU test on a machine without CUDA fails, it does not skip."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu test needs CUDA, none is available")
    return torch.device("cuda:0")


_INPUT_CACHE = {}


@pytest.fixture(scope="session")
def workload_inputs():
    """Session cache: name -> (CPU Inputs, device Inputs) for the named workloads."""
    import torch
    from workloads import WORKLOADS, make_inputs, to_device

    def get(name):
        if name not in _INPUT_CACHE:
            cpu = make_inputs(WORKLOADS[name])
            dev = to_device(cpu, torch.device("cuda:0"))
            _INPUT_CACHE[name] = (cpu, dev)
        return _INPUT_CACHE[name]

    yield get
    _INPUT_CACHE.clear()
