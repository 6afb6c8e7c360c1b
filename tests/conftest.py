import os
import sys
import threading

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the compiled libbigemm.so")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu-marked test run without a CUDA device")
    return torch.device("cuda:0")


_BUILTIN_SCRATCH = threading.Lock()


@pytest.fixture
def builtin_scratch(cuda_device):
    """Held by every test that uses the library's built-in scratch array
    (bigemm_run_splitk_static and the failure self-tests): calls that overlap
    on the GPU would race on it, so such tests never run at the same time,
    whatever runner or thread runs them, and each leaves the device idle."""
    import torch
    with _BUILTIN_SCRATCH:
        torch.cuda.synchronize()
        yield
        torch.cuda.synchronize()
