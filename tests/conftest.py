import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# the library's test-only switches (include/sgemm_testing.h) act only in a
# process whose environment allows them
os.environ["SGEMM_TEST_SWITCHES"] = "1"


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libsgemm")
    config.addinivalue_line("markers", "slow: CPU test that takes more than a few seconds")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


@pytest.fixture(scope="session")
def lib():
    """The built GPU library; a missing library is an error on a GPU machine, never a skip."""
    import dense_fp32_matrix_04_gb300 as sg
    return sg.load()
