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
    config.addinivalue_line("markers", "tiny: GPU test that keeps the one-thread-per-output path for tiny products on")


@pytest.fixture(autouse=True)
def _tiny_path(request):
    """GPU tests run with the tiny-product kernel off, so that their small shapes
    reach the tiled kernels' edge handling; tests marked `tiny` keep it on."""
    if request.node.get_closest_marker("gpu") is None:
        yield
        return
    import dense_fp32_matrix_04_gb300 as sg
    sg.sgemm_test_tiny_path(request.node.get_closest_marker("tiny") is not None)
    yield
    sg.sgemm_test_tiny_path(True)


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
