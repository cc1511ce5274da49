"""The bounded waits of the TMA kernel: when its copies never arrive (a test-only
switch stops them from being issued), every block gives up after the wait
limit, writes nothing, and the device status reports the timeout; the GPU stays
usable and the next product is correct.  No fault, trap or endless loop is
involved."""

import numpy as np
import pytest

import gen
from helpers import CANARY_BITS, check_full, run_sgemm

pytestmark = pytest.mark.gpu


@pytest.fixture
def sg(cuda_device, lib):
    import dense_fp32_matrix_04_gb300 as sg
    sg.sgemm_device_status()          # start from a clear error word
    yield sg
    sg.sgemm_test_switches(0, 2_000_000_000)
    sg.sgemm_device_status()


def test_status_ok_after_normal_products(sg):
    A, B = gen.operands(64, 256, 96, seed=30)
    check_full(run_sgemm(sg, A, B), A, B)
    assert sg.sgemm_device_status() == sg.SGEMM_OK


@pytest.mark.parametrize("K", [64, 96])   # the small-K tile and the main tile
def test_timeout_is_reported_and_nothing_is_written(sg, K):
    import torch
    A, B = gen.operands(128, 256, K, seed=31)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.from_numpy(np.full((128, 256), CANARY_BITS, np.int32).view(np.float32)).cuda()
    sg.sgemm_test_switches(1, 50_000_000)     # copies never issued; 50 ms bound per wait
    sg.sgemm_f32(128, 256, K, dA, K, dB, 256, dC, 256)
    assert sg.sgemm_device_status() == sg.SGEMM_ERR_TIMEOUT
    assert np.all(dC.cpu().numpy().view(np.int32) == CANARY_BITS)
    # the status is cleared by reading it
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    # and the device is still usable
    sg.sgemm_test_switches(0, 2_000_000_000)
    sg.sgemm_f32(128, 256, K, dA, K, dB, 256, dC, 256)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    check_full(dC.cpu().numpy(), A, B)
