"""Failure detection on the device, without a GPU fault.

Every wait of the library's kernels is bounded: when a copy or an MMA never
completes, the waiting role records QG_ERR_TIMEOUT in a device status word
and the kernel returns.  qg_selftest_wait_timeout makes one wait run out on
purpose (an mbarrier that nothing arrives on, a short limit); the host must
read QG_ERR_TIMEOUT once through qg_device_status, the word must be cleared
by that read, and the context must still run work afterwards.
"""
import numpy as np
import pytest

import bit_quantized_tensor_gb300 as qg
from bit_quantized_tensor_gb300 import inputs


def test_selftest_rejects_bad_limits():
    L = qg.lib()
    assert L.qg_selftest_wait_timeout(0, None) == qg.QG_ERR_INVALID_ARG
    assert L.qg_selftest_wait_timeout(2_000_000_000, None) == qg.QG_ERR_INVALID_ARG


@pytest.mark.gpu
def test_wait_that_runs_out_is_reported_and_context_survives(oracle):
    import torch
    assert torch.cuda.is_available()
    L = qg.lib()
    assert qg.device_status() == qg.QG_OK
    assert L.qg_selftest_wait_timeout(5_000_000, None) == qg.QG_OK  # 5 ms limit
    assert qg.device_status() == qg.QG_ERR_TIMEOUT
    assert qg.device_status() == qg.QG_OK  # reading cleared it
    # twice more on another stream: each run is reported once
    s = torch.cuda.Stream()
    assert L.qg_selftest_wait_timeout(1_000_000, s.cuda_stream) == qg.QG_OK
    assert qg.device_status(s) == qg.QG_ERR_TIMEOUT
    assert qg.device_status(s) == qg.QG_OK
    # the context still computes correctly
    A = inputs.s8_uniform(300, 512, 1900)
    B = inputs.s8_uniform(260, 512, 2900)
    C = qg.qgemm_s8(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()).cpu().numpy()
    assert np.array_equal(C, oracle.gemm_s8(A, B))
    assert qg.device_status() == qg.QG_OK
