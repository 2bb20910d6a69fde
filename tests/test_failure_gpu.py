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
    for pattern in (0, 4, -1):
        assert L.qg_selftest_deadlock(pattern, 1_000_000, None) == qg.QG_ERR_INVALID_ARG
    assert L.qg_selftest_deadlock(1, 0, None) == qg.QG_ERR_INVALID_ARG
    assert L.qg_selftest_deadlock(3, 1_000_000_001, None) == qg.QG_ERR_INVALID_ARG


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


# pattern -> (site tags the role that gives up may record, parity it waited on)
DEADLOCKS = {
    1: ({901}, 0),       # incomplete arrival count
    2: ({902}, 1),       # phase mismatch: waits on parity 1 after phase 0 closed
    3: ({903, 904}, 0),  # dependency cycle between a drain and an MMA role
}


@pytest.mark.gpu
@pytest.mark.parametrize("pattern", sorted(DEADLOCKS))
def test_staged_deadlocks_end_in_a_reported_timeout(oracle, pattern):
    """Each of the three deadlock patterns of a hand-built pipeline, staged
    with bounded waits, ends in QG_ERR_TIMEOUT with the stalled role's tag,
    and the parity it waited for in the status word; the call
    returns within a few multiples of the limit and the context still runs
    work afterwards."""
    import time

    import torch
    assert torch.cuda.is_available()
    L = qg.lib()
    assert qg.device_status() == qg.QG_OK
    t0 = time.perf_counter()
    assert L.qg_selftest_deadlock(pattern, 20_000_000, None) == qg.QG_OK  # 20 ms limit
    d = qg.device_status_detail()
    elapsed = time.perf_counter() - t0
    sites, parity = DEADLOCKS[pattern]
    assert d["code"] == qg.QG_ERR_TIMEOUT
    assert d["site"] in sites
    assert d["count"] >= 1 and d["block"] == 0
    assert d["parity"] == parity
    assert elapsed < 5.0
    assert qg.device_status_detail()["code"] == qg.QG_OK  # reading cleared it
    A = inputs.s8_uniform(130, 256, 1910 + pattern)
    B = inputs.s8_uniform(70, 256, 2910 + pattern)
    C = qg.qgemm_s8(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()).cpu().numpy()
    assert np.array_equal(C, oracle.gemm_s8(A, B))
    assert qg.device_status() == qg.QG_OK
