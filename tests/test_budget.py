"""Resource accounting of every kernel instance the library launches.

Smoke tests do not see a kernel that asks an SM for more than it has, or a
design that relies on two CTAs per SM when registers or shared memory only
allow one ("Warp-Specialized Kernel Implementation for W4A4 MatMul ...", on
budget tables and unit tests for resource accounting).  On the host the
table's own numbers are checked against the SM's shared memory and tensor
memory; on a device the compiled kernels' real residency (registers
included) must reach what the design counts on, and the tensor-memory
kernels must never fit two CTAs on one SM, since a second CTA's allocation
would wait on the first (and, for CTA pairs, could wait in a cycle).
"""
import pytest

import bit_quantized_tensor_gb300 as qg
from bit_quantized_tensor_gb300 import budget


@pytest.fixture(scope="module")
def rows():
    return qg.kernel_budgets()


def test_table_lists_every_launched_kernel(rows):
    names = [r["kernel"] for r in rows]
    assert len(names) == len(set(names)), "kernel registered twice"
    for stem in ("tc_gemm_kernel<", "tc_gemm2_kernel<", "k_expand<", "k_w4a16_gemv<", "k_w4a16_gemv16<",
                 "w4a16_tc_kernel", "k_w4a16<", "k_w4a16_dec<", "k_w4a4_quantize<", "k_scales_transposed",
                 "w4a4_gemm_kernel", "w4a4_gemm2_kernel", "tc_gemm2_s4raw_kernel"):
        assert any(n.startswith(stem) for n in names), stem
    assert len(names) == 33


def test_host_accounting(rows):
    bad = {r["kernel"]: budget.accounting_errors(r) for r in rows if budget.accounting_errors(r)}
    assert not bad, bad


def test_tensor_memory_kernels_stay_alone_on_their_sm(rows):
    for r in rows:
        if r["tmem_cols"]:
            # even with room in tensor memory for a second CTA, shared memory
            # must keep one per SM (the CTA-pair kernels take all 512 columns)
            assert 2 * (r["smem_bytes"] + budget.CTA_RESERVED_SMEM) > budget.SM_SMEM_BYTES, r["kernel"]


def test_planted_overbudget_entries_are_caught():
    ok = {"kernel": "x", "threads": 512, "smem_bytes": 110 * 1024, "tmem_cols": 0, "cluster": 1,
          "min_ctas_per_sm": 2}
    assert budget.accounting_errors(ok) == []
    assert budget.accounting_errors(dict(ok, smem_bytes=115 * 1024))  # two no longer fit
    assert budget.accounting_errors(dict(ok, smem_bytes=232449, min_ctas_per_sm=1))
    assert budget.accounting_errors(dict(ok, tmem_cols=512))  # two CTAs x 512 columns
    assert budget.accounting_errors(dict(ok, tmem_cols=96, min_ctas_per_sm=1))  # not a power of two
    assert budget.accounting_errors(dict(ok, threads=1056))
    assert budget.accounting_errors(dict(ok, cluster=16))


def test_table_prints(rows):
    text = budget.format_table(rows)
    assert text.count("\n") == len(rows)
    assert "w4a16_tc_kernel" in text


def test_measure_without_a_device_reports_a_cuda_error():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    a, b, c = qg._int(), qg._int(), qg._int()
    import ctypes
    rc = qg.lib().qg_kernel_budget_measure(0, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c))
    assert rc == qg.QG_ERR_CUDA
    assert qg.lib().qg_kernel_budget_measure(-1, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)) \
        == qg.QG_ERR_INVALID_ARG


@pytest.mark.gpu
def test_device_residency_matches_the_design():
    rows = qg.kernel_budgets(measure=True)
    for r in rows:
        assert r["regs_per_thread"] > 0, r
        assert r["static_smem_bytes"] + r["smem_bytes"] <= budget.CTA_SMEM_LIMIT, r
        assert r["ctas_per_sm"] >= r["min_ctas_per_sm"], r
        if r["tmem_cols"]:
            assert r["ctas_per_sm"] * r["tmem_cols"] <= budget.TMEM_COLUMNS, r
            assert r["ctas_per_sm"] == 1, r
