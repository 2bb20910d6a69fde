"""Host logic of bench.py that needs no device: regression floors and the
ablation table."""
import bench


def _breakdown(scale=1.0):
    return {entry: {key: floor * scale} for (entry, key), floor in bench.FLOORS.items()}


def test_floors_pass_at_and_above_the_floor():
    assert bench.check_floors(_breakdown(1.0)) == {"ok": True, "failed": []}
    assert bench.check_floors(_breakdown(1.2))["ok"]


def test_a_planted_regression_is_reported():
    b = _breakdown(1.1)
    b["w4a16_m1_4096"]["frac_of_hbm"] = 0.05
    out = bench.check_floors(b)
    assert not out["ok"]
    assert [f["op"] for f in out["failed"]] == ["w4a16_m1_4096"]
    assert out["failed"][0]["value"] == 0.05


def test_a_missing_entry_counts_as_a_miss():
    b = _breakdown(1.1)
    del b["int4_gemm_8192"]
    out = bench.check_floors(b)
    assert [f["op"] for f in out["failed"]] == ["int4_gemm_8192"]


def test_ablation_knobs_name_library_setters_and_known_ops():
    import bit_quantized_tensor_gb300 as qg
    for name, (setter, values, ops) in bench.ABLATIONS.items():
        assert setter in qg.SIGNATURES, name
        assert len(values) >= 2 and len(set(values)) == len(values), name
        assert set(ops) <= set(bench.OPS), name


def test_sweep_working_sets_and_l2_labels():
    # int8: A, B (1 B each), C (4 B), fp16 copies of A and B (2 B each)
    assert bench.sweep_working_set("s8", 512) == (2 + 4 + 4) * 512 * 512
    # int4: packed A, B (n^2 bytes together), C, e4m3 copies (1 B each)
    assert bench.sweep_working_set("s4", 2048) == (1 + 4 + 2) * 2048 * 2048
    assert bench.sweep_working_set("f16", 4096) == 6 * 4096 * 4096
    # the two small workload definitions fit in a 126 MiB L2, 4096^3 INT8 does not
    l2 = 126 << 20
    assert bench.sweep_working_set("s8", 512) <= l2 and bench.sweep_working_set("s4", 2048) <= l2
    assert bench.sweep_working_set("s8", 4096) > l2


def test_w4a4_floor_is_against_the_fp8_kind():
    keys = [k for (e, k) in bench.FLOORS if e.startswith("w4a4")]
    assert keys == ["frac_of_fp8_peak"]
