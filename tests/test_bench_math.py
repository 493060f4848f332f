"""The measurement arithmetic of bench.py (no GPU): algorithmic bytes and
FLOPs per launch, the peaks they are divided by, and the committed traffic
record lookup."""
import pytest

import bench
from group_limited_routing_03_b300 import inputs

PK = dict(hbm=6500.0, bf16=1800.0, bf16_sustained=1400.0, source="test")


def _m(ms_gate_up, touched):
    st = [0.0] * len(bench.STAGES)
    st[bench.STAGES.index("gate_up")] = ms_gate_up
    return {"stage_ms": st, "touched": touched}


def test_weight_bytes_per_expert():
    wl = inputs.workload("decode")
    assert bench.weight_bytes_per_expert(wl) == 3 * 5120 * 2560 * 2
    assert bench.weight_bytes_per_expert(inputs.workload("fp8")) == 3 * 5120 * 2560 + 4 * (2 * 2560 + 5120)
    nv = bench.weight_bytes_per_expert(inputs.workload("nvfp4"))
    assert nv == 3 * 5120 * 2560 // 2 + 3 * 5120 * 2560 // 16 + 12


def test_roofline_bf16_decode_bytes_and_fraction():
    wl = inputs.workload("decode")
    hbm, tc = bench.roofline(wl, _m(1.5, 222), PK)
    R = 64 * 8
    wbytes = 222 * 2 * 2560 * 5120 * 2
    act = R * 5120 * 2 + R * 2560 * 2
    assert hbm["algorithmic_bytes"] == wbytes + act
    assert hbm["achieved"] == pytest.approx((wbytes + act) / 1.5e-3 / 1e9, rel=1e-3)
    assert hbm["frac"] == pytest.approx(hbm["achieved"] / 6500.0, rel=1e-3)
    assert tc["algorithmic_flops"] == 2.0 * R * 2 * 2560 * 5120
    assert tc["peak"] == 1800.0 and tc["peak_sustained"] == 1400.0


def test_roofline_fp8_uses_twice_the_bf16_peak_and_one_byte_weights():
    wl = inputs.workload("fp8")
    hbm, tc = bench.roofline(wl, _m(1.6, 256), PK)
    R = 8192 * 8
    wbytes = 256 * 2 * 2560 * 5120 + 256 * 2 * 2560 * 4
    act = R * 5120 * 1 + R * 2560 * 2
    assert hbm["algorithmic_bytes"] == wbytes + act
    assert tc["peak"] == 3600.0 and tc["peak_sustained"] == 2800.0
    assert tc["frac"] == pytest.approx(tc["achieved"] / 3600.0, rel=1e-3)


def test_residual_numbers_bytes():
    wl = inputs.workload("prefill")
    st = [0.0] * len(bench.STAGES)
    c = bench.STAGES.index("combine")
    st[c] = 0.15
    plain = {"stage_ms": list(st), "total_ms": 50.0}
    res = {"stage_ms": list(st), "total_ms": 50.0, "clocks": {}}
    out = bench.residual_numbers(wl, plain, res, 10, PK, 105)
    T, H = 8192, 5120
    assert out["roofline"]["algorithmic_bytes"] == T * 8 * H * 2 + 2 * T * H * 2 + H * 4 + T * 8 * 8
    assert out["step_k"] == 105 and out["in_place"]


def test_job_throughput_counts_every_rank():
    assert bench.job_throughput(64, 50, 4, 100.0) == pytest.approx(64 * 50 * 4 / 0.1)


def test_traffic_record_lookup():
    assert bench.traffic_record("moe_gemm_gate_up", "no_such_workload", 1e9) is None
    assert bench.traffic_record("moe_gemm_gate_up", "prefill", 1e9) is None  # no record for prefill-sized layers
    v = bench.traffic_record("moe_gemm_gate_up", "decode", 1.128e10)
    # the small-case ratio times this launch's algorithmic bytes, or None once the kernel source changed
    assert v is None or 0.95e10 * 1.128 < v < 1.05e10 * 1.128


def test_code_hash_ignores_comments_only():
    a = 'int f() { return 1; }  // one\n/* block */ const char* s = "// kept";\n'
    b = 'int f() {\n  return 1;\n}\nconst char* s = "// kept";\n'
    assert bench.code_hash([a]) == bench.code_hash([b])
    assert bench.code_hash([a]) != bench.code_hash([a.replace("return 1", "return 2")])
    assert bench.code_hash([a]) != bench.code_hash([a.replace('"// kept"', '""')])


def test_line_contract_check():
    """bench.py refuses to print a line whose contract objects are malformed
    (a stray float in cpu_baseline once slipped through)."""
    good = {"metric": "m", "value": 1.0, "unit": "tokens/s", "n_gpus": 1, "steps": 5, "warmup": 3,
            "ms_per_step": 2.4, "higher_is_better": True, "scaling": "weak", "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "decode"}, "gpu_launches": 40, "clocks": {"sm_mhz": 2032.0},
            "roofline": {"bound": "hbm", "achieved": 1.0, "peak": 2.0, "unit": "GB/s", "frac": 0.5, "traffic": None},
            "cpu_baseline": {"value": 4.0, "unit": "tokens/s", "cores": 16, "kind": "oracle", "sample": "s"},
            "e2e": {"value": 1.0, "unit": "tokens/s", "h2d_bytes_per_step": 1, "d2h_bytes_per_step": 1}}
    assert bench.line_problems(good) == []
    assert bench.line_problems(dict(good, cpu_baseline=3.0)) == ["cpu_baseline malformed: float"]
    assert bench.line_problems(dict(good, e2e=None), full=False) == []
    assert bench.line_problems(dict(good, roofline={"bound": "hbm"}))
    assert bench.line_problems(dict(good, gpu_launches=None))
