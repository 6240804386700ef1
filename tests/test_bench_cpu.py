"""Host-side helpers of bench.py (CPU only): the clock-sample summary, the ncu
traffic lookup and its staleness rule, and the workload names."""
import bench
from bit_moe_expert_w2_gb300 import inputs


def _sample(sm, mx, hw="Not Active", thermal="Not Active", sw_thermal="Not Active", power="Not Active"):
    return f"0, {sm}, {mx}, 900.00, 0x0000000000000000, {hw}, {thermal}, {sw_thermal}, {power}"


def test_clock_summary_median_max_and_reasons():
    c = bench.ClockSampler(0)
    c.lines = [_sample(2070, 2070), _sample(2055, 2070, power="Active"), _sample(2070, 2070),
               "garbage line", _sample(1980, 2070, hw="Active")]
    s = c.summary()
    assert s["sm_mhz"] == 2062.5 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 4
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_clock_summary_without_samples_says_so():
    s = bench.ClockSampler(0).summary()
    assert s["samples"] == 0 and s["reasons"] == ["unsampled"]


def test_ncu_traffic_is_reported_only_for_its_workload_and_source(monkeypatch, tmp_path):
    import json
    (tmp_path / "profiles").mkdir()
    (tmp_path / "k.cu").write_text("__global__ void k() {}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    entry = {"workload": "decode_t32", "source": "k.cu", "source_sha": bench.file_sha("k.cu"),
             "traffic_bytes_per_launch": 1234}
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps({"k": entry}))
    assert bench.ncu_traffic("k", "decode_t32") == 1234
    assert bench.ncu_traffic("k", "decode_t1") is None        # another workload
    assert bench.ncu_traffic("other", "decode_t32") is None   # no capture of that kernel
    (tmp_path / "k.cu").write_text("__global__ void k() { }\n")
    assert bench.ncu_traffic("k", "decode_t32") is None       # the source changed since the capture


def test_every_workload_has_a_name_with_its_shape():
    for name, cfg in inputs.CONFIGS.items():
        w = bench.workload_name(name)
        assert w.startswith(name + ":") and f"H={cfg.hidden}" in w and f"T={cfg.tokens}" in w
    for name, n in inputs.REQUANT_CASES.items():
        w = bench.workload_name(name)
        assert w.startswith(name + ":") and f"{n or inputs.REQUANT.num_experts} experts" in w
