"""Host-side helpers of bench.py (CPU only): the clock-sample summary, the ncu
traffic lookup and its staleness rule, and the workload names."""
import bench
from bit_moe_expert_w2_gb300 import inputs


def _sample(sm, mx, hw="Not Active", thermal="Not Active", sw_thermal="Not Active", power="Not Active"):
    return f"0, {sm}, {mx}, 900.00, 0x0000000000000000, {hw}, {thermal}, {sw_thermal}, {power}"


def test_clock_summary_median_max_and_reasons():
    c = bench.ClockSampler("0")
    lines = [_sample(2070, 2070), _sample(2055, 2070, power="Active"), _sample(2070, 2070),
             "garbage line", _sample(1980, 2070, hw="Active")]
    c.samples = [(10.0 + i, line) for i, line in enumerate(lines)]
    s = c.summary(10.0, 14.0, want=1)
    assert s["sm_mhz"] == 2062.5 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 4
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"] and s["window"] == "timed steps"


def test_clock_summary_takes_the_timed_window_or_widens_it_to_the_warm_replays():
    c = bench.ClockSampler("0")
    # warm replays at t = 0..9 (1500 MHz), timed steps at t = 20..22 (2070 MHz), idle after
    c.samples = [(float(t), _sample(1500, 2070)) for t in range(10)] + \
                [(float(t), _sample(2070, 2070)) for t in (20, 21, 22)] + [(40.0, _sample(300, 2070))]
    s = c.summary(20.0, 22.0, warm0=0.0, want=3)
    assert s["samples"] == 3 and s["sm_mhz"] == 2070.0 and s["window"] == "timed steps"
    s = c.summary(20.0, 22.0, warm0=0.0, want=10)       # too few in the timed window: widened
    assert s["samples"] == 13 and s["sm_mhz"] == 1500.0 and s["window"] == "warm replays and timed steps"


def test_clock_summary_without_samples_says_so():
    s = bench.ClockSampler("0").summary(0.0, 1.0)
    assert s["samples"] == 0 and s["reasons"] == ["unsampled"]


def test_ncu_traffic_is_reported_only_for_its_workload_and_sources(monkeypatch, tmp_path):
    import json
    (tmp_path / "profiles").mkdir()
    files = {"k.cu": "__global__ void k() {}\n", "common.cuh": "// helpers\n", "api.h": "// abi\n"}
    for f, text in files.items():
        (tmp_path / f).write_text(text)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", {"k": ["k.cu"], "other": ["o.cu"]})
    monkeypatch.setattr(bench, "COMMON_SOURCES", ["common.cuh", "api.h"])
    srcs = bench.kernel_sources("k")
    entry = {"workload": "decode_t32", "sources": srcs, "sources_sha": bench.sources_sha(srcs),
             "traffic_bytes_per_launch": 1234}
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps({"k": entry}))
    assert bench.ncu_traffic("k", "decode_t32") == 1234
    assert bench.ncu_traffic("k", "decode_t1") is None        # another workload
    assert bench.ncu_traffic("other", "decode_t32") is None   # no capture of that kernel
    (tmp_path / "common.cuh").write_text("// helpers, changed\n")
    assert bench.ncu_traffic("k", "decode_t32") is None       # a shared header changed since the capture
    (tmp_path / "common.cuh").write_text(files["common.cuh"])
    assert bench.ncu_traffic("k", "decode_t32") == 1234
    (tmp_path / "k.cu").write_text("__global__ void k() { }\n")
    assert bench.ncu_traffic("k", "decode_t32") is None       # the kernel source changed


def test_every_workload_has_a_name_with_its_shape():
    for name, cfg in inputs.CONFIGS.items():
        w = bench.workload_name(name)
        assert w.startswith(name + ":") and f"H={cfg.hidden}" in w and f"T={cfg.tokens}" in w
    for name, n in inputs.REQUANT_CASES.items():
        w = bench.workload_name(name)
        assert w.startswith(name + ":") and f"{n or inputs.REQUANT.num_experts} experts" in w
    for name, n in inputs.REQUANT_FP8_CASES.items():
        w = bench.workload_name(name)
        assert w.startswith(name + ":") and f"{n} experts FP8" in w
    for name, cfg in inputs.W4_CONFIGS.items():
        w = bench.workload_name(name)
        assert w.startswith(name + ":") and "FP4 layer" in w and f"H={cfg.hidden}" in w and f"E={cfg.num_experts}" in w
    for name, n in inputs.REQUANT_MXFP4_CASES.items():
        w = bench.workload_name(name)
        assert w.startswith(name + ":") and f"{n} experts MXFP4" in w
