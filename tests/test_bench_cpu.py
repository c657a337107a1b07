"""Host logic of bench.py (no GPU): the roofline peak follows the timed
window's clock record, and the roofline figures are the algorithmic work of
the two grouped-GEMM launches over their summed time."""
import bench
from top_routing_grouped_fp32_gb300.inputs import WORKLOADS

PEAKS = {"hbm_gbs": 6700.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1800.0}
STAGES = {"route": 0.01, "dispatch": 0.09, "gate_up_gemm": 0.70, "down_gemm": 0.40, "combine": 0.07}


def test_peak_is_burst_only_at_max_clock_without_power_cap():
    burst = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    capped = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    slow = {"sm_mhz": 1600.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert bench.tensor_peak(PEAKS, "measured", burst)[0] == 2000.0
    assert bench.tensor_peak(PEAKS, "measured", capped)[0] == 1800.0
    assert bench.tensor_peak(PEAKS, "measured", slow)[0] == 1800.0
    # no clock record: the larger (burst) denominator, the conservative fraction
    assert bench.tensor_peak(PEAKS, "measured", {})[0] == 2000.0


def test_tensor_roofline_is_both_gemm_launches():
    wl = WORKLOADS["finegrained_bf16"]
    clocks = {"sm_mhz": 1600.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    r = bench.roofline_for(wl, STAGES, 64, clocks, PEAKS, "measured", traffic=1.2e9)
    flop = 6.0 * wl.T * wl.top_k * wl.H * wl.I
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - flop / 1.10e-3 / 1e12) < 1e-6 * r["achieved"]
    assert r["peak"] == 1800.0 and abs(r["frac"] - r["achieved"] / 1800.0) < 1e-12
    assert abs(r["frac_of_burst"] - r["achieved"] / 2000.0) < 1e-12
    assert abs(r["gate_up"]["achieved"] - 4.0 * wl.T * wl.top_k * wl.H * wl.I / 0.70e-3 / 1e12) < 1e-6
    assert r["traffic"] == 1.2e9


def test_decode_roofline_is_touched_weight_bytes_over_hbm():
    wl = WORKLOADS["decode_bf16"]
    st = dict(STAGES, gate_up_gemm=1.35, down_gemm=0.68)
    r = bench.roofline_for(wl, st, 160, {}, PEAKS, "measured")
    wbytes = 160 * 3.0 * wl.H * wl.I * 2
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6700.0
    assert abs(r["achieved"] - wbytes / 2.03e-3 / 1e9) < 1e-6 * r["achieved"]


def test_fp32_roofline_is_the_ffma_pipe():
    wl = WORKLOADS["tiny_fp32"]
    r = bench.roofline_for(wl, STAGES, 4, {"sm_max_mhz": 2070.0}, PEAKS, "measured")
    assert r["bound"] == "alu"
    assert abs(r["peak"] - 152 * 128 * 2 * 2070e6 / 1e12) < 1e-9


def test_traffic_is_dropped_when_the_kernel_source_changes(monkeypatch):
    wl = WORKLOADS["finegrained_bf16"]
    sha = bench.code_sha256("top_routing_grouped_fp32_gb300/csrc/gemm_tc.cu")
    monkeypatch.setitem(bench.GEMM_TRAFFIC, wl.name, {"bytes_per_launch": 123.0, "code_sha256": sha})
    assert bench.gemm_traffic(wl) == 123.0
    monkeypatch.setitem(bench.GEMM_TRAFFIC, wl.name, {"bytes_per_launch": 123.0, "code_sha256": "0" * 64})
    assert bench.gemm_traffic(wl) is None
    assert bench.gemm_traffic(WORKLOADS["mixtral_bf16"]) is None  # no capture of that workload


def test_launch_count_per_step():
    # route, count, scatter (scan fused), gather, two GEMMs, combine
    assert bench.launches_per_step(16384, 64) == 7
    # a large chunk-histogram table adds the scan kernel
    assert bench.launches_per_step(65536 * 4, 1024) == 8


def test_code_fingerprint_ignores_comments_not_code(tmp_path, monkeypatch):
    src = 'int f(int a) {  // add one\n  /* "x" */ return a + 1; }\nconst char* s = "// kept";\n'
    (tmp_path / "a.cu").write_text(src)
    (tmp_path / "b.cu").write_text(src.replace("// add one", "// adds one, see below").replace("  ", " "))
    (tmp_path / "c.cu").write_text(src.replace("a + 1", "a + 2"))
    (tmp_path / "d.cu").write_text(src.replace('"// kept"', '"// changed"'))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    a, b, c, d = (bench.code_sha256(n) for n in ("a.cu", "b.cu", "c.cu", "d.cu"))
    assert a == b
    assert a != c and a != d


def test_traffic_record_matches_the_committed_kernel():
    """The committed capture was taken on the code now in gemm_tc.cu."""
    rec = bench.GEMM_TRAFFIC["finegrained_bf16"]
    assert rec["code_sha256"] == bench.code_sha256("top_routing_grouped_fp32_gb300/csrc/gemm_tc.cu")
