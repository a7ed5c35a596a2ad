"""Host arithmetic of bench.py's step roofline (no GPU): algorithmic bytes
per launch for the decode workload M=16, N=5120, K=2048 with bias, for the
fused schedule (one launch per step) and the unfused one."""
import os
import sys
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

D = types.SimpleNamespace(m=16, n=5120, k=2048)
WB = 5120 * 2048 + 5120 * 2048 // 32      # E4M3 weights + E8M0 scales
ACT_SF = 16 * 2048 // 32                   # 8x4 scales of 16 rows


def test_weight_bytes_helper():
    assert bench.weight_bytes(5120, 2048) == WB == 10_813_440


def test_fused_step_is_the_dominant_launch():
    r = bench.step_roofline(D, WB, 1, 0.005, 0.004, 6800.0, None, ACT_SF)
    nbytes = 2 * 16 * 2048 + WB + 2 * 5120 + 2 * 16 * 5120
    assert r["alg_bytes_per_launch"] == nbytes == 11_053_056
    assert abs(r["us_per_launch"] - 5.0) < 1e-9
    assert abs(r["achieved"] - nbytes / 5e-6 / 1e9) < 1e-6
    assert abs(r["frac"] - r["achieved"] / 6800.0) < 1e-12
    g = r["gemm_prequantized_alone"]  # dropped from the printed line by main()
    assert g["alg_bytes_per_launch"] == 11_021_312 and abs(g["us_per_launch"] - 4.0) < 1e-9


def test_unfused_step_reports_the_gemm():
    r = bench.step_roofline(D, WB, 2, 0.005, 0.004, 6800.0, 123.0, ACT_SF)
    assert r["alg_bytes_per_launch"] == 11_021_312
    assert abs(r["us_per_launch"] - 4.0) < 1e-9
    assert r["traffic"] == 123.0 and r["bound"] == "hbm" and r["unit"] == "GB/s"


def test_compact_keeps_four_significant_digits():
    v = bench.compact({"a": 1599.9999875, "b": [0.241178353, 3], "c": {"d": 1e-7 / 3}, "e": "s"})
    assert v == {"a": 1600.0, "b": [0.2412, 3], "c": {"d": 3.333e-08}, "e": "s"}


def test_large_m_block_uses_the_fp8_peak():
    peaks = {"bf16_tflops": 1897.8, "source": "measured"}
    cfg = {"prefill_m8192_n8192_k8192": {"us_per_call": 424.0, "tflops": 2593.2, "gemm_us": 387.0,
                                         "gemm_tflops": 2841.1}}
    lm = bench.large_m_block(cfg, peaks)
    assert abs(lm["peak_tflops"] - 3795.6) < 1e-9
    assert abs(lm["frac"] - 2593.2 / 3795.6) < 1e-12
    assert abs(lm["gemm_frac"] - 2841.1 / 3795.6) < 1e-12
    assert bench.large_m_block({}, peaks) is None


def test_host_description_names_cores_and_model():
    h = bench.host_description()
    assert h["host_cores"] == os.cpu_count() and isinstance(h["cpu_model"], str) and h["cpu_model"]


def test_timing_method_is_named():
    """The timed region's bounds: events inside the captured graphs where
    this PyTorch records them there, else events around the replays."""
    assert bench.timing_method() in bench.TIMING.values()


def test_code_sha_ignores_comments_only(tmp_path):
    """Captured traffic stays valid across comment edits of the kernel
    source, not across code edits (bench.code_sha)."""
    a = tmp_path / "a.cu"
    a.write_text('int f(int x) {  // twice\n  /* body */ return 2 * x; }\nconst char* s = "//x";\n')
    b = tmp_path / "b.cu"
    b.write_text('// header\nint f(int x) {  // doubled\n\n  return 2 * x; }\nconst char* s = "//x";\n')
    c = tmp_path / "c.cu"
    c.write_text('int f(int x) {  // twice\n  return 3 * x; }\nconst char* s = "//x";\n')
    d = tmp_path / "d.cu"
    d.write_text('int f(int x) {  // twice\n  return 2 * x; }\nconst char* s = "//y";\n')
    assert bench.code_sha(str(a)) == bench.code_sha(str(b))
    assert bench.code_sha(str(a)) != bench.code_sha(str(c))
    assert bench.code_sha(str(a)) != bench.code_sha(str(d))
