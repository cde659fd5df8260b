"""Host-side logic of bench.py that needs no GPU: the comment-insensitive
code hash that links a profile summary to the kernel source it was taken
on, and the lookup of a profiled DRAM traffic figure."""
import bench


def _hash_of(tmp_path, text):
    p = tmp_path / "k.cu"
    p.write_text(text)
    return bench.code_hash(str(p))


BASE = """// header comment
__global__ void k(float* x) {  /* block comment */
    x[0] = 1.0f;  // trailing comment
    const char* s = "a // not a comment";
}
"""


def test_code_hash_ignores_comments_and_whitespace(tmp_path):
    h = _hash_of(tmp_path, BASE)
    assert len(h) == 16
    edited = BASE.replace("// header comment", "// a different header\n// over two lines")
    edited = edited.replace("/* block comment */", "/* another\n   block */")
    edited = edited.replace("x[0] = 1.0f;", "x[0]  =  1.0f ;")
    assert _hash_of(tmp_path, edited) == h


def test_code_hash_sees_code_changes(tmp_path):
    h = _hash_of(tmp_path, BASE)
    assert _hash_of(tmp_path, BASE.replace("1.0f", "2.0f")) != h
    # text inside a string literal is code, even when it looks like a comment
    assert _hash_of(tmp_path, BASE.replace("not a comment", "still code")) != h


def test_profiled_traffic_follows_the_recorded_hash(tmp_path, monkeypatch):
    csrc = tmp_path / "fp8_fine_grained_25_b300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "k.cu").write_text(BASE)
    h = bench.code_hash(str(csrc / "k.cu"))
    (tmp_path / "profiles" / "k.md").write_text(
        f"code-sha256-16 (source without comments or whitespace): k.cu {h}\n\n"
        "traffic_bytes_per_launch: 123456 (k)\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("k.md", "k.cu") == 123456
    (csrc / "k.cu").write_text(BASE.replace("// trailing comment", "// edited"))
    assert bench.profiled_traffic("k.md", "k.cu") == 123456  # comment edit: still linked
    (csrc / "k.cu").write_text(BASE.replace("1.0f", "2.0f"))
    assert bench.profiled_traffic("k.md", "k.cu") is None  # code changed: unlinked
    assert bench.profiled_traffic("missing.md", "k.cu") is None


PEAKS = {"hbm_gbs": 6488.3, "bf16_tflops": 1771.9, "bf16_tflops_sustained": 1393.5}


def test_fp8_peak_burst_for_a_short_uncapped_region():
    fp8 = {"burst_tflops": 3500.0, "sustained_tflops": 2700.0}
    peak, burst, sus, desc = bench.choose_fp8_peak(fp8, PEAKS, "measured", 0.008, {"reasons": []})
    assert burst == 3543.8 and peak == burst          # 2 x bf16 burst beats the cuBLAS burst
    assert sus == 2787.0                              # 2 x bf16 sustained beats 2700
    assert desc.startswith("burst")


def test_fp8_peak_sustained_when_long_or_capped():
    fp8 = {"burst_tflops": 3700.0, "sustained_tflops": 2900.0}
    p_long, _, sus, d_long = bench.choose_fp8_peak(fp8, PEAKS, "measured", 5.0, {"reasons": []})
    assert p_long == sus == 2900.0 and d_long.startswith("sustained: measured fp8")
    p_cap, burst, _, _ = bench.choose_fp8_peak(fp8, PEAKS, "measured", 0.01, {"reasons": ["sw_power_cap"]})
    assert p_cap == 2900.0 and burst == 3700.0
    p_none, _, _, _ = bench.choose_fp8_peak({}, PEAKS, "fallback", 0.01, {"reasons": []})
    assert p_none == 3543.8


def test_clock_summary_windows_and_reasons():
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.source = "test"
    c.samples = [(0.0, 1200.0, 2032.0, 0x0), (1.0, 2032.0, 2032.0, 0x4), (2.0, 1900.0, 2032.0, 0x8),
                 (3.0, 2032.0, 2032.0, 0x0)]
    full = c.summary()
    assert full["samples"] == 4 and full["sm_max_mhz"] == 2032.0
    assert full["reasons"] == ["sw_power_cap", "hw_slowdown"]
    w = c.summary(0.5, 2.5)
    assert w["samples"] == 2 and w["sm_mhz"] == (2032.0 + 1900.0) / 2
    assert c.summary(10.0, 11.0)["samples"] == 0


def test_both_arms_describe_the_same_config():
    from fp8_fine_grained_25_b300 import workloads
    w = workloads.tiny(seed=0, device="cpu")
    cfg = bench.run_config(w, 1)
    assert cfg == bench.run_config(workloads.tiny(seed=0, device="cpu"), 1)
    assert cfg["workload"].startswith("tiny 128x256x512: quant_act(A) + quant_weight(W) + dense")
    assert cfg["parallelism"] == "replicas x1"
