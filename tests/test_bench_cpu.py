"""bench.py helpers that need no GPU."""
import bench


def test_profiled_traffic_follows_the_kernel_sources(monkeypatch):
    v = bench.profiled_traffic("flp_bwd_kernel/dx_dw", "m4096_h4096_v131072")
    digest = bench.kernel_sources_digest()
    line = [ln for ln in open(bench.os.path.join(bench.ROOT, "profiles",
                                                  "dram_traffic_m4096_h4096_v131072.md"))
            if ln.startswith("traffic-per-launch flp_bwd_kernel/dx_dw ")][0].split()
    if line[4] == digest:
        assert v == float(line[2])
    else:
        assert v is None
    monkeypatch.setattr(bench, "kernel_sources_digest", lambda: "0" * 64)
    assert bench.profiled_traffic("flp_bwd_kernel/dx_dw", "m4096_h4096_v131072") is None
    assert bench.profiled_traffic("no_such_kernel", "m4096_h4096_v131072") is None
    assert bench.profiled_traffic("flp_bwd_kernel/dx_dw", "no_such_workload") is None


def test_reference_arm_prints_its_json_line():
    """`bench.py --impl reference` on the tiny workload: one JSON line with the
    contract's keys, the oracle on the host cores as its CPU baseline."""
    import json
    import subprocess
    import sys
    out = subprocess.run([sys.executable, bench.os.path.join(bench.ROOT, "bench.py"), "--impl",
                          "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3"],
                         capture_output=True, text=True, timeout=600, check=True).stdout
    d = json.loads(out.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["config"]["workload"] == "tiny"


def test_peak_follows_the_timed_region_and_the_clock():
    peaks = {"bf16_tflops": 1878.3, "bf16_tflops_sustained": 1704.2}
    key, peak, _ = bench.choose_peak(peaks, 0.3, {"sm_mhz": 1500.0, "sm_max_mhz": 2070.0})
    assert (key, peak) == ("bf16_tflops", 1878.3)          # short region: burst
    key, peak, _ = bench.choose_peak(peaks, 5.0, {"sm_mhz": 2040.0, "sm_max_mhz": 2070.0})
    assert (key, peak) == ("bf16_tflops", 1878.3)          # clock near its maximum: burst
    key, peak, _ = bench.choose_peak(peaks, 5.0, {"sm_mhz": 1455.0, "sm_max_mhz": 2070.0})
    assert (key, peak) == ("bf16_tflops_sustained", 1704.2)
    key, _, _ = bench.choose_peak(peaks, 5.0, None)
    assert key == "bf16_tflops_sustained"


def test_profiled_counters_follow_the_kernel_sources(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "kernel_sources_digest", lambda: "ab" * 32)
    (tmp_path / "profiles" / "counters_w.md").write_text(
        "# text\nncu-counters flp_fwd_kernel tensor_pipe_pct=88.5 dram_gb=1.2 case=q sources-sha256 "
        + "ab" * 32 + "\n")
    got = bench.profiled_counters("w")
    assert got == {"flp_fwd_kernel": {"tensor_pipe_pct": 88.5, "dram_gb": 1.2, "case": "q"}}
    monkeypatch.setattr(bench, "kernel_sources_digest", lambda: "cd" * 32)
    assert bench.profiled_counters("w") is None
    assert bench.profiled_counters("missing") is None


def test_strip_comments_keeps_code_and_literals():
    src = ('int a = 1; // tail\n'
           '/* block\n   over lines */ int b = 2;\n'
           'const char* s = "not // a comment /* nor this */";\n'
           "char c = '/'; char d = '\\''; /**/ int e;\n"
           '   \n')
    assert bench.strip_comments(src) == (
        'int a = 1;\n'
        ' int b = 2;\n'
        'const char* s = "not // a comment /* nor this */";\n'
        "char c = '/'; char d = '\\'';  int e;")


def test_kernel_sources_digest_ignores_comments_only(tmp_path, monkeypatch):
    csrc = tmp_path / "entropy_loss_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cuh").write_text("// header\nint f() { return 1; }  // one\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d0 = bench.kernel_sources_digest()
    (csrc / "k.cuh").write_text("/* another header */\n\nint f() { return 1; }\n")
    assert bench.kernel_sources_digest() == d0
    (csrc / "k.cuh").write_text("int f() { return 2; }\n")
    assert bench.kernel_sources_digest() != d0
