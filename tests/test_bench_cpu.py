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
