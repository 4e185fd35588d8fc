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
