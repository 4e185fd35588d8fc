"""bench.py end to end on the GPU for each backward schedule, on the tiny
workload: one JSON line per run carrying the contract's keys."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("schedule", ["auto", "split", "fused", "vsplit"])
def test_bench_line(schedule):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "tiny",
                          "--steps", "3", "--warmup", "3", "--no-cpu-baseline", "--schedule",
                          schedule], capture_output=True, text=True, timeout=600, check=True).stdout
    d = json.loads(out.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "dtype", "data", "config", "roofline", "e2e",
              "gpu_launches", "clocks", "phase_ms"):
        assert k in d, k
    assert d["value"] > 0 and d["e2e"]["value"] > 0
    assert d["config"]["bwd_schedule"] == ("split" if schedule == "auto" else schedule)
    assert d["gpu_launches"] >= 3 * 3
    assert set(d["roofline"]) >= {"bound", "achieved", "peak", "unit", "frac", "traffic"}
