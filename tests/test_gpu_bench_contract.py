"""bench.py's own arm on the GPU, on the small workload: one JSON line with the keys and
types the contract names (metric, value, steps, roofline with its fractions, cpu_baseline,
e2e with the copied bytes, gpu_launches, clocks, oracle_check), each sane."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_our_arm_prints_the_contract_line():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "tiny",
                          "--steps", "5", "--warmup", "3", "--no-other-workloads",
                          "--no-unfused-memory", "--cpu-seconds", "1", "--e2e-steps", "5"],
                         capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    sys.path.insert(0, ROOT)
    import bench
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["n_gpus"] == 1
    assert d["steps"] == 5 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["scaling"] == "weak" and d["data"] == "synthetic" and d["dtype"] == "bf16"
    assert d["config"]["workload"] == "tiny" and "l2" in d["config"]
    # the step is N tokens: value and ms_per_step agree
    assert abs(d["value"] - 256 / (d["ms_per_step"] / 1e3)) <= 1e-6 * d["value"]
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert "frac_burst" in r and "traffic" in r
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == d["unit"]
    # hidden + weight + labels + both upstream gradients of one tiny step, as copied
    assert e["h2d_bytes_per_step"] == 256 * 512 * 2 + 512 * 4096 * 2 + 256 * 8 + 4 + 4
    assert e["d2h_bytes_per_step"] == 8
    assert d["gpu_launches"] == 5 * 7  # forward 3 + backward 4 kernels per step
    assert set(d["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons", "samples"}
    assert d["oracle_check"]["pass"] is True
    g = d["grad_in_forward"]
    assert g["value"] > 0 and g["gpu_launches"] > 0
