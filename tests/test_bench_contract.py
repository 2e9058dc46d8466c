"""bench.py's output contract, checked on the CPU through its reference arm (the fp64
oracle timed on the host): one JSON line with the keys and types its readers rely on."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_the_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "1", "--warmup", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    sys.path.insert(0, ROOT)
    import bench
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 1
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["vs_baseline"] is None and d["data"] == "synthetic"
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    """Launched like the multi-GPU bench (torchrun, 2 ranks, rendezvous on 127.0.0.1):
    rank 0 alone runs the oracle and prints; the other rank exits 0 without work."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
           "--gpus", "2", "--steps", "1", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    # rank 0 works alone, so its oracle runs on every host core despite torchrun's
    # one-thread default
    sys.path.insert(0, ROOT)
    import bench
    assert d["cpu_baseline"]["cores"] == bench.host_cores()


def test_peak_comes_from_the_measured_file_when_present(tmp_path):
    sys.path.insert(0, ROOT)
    import bench
    assert bench.load_peaks(str(tmp_path)) == (1900.0, "of fallback (1.9 PFLOP/s bf16 burst)")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 7100.0, "bf16_tflops": 2050.0, "bf16_tflops_sustained": 1720.0}))
    # the burst figure is the larger measured rate: the peak a fraction is taken of
    assert bench.load_peaks(str(tmp_path)) == (2050.0, "of measured (bf16_tflops)")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"bf16_tflops_sustained": 1720.0}))
    assert bench.load_peaks(str(tmp_path)) == (1720.0, "of measured (bf16_tflops_sustained)")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"bf16_tflops": {"value": 2010.0}}))
    assert bench.load_peaks(str(tmp_path)) == (2010.0, "of measured (bf16_tflops)")
    (tmp_path / "MEASURED_PEAKS.json").write_text("not json")
    assert bench.load_peaks(str(tmp_path))[0] == 1900.0


def test_roofline_fractions_against_burst_sustained_and_per_clock(tmp_path):
    sys.path.insert(0, ROOT)
    import bench
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0,
         "clocks_under_load": {"sm_mhz_median": 1600.0}}))
    f = bench.roofline_fractions(1800.0, 2000.0, str(tmp_path))
    assert abs(f["frac_burst"] - 0.9) < 1e-12
    assert abs(f["frac_sustained"] - 1.125) < 1e-12
    cn = f["clock_normalised"]
    # 1800 TF/s at 2000 MHz is 0.9 TF/s per MHz; the sustained peak is 1.0 per MHz
    assert abs(cn["achieved_tflops_per_mhz"] - 0.9) < 1e-12
    assert abs(cn["peak_tflops_per_mhz"] - 1.0) < 1e-12
    assert abs(cn["frac"] - 0.9) < 1e-12
    # no sampled clock: no per-clock fraction; no file: nothing
    assert "clock_normalised" not in bench.roofline_fractions(1800.0, None, str(tmp_path))
    assert bench.roofline_fractions(1800.0, 2000.0, str(tmp_path / "absent")) == {}


def test_reported_peak_is_the_largest_measured_rate():
    """The roofline's `peak` is the burst figure when both are measured, so `frac`
    (achieved / peak) can exceed 1 only if the kernel beat the burst matmul itself."""
    sys.path.insert(0, ROOT)
    import bench
    t = bench.load_peak_table()
    if "bf16_tflops" not in t:
        return
    peak, _ = bench.load_peaks()
    assert peak == max(v for k, v in t.items() if k.startswith("bf16_tflops"))


def test_oracle_check_compares_the_sampled_rows():
    """bench.py's oracle_check: per-row outputs of the GPU run against the oracle's on the
    CPU-baseline sample, with the parity tests' 2e-3 absolute tolerance."""
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    import bench
    rng = np.random.default_rng(0)
    o = {k: rng.normal(size=5) for k in ("lse", "ez", "loss", "entropy")}
    full = {k: torch.tensor(np.concatenate([v, rng.normal(size=3)]), dtype=torch.float32)
            for k, v in o.items()}
    res = bench.oracle_check(o, full["lse"], full["ez"], full["loss"], full["entropy"], "none")
    assert res["rows"] == 5 and res["pass"]
    assert set(res["max_abs_err"]) == {"lse", "ez", "loss", "entropy"}
    bad = full["ez"].clone()
    bad[4] += 0.01  # a sampled row off by more than the tolerance
    res = bench.oracle_check(o, full["lse"], bad, full["loss"], full["entropy"], "mean")
    assert not res["pass"] and set(res["max_abs_err"]) == {"lse", "ez"}
    bad = full["ez"].clone()
    bad[6] += 1.0  # a row outside the sample is not compared
    assert bench.oracle_check(o, full["lse"], bad, full["loss"], full["entropy"], "mean")["pass"]


def test_cpu_baseline_sample_is_fitted_to_the_time_budget(monkeypatch):
    """calibrate_rows reads the row count from a line through its last two trial samples
    (a fixed set-up cost plus a cost per row), so the timed sample lands on the budget
    even when the set-up cost is a large part of the trial samples."""
    sys.path.insert(0, ROOT)
    import bench
    clock = [0.0]

    def fake_step(w, *args, rows):
        clock[0] += 0.8 + 0.02 * rows  # seconds: 0.8 of set-up, 20 ms per row

    monkeypatch.setattr(bench, "oracle_sample_step", fake_step)
    monkeypatch.setattr(bench.time, "perf_counter", lambda: clock[0])

    class W:
        N = 8192

    rows, _ = bench.calibrate_rows(W(), (), 15.0)
    assert rows == int((15.0 - 0.8) / 0.02)
    # never more rows than the workload has
    W.N = 100
    assert bench.calibrate_rows(W(), (), 15.0)[0] == 100
