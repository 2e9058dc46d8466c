#!/usr/bin/env python
"""Benchmark of fused linear cross-entropy + entropy (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = flce_forward + flce_backward over one batch of the workload (every
kernel of the path).  Default workload: the Llama-3-8B LM-head shape
(N=8192 tokens, H=4096, V=128256, 20 % ignored, z-loss 1e-4, mean).  Inputs are
seeded synthetic tensors, resident in HBM before the timed region; the weight
(about 1 GB) is larger than L2, so every pass streams it from HBM.

Prints one JSON line (rank 0).  With N > 1 (torchrun) each rank runs an
independent replica on its own GPU; value = all ranks' tokens / max rank time.

`--impl reference` times the fp64 CPU oracle on the host cores instead (the
baseline arm), on bounded row samples of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fwd+bwd tokens/sec and TFLOP/s (% of GB300 BF16 dense peak) at N×H×V"
UNIT = "tokens/s"
FALLBACK_BF16_TFLOPS = 1900.0  # profiling recipe fallback (burst), used only without a peaks file


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # about a second of timed steps on the Llama-3 head: long enough for the clock samples
    # (every 100 ms) to describe the window
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama3_8b_head")
    ap.add_argument("--tokens", type=int, default=0,
                    help="reduced case: replace the workload's N (for small ncu captures)")
    ap.add_argument("--vocab", type=int, default=0,
                    help="reduced case: replace the workload's V (for small ncu captures)")
    ap.add_argument("--softcap", type=float, default=None,
                    help="reduced case: replace the workload's logit soft-cap (0 = none)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-unfused-memory", action="store_true",
                    help="skip the unfused PyTorch baseline (its peak memory and its time)")
    ap.add_argument("--no-grad-in-forward", action="store_true",
                    help="skip timing the one-call forward+backward (gradient in forward)")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end run from host buffers (launch-list captures)")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip timing the two-call step of the other workloads")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def blas_threads() -> int:
    """Threads the oracle's BLAS runs on: the OpenBLAS / OpenMP thread variables when
    set (read when numpy loads), else every host core."""
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        v = os.environ.get(var, "")
        if v.isdigit() and int(v) > 0:
            return min(int(v), host_cores())
    return host_cores()


L2_BYTES = 129 * 10**6     # GB300 L2
# clock-event reasons that invalidate a timed window (a power cap is normal under load)
REJECTED_CLOCK_REASONS = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
FLUSH_BYTES = 512 << 20     # written between timed steps when the inputs fit in L2


def needs_flush(w):
    return w.H * w.V * 2 + w.N * w.H * 2 <= L2_BYTES


def workload_config(w, world):
    if needs_flush(w):
        l2 = ("inputs fit in L2 (%.1f MB): a %d MB buffer is written before every timed step "
              "(not timed) to flush it" % ((w.H * w.V * 2 + w.N * w.H * 2) / 1e6,
                                          FLUSH_BYTES >> 20))
    else:
        l2 = "inputs larger than L2: weight %.2f GB streamed from HBM every pass" % (
            w.H * w.V * 2 / 1e9)
    return {"workload": w.name, "N": w.N, "H": w.H, "V": w.V, "reduction": w.reduction,
            "zloss_coef": w.zloss_coef, "softcap": w.softcap, "ignore_frac": w.ignore_frac,
            "label_mode": w.label_mode, "grad_mode": w.grad_mode, "global_batch": w.N * world,
            "seq_len": w.N, "parallelism": "replicas" if world > 1 else "single", "l2": l2}


def select_workload(args):
    """The named workload, or a reduced case of it when --tokens / --vocab are given
    (same recipe, other sizes; its name says so)."""
    from linear_cross_entropy_forward_gb300.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.tokens or args.vocab:
        N = args.tokens or w.N
        V = args.vocab or w.V
        w = w.scaled(f"{w.name}_N{N}_V{V}", N, w.H, V)
    if args.softcap is not None:
        w = dataclasses.replace(w, name=f"{w.name}_cap{args.softcap:g}", softcap=args.softcap)
    return w


# ---------------------------------------------------------------- CPU oracle leg
def oracle_sample_step(w, h64, W64, labels_np, gl_np, ge_np, rows):
    """fwd + bwd of the fp64 oracle on a row sample (dhidden of those rows and their
    dweight contribution), as the oracle stands."""
    from oracle import flce_oracle as orc
    hs = h64[:rows]
    ys = labels_np[:rows]
    if w.reduction == "none":
        gl, ge = gl_np[:rows], ge_np[:rows]
    else:
        gl, ge = gl_np, ge_np
    o = orc.forward(hs, W64, ys, w.reduction, zloss_coef=w.zloss_coef, softcap=w.softcap)
    orc.backward(hs, W64, ys, o["lse"], o["ez"], gl, ge, w.reduction,
                 zloss_coef=w.zloss_coef, softcap=w.softcap)
    return o


def oracle_inputs(w, hidden, weight, labels, g_loss, g_ent):
    from linear_cross_entropy_forward_gb300.workloads import bf16_bits
    from oracle import flce_oracle as orc
    h64 = orc.bf16_bits_to_f64(bf16_bits(hidden))
    W64 = orc.bf16_bits_to_f64(bf16_bits(weight))
    return h64, W64, labels.numpy(), g_loss.numpy(), g_ent.numpy()


def calibrate_rows(w, args_oracle, seconds):
    """Rows per oracle sample so that one sample takes about `seconds`.  A sample costs a
    fixed set-up plus a cost per row, so the last two trial samples (4x apart in rows)
    give the line a + b * rows that the row count is read from."""
    rows, trials = 4, []
    while True:
        t0 = time.perf_counter()
        oracle_sample_step(w, *args_oracle, rows=rows)
        trials.append((rows, max(time.perf_counter() - t0, 1e-3)))
        if trials[-1][1] >= 0.1 * seconds or rows >= w.N:
            break
        rows = min(w.N, rows * 4)
    r1, t1 = trials[-1]
    b = t1 / r1
    if len(trials) > 1:
        r0, t0_ = trials[-2]
        if t1 > t0_ and r1 > r0:
            b = (t1 - t0_) / (r1 - r0)
    a = max(0.0, t1 - b * r1)
    return max(1, min(w.N, int((seconds - a) / b))), t1


def cpu_baseline(w, hidden, weight, labels, g_loss, g_ent, seconds):
    """The oracle timed on a row sample; also returns its forward outputs for those rows,
    which the bench line compares with the GPU's."""
    ai = oracle_inputs(w, hidden, weight, labels, g_loss, g_ent)
    rows, _ = calibrate_rows(w, ai, seconds)
    t0 = time.perf_counter()
    o = oracle_sample_step(w, *ai, rows=rows)
    dt = time.perf_counter() - t0
    return {"value": rows / dt, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": f"fp64 numpy oracle fwd+bwd on the first {rows} of {w.N} rows "
                      f"(full H={w.H}, V={w.V}), {dt:.1f} s on {blas_threads()} BLAS threads"}, o


def oracle_check(o, lse, ez, loss, ent, reduction):
    """Max abs error of the GPU's per-row outputs of the timed runs against the oracle's
    on the CPU-baseline sample (the tolerance of the parity tests: 2e-3)."""
    import numpy as np
    r = len(o["lse"])
    f64 = lambda t: t[:r].float().cpu().numpy().astype(np.float64)  # noqa: E731
    errs = {"lse": float(np.abs(f64(lse) - o["lse"]).max()),
            "ez": float(np.abs(f64(ez) - o["ez"]).max())}
    if reduction == "none":
        errs["loss"] = float(np.abs(f64(loss) - o["loss"]).max())
        errs["entropy"] = float(np.abs(f64(ent) - o["entropy"]).max())
    return {"rows": r, "max_abs_err": errs, "tolerance_abs": 2e-3,
            "pass": all(e <= 2e-3 for e in errs.values())}


# ---------------------------------------------------------------- clocks sampler
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(gpu_id)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [s for (t, s) in self.samples if t0 <= t <= t1]
        if not rows:  # a window shorter than the sampling interval: the nearest samples
            rows = [s for (_, s) in sorted(self.samples, key=lambda ts: abs(ts[0] - t1))[:2]]
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w": statistics.median(power), "reasons": sorted(reasons),
                "samples": len(sm)}


def nvsmi_id(torch, dev_index):
    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[dev_index]
        return str(dev_index)


def load_peak_table(root=None):
    """Measured bf16 dense peaks from MEASURED_PEAKS.json: the burst and sustained
    matmul figures (TFLOP/s) and the median SM clock seen under the sustained loop;
    {} when the file is absent or unreadable."""
    path = os.path.join(root or ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(path):
        return {}
    try:
        d = json.load(open(path))
    except (OSError, ValueError):
        return {}
    if not isinstance(d, dict):
        return {}
    out = {}
    for key in ("bf16_tflops", "bf16_tflops_sustained"):
        v = d.get(key)
        if isinstance(v, dict):  # {"value": ..., ...}
            v = v.get("value", v.get("tflops"))
        if isinstance(v, (int, float)) and v > 0:
            out[key] = float(v)
    clk = d.get("clocks_under_load")
    if isinstance(clk, dict) and isinstance(clk.get("sm_mhz_median"), (int, float)):
        out["sustained_sm_mhz"] = float(clk["sm_mhz_median"])
    return out


def load_peaks(root=None):
    """The bf16 dense peak (TFLOP/s) to report against: the measured burst figure (the
    largest measured rate, so a fraction of it stays below 1), else the measured
    sustained figure, else the recipe's fallback."""
    t = load_peak_table(root)
    for key in ("bf16_tflops", "bf16_tflops_sustained"):
        if key in t:
            return t[key], f"of measured ({key})"
    return FALLBACK_BF16_TFLOPS, "of fallback (1.9 PFLOP/s bf16 burst)"


def roofline_fractions(achieved, sm_mhz, root=None):
    """The achieved rate as a fraction of each measured peak, and per clock: achieved /
    sampled SM MHz against the sustained peak / the SM MHz it was measured at (the
    sustained loop runs power-capped at a lower clock than a short burst)."""
    t = load_peak_table(root)
    out = {}
    if "bf16_tflops" in t:
        out["frac_burst"] = achieved / t["bf16_tflops"]
    if "bf16_tflops_sustained" in t:
        out["frac_sustained"] = achieved / t["bf16_tflops_sustained"]
        if sm_mhz and t.get("sustained_sm_mhz"):
            per = achieved / sm_mhz
            peak_per = t["bf16_tflops_sustained"] / t["sustained_sm_mhz"]
            out["clock_normalised"] = {
                "achieved_tflops_per_mhz": per, "peak_tflops_per_mhz": peak_per,
                "frac": per / peak_per, "sm_mhz": sm_mhz,
                "peak_sm_mhz": t["sustained_sm_mhz"]}
    return out


def load_traffic(workload):
    """Per-launch DRAM bytes of the forward GEMM from the committed ncu summary (None
    when it has not been measured since the kernel last changed)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(path))
        return d.get(workload, {}).get("fwd_stats_bytes_per_launch")
    except (OSError, ValueError):
        return None


def unfused_step(torch, w, hd, Wd, yd, gld, ged):
    """One forward + backward of the unfused computation: logits in fp32 from fp32
    copies of hidden and weight, log-softmax, entropy and cross-entropy as written out
    on the pages (verl PR #462, "Equivalent compute logic"), masking of ignored rows,
    z-loss and soft-cap when the workload has them, and autograd's backward.  Returns
    the two leaf tensors (their .grad hold the gradients)."""
    import torch.nn.functional as F
    h = hd.detach().requires_grad_(True)
    W = Wd.detach().requires_grad_(True)
    logits = torch.matmul(h.float(), W.float())
    if w.softcap:
        logits = w.softcap * torch.tanh(logits / w.softcap)
    lse = torch.logsumexp(logits, dim=-1)
    p = torch.softmax(logits, dim=-1)
    ent = lse - (p * logits).sum(-1)
    ce = F.cross_entropy(logits, yd, ignore_index=-100, reduction="none")
    valid = (yd != -100).float()
    loss_t = (ce + w.zloss_coef * lse * lse) * valid
    ent_t = ent * valid
    if w.reduction == "none":
        obj = (loss_t * gld).sum() + (ent_t * ged).sum()
    else:
        den = valid.sum() if w.reduction == "mean" else 1.0
        obj = (loss_t.sum() * gld[0] + ent_t.sum() * ged[0]) / den
    obj.backward()
    return h, W


def unfused_baseline(torch, w, hd, Wd, yd, gld, ged, dev, warmup=2, steps=3):
    """The unfused computation as a stated baseline (not the target): peak bytes it
    allocates above its inputs (the gradients, outputs both paths produce, excluded),
    and its time per fwd+bwd step (CUDA events, after `warmup` steps)."""
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    h, W = unfused_step(torch, w, hd, Wd, yd, gld, ged)
    torch.cuda.synchronize()
    grads = h.grad.numel() * h.grad.element_size() + W.grad.numel() * W.grad.element_size()
    peak = torch.cuda.max_memory_allocated(dev) - base - grads
    del h, W
    for _ in range(warmup):
        unfused_step(torch, w, hd, Wd, yd, gld, ged)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        unfused_step(torch, w, hd, Wd, yd, gld, ged)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    torch.cuda.empty_cache()
    return {"peak_extra_bytes": int(peak), "ms_per_step": ms, "tokens_per_s": w.N / (ms / 1e3),
            "steps": steps, "warmup": warmup,
            "what": "verl PR #462 equivalent compute logic in PyTorch (fp32 logits, softmax, "
                    "entropy, cross-entropy, autograd backward), masked like the fused path"}


def time_other_workload(torch, w, steps, warmup, dev, local, min_seconds=1.0):
    """The two-call step (flce_forward + flce_backward) of another workload: the same
    timing and clock sampling as the headline line's (the forward call timed apart too),
    over at least `steps` steps and at least `min_seconds` of them."""
    from linear_cross_entropy_forward_gb300 import (flce_backward, flce_forward, make_params,
                                                    workspace_size)
    from linear_cross_entropy_forward_gb300.workloads import make_inputs
    label_dev = "cuda" if w.label_mode == "self" else "cpu"
    hidden, weight, labels, g_loss, g_ent = make_inputs(w, label_device=label_dev)
    hd, Wd, yd = hidden.to(dev), weight.to(dev), labels.to(dev)
    gld, ged = g_loss.to(dev), g_ent.to(dev)
    del hidden, weight
    N, H, V = w.N, w.H, w.V
    n_out = N if w.reduction == "none" else 1
    out_f = (torch.empty(n_out, device=dev), torch.empty(n_out, device=dev),
             torch.empty(N, device=dev), torch.empty(N, device=dev))
    out_b = (torch.empty(N, H, dtype=torch.bfloat16, device=dev),
             torch.empty(H, V, dtype=torch.bfloat16, device=dev))
    p = make_params(N, H, V, w.reduction, zloss_coef=w.zloss_coef, softcap=w.softcap)
    ws_f = torch.empty(workspace_size(p, 0), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(workspace_size(p, 1), dtype=torch.uint8, device=dev)
    kw = dict(zloss_coef=w.zloss_coef, softcap=w.softcap)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if needs_flush(w) else None

    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        flce_forward(hd, Wd, yd, w.reduction, workspace=ws_f, out=out_f, **kw)
        if ev is not None:
            ev[1].record(stream)
        flce_backward(hd, Wd, yd, out_f[2], out_f[3], gld, ged, w.reduction, workspace=ws_b,
                      out=out_b, **kw)
        if ev is not None:
            ev[2].record(stream)

    w0 = torch.cuda.Event(enable_timing=True)
    w1 = torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for _ in range(warmup):
        step()
    w1.record(stream)
    torch.cuda.synchronize()
    # at least min_seconds of timed steps, so that the clock record holds several samples
    # under load (a short workload's K steps alone take a fraction of a sampling period)
    est = w0.elapsed_time(w1) / max(warmup, 1)
    steps = max(steps, min(20000, math.ceil(min_seconds * 1e3 / max(est, 1e-3))))
    sampler = ClockSampler(nvsmi_id(torch, local))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    t0 = time.time()
    for i in range(steps):
        if flush is not None:
            flush.fill_(i & 255)
        step(ev[i])
    torch.cuda.synchronize()
    t1 = time.time()
    sampler.stop()
    ms = sum(e[0].elapsed_time(e[2]) for e in ev) / steps
    f_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
    tflops = 8.0 * N * H * V / (ms / 1e3) / 1e12
    f_tflops = 2.0 * N * H * V / (f_ms / 1e3) / 1e12
    peak, _ = load_peaks()
    clocks = sampler.summary(t0, t1)
    res = {"N": N, "H": H, "V": V, "ms_per_step": ms, "tokens_per_s": N / (ms / 1e3),
           "tflops": tflops, "frac_of_peak": tflops / peak,
           "fwd_ms": f_ms, "fwd_tflops": f_tflops, "fwd_frac_of_peak": f_tflops / peak,
           "clocks": clocks, "steps": steps, "warmup": warmup,
           "l2": "flushed between steps" if flush is not None else "inputs larger than L2"}
    del hd, Wd, yd, out_f, out_b, ws_f, ws_b, flush
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    from linear_cross_entropy_forward_gb300 import (flce_backward, flce_forward,
                                                    flce_forward_backward, kernel_launches,
                                                    make_params, workspace_size)
    from linear_cross_entropy_forward_gb300.build import build
    from linear_cross_entropy_forward_gb300.workloads import WORKLOADS, make_inputs

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    if rank == 0 or world == 1:
        build()
    if pg:
        pg.barrier()
    build()  # no-op once built; loads nothing yet

    w = select_workload(args)
    label_dev = "cuda" if w.label_mode == "self" else "cpu"
    hidden, weight, labels, g_loss, g_ent = make_inputs(w, label_device=label_dev)
    hd, Wd, yd = hidden.to(dev), weight.to(dev), labels.to(dev)
    gld, ged = g_loss.to(dev), g_ent.to(dev)
    N, H, V = w.N, w.H, w.V
    n_out = N if w.reduction == "none" else 1
    loss = torch.empty(n_out, device=dev)
    ent = torch.empty(n_out, device=dev)
    lse = torch.empty(N, device=dev)
    ez = torch.empty(N, device=dev)
    dh = torch.empty(N, H, dtype=torch.bfloat16, device=dev)
    dw = torch.empty(H, V, dtype=torch.bfloat16, device=dev)
    p = make_params(N, H, V, w.reduction, zloss_coef=w.zloss_coef, softcap=w.softcap)
    # memory above the inputs, outputs and saved per-row statistics: the workspaces
    torch.cuda.synchronize()
    mem_base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    ws_f = torch.empty(workspace_size(p, 0), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(workspace_size(p, 1), dtype=torch.uint8, device=dev)
    kw = dict(zloss_coef=w.zloss_coef, softcap=w.softcap)

    def fwd():
        flce_forward(hd, Wd, yd, w.reduction, workspace=ws_f, out=(loss, ent, lse, ez), **kw)

    def bwd():
        flce_backward(hd, Wd, yd, lse, ez, gld, ged, w.reduction, workspace=ws_b, out=(dh, dw),
                      **kw)

    fwd()
    bwd()
    torch.cuda.synchronize()
    peak_extra = torch.cuda.max_memory_allocated(dev) - mem_base
    stream = torch.cuda.current_stream()
    K = args.steps
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if needs_flush(w) else None

    def timed_two_call():
        """W warm-up steps, then K timed steps; the SM clocks are sampled throughout."""
        sampler = ClockSampler(nvsmi_id(torch, local))
        for _ in range(args.warmup):
            fwd()
            bwd()
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
        t_host0 = time.time()
        e_start = torch.cuda.Event(enable_timing=True)
        e_end = torch.cuda.Event(enable_timing=True)
        e_start.record(stream)
        for i in range(K):
            if flush is not None:
                flush.fill_(i & 255)
            ev[i][0].record(stream)
            fwd()
            ev[i][1].record(stream)
            bwd()
            ev[i][2].record(stream)
        e_end.record(stream)
        torch.cuda.synchronize()
        t_host1 = time.time()
        f_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
        b_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
        # with flushes between steps only the steps are timed
        tot = e_start.elapsed_time(e_end) if flush is None else sum(f_ms) + sum(b_ms)
        if pg:
            t = torch.tensor([tot], device=dev)
            pg.all_reduce(t, op=pg.ReduceOp.MAX)
            tot = float(t.item())
            pg.barrier()
        sampler.stop()
        return tot, f_ms, b_ms, sampler.summary(t_host0, t_host1)

    # a window whose clock record shows a hardware or thermal slowdown is measured once more
    total_ms, fwd_ms, bwd_ms, clocks = timed_two_call()
    slowed = 1.0 if REJECTED_CLOCK_REASONS & set(clocks["reasons"]) else 0.0
    if pg:
        t = torch.tensor([slowed], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        slowed = float(t.item())
    if slowed:
        first = clocks["reasons"]
        total_ms, fwd_ms, bwd_ms, clocks = timed_two_call()
        clocks["remeasured_after"] = first

    # the same step as one flce_forward_backward call (gradient in forward, no recompute)
    gif = None
    if not args.no_grad_in_forward:
        ws_g = torch.empty(workspace_size(p, 3), dtype=torch.uint8, device=dev)

        def fused():
            flce_forward_backward(hd, Wd, yd, gld, ged, w.reduction, workspace=ws_g,
                                  out=(loss, ent, lse, ez, dh, dw), **kw)

        for _ in range(args.warmup):
            fused()
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for i in range(K):
            if flush is not None:
                flush.fill_(i & 255)
            gev[i][0].record(stream)
            fused()
            gev[i][1].record(stream)
        g1.record(stream)
        torch.cuda.synchronize()
        gif_ms = (g0.elapsed_time(g1) if flush is None
                  else sum(a.elapsed_time(b) for a, b in gev)) / K
        if pg:
            t = torch.tensor([gif_ms], device=dev)
            pg.all_reduce(t, op=pg.ReduceOp.MAX)
            gif_ms = float(t.item())
        gif = {"value": N * world / (gif_ms / 1e3), "unit": UNIT, "ms_per_step": gif_ms,
               "tflops_algorithmic": 6.0 * N * H * V / (gif_ms / 1e3) / 1e12,
               "algorithmic": "6*N*H*V flops per step (no recompute)",
               "workspace_bytes": int(ws_g.numel()),
               "gpu_launches": kernel_launches(p, 4) * K}
        del ws_g

    # end to end through HostPipeline: every step's inputs copied in from pinned host memory
    # (on a side stream, the next step's copy overlapping this step's compute) and its loss and
    # entropy copied back, all inside the timed region
    from linear_cross_entropy_forward_gb300.pipeline import HostPipeline
    host_in = (hidden.pin_memory(), weight.pin_memory(), labels.cpu().pin_memory(),
               g_loss.pin_memory(), g_ent.pin_memory())

    def e2e(gif):
        pipe = HostPipeline(N, H, V, w.reduction, zloss_coef=w.zloss_coef, softcap=w.softcap,
                            grad_in_forward=gif, device=dev)
        pipe.submit(*host_in)
        pipe.step()
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        steps = args.e2e_steps
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        sampler = ClockSampler(nvsmi_id(torch, local))
        t0 = time.time()
        ev[0].record(stream)
        pipe.copy_stream.wait_stream(stream)
        pipe.submit(*host_in)
        for i in range(steps):
            if i + 1 < steps:
                pipe.submit(*host_in)
            pipe.step()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        t1 = time.time()
        sampler.stop()
        ms = ev[0].elapsed_time(ev[steps]) / steps
        med = statistics.median(ev[i].elapsed_time(ev[i + 1]) for i in range(steps))
        if pg:
            t = torch.tensor([ms], device=dev)
            pg.all_reduce(t, op=pg.ReduceOp.MAX)
            ms = float(t.item())
        res = (ms, med, pipe.h2d_bytes(), pipe.d2h_bytes(), sampler.summary(t0, t1))
        del pipe
        return res

    e2e_res = None
    if not args.no_e2e:
        e2e_res = e2e(False)
        if gif is not None:
            gms, gmed, _, _, gclk = e2e(True)
            gif["e2e"] = {"value": N * world / (gms / 1e3), "unit": UNIT, "ms_per_step": gms,
                          "median_step_ms": gmed, "clocks": gclk}

    # the unfused baseline: the pages' equivalent compute logic in plain PyTorch (fp32
    # logits, softmax, entropy, cross-entropy, autograd backward), run outside every
    # timed region of the fused path; its peak memory above the inputs (the gradients
    # excluded as outputs) and its time per step
    unfused = None
    if not args.no_unfused_memory:
        del ws_f, ws_b
        unfused = unfused_baseline(torch, w, hd, Wd, yd, gld, ged, dev)

    ms_step = total_ms / K
    tokens = N * world
    value = tokens / (ms_step / 1e3)
    flops_step = 8.0 * N * H * V
    tflops = flops_step / (ms_step / 1e3) / 1e12
    peak, peak_src = load_peaks()
    fracs = roofline_fractions(2.0 * N * H * V / (statistics.mean(fwd_ms) / 1e3) / 1e12,
                               clocks.get("sm_mhz"))
    fwd_avg = statistics.mean(fwd_ms)
    bwd_avg = statistics.mean(bwd_ms)
    fwd_tflops = 2.0 * N * H * V / (fwd_avg / 1e3) / 1e12
    bwd_tflops = 6.0 * N * H * V / (bwd_avg / 1e3) / 1e12
    launches = (kernel_launches(p, 0) + kernel_launches(p, 1)) * K

    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w, world),
        "tflops": tflops * world, "pct_peak": 100.0 * tflops / peak,
        "peak_tflops": peak, "peak_source": peak_src,
        "fwd_ms": fwd_avg, "bwd_ms": bwd_avg, "fwd_tflops": fwd_tflops, "bwd_tflops": bwd_tflops,
        "roofline": {"bound": "tensor",
                     "kernel": "flce_gemm_pair_kernel<EPI_FWD_STATS> (timed as the flce_forward call)",
                     "achieved": fwd_tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": fwd_tflops / peak, "peak_note": peak_src,
                     **fracs,
                     "algorithmic": "2*N*H*V flops per launch",
                     "traffic": load_traffic(w.name)},
        "roofline_step": {"bound": "tensor", "achieved": tflops, "peak": peak,
                          "unit": "TFLOP/s", "frac": tflops / peak,
                          "algorithmic": "8*N*H*V flops per step (fwd 2, bwd 6 incl. recompute)"},
        "memory": {"peak_extra_bytes": int(peak_extra),
                   "unfused_peak_extra_bytes": unfused and unfused["peak_extra_bytes"],
                   "workspace_fwd_bytes": int(workspace_size(p, 0)),
                   "workspace_bwd_bytes": int(workspace_size(p, 1)),
                   "unfused_fp32_logits_bytes": int(N * V * 4)},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if e2e_res is not None:
        e2e_ms, e2e_med, h2d, d2h, e2e_clk = e2e_res
        # its own window's clock record: under the power cap the clock settles a little
        # differently from one window to the next, so compare the two per clock
        out["e2e"] = {"value": tokens / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                      "median_step_ms": e2e_med, "clocks": e2e_clk}
    if unfused is not None:
        unfused["speedup_of_fused"] = unfused["ms_per_step"] / ms_step
        out["unfused_baseline"] = unfused
    if gif is not None:
        gif["speedup_vs_two_call"] = ms_step / gif["ms_per_step"]
        out["grad_in_forward"] = gif
    if gif is not None:
        out["memory"]["grad_in_forward_extra_bytes"] = gif["workspace_bytes"]
    reduced = args.tokens or args.vocab or args.softcap is not None
    if world == 1 and not args.no_other_workloads and not reduced:
        # the other workloads' two-call step, measured the same way (no e2e, no baselines)
        from linear_cross_entropy_forward_gb300.workloads import WORKLOADS
        others = {}
        for name, ow in WORKLOADS.items():
            if name == w.name:
                continue
            others[name] = time_other_workload(torch, ow, args.steps, args.warmup, dev, local)
        out["other_workloads"] = others
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"], o_sample = cpu_baseline(w, hidden, weight, labels, g_loss, g_ent,
                                                     args.cpu_seconds)
        # the outputs of the last timed call against the oracle on the same rows
        out["oracle_check"] = oracle_check(o_sample, lse, ez, loss, ent, w.reduction)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


# ---------------------------------------------------------------- reference arm
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from linear_cross_entropy_forward_gb300.workloads import make_inputs
    w = select_workload(args)
    if w.label_mode == "self":
        import torch
        label_dev = "cuda" if torch.cuda.is_available() else "cpu"
    else:
        label_dev = "cpu"
    hidden, weight, labels, g_loss, g_ent = make_inputs(w, label_device=label_dev)
    ai = oracle_inputs(w, hidden, weight, labels, g_loss, g_ent)
    per_step = max(1.0, 150.0 / max(1, args.steps + args.warmup))
    rows, _ = calibrate_rows(w, ai, per_step)
    for _ in range(args.warmup):
        oracle_sample_step(w, *ai, rows=rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample_step(w, *ai, rows=rows)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    value = rows / dt
    sample = (f"fp64 numpy oracle fwd+bwd on the first {rows} of {w.N} rows per step "
              f"(full H={w.H}, V={w.V})")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": workload_config(w, 1),
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(),
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        rank, world, _ = dist_env()
        if world > 1 and rank == 0:
            # torchrun sets one OpenMP thread per rank; here the other ranks do no work,
            # so rank 0's oracle gets every core (numpy is not loaded yet)
            os.environ["OPENBLAS_NUM_THREADS"] = os.environ["OMP_NUM_THREADS"] = \
                str(host_cores())
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
