#!/usr/bin/env python
"""Fused transformer MLP benchmark on GB300: us/call, TFLOP/s and roofline fraction.

One "step" is one call of the whole hot path -- the up projection with its fused
bias/activation/rounding epilogue and the down projection -- on one batch of
seeded synthetic input already resident in HBM.  The default workload is the F16
SigLIP MLP X[1,729,1152] -> 4304 -> 1152 with tanh GELU and no biases.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl kt|reference]
                    [--block ln,res] [--weights in_out|out_in]

``--block`` runs the feed-forward as a transformer block applies it (LayerNorm
prologue kernel and / or the residual add fused into the down projection);
``--weights out_in`` passes the weights in PyTorch's nn.Linear order.  The
FLOP count stays that of the two GEMMs.

Timing: W untimed warm-up steps, then K steps bracketed by a barrier and a
device synchronize on both sides.  Each step's device time is taken with CUDA
events on the launching stream; a 256 MiB buffer (> the 129 MB L2) is written
between steps, outside the events, so every step reads its inputs from HBM
("cold", the headline: mean, median and p90 of the K steps).  The same steps are
then timed without the scrub ("warm": weights and X resident in L2).  Unless
``--no-configs``, every other workload of the suite (the tiny case, both SDXL
feed-forward levels and the ragged-M sweep) is timed in the same run with the same
cold protocol and reported under ``configs``.
For N > 1 (torchrun, one rank per GPU) every rank runs its own replica of the
workload (no collective on the data path: "scaling": "weak"); the time is the
maximum over ranks and the value the work of all ranks over that time.

The JSON line also carries: the per-kernel roofline of the dominant kernel
(device time per launch from CUDA events, against MEASURED_PEAKS.json), the
end-to-end number through the C ABI with host buffers (kt_mlp_run_host), the
SM clocks sampled with nvidia-smi every 20 ms (over the timed region, and over a
clock soak of about two seconds of the same steps whose per-step times are binned
by the sampled SM clock), and the float64 CPU oracle timed on the host cores as a
reported baseline (with the CPU model and the threads it used).

``--impl reference`` times the oracle itself (the reference arm of this build):
each step computes a bounded sample of the workload's rows on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused MLP µs/call and TFLOP/s at 1 GB300; % of dense FP16/BF16 tensor peak"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_LABEL = f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write)"
CLOCK_PERIOD_MS = 20
CONFIG_SUITE = ("tiny", "siglip", "sdxl_l2", "sdxl_l1", "sweep_M256", "sweep_M1000", "sweep_M4096", "sweep_M16384")


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="siglip")
    ap.add_argument("--block", default="", help="comma list of block options: ln (LayerNorm prologue), "
                                                 "res (residual add in the down epilogue)")
    ap.add_argument("--weights", choices=["in_out", "out_in"], default="in_out")
    ap.add_argument("--h-path", choices=["memory", "on_chip", "auto"], default="memory",
                    help="where H lives between the projections (on_chip: the fused kernel, D <= 256)")
    ap.add_argument("--launches", choices=["auto", "one", "two"], default="auto",
                    help="both projections in one persistent launch (one) or two launches (two; auto: the "
                         "planner's choice)")
    ap.add_argument("--shape", default=None,
                    help="a custom workload instead of --workload: M,D,F,act,dtype,bias with act one of "
                         "gelu_erf|gelu_tanh|geglu|none|gelu_sigmoid|silu and dtype f16|bf16")
    ap.add_argument("--impl", choices=["kt", "reference"], default="kt")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="minimum CPU time of the oracle baseline sample (kt arm)")
    ap.add_argument("--reference-seconds", type=float, default=90.0,
                    help="target total CPU time of the reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="time the selected workload only")
    ap.add_argument("--config-steps", type=int, default=200, help="cold steps per workload of the configs table")
    ap.add_argument("--soak-seconds", type=float, default=2.0, help="length of the clock soak (0: none)")
    ap.add_argument("--json-out", default=None, help="also write the JSON line to this file")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(values, dist, device):
    """Element-wise maximum of a list of floats over all ranks (the slowest rank's times)."""
    import torch
    v = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(v, op=dist.ReduceOp.MAX)
    return [float(x) for x in v]


def job_value(world: int, steps: int, flops_per_step: float, seconds: float) -> float:
    """Whole-job TFLOP/s: the work of every rank (weak scaling) over the slowest rank's time."""
    return world * steps * flops_per_step / seconds / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = ("kt_gemm.cuh", "kt_gemm_act.cu", "kt_gemm_geglu.cu", "kt_gemm_down.cu", "kt_mlp_two_act_f16.cu",
                  "kt_mlp_two_act_bf16.cu", "kt_mlp_two_geglu.cu", "kt_mlp_kernels.cu",
                  "kt_internal.h")


def _code_only(text: str) -> str:
    """The source without comments and blank lines: what the compiler sees (comment edits
    leave the measured kernels, and so their ncu counters, unchanged)."""
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif text[i] == '"':  # string literal, kept whole
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "transformer_mlp_gemms_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()


def ncu_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it is still current."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_sha256") != kernel_source_hash():
        return None
    entry = d.get("workloads", {}).get(workload, {}).get(kernel)
    return entry.get("dram_bytes_per_launch") if entry else None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons every CLOCK_PERIOD_MS in the background; each
    sample is stamped with the host's clock when it is read."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        import threading
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", str(CLOCK_PERIOD_MS)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            row = parse_clock_line(line)
            if row is not None:
                row["t"] = time.perf_counter()
                self.rows.append(row)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)
        return list(self.rows)


def parse_clock_line(line: str):
    parts = [x.strip() for x in line.split(",")]
    if len(parts) < 9:
        return None
    try:
        return {"sm": float(parts[1]), "max": float(parts[2]),
                "power": float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else None,
                "hw_slowdown": parts[5], "hw_thermal": parts[6], "sw_thermal": parts[7],
                "sw_power_cap": parts[8]}
    except ValueError:
        return None


def summarize_clocks(rows, window=None):
    """Median SM clock under load and the throttle reasons seen.  ``window`` = (t0, t1)
    restricts the summary to the samples read in that host-time interval."""
    if window is not None:
        rows = [r for r in rows if window[0] <= r.get("t", -1.0) <= window[1]]
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
    powers = [r["power"] for r in rows if r["power"] is not None]
    pmax = max(powers) if powers else None
    loaded = [r for r in rows if r["power"] is not None and pmax and r["power"] >= 0.5 * pmax] or rows
    reasons = []
    for key, name in (("hw_slowdown", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                      ("sw_thermal", "sw_thermal_slowdown"), ("sw_power_cap", "sw_power_cap")):
        if any(r[key] == "Active" for r in loaded):
            reasons.append(name)
    return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
            "sm_max_mhz": max(r["max"] for r in rows), "reasons": reasons,
            "samples": len(rows), "samples_under_load": len(loaded), "power_w_max": pmax}


def bin_by_clock(chunks, rows, bin_mhz: float = 30.0):
    """Per-step device time binned by the SM clock: each chunk (host-time interval, its
    steps' device times in ms) takes the clock samples read inside its interval."""
    bins = {}
    for t0, t1, times in chunks:
        near = [r["sm"] for r in rows if t0 <= r.get("t", -1.0) <= t1]
        if not near:
            continue
        mhz = bin_mhz * round(statistics.median(near) / bin_mhz)
        bins.setdefault(mhz, []).extend(times)
    return [{"sm_mhz": m, "steps": len(v), "us_per_step_median": 1e3 * statistics.median(v),
             "us_x_ghz": 1e3 * statistics.median(v) * m / 1e3}
            for m, v in sorted(bins.items())]


def step_stats(ms_list):
    """Mean, median and p90 of per-step device times (ms) in us."""
    v = sorted(ms_list)
    p90 = v[min(len(v) - 1, int(round(0.9 * (len(v) - 1))))]
    return {"mean": 1e3 * statistics.mean(v), "median": 1e3 * statistics.median(v), "p90": 1e3 * p90,
            "min": 1e3 * v[0], "steps": len(v)}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform string)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_baseline(w, t_bits, min_seconds: float, max_seconds: float = 30.0):
    """The float64 oracle, as it stands, on the host cores: whole workload, repeated."""
    import numpy as np
    import oracle
    flops_row = 2 * (w.D * w.F_up + w.F * w.D)
    rows = np.arange(w.M, dtype=np.int64)
    if w.M * flops_row > 5e11:  # very large M: a fixed row sample keeps one pass near seconds
        rows = np.linspace(0, w.M - 1, num=max(1, int(5e11 // flops_row)), dtype=np.int64)
    done_rows, t_total, passes = 0, 0.0, 0
    while True:
        t0 = time.perf_counter()
        oracle.mlp(t_bits["X"], t_bits["W_up"], t_bits["W_down"], t_bits.get("b_up"), t_bits.get("b_down"),
                   act=w.act, dtype=w.dtype, rows=rows)
        t_total += time.perf_counter() - t0
        done_rows += rows.size
        passes += 1
        if t_total >= min_seconds or t_total + t_total / passes > max_seconds:
            break
    value = done_rows * flops_row / t_total / 1e12
    return {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "cpu_model": cpu_model(), "kind": "oracle",
            "sample": f"{passes} pass(es) over {rows.size} of {w.M} rows of {w.name} "
                      f"({done_rows * flops_row / 1e9:.1f} GFLOP in {t_total:.1f} s, float64, OpenMP over rows)"}


def block_options(args):
    opts = {o for o in args.block.split(",") if o}
    bad = opts - {"ln", "res"}
    if bad:
        raise SystemExit(f"unknown --block option(s): {sorted(bad)}")
    return "ln" in opts, "res" in opts, args.weights == "out_in"


def h_path_code(args):
    from transformer_mlp_gemms_gb300 import kt_mlp
    return {"memory": kt_mlp.KT_H_MEMORY, "on_chip": kt_mlp.KT_H_ON_CHIP, "auto": kt_mlp.KT_H_AUTO}[args.h_path]


def launches_code(args):
    from transformer_mlp_gemms_gb300 import kt_mlp
    return {"auto": kt_mlp.KT_LAUNCH_AUTO, "one": kt_mlp.KT_LAUNCH_ONE, "two": kt_mlp.KT_LAUNCH_TWO}[
        getattr(args, "launches", "auto")]


def pick_workload(args):
    from transformer_mlp_gemms_gb300 import workloads as wl
    if not args.shape:
        return wl.WORKLOADS[args.workload]
    M, D, F, act, dt, bias = args.shape.split(",")
    acts = {v: k for k, v in wl.ACT_NAMES.items()}
    dts = {v: k for k, v in wl.DT_NAMES.items()}
    return wl.custom(int(M), int(D), int(F), acts[act], dts[dt], bias in ("1", "true", "yes"), seed=11,
                     name=f"custom_{M}x{D}x{F}")


def kernel_bytes(w, kernel: str, residual: bool) -> int:
    """Algorithmic DRAM bytes of one launch: every operand read once, every result written once."""
    e = 2
    x, y, h = w.M * w.D * e, w.M * w.D * e, w.M * w.F * e
    wu, wd = w.D * w.F_up * e, w.F * w.D * e
    bu, bd = (w.F_up * e, w.D * e) if w.bias else (0, 0)
    r = y if residual else 0
    if kernel == "up":
        return x + wu + bu + h
    if kernel == "down":
        return h + wd + bd + r + y
    if kernel == "one":  # both projections in one kernel, H through memory
        return x + wu + bu + 2 * h + wd + bd + r + y
    return x + wu + bu + wd + bd + r + y  # both projections in one kernel, H on chip


def traffic_key(w, args) -> str:
    ln, res, outin = block_options(args)
    tags = [t for t, on in (("ln", ln), ("res", res), ("out_in", outin), ("h_on_chip", args.h_path != "memory"),
                            ("one_launch", getattr(args, "launches", "auto") == "one")) if on]
    return w.name + (f"[{','.join(tags)}]" if tags else "")


def workload_config(w, l2, args=None):
    from transformer_mlp_gemms_gb300 import workloads as wl
    cfg = {"workload": f"{w.name}: X[{w.batch},{w.tokens},{w.D}] -> {w.F_up} -> {w.D}",
           "M": w.M, "D": w.D, "F": w.F, "F_up": w.F_up, "act": wl.ACT_NAMES[w.act],
           "io_dtype": wl.DT_NAMES[w.dtype], "bias": w.bias, "seed": w.seed,
           "flops_per_call": w.flops, "l2": l2}
    if args is not None:
        ln, res, outin = block_options(args)
        cfg["block"] = {"layernorm": ln, "residual": res, "weights": "out_in" if outin else "in_out",
                        "h_path": args.h_path, "launches": getattr(args, "launches", "auto")}
    return cfg


def emit(line, args):
    s = json.dumps(line)
    print(s, flush=True)
    if args.json_out:
        with open(args.json_out, "w") as f:
            f.write(s + "\n")


def run_reference(args, w, rank, world):
    """The reference arm: the float64 oracle on the host cores, bounded samples per step."""
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    from transformer_mlp_gemms_gb300 import workloads as wl
    b = {k: wl.bits(v) for k, v in wl.generate(w).items()}
    flops_row = 2 * (w.D * w.F_up + w.F * w.D)
    oracle.build()
    cal = np.arange(min(w.M, 32), dtype=np.int64)
    t0 = time.perf_counter()
    oracle.mlp(b["X"], b["W_up"], b["W_down"], b.get("b_up"), b.get("b_down"), act=w.act, dtype=w.dtype, rows=cal)
    rate = cal.size * flops_row / max(time.perf_counter() - t0, 1e-6)
    steps_total = args.steps + args.warmup
    rows_per_step = int(max(1, min(w.M, args.reference_seconds * rate / (steps_total * flops_row))))
    rng = np.random.default_rng(w.seed)
    samples = [np.sort(rng.choice(w.M, size=rows_per_step, replace=False)).astype(np.int64)
               for _ in range(steps_total)]

    def step(i):
        oracle.mlp(b["X"], b["W_up"], b["W_down"], b.get("b_up"), b.get("b_down"), act=w.act, dtype=w.dtype,
                   rows=samples[i])

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.warmup, steps_total):
        step(i)
    dt = time.perf_counter() - t0
    value = args.steps * rows_per_step * flops_row / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, l2=L2_LABEL, args=args),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "cpu_model": cpu_model(),
                         "kind": "oracle",
                         "sample": f"{rows_per_step} random rows of {w.M} per step, float64 oracle on the host "
                                   f"cores (operands in host memory)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    emit(line, args)
    return 0


def time_config(w, steps: int, flush, stream) -> dict:
    """One workload of the suite on the planner's default plan: cold steps (L2 scrubbed
    before each), CUDA events per step; us/call, TFLOP/s and the fraction of the measured
    dense peak."""
    import torch
    from transformer_mlp_gemms_gb300 import kt_mlp
    from transformer_mlp_gemms_gb300 import workloads as wl
    t = wl.generate(w)
    d = {k: v.cuda() for k, v in t.items()}
    Y = torch.empty((w.M, w.D), dtype=wl.TORCH_DTYPES[w.dtype], device="cuda")
    plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias)
    info = plan.info()

    def once():
        plan.run(d["X"], d["W_up"], d["W_down"], d.get("b_up"), d.get("b_down"), Y)

    for _ in range(5):
        flush.zero_()
        once()
    evs = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.zero_()
        a.record(stream)
        once()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    ok = plan.status() == kt_mlp.KT_OK
    plan.close()
    if not ok:
        raise RuntimeError(f"device status after {w.name}: " + kt_mlp.kt_last_error())
    st = step_stats([a.elapsed_time(b) for a, b in evs])
    peaks, _ = load_peaks()
    peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    tflops = w.flops / (st["mean"] * 1e-6) / 1e12
    up, dn = info["up"], info["down"]
    return {"workload": f"X[{w.batch},{w.tokens},{w.D}] -> {w.F_up} -> {w.D}, {wl.ACT_NAMES[w.act]}, "
                        f"{wl.DT_NAMES[w.dtype]}, bias={int(w.bias)}",
            "us_per_call": st["mean"], "us_median": st["median"], "us_p90": st["p90"], "steps": steps,
            "tflops": tflops, "frac_of_measured_peak": tflops / peak,
            "plan": {"one_launch": info["one_launch"], "h_on_chip": info["h_on_chip"],
                     "up": f"{up['BM']}x{up['BN']} BK{up['BK']} grid {up['grid']}",
                     "down": f"{dn['BM']}x{dn['BN']} BK{dn['BK']} split {dn['split_k']}"
                             f"{' cluster' if dn['cluster_sk'] else ''} grid {dn['grid']}"}}


def main():
    args = parse_args()
    rank, world, local = dist_env()
    from transformer_mlp_gemms_gb300 import workloads as wl
    w = pick_workload(args)
    if args.impl == "reference":
        return run_reference(args, w, rank, world)

    import torch
    from transformer_mlp_gemms_gb300 import build as kbuild
    from transformer_mlp_gemms_gb300 import kt_mlp

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0:
        kbuild.build()
    if dist is not None:
        dist.barrier()
    kt_mlp.load()

    ln, res, outin = block_options(args)
    plain = not (ln or res) and args.h_path == "memory"
    t = wl.generate(w, residual=res, layernorm=ln)
    dev_t = wl.torch_order(t) if outin else t
    d = {k: v.cuda() for k, v in dev_t.items()}
    tdt = wl.TORCH_DTYPES[w.dtype]
    Y = torch.empty((w.M, w.D), dtype=tdt, device="cuda")
    plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias, residual=res, layernorm=ln,
                       weight_layout=kt_mlp.KT_W_OUT_IN if outin else kt_mlp.KT_W_IN_OUT, h_path=h_path_code(args),
                       launches=launches_code(args))
    info = plan.info()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    args_run = (d["X"], d["W_up"], d["W_down"], d.get("b_up"), d.get("b_down"), Y)
    ex_kw = dict(b_up=d.get("b_up"), b_down=d.get("b_down"), R=d.get("R"), ln_gamma=d.get("ln_gamma"),
                 ln_beta=d.get("ln_beta"))

    def run_once(X=d["X"], Yo=Y):
        if plain:
            plan.run(X, d["W_up"], d["W_down"], d.get("b_up"), d.get("b_down"), Yo)
        else:
            plan.run_ex(X, d["W_up"], d["W_down"], Yo, **ex_kw)

    props = torch.cuda.get_device_properties(local)
    gpu_id = str(local)
    uuid = getattr(props, "uuid", None)
    if uuid is not None:
        gpu_id = str(uuid) if str(uuid).startswith("GPU-") else "GPU-" + str(uuid)
    sampler = ClockSampler(gpu_id)

    for _ in range(args.warmup):
        flush.zero_()
        run_once()
    torch.cuda.synchronize()
    if plan.status() != kt_mlp.KT_OK:
        raise RuntimeError("device status after warm-up: " + kt_mlp.kt_last_error())

    # ---------------- timed region: K steps, barrier + synchronize on both sides ----------------
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()                 # L2 scrub, outside the step's events
        starts[i].record(stream)
        run_once()
        ends[i].record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    wall1 = time.perf_counter()
    wall = wall1 - wall0
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(step_ms)
    if plan.status() != kt_mlp.KT_OK:
        raise RuntimeError("device status after the timed steps: " + kt_mlp.kt_last_error())

    # ---------------- warm: the same steps without the L2 scrub ----------------
    warm_ms = []
    for _ in range(max(1, min(args.steps, 500))):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run_once()
        b.record(stream)
        warm_ms.append((a, b))
    torch.cuda.synchronize()
    warm_ms = [a.elapsed_time(b) for a, b in warm_ms]

    # ---------------- clock soak: cold steps in chunks, binned by the sampled SM clock ----------------
    soak_chunks = []
    soak_end = time.perf_counter() + max(0.0, args.soak_seconds)
    while time.perf_counter() < soak_end:
        evs = []
        c0 = time.perf_counter()
        for _ in range(20):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            flush.zero_()
            a.record(stream)
            run_once()
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        soak_chunks.append((c0, time.perf_counter(), [a.elapsed_time(b) for a, b in evs]))

    # ---------------- per-kernel device time (same steps, events between the kernels) ----------------
    ms_ln, ms_up, ms_dn = [], [], []
    for _ in range(max(1, min(args.steps, 500))):
        flush.zero_()
        if plain:
            a, b = plan.run_timed(*args_run)
            c0 = 0.0
        else:
            c0, a, b = plan.run_ex_timed(d["X"], d["W_up"], d["W_down"], Y, **ex_kw)
        ms_ln.append(c0)
        ms_up.append(a)
        ms_dn.append(b)

    # ---------------- end to end through the C ABI with host buffers ----------------
    Xh = t["X"].pin_memory()
    Yh = torch.empty((w.M, w.D), dtype=tdt).pin_memory()
    Xs = torch.empty_like(d["X"])
    e2e_steps = max(1, min(args.steps, 500))

    def e2e_once():
        if plain:  # the library's own host-buffer entry point
            plan.run_host(Xh, d["W_up"], d["W_down"], d.get("b_up"), d.get("b_down"), Yh)
        else:      # copies on the stream around kt_mlp_run_ex, read back before the clock stops
            Xs.copy_(Xh, non_blocking=True)
            kw = dict(ex_kw)
            if res:
                kw["R"] = Xs   # the block's residual is its own input: x = ff(LayerNorm(x)) + x
            plan.run_ex(Xs, d["W_up"], d["W_down"], Y, **kw)
            Yh.copy_(Y, non_blocking=True)
            torch.cuda.current_stream().synchronize()

    for _ in range(min(args.warmup, 5)):
        e2e_once()
    e2e_s = 0.0
    for _ in range(e2e_steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_once()
        e2e_s += time.perf_counter() - t0
    # ---------------- the other workloads of the suite, same cold protocol ----------------
    configs = {}
    if not args.no_configs and args.shape is None and not (ln or res or outin) and args.h_path == "memory" \
            and getattr(args, "launches", "auto") == "auto":
        for name in CONFIG_SUITE:
            if name == w.name:
                continue
            configs[name] = time_config(wl.WORKLOADS[name], args.config_steps, flush, stream)
    clock_rows = sampler.stop()
    clocks = summarize_clocks(clock_rows, window=(wall0, wall1))
    clocks_all = summarize_clocks(clock_rows)
    clock_bins = bin_by_clock(soak_chunks, clock_rows)
    if clocks["samples"] == 0:  # a timed region shorter than the sampling period: the soak's samples
        clocks = dict(clocks_all, note=f"no sample fell inside the {wall * 1e3:.1f} ms timed region; "
                                       f"summary over the whole run ({CLOCK_PERIOD_MS} ms sampling)")

    if dist is not None:
        total_ms, e2e_s = reduce_max([total_ms, e2e_s], dist, "cuda")
    if rank != 0:
        plan.close()
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    value = job_value(world, args.steps, w.flops, total_ms * 1e-3)
    ms_per_step = total_ms / args.steps
    e2e_value = job_value(world, e2e_steps, w.flops, e2e_s)
    up_flops = 2 * w.M * w.D * w.F_up
    dn_flops = 2 * w.M * w.F * w.D
    mu, md, ml = statistics.mean(ms_up), statistics.mean(ms_dn), statistics.mean(ms_ln)
    fused = bool(info.get("h_on_chip"))
    one = bool(info.get("one_launch"))
    dominant = "fused" if fused else "one" if one else ("up" if mu >= md else "down")
    k_ms, k_flops = {"fused": (mu, w.flops), "one": (mu, w.flops), "up": (mu, up_flops),
                     "down": (md, dn_flops)}[dominant]
    peak_tflops = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])  # fp16 : bf16 nominal 1 : 1
    peak_gbs = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    achieved = k_flops / (k_ms * 1e-3) / 1e12
    # the dominant kernel's algorithmic bytes (each operand read once, each result written
    # once) and the roofline that binds: the larger of its FLOP floor and its byte floor
    k_bytes = kernel_bytes(w, dominant, res)
    t_tensor = k_flops / (peak_tflops * 1e12)
    t_hbm = k_bytes / (peak_gbs * 1e9)
    achieved_gbs = k_bytes / (k_ms * 1e-3) / 1e9
    hbm_bound = t_hbm > t_tensor
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.DT_NAMES[w.dtype], "data": "synthetic",
        "config": workload_config(w, l2=L2_LABEL, args=args),
        "us_per_call": ms_per_step * 1e3,
        "us_per_call_stats": {"cold": step_stats(step_ms), "warm": step_stats(warm_ms),
                              "note": "cold = L2 scrubbed before every step (the headline, its mean); warm = "
                                      "weights and X left resident in L2 by the previous step"},
        "pct_of_peak": 100.0 * value / world / peak_tflops,
        "peak_tflops": peak_tflops, "peak_source": peak_src,
        "roofline": {"bound": "hbm" if hbm_bound else "tensor",
                     "kernel": ("kt_fused_kernel (both projections, H on chip)" if fused else
                                "kt_gemm_kernel (both projections in one launch)" if one else
                                f"kt_gemm_kernel ({dominant} projection)"),
                     "achieved": achieved_gbs if hbm_bound else achieved,
                     "peak": peak_gbs if hbm_bound else peak_tflops,
                     "unit": "GB/s" if hbm_bound else "TFLOP/s",
                     "frac": achieved_gbs / peak_gbs if hbm_bound else achieved / peak_tflops,
                     "traffic": ncu_traffic(traffic_key(w, args), dominant),
                     "algorithmic_flops_per_launch": k_flops, "algorithmic_bytes_per_launch": k_bytes,
                     "tensor_frac": achieved / peak_tflops, "hbm_frac": achieved_gbs / peak_gbs,
                     "hbm_peak_gbs": peak_gbs, "ms_per_launch": k_ms,
                     "peak_note": (f"{peak_src} bf16 dense burst from MEASURED_PEAKS.json (fp16 has the "
                                   f"same nominal rate)") if peak_src == "measured" else "fallback"},
        "kernels_ms": ({"fused": mu, "fused_tflops": w.flops / (mu * 1e-3) / 1e12} if fused else
                       {"one_launch": mu, "one_launch_tflops": w.flops / (mu * 1e-3) / 1e12} if one else
                       {"up": mu, "down": md, "up_tflops": up_flops / (mu * 1e-3) / 1e12,
                        "down_tflops": dn_flops / (md * 1e-3) / 1e12}),
        **({"layernorm_kernel": {"ms": ml, "bytes": 2 * w.M * w.D * 2 + 2 * w.D * 2,
                                 "gbs": (2 * w.M * w.D * 2 + 2 * w.D * 2) / (ml * 1e-3) / 1e9 if ml > 0 else None}}
           if ln else {}),
        "plan": {"up": {k: info["up"][k] for k in ("BM", "BN", "BK", "stages", "split_k", "grid", "waves")},
                 "down": {k: info["down"][k] for k in ("BM", "BN", "BK", "stages", "split_k", "cluster_sk", "grid",
                                                       "waves")},
                 "h_on_chip": int(fused), "one_launch": int(one),
                 **({"fused": {"grid": info["fused_grid"], "stages": info["fused_stages"]}} if fused else {})},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": w.M * w.D * 2,
                "d2h_bytes_per_step": w.M * w.D * 2, "us_per_call": e2e_s / e2e_steps * 1e6,
                "entry_point": ("kt_mlp_run_host (pinned X in, Y out; weights resident)" if plain else
                                "kt_mlp_run_ex between a pinned X copy in and a Y copy out (weights resident)")},
        "gpu_launches": ((1 if fused or one else 2) + (1 if ln else 0)) * args.steps,
        "clocks": clocks,
        "clocks_whole_run": clocks_all,
        "clock_bins": clock_bins,
        **({"configs": configs} if configs else {}),
        "wall_s_timed_region": wall,
        "gpu": props.name, "sms": props.multi_processor_count,
    }
    plan.close()
    if dist is not None:
        dist.destroy_process_group()
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        line["cpu_baseline"] = oracle_baseline(w, {k: wl.bits(v) for k, v in t.items()}, args.cpu_seconds)
    emit(line, args)
    return 0


if __name__ == "__main__":
    sys.exit(main())
