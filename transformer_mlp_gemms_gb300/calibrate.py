"""Planner calibration: the planner's modelled time against measured time.

The planner (``csrc/kt_planner.cpp``) ranks tile configurations with an analytic
model and never autotunes at run time.  Its second opinion is a measured sweep,
the same check the IPU layout-sweep page applies to its own cost models (rank
correlation of modelled against measured time, and the selection regret of the
model's pick):

    python -m transformer_mlp_gemms_gb300.calibrate sweep siglip sdxl_l2 ... [--out DIR]
    python -m transformer_mlp_gemms_gb300.calibrate evaluate [--dir DIR] [workloads...]
    python -m transformer_mlp_gemms_gb300.calibrate sweep-one siglip ... [--out DIR]
    python -m transformer_mlp_gemms_gb300.calibrate evaluate-one [--dir DIR] [workloads...]

``sweep`` (needs the GPU) forces every feasible configuration of each GEMM of a
workload through the planner's override variables (``KT_FORCE_UP`` =
``BN,PAIR,BK``; ``KT_FORCE_DOWN`` = ``BN,SK,PAIR,BK,CLUSTER``), skips those of more
than 10 waves, and times each with ``kt_mlp_run_timed`` (CUDA events around each
kernel, 256 MiB L2 scrub before each call, mean of the calls after warm-up).  It
writes ``calib_<workload>.json``.  ``evaluate`` (host only) recomputes the model's
estimate of every measured configuration with the current library, and prints per
GEMM the Spearman rank correlation, the planner's pick, its measured time, the best
measured time and the regret.

``sweep-one`` (needs the GPU) does the same for the whole call in one launch: every
pairing of the model's two best up tiles of each CTA pairing with every down tile and
split the one-launch planner considers (K splits of up to four, all items in one round), forced with
``KT_FORCE_LAUNCHES=1``, plus the two-launch plan and the planner's own choice, each
timed as whole calls (CUDA events around ``kt_mlp_run``, the L2 scrub before each call).
``evaluate-one`` prints per workload the Spearman rank correlation of the one-launch
model against measurement, the model's one-launch pick and its regret, and the launch
decision (one or two launches) against the measured better of the two.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys

from . import kt_mlp
from . import workloads as wl

ENV = ("KT_FORCE_UP", "KT_FORCE_DOWN")


def _clear_env():
    for k in ENV:
        os.environ.pop(k, None)
    # each GEMM is measured and modelled on its own: two launches, never the one-launch schedule
    os.environ["KT_FORCE_LAUNCHES"] = "2"


def _restore_env():
    for k in ENV + ("KT_FORCE_LAUNCHES",):
        os.environ.pop(k, None)


def _configs():
    """(gemm, override value) for every candidate shape the planner considers."""
    out = []
    for pr in (1, 2):
        for bk in (64, 128):
            for bn in range(32 * pr, 257, 32 * pr):
                out.append(("up", f"{bn},{pr},{bk}"))
                for sk in (1, 2, 3, 4, 6, 8):
                    out.append(("down", f"{bn},{sk},{pr},{bk},0"))
                    if pr == 1 and sk > 1:
                        out.append(("down", f"{bn},{sk},{pr},{bk},1"))
    return out


def sweep(name: str, out_dir: str, calls: int = 40, warm: int = 5) -> list:
    import torch
    w = wl.WORKLOADS[name]
    t = wl.generate(w)
    d = {k: v.cuda() for k, v in t.items()}
    Y = torch.empty((w.M, w.D), dtype=wl.TORCH_DTYPES[w.dtype], device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    args = (d["X"], d["W_up"], d["W_down"], d.get("b_up"), d.get("b_down"), Y)
    rows = []
    for gemm, val in _configs():
        _clear_env()
        os.environ["KT_FORCE_UP" if gemm == "up" else "KT_FORCE_DOWN"] = val
        try:
            p = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias)
        except kt_mlp.KtError:
            continue  # infeasible: the planner rejects the override
        g = p.info()[gemm]
        if g["waves"] > 10:
            p.close()
            continue
        ms = []
        for i in range(calls + warm):
            flush.zero_()
            a, b = p.run_timed(*args)
            if i >= warm:
                ms.append((a if gemm == "up" else b) * 1e3)
        status = p.status()
        p.close()
        if status != kt_mlp.KT_OK:
            raise RuntimeError(f"{name} {gemm} {val}: device status {status}")
        r = {"gemm": gemm, "force": val, "BM": g["BM"], "BN": g["BN"], "BK": g["BK"], "SK": g["split_k"],
             "CL": g["cluster_sk"], "stages": g["stages"], "grid": g["grid"], "waves": g["waves"],
             "model_us": g["est_us"], "us_mean": statistics.mean(ms), "us_median": statistics.median(ms)}
        rows.append(r)
        print(json.dumps(r), flush=True)
    _restore_env()
    with open(os.path.join(out_dir, f"calib_{name}.json"), "w") as f:
        json.dump(rows, f)
    return rows


def _spearman(a, b) -> float:
    def ranks(x):
        order = sorted(range(len(x)), key=lambda i: x[i])
        r = [0.0] * len(x)
        i = 0
        while i < len(order):
            j = i
            while j + 1 < len(order) and x[order[j + 1]] == x[order[i]]:
                j += 1
            for k in range(i, j + 1):
                r[order[k]] = (i + j) / 2.0
            i = j + 1
        return r
    ra, rb = ranks(a), ranks(b)
    ma, mb = statistics.mean(ra), statistics.mean(rb)
    num = sum((x - ma) * (y - mb) for x, y in zip(ra, rb))
    den = (sum((x - ma) ** 2 for x in ra) * sum((y - mb) ** 2 for y in rb)) ** 0.5
    return num / den if den else float("nan")


def evaluate(names, in_dir: str, num_sms: int = 152) -> float:
    kt_mlp.load()
    total = 0.0
    print("| workload | GEMM | configs | Spearman | pick | pick measured µs | best measured µs | regret µs |")
    print("|---|---|---:|---:|---|---:|---:|---:|")
    for name in names:
        path = os.path.join(in_dir, f"calib_{name}.json")
        if not os.path.exists(path):
            continue
        w = wl.WORKLOADS[name]
        rows = json.load(open(path))
        for gemm in ("up", "down"):
            mod, meas, keep = [], [], []
            for r in (x for x in rows if x["gemm"] == gemm):
                _clear_env()
                os.environ["KT_FORCE_UP" if gemm == "up" else "KT_FORCE_DOWN"] = r["force"]
                try:
                    est = kt_mlp.kt_mlp_plan_info(w.M, w.D, w.F, w.act, w.dtype, w.bias, num_sms)[gemm]["est_us"]
                except kt_mlp.KtError:
                    continue  # no longer a candidate of the planner
                mod.append(est)
                meas.append(r["us_mean"])
                keep.append(r)
            _clear_env()
            pick = kt_mlp.kt_mlp_plan_info(w.M, w.D, w.F, w.act, w.dtype, w.bias, num_sms)[gemm]
            hit = [r for r in keep if (r["BM"], r["BN"], r["BK"], r["SK"], r["CL"]) ==
                   (pick["BM"], pick["BN"], pick["BK"], pick["split_k"], pick["cluster_sk"])]
            if not meas:
                continue
            best = min(meas)
            pm = hit[0]["us_mean"] if hit else float("nan")
            regret = pm - best
            if regret == regret:
                total += regret
            tag = f"{pick['BM']}x{pick['BN']}x{pick['BK']} SK {pick['split_k']}" + (" cluster" if pick["cluster_sk"] else "")
            print(f"| {name} | {gemm} | {len(keep)} | {_spearman(mod, meas):.2f} | {tag} | {pm:.2f} | {best:.2f} | "
                  f"{regret:.2f} |")
    _restore_env()
    print(f"\ntotal regret {total:.2f} µs")
    return total


def _force(up=None, down=None, launches=None):
    for k, v in (("KT_FORCE_UP", up), ("KT_FORCE_DOWN", down), ("KT_FORCE_LAUNCHES", launches)):
        if v:
            os.environ[k] = v
        else:
            os.environ.pop(k, None)


def _one_candidates(w, num_sms: int = 152, n_up: int = 2):
    """(up, down) overrides of the one-launch sweep: the n_up best up tiles of each pairing
    by the model, each with every down tile and split the one-launch planner's own search
    considers (no 16-column weight boxes; K splits only while all items fit one round)."""
    out = []
    for pr in (1, 2):
        ups = []
        for bk in (64, 128):
            for bn in range(32, 257, 32):
                _force(up=f"{bn},{pr},{bk}", launches="2")
                try:
                    g = kt_mlp.kt_mlp_plan_info(w.M, w.D, w.F, w.act, w.dtype, w.bias, num_sms)["up"]
                except kt_mlp.KtError:
                    continue
                ups.append((g["est_us"], f"{bn},{pr},{bk}"))
        for _, up in sorted(ups)[:n_up]:
            for bk in (64, 128):
                for bn in range(32, 257, 32):
                    if pr == 2 and (bn // 2) % 32:
                        continue  # 16-column weight boxes
                    for sk in (1, 2, 3, 4):
                        down = f"{bn},{sk},{pr},{bk},0"
                        _force(up=up, down=down, launches="1")
                        try:
                            info = kt_mlp.kt_mlp_plan_info(w.M, w.D, w.F, w.act, w.dtype, w.bias, num_sms)
                        except kt_mlp.KtError:
                            continue
                        dn = info["down"]
                        items = dn["tiles_m"] * dn["tiles_n"] * sk
                        if info["one_launch"] and (sk == 1 or items <= num_sms // pr):
                            out.append((up, down))
    _force()
    return out


def _time_calls(w, d, flush, calls: int, warm: int) -> float:
    import torch
    Y = torch.empty((w.M, w.D), dtype=wl.TORCH_DTYPES[w.dtype], device="cuda")
    p = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias)
    args = (d["X"], d["W_up"], d["W_down"], d.get("b_up"), d.get("b_down"), Y)
    stream = torch.cuda.current_stream()
    evs = []
    for i in range(calls + warm):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.zero_()
        a.record(stream)
        p.run(*args)
        b.record(stream)
        if i >= warm:
            evs.append((a, b))
    torch.cuda.synchronize()
    status = p.status()
    p.close()
    if status != kt_mlp.KT_OK:
        raise RuntimeError(f"device status {status}")
    return statistics.mean(a.elapsed_time(b) * 1e3 for a, b in evs)


def sweep_one(name: str, out_dir: str, calls: int = 20, warm: int = 3) -> list:
    import torch
    w = wl.WORKLOADS[name]
    t = wl.generate(w)
    d = {k: v.cuda() for k, v in t.items()}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    rows = []
    for up, down, launches in [(u, dn, "1") for u, dn in _one_candidates(w)] + [(None, None, "2"), (None, None, None)]:
        _force(up=up, down=down, launches=launches)
        try:
            us = _time_calls(w, d, flush, calls, warm)
        except kt_mlp.KtError:
            continue
        r = {"up": up, "down": down, "launches": launches, "us_mean": us}
        rows.append(r)
        print(json.dumps(r), flush=True)
    _force()
    with open(os.path.join(out_dir, f"calib_one_{name}.json"), "w") as f:
        json.dump(rows, f)
    return rows


def evaluate_one(names, in_dir: str, num_sms: int = 152) -> float:
    kt_mlp.load()
    total = 0.0
    print("| workload | one-launch configs | Spearman | one-launch pick | pick µs | best one-launch µs | regret µs "
          "| two launches µs | decision | decision regret µs |")
    print("|---|---:|---:|---|---:|---:|---:|---:|---|---:|")
    for name in names:
        path = os.path.join(in_dir, f"calib_one_{name}.json")
        if not os.path.exists(path):
            continue
        w = wl.WORKLOADS[name]
        rows = json.load(open(path))
        mod, meas, keep = [], [], []
        for r in rows:
            if r["launches"] != "1":
                continue
            _force(up=r["up"], down=r["down"], launches="1")
            try:
                info = kt_mlp.kt_mlp_plan_info(w.M, w.D, w.F, w.act, w.dtype, w.bias, num_sms)
            except kt_mlp.KtError:
                continue
            if not info["one_launch"]:
                continue
            mod.append(info["one_launch_est_us"])
            meas.append(r["us_mean"])
            keep.append(r)
        two = [r["us_mean"] for r in rows if r["launches"] == "2"]
        _force(launches="1")
        pick = kt_mlp.kt_mlp_plan_info(w.M, w.D, w.F, w.act, w.dtype, w.bias, num_sms)
        _force()
        auto = kt_mlp.kt_mlp_plan_info(w.M, w.D, w.F, w.act, w.dtype, w.bias, num_sms)
        if not meas:
            continue

        def key_of(info):
            u, dn = info["up"], info["down"]
            return (f"{u['BN']},{u['BM'] // 128},{u['BK']}", f"{dn['BN']},{dn['split_k']},{dn['BM'] // 128},{dn['BK']},0")

        pk = key_of(pick)
        hit = [r["us_mean"] for r in keep if (r["up"], r["down"]) == pk]
        pm = hit[0] if hit else float("nan")
        best = min(meas)
        regret = pm - best
        if regret == regret:
            total += regret
        two_us = two[0] if two else float("nan")
        chosen = min(best, two_us)
        dec = "one" if auto["one_launch"] else "two"
        dec_us = pm if auto["one_launch"] else two_us
        print(f"| {name} | {len(keep)} | {_spearman(mod, meas):.2f} | up {pk[0]}, down {pk[1]} | {pm:.2f} | {best:.2f} | "
              f"{regret:.2f} | {two_us:.2f} | {dec} | {dec_us - chosen:.2f} |")
    _force()
    print(f"\ntotal one-launch regret {total:.2f} µs")
    return total


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    sub = ap.add_subparsers(dest="cmd", required=True)
    s = sub.add_parser("sweep")
    s.add_argument("workloads", nargs="+")
    s.add_argument("--out", default=".")
    e = sub.add_parser("evaluate")
    e.add_argument("workloads", nargs="*")
    e.add_argument("--dir", default=".")
    so = sub.add_parser("sweep-one")
    so.add_argument("workloads", nargs="+")
    so.add_argument("--out", default=".")
    eo = sub.add_parser("evaluate-one")
    eo.add_argument("workloads", nargs="*")
    eo.add_argument("--dir", default=".")
    a = ap.parse_args(argv)
    if a.cmd in ("sweep", "sweep-one"):
        from . import build
        build.build()
        kt_mlp.load()
        os.makedirs(a.out, exist_ok=True)
        for n in a.workloads:
            (sweep if a.cmd == "sweep" else sweep_one)(n, a.out)
    elif a.cmd == "evaluate-one":
        names = a.workloads or ["siglip", "sdxl_l1", "sweep_M256", "sweep_M1000", "sweep_M4096"]
        evaluate_one(names, a.dir)
    else:
        names = a.workloads or ["siglip", "sdxl_l2", "sdxl_l1", "sweep_M256", "sweep_M1000", "sweep_M4096"]
        evaluate(names, a.dir)
    return 0


if __name__ == "__main__":
    sys.exit(main())
