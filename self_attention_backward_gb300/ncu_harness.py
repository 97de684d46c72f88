"""ncu evidence harness for the backward kernels.

On a machine with the GPU it runs the benchmark once plainly, then under
Nsight Compute (`--clock-control none` always):

1. the launch list (`gpu__time_duration.sum` only, one pass per launch) of the
   whole benchmark command;
2. for each backward kernel of the family, its own capture of ONE launch (the
   first timed step's) with DRAM bytes, duration and tensor-pipe utilisation
   (a handful of passes for that launch only; every other launch runs
   unprofiled);

and writes Markdown summaries: per kernel its launches, total time and share,
and per captured launch its DRAM traffic, achieved DRAM bandwidth against the
measured HBM peak, and tensor-pipe busy fraction.  The summarising half reads
ncu's `--csv` output and runs anywhere.

    python -m self_attention_backward_gb300.ncu_harness run --out DIR [--algo tc|tc2|simt|auto]
    python -m self_attention_backward_gb300.ncu_harness launches DIR/launches.csv
    python -m self_attention_backward_gb300.ncu_harness kernels DIR/kernels.csv

ncu's per-launch times are cold-cache and serialised: compare shares, not
absolute times, with the benchmark's CUDA-event numbers.
"""
from __future__ import annotations

import argparse
import csv
import json
import os
import subprocess
import sys
from collections import OrderedDict

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

KERNEL_METRICS = ["gpu__time_duration.sum", "dram__bytes_read.sum", "dram__bytes_write.sum",
                  "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active"]
# the backward kernels of each family, by function name, in launch order
FAMILY_KERNELS = {
    "tc": ["pre_stats_kernel", "bwd_main_kernel", "dq_finalize_kernel"],
    "tc2": ["pre_kernel", "bwd_kv_pair_kernel", "bwd_q_pair_kernel", "bwd_dkdv_kernel", "dq_kernel"],
    "simt": ["pre_kernel", "dkdv_kernel", "dq_kernel"],
}
WARMUP_STEPS = 3

_TIME_SCALE_US = {"ns": 1e-3, "nsecond": 1e-3, "us": 1.0, "usecond": 1.0, "ms": 1e3, "msecond": 1e3,
                  "s": 1e6, "second": 1e6}
_BYTE_SCALE = {"byte": 1.0, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "tbyte": 1e12}


def _number(text: str) -> float:
    return float(text.replace(",", "").strip())


def read_metric_rows(path: str):
    """Rows of an ncu `--csv` metrics log: (launch id, kernel, metric, unit, value)."""
    with open(path, newline="") as f:
        lines = [ln for ln in f if ln.startswith('"')]   # ncu may prepend its own log lines
    rows = list(csv.reader(lines))
    if not rows:
        return []
    hdr = rows[0]
    idx = {k: hdr.index(k) for k in ("ID", "Kernel Name", "Metric Name", "Metric Unit", "Metric Value")}
    out = []
    for r in rows[1:]:
        if len(r) < len(hdr):
            continue
        try:
            val = _number(r[idx["Metric Value"]])
        except ValueError:
            continue
        out.append((r[idx["ID"]], r[idx["Kernel Name"]], r[idx["Metric Name"]], r[idx["Metric Unit"]], val))
    return out


def short_name(kernel: str) -> str:
    """`void psa::<unnamed>::bwd_main_kernel<32>(CUtensorMap_st, ...)` -> `bwd_main_kernel<32>`."""
    s = kernel.strip()
    if s.startswith("void "):
        s = s[5:]
    s = s.replace("(anonymous namespace)", "")
    depth, cut, last = 0, len(s), 0
    for i, ch in enumerate(s):
        if ch == "<":
            depth += 1
        elif ch == ">":
            depth = max(0, depth - 1)
        elif ch == "(" and depth == 0:
            cut = i
            break
        elif ch == ":" and depth == 0 and s[i:i + 2] == "::":
            last = i + 2
    return s[last:cut].strip()


def time_us(value: float, unit: str) -> float:
    return value * _TIME_SCALE_US[unit.strip().lower()]


def nbytes(value: float, unit: str) -> float:
    return value * _BYTE_SCALE[unit.strip().lower()]


def summarize_launches(rows):
    """Per kernel: launches, total microseconds, share of the listed time."""
    agg: "OrderedDict[str, list]" = OrderedDict()
    for _, kernel, metric, unit, val in rows:
        if metric != "gpu__time_duration.sum":
            continue
        a = agg.setdefault(short_name(kernel), [0, 0.0])
        a[0] += 1
        a[1] += time_us(val, unit)
    total = sum(t for _, t in agg.values())
    table = [(k, n, t, 100.0 * t / total if total else 0.0, t / n) for k, (n, t) in agg.items()]
    table.sort(key=lambda x: -x[2])
    return table, total


def summarize_kernels(rows, hbm_gbs: float):
    """Per captured launch: duration, DRAM bytes, achieved GB/s and its fraction
    of `hbm_gbs`, tensor-pipe busy percentage."""
    per: "OrderedDict[str, dict]" = OrderedDict()
    for lid, kernel, metric, unit, val in rows:
        d = per.setdefault(lid, {"kernel": short_name(kernel)})
        if metric == "gpu__time_duration.sum":
            d["us"] = time_us(val, unit)
        elif metric == "dram__bytes_read.sum":
            d["read"] = nbytes(val, unit)
        elif metric == "dram__bytes_write.sum":
            d["write"] = nbytes(val, unit)
        elif metric.startswith("sm__pipe_tensor_cycles_active"):
            d["tensor_pct"] = val
    out = []
    for lid, d in per.items():
        traffic = d.get("read", 0.0) + d.get("write", 0.0)
        gbs = traffic / (d["us"] * 1e-6) / 1e9 if d.get("us") else 0.0
        out.append({"id": lid, "kernel": d["kernel"], "us": d.get("us", 0.0), "dram_read": d.get("read", 0.0),
                    "dram_write": d.get("write", 0.0), "gbs": gbs, "hbm_frac": gbs / hbm_gbs if hbm_gbs else 0.0,
                    "tensor_pct": d.get("tensor_pct")})
    return out


def launches_markdown(table, total) -> str:
    lines = ["| kernel | launches | total (us) | share | per launch (us) |", "|---|---|---|---|---|"]
    for k, n, t, share, per in table:
        lines.append(f"| {k} | {n} | {t:.1f} | {share:.1f} % | {per:.1f} |")
    lines.append(f"| all | {sum(r[1] for r in table)} | {total:.1f} | 100 % | |")
    return "\n".join(lines)


def kernels_markdown(items, hbm_gbs: float) -> str:
    lines = [f"| launch | kernel | time (us) | DRAM read (MB) | DRAM write (MB) | achieved GB/s | of {hbm_gbs:.0f} GB/s "
             "| tensor pipe busy |", "|---|---|---|---|---|---|---|---|"]
    for it in items:
        tp = "n/a" if it["tensor_pct"] is None else f"{it['tensor_pct']:.1f} %"
        lines.append(f"| {it['id']} | {it['kernel']} | {it['us']:.1f} | {it['dram_read'] / 1e6:.2f} | "
                     f"{it['dram_write'] / 1e6:.2f} | {it['gbs']:.0f} | {100 * it['hbm_frac']:.1f} % | {tp} |")
    return "\n".join(lines)


def measured_hbm_gbs() -> float:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"])
    except Exception:
        return 6800.0   # the profiling recipe's fallback


# the library's profiling slot (bench.py's kernels_ms_per_step keys) of each kernel
SLOT_OF = {"bwd_main_kernel": "bwd_main", "bwd_kv_pair_kernel": "bwd_main", "bwd_dkdv_kernel": "bwd_main",
           "dkdv_kernel": "bwd_main", "bwd_q_pair_kernel": "bwd_dq", "dq_kernel": "bwd_dq",
           "dq_finalize_kernel": "bwd_dq", "pre_kernel": "bwd_pre", "pre_stats_kernel": "bwd_pre",
           "pre_stats_view_kernel": "bwd_pre"}


def record_traffic(items, workload: str, algo: str, path=None) -> dict:
    """Writes each captured backward kernel's DRAM bytes per launch into
    profiles/traffic.json under (workload, algo, slot), with the hash of the
    sources the kernel family is built from (bench.py nulls a record whose
    sources changed since)."""
    sys.path.insert(0, ROOT)
    import bench  # noqa: E402  (the benchmark owns the source lists and the hash)
    path = path or os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        rec = {}
    fam = rec.setdefault(workload, {}).setdefault(algo, {})
    for it in items:
        slot = SLOT_OF.get(it["kernel"].split("<", 1)[0])
        if slot is None:
            continue
        fam[slot] = {"dram_bytes_per_launch": it["dram_read"] + it["dram_write"],
                     "source_hash": bench.source_hash(algo), "sources": ", ".join(bench.TRAFFIC_SOURCES[algo]),
                     "ncu": f"dram__bytes_read.sum + dram__bytes_write.sum of {it['kernel']}, one launch "
                            "(ncu_harness run), cache control all"}
    with open(path, "w") as f:
        json.dump(rec, f, indent=1)
    return rec


def _run(cmd, log_path: str) -> int:
    with open(log_path, "w") as log:
        return subprocess.call(cmd, cwd=ROOT, stdout=log, stderr=subprocess.STDOUT)


def kernel_capture_cmd(name: str, csv_path: str, bench_cmd) -> list:
    """ncu command line that profiles ONE launch of kernel `name`: the first
    launch after the warm-up steps (`-s` counts only launches that match the
    name filter), with the DRAM, duration and tensor-pipe metrics."""
    return ["ncu", "--metrics", ",".join(KERNEL_METRICS), "--clock-control", "none",
            "-k", f"regex:^{name}$|^{name}<", "-s", str(WARMUP_STEPS), "-c", "1", "--csv",
            "--log-file", csv_path] + list(bench_cmd)


def run(out_dir: str, algo: str, workload: str | None, record: bool = False) -> int:
    os.makedirs(out_dir, exist_ok=True)
    bench = [sys.executable, "bench.py", "--steps", "2", "--warmup", str(WARMUP_STEPS), "--no-cpu",
             "--no-secondary", "--no-extras", "--algo", algo]
    if workload:
        bench += ["--workload", workload]
    # the same command must exit 0 without ncu before ncu runs it
    if _run(bench, os.path.join(out_dir, "plain.log")) != 0:
        print("plain benchmark run failed; see plain.log", file=sys.stderr)
        return 1
    launches = os.path.join(out_dir, "launches.csv")
    rc = _run(["ncu", "--metrics", "gpu__time_duration.sum", "--clock-control", "none", "-c", "400", "--csv",
               "--log-file", launches] + bench, os.path.join(out_dir, "ncu_launches.log"))
    if rc != 0:
        return rc
    # one capture per backward kernel that the launch list shows, one launch each
    family = algo if algo in FAMILY_KERNELS else "tc"
    seen = {short_name(k).split("<", 1)[0] for _, k, _, _, _ in read_metric_rows(launches)}
    rows = []
    for name in FAMILY_KERNELS[family]:
        if name not in seen:
            continue
        csv_path = os.path.join(out_dir, f"kernel_{name}.csv")
        rc = _run(kernel_capture_cmd(name, csv_path, bench), os.path.join(out_dir, f"ncu_{name}.log"))
        if rc != 0:
            return rc
        # launch ids restart in every capture: key them by the kernel name too
        rows += [(f"{name}:{lid}", k, m, u, v) for lid, k, m, u, v in read_metric_rows(csv_path)]
    hbm = measured_hbm_gbs()
    table, total = summarize_launches(read_metric_rows(launches))
    items = summarize_kernels(rows, hbm)
    text = ("# ncu evidence: " + " ".join(bench[1:]) + "\n\n## Launch list (cold-cache, serialised)\n\n" +
            launches_markdown(table, total) + "\n\n## One launch of each backward kernel (separate captures)\n\n" +
            kernels_markdown(items, hbm) + "\n")
    with open(os.path.join(out_dir, "summary.md"), "w") as f:
        f.write(text)
    print(text)
    if record and algo in ("tc", "tc2", "simt"):
        sys.path.insert(0, ROOT)
        import bench  # noqa: E402
        record_traffic(items, workload or bench.HEADLINE, algo, os.path.join(out_dir, "traffic.json"))
    return 0


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    sub = ap.add_subparsers(dest="cmd", required=True)
    r = sub.add_parser("run")
    r.add_argument("--out", required=True)
    r.add_argument("--algo", default="auto", choices=["auto", "tc", "tc2", "simt"])
    r.add_argument("--workload", default=None)
    r.add_argument("--record-traffic", action="store_true",
                   help="also write the DRAM bytes per launch to OUT/traffic.json (profiles/traffic.json format)")
    la = sub.add_parser("launches")
    la.add_argument("csv")
    ke = sub.add_parser("kernels")
    ke.add_argument("csv")
    ke.add_argument("--hbm-gbs", type=float, default=None)
    a = ap.parse_args(argv)
    if a.cmd == "run":
        return run(a.out, a.algo, a.workload, a.record_traffic)
    if a.cmd == "launches":
        table, total = summarize_launches(read_metric_rows(a.csv))
        print(launches_markdown(table, total))
        return 0
    hbm = a.hbm_gbs or measured_hbm_gbs()
    print(kernels_markdown(summarize_kernels(read_metric_rows(a.csv), hbm), hbm))
    return 0


if __name__ == "__main__":
    sys.exit(main())
