"""Summarise an ncu launch list (``ncu --csv --log-file``) of the blended prefill.

    python ncu_summary.py launches.csv --steps 2 --markdown out.md
    python ncu_summary.py --gemm-shapes "q|k|v:1357:9216:7168:store:gemm_qkv.csv" ... \\
        --traffic-json profiles/gemm_traffic.json --command "<the ncu command>"

Per kernel: launches, total device time, share of the listed time and, when the capture
has ``dram__bytes_read.sum`` / ``dram__bytes_write.sum``, the average DRAM bytes per
launch.  A launch list over a full-size workload carries ``gpu__time_duration.sum`` only;
DRAM counters come from single-kernel captures of a small case (``-k``, ``-c 1..3``).
``--gemm-shapes`` takes one such capture per projection shape (``name:M:N:K:epilogue:csv``)
and ``--traffic-json`` records each shape's DRAM bytes against its algorithmic bytes
(weights + A + C: fp32 C written for ``store``, read and written for ``add``, bf16 C of N/2
columns for ``swiglu``) with a hash of the GEMM's sources; ``bench.py`` reports the ratio
of the sums as ``roofline.traffic`` only while those sources are unchanged.  Durations under ncu are serialised and cold-cache:
compare shares, not absolute times.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import json
import os
import re
from collections import OrderedDict

ROOT = os.path.dirname(os.path.abspath(__file__))
GEMM_SOURCES = ["rag_non_prefix_gb300/csrc/gemm.cu", "rag_non_prefix_gb300/csrc/gemm_pair.cu",
                "rag_non_prefix_gb300/csrc/common.cuh"]
GEMM_KERNELS = ("gemm_bf16_tc", "gemm_pair_kernel")
_UNIT = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "ns": 1e-3, "us": 1.0, "usecond": 1.0,
         "nsecond": 1e-3, "msecond": 1e3, "ms": 1e3}


def short_name(name: str) -> str:
    """'void cb::tc::gemm_bf16_tc<256, true>(CUtensorMap_st, ...)' -> 'tc::gemm_bf16_tc<256, true>'."""
    n = re.sub(r"^void\s+", "", name)
    n = n.split("(")[0]
    return n.replace("cb::", "")


def read_launches(path: str):
    """Rows of (launch id, kernel, metric, value in us or bytes)."""
    with open(path) as f:
        lines = f.read().splitlines()
    start = next(i for i, l in enumerate(lines) if l.startswith('"ID"'))
    rows = list(csv.DictReader(lines[start:]))
    out = []
    for r in rows:
        unit = r.get("Metric Unit", "")
        val = float(r["Metric Value"].replace(",", ""))
        out.append((int(r["ID"]), r["Kernel Name"], r["Metric Name"], val * _UNIT.get(unit, 1.0)))
    return out


def summarise(path: str):
    per = OrderedDict()
    launches = {}
    for lid, kern, metric, val in read_launches(path):
        k = short_name(kern)
        launches.setdefault(k, set()).add(lid)
        d = per.setdefault(k, {"us": 0.0, "dram": 0.0, "has_dram": False})
        if metric == "gpu__time_duration.sum":
            d["us"] += val
        elif metric in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            d["dram"] += val
            d["has_dram"] = True
    total = sum(d["us"] for d in per.values())
    table = []
    for k, d in sorted(per.items(), key=lambda kv: -kv[1]["us"]):
        n = len(launches[k])
        table.append({"kernel": k, "launches": n, "total_us": round(d["us"], 1),
                      "share": round(100.0 * d["us"] / total, 2) if total else 0.0,
                      "dram_mb_per_launch": round(d["dram"] / n / 1e6, 1) if d["has_dram"] else None})
    return table, total


def sources_sha256(sources) -> str:
    h = hashlib.sha256()
    for src in sources:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def algorithmic_bytes(M: int, N: int, K: int, epilogue: str) -> int:
    """Weights + A + C of one projection launch (bf16 operands)."""
    c = {"store": M * N * 4, "add": M * N * 8, "swiglu": M * (N // 2) * 2}[epilogue]
    return N * K * 2 + M * K * 2 + c


def gemm_shapes_record(specs, command: str):
    shapes = []
    for spec in specs:
        name, M, N, K, epi, path = spec.split(":")
        M, N, K = int(M), int(N), int(K)
        table, total = summarise(path)
        rows = [r for r in table if any(g in r["kernel"] for g in GEMM_KERNELS)]
        if len(rows) != 1 or rows[0]["launches"] != 1 or rows[0]["dram_mb_per_launch"] is None:
            raise SystemExit(f"{path}: expected one captured GEMM launch with DRAM counters")
        r = rows[0]
        dram = r["dram_mb_per_launch"] * 1e6
        alg = algorithmic_bytes(M, N, K, epi)
        shapes.append({"projection": name, "M": M, "N": N, "K": K, "epilogue": epi, "kernel": r["kernel"],
                       "dram_bytes": round(dram), "algorithmic_bytes": alg, "ratio": round(dram / alg, 3),
                       "us_under_ncu": r["total_us"]})
    ratio = sum(x["dram_bytes"] for x in shapes) / sum(x["algorithmic_bytes"] for x in shapes)
    return {"kernel": "projection GEMM (tc::gemm_bf16_tc, pr::gemm_pair_kernel)", "source_sha256": sources_sha256(GEMM_SOURCES),
            "sources": GEMM_SOURCES,
            "metrics": "dram__bytes_read.sum + dram__bytes_write.sum of one launch per shape (single-kernel capture, "
                       "small case, the first launch after an L2 flush)",
            "shapes": shapes, "ratio": round(ratio, 4),
            "use": "bench.py reports roofline.traffic = ratio x the step's algorithmic bytes per GEMM launch",
            "command": command}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("csv", nargs="?")
    ap.add_argument("--steps", type=int, default=1, help="timed steps the capture covers (per-step figures)")
    ap.add_argument("--markdown", default=None)
    ap.add_argument("--gemm-shapes", nargs="*", default=None, help="name:M:N:K:epilogue:csv per projection shape")
    ap.add_argument("--traffic-json", default=None)
    ap.add_argument("--command", default="")
    a = ap.parse_args()
    if a.gemm_shapes:
        rec = gemm_shapes_record(a.gemm_shapes, a.command)
        print(json.dumps(rec, indent=1))
        if a.traffic_json:
            with open(a.traffic_json, "w") as f:
                json.dump(rec, f, indent=1)
                f.write("\n")
        return
    table, total = summarise(a.csv)
    lines = ["| kernel | launches | total us | share | DRAM MB / launch |", "|---|---:|---:|---:|---:|"]
    for r in table:
        mb = "" if r["dram_mb_per_launch"] is None else f"{r['dram_mb_per_launch']}"
        lines.append(f"| {r['kernel']} | {r['launches']} | {r['total_us']} | {r['share']} % | {mb} |")
    lines.append(f"\n{sum(r['launches'] for r in table)} launches, {total / 1e3:.2f} ms listed "
                 f"({total / 1e3 / max(1, a.steps):.2f} ms per step).")
    text = "\n".join(lines)
    print(text)
    if a.markdown:
        with open(a.markdown, "w") as f:
            f.write(text + "\n")


if __name__ == "__main__":
    main()
