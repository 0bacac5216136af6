"""DRAM traffic per launch from an ncu report, kept beside the kernel source it was
measured on.

    python -m host_offloaded_weight_gb300.profiling REPORT.ncu-rep WORKLOAD NAME=REGEX [NAME=REGEX ...]

reads ``dram__bytes_read.sum`` and ``dram__bytes_write.sum`` of every captured launch
whose kernel name matches REGEX (``ncu -i REPORT --page raw --csv --print-units base``),
averages them per
NAME and records the result in ``profiles/traffic.json`` under (WORKLOAD, NAME), with
the SHA-256 of the source file that defines the kernel. ``traffic()`` gives the figure
back only while that source is unchanged: counters taken from an older kernel are not
reported as the current kernel's.
"""
from __future__ import annotations

import csv
import hashlib
import io
import json
import os
import re
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")

# the source file of each kernel class the runtime times
SOURCES = {
    "gemm_up": "csrc/k_gemm.cu", "gemm_down": "csrc/k_gemm.cu", "gemm_proj": "csrc/k_gemm.cu",
    "copy_h2slot": "csrc/k_copy.cu", "wait_ready": "csrc/k_copy.cu",
    "linear_gelu_f32": "csrc/k_simt.cu",
    "moe_route_group": "csrc/k_moe.cu", "moe_gather": "csrc/k_moe.cu", "moe_combine": "csrc/k_moe.cu",
}


def source_sha(kernel: str) -> str | None:
    rel = SOURCES.get(kernel)
    if rel is None:
        return None
    with open(os.path.join(PKG, rel), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def _load() -> dict:
    try:
        with open(TRAFFIC_FILE) as f:
            return json.load(f)
    except FileNotFoundError:
        return {"entries": []}


def traffic(workload: str, kernel: str) -> int | None:
    """DRAM bytes (read + write) per launch of `kernel` in `workload`, or None when no
    capture exists or the kernel's source has changed since it was taken."""
    sha = source_sha(kernel)
    for e in _load()["entries"]:
        if e["workload"] == workload and e["kernel"] == kernel:
            return int(e["dram_bytes_per_launch"]) if sha is not None and e["source_sha256"] == sha else None
    return None


_SCALE = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KiB": 1024, "MiB": 1 << 20, "GiB": 1 << 30}


def _raw_rows(report: str) -> list:
    """Rows of the raw page, each value paired with its unit: {metric: (value, unit)}."""
    out = subprocess.run(["ncu", "-i", report, "--page", "raw", "--csv", "--print-units", "base"],
                         capture_output=True, text=True, check=True).stdout
    rows = list(csv.reader(io.StringIO(out)))
    head, units = rows[0], rows[1]
    body = [r for r in rows[2:] if len(r) == len(head)]
    return [{h: (v, u) for h, v, u in zip(head, r, units)} for r in body]


def _bytes(vu) -> float:
    v, u = vu
    return float(v.replace(",", "")) * _SCALE.get(u.strip(), 1)


def record(report: str, workload: str, pairs: list) -> dict:
    rows = _raw_rows(report)
    data = _load()
    done = {}
    for name, rx in pairs:
        hits = [r for r in rows if re.search(rx, r.get("Kernel Name", ("", ""))[0])]
        if not hits:
            raise SystemExit(f"no launch of {rx!r} in {report}")
        per = [_bytes(r["dram__bytes_read.sum"]) + _bytes(r["dram__bytes_write.sum"]) for r in hits]
        value = int(round(sum(per) / len(per)))
        data["entries"] = [e for e in data["entries"] if not (e["workload"] == workload and e["kernel"] == name)]
        data["entries"].append({"workload": workload, "kernel": name, "dram_bytes_per_launch": value,
                                "launches": len(per), "source": SOURCES[name], "source_sha256": source_sha(name),
                                "report": os.path.basename(report)})
        done[name] = value
    data["entries"].sort(key=lambda e: (e["workload"], e["kernel"]))
    os.makedirs(os.path.dirname(TRAFFIC_FILE), exist_ok=True)
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(data, f, indent=1)
        f.write("\n")
    return done


def main(argv: list) -> int:
    if len(argv) < 3:
        print(__doc__)
        return 2
    report, workload = argv[0], argv[1]
    pairs = [a.split("=", 1) for a in argv[2:]]
    print(json.dumps(record(report, workload, pairs)))
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
