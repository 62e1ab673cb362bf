"""Record a kernel's measured DRAM traffic per launch from an ncu capture.

    ncu -i CAPTURE.ncu-rep --page raw --csv > RAW.csv
    python -m long_context_self_gb300.ncu_record RAW.csv --kernel verify_heads \\
        --source long_context_self_gb300/csrc/attn_heads.cu --workload llama8b_b128_l32k \\
        --captured "B=32, L=32000" --scale 4 --out profiles/verify_attn_llama8b_b128_l32k.json

The record holds dram__bytes_read.sum + dram__bytes_write.sum of the captured
launch(es) (mean per launch), that value scaled to one launch of the full
workload (`--scale`: the ratio of units processed, used when the full
workload is too large to capture), and the sha256 prefix of the kernel's
source, so that readers of the record can tell when the kernel has changed
since the counters were taken.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import json
import sys

UNITS = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12,
         "KB": 1e3, "MB": 1e6, "GB": 1e9, "TB": 1e12}


def source_sha16(path: str) -> str:
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def launch_traffic(raw_csv: str, kernel: str):
    """Per captured launch of a kernel whose name contains `kernel`: read + write DRAM bytes."""
    with open(raw_csv, newline="") as f:
        rows = list(csv.reader(f))
    hdr = rows[0]
    col = {name: i for i, name in enumerate(hdr)}
    units = rows[1] if len(rows) > 1 and not rows[1][0].strip().isdigit() else None
    data = rows[2:] if units else rows[1:]
    out = []
    for r in data:
        if kernel not in r[col["Kernel Name"]]:
            continue
        tot = 0.0
        for m in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            v = float(r[col[m]].replace(",", ""))
            scale = UNITS.get(units[col[m]], 1.0) if units else 1.0
            tot += v * scale
        out.append(tot)
    return out


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("raw_csv")
    ap.add_argument("--kernel", required=True)
    ap.add_argument("--source", required=True, help="the kernel's .cu file")
    ap.add_argument("--workload", required=True, help="the full workload the record is for")
    ap.add_argument("--captured", required=True, help="the captured case, in words")
    ap.add_argument("--scale", type=float, default=1.0, help="full-workload units / captured units")
    ap.add_argument("--out", required=True)
    args = ap.parse_args(argv)
    per = launch_traffic(args.raw_csv, args.kernel)
    if not per:
        sys.exit(f"no launch of a kernel matching {args.kernel!r} in {args.raw_csv}")
    mean = sum(per) / len(per)
    rec = {"kernel": args.kernel, "source": args.source, "source_sha16": source_sha16(args.source),
           "workload": args.workload, "captured_case": args.captured, "captured_launches": len(per),
           "dram_bytes_per_captured_launch": mean, "scale": args.scale,
           "dram_bytes_per_launch": mean * args.scale}
    with open(args.out, "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    print(json.dumps(rec))


if __name__ == "__main__":
    main()
