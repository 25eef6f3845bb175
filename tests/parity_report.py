"""Turn the parity log of a GPU test run into a markdown table.

    ECA_PARITY_LOG=parity.jsonl python -m pytest tests -m gpu
    python tests/parity_report.py parity.jsonl > report.md

Each line of the log is one named comparison of the CUDA path with the FP64 oracle
(tests/helpers.py `compare`).  The table gives, per comparison, the rows compared,
the measured O and lse errors and whether the stated tolerances hold (O max-abs
4e-3 and mean-abs 5e-4, lse 1e-4); for bf16 also bf16's own rounding floor measured
on the oracle, whether the floor bound holds without the term for P's rounding,
and the margin left under the derived bound.
"""
from __future__ import annotations

import json
import sys


def fmt(x):
    if isinstance(x, bool):
        return "yes" if x else "no"
    if isinstance(x, float):
        return f"{x:.3e}"
    return str(x)


def main(path: str) -> None:
    recs = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line:
                r = json.loads(line)
                recs[r["name"]] = r  # a repeated name keeps its last run
    cols = ["name", "dtype", "rows", "o_max_abs", "o_mean_abs", "lse_max_abs", "meets_stated_o_tolerance",
            "meets_stated_lse_tolerance"]
    print("| " + " | ".join(cols) + " |")
    print("|" + "---|" * len(cols))
    for r in recs.values():
        print("| " + " | ".join(fmt(r.get(c, "")) for c in cols) + " |")
    bf = [r for r in recs.values() if r.get("dtype") == "bf16"]
    if bf:
        cols_b = ["name", "o_max_abs", "o_mean_abs", "bf16_floor_max", "bf16_floor_mean",
                  "floor_bound_without_p_term_met", "excess_over_floor_bound_without_p_term",
                  "excess_over_derived_bound", "mean_bound"]
        print()
        print("bf16 comparisons against bf16's own floor (elementwise 4e-3 + ulp_bf16(oracle); the derived bound "
              "adds 2^-8 times the oracle on |V|; mean bound 5e-4 + mean |rn_bf16(oracle) - oracle|):")
        print()
        print("| " + " | ".join(cols_b) + " |")
        print("|" + "---|" * len(cols_b))
        for r in bf:
            print("| " + " | ".join(fmt(r.get(c, "")) for c in cols_b) + " |")


if __name__ == "__main__":
    main(sys.argv[1])
