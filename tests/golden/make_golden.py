"""Writes the stored fixtures under tests/golden/.  Calls only the input module and oracle/.

* inputs_sha256.json: SHA-256 of the q, k, v bit patterns of every named workload,
  so that any change in the seeded recipe shows up.
* oracle_rows.json: oracle O rows and lse of the small causal workload
  (B=1, H=2, N=256, D=64, fp16, seed 0) at a few (bh, i) positions, as a
  regression record of the oracle's arithmetic.

The pages print no worked numeric example for attention, so no stored value here
comes from them; the hand-derived examples live in tests/test_oracle.py.
Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from exact_causal_attention_gb300 import inputs  # noqa: E402

ROWS = [(0, 0), (0, 1), (0, 127), (0, 128), (1, 200), (1, 255)]


def main():
    hashes = {}
    for name, w in inputs.WORKLOADS.items():
        q, k, v = inputs.workload_qkv(w)
        hashes[name] = {"q": inputs.sha256(q), "k": inputs.sha256(k), "v": inputs.sha256(v)}
    with open(os.path.join(HERE, "inputs_sha256.json"), "w") as f:
        json.dump(hashes, f, indent=1, sort_keys=True)
        f.write("\n")
    w = inputs.WORKLOADS["causal_b1_h2_n256_d64_fp16"]
    q, k, v = inputs.workload_qkv(w)
    o, lse = oracle.attention_from_bits(inputs.bits(q), inputs.bits(k), inputs.bits(v), w.dtype,
                                        w.causal, w.scale, rows=ROWS)
    rec = {"workload": w.name, "rows": ROWS, "o": [[float.hex(float(x)) for x in r] for r in o],
           "lse": [float.hex(float(x)) for x in lse]}
    with open(os.path.join(HERE, "oracle_rows.json"), "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
