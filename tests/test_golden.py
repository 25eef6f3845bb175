"""Stored fixtures (written by tests/golden/make_golden.py, which calls only oracle/ and the input module)."""
import json
import os

import numpy as np

import oracle
from exact_causal_attention_gb300 import inputs

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_seeded_inputs_are_byte_identical_to_the_record():
    rec = json.load(open(os.path.join(HERE, "inputs_sha256.json")))
    assert set(rec) == set(inputs.WORKLOADS)
    for name, w in inputs.WORKLOADS.items():
        q, k, v = inputs.workload_qkv(w)
        got = {"q": inputs.sha256(q), "k": inputs.sha256(k), "v": inputs.sha256(v)}
        assert got == rec[name], name


def test_oracle_rows_match_the_record():
    rec = json.load(open(os.path.join(HERE, "oracle_rows.json")))
    w = inputs.WORKLOADS[rec["workload"]]
    q, k, v = inputs.workload_qkv(w)
    o, lse = oracle.attention_from_bits(inputs.bits(q), inputs.bits(k), inputs.bits(v), w.dtype,
                                        w.causal, w.scale, rows=rec["rows"])
    ref_o = np.array([[float.fromhex(x) for x in r] for r in rec["o"]])
    ref_l = np.array([float.fromhex(x) for x in rec["lse"]])
    # libm exp/log may differ in the last bit between hosts: allow a few ulps.
    np.testing.assert_allclose(o, ref_o, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-13, atol=1e-15)
