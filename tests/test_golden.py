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


def test_device_draws_are_seeded_and_shaped():
    """inputs.make_qkv_device (the largest-size test's generator), run on the host's device
    type: the same seed gives the same bytes, another seed other bytes, and the three
    tensors are distinct draws of the asked shape and 16-bit type with unit spread."""
    import torch

    for dtype, t in (("fp16", torch.float16), ("bf16", torch.bfloat16)):
        a = inputs.make_qkv_device(2, 3, 64, 32, dtype, seed=5, device="cpu")
        b = inputs.make_qkv_device(2, 3, 64, 32, dtype, seed=5, device="cpu")
        c = inputs.make_qkv_device(2, 3, 64, 32, dtype, seed=6, device="cpu")
        for x, y, z in zip(a, b, c):
            assert x.shape == (2, 3, 64, 32) and x.dtype == t
            assert torch.equal(x.view(torch.int16), y.view(torch.int16))
            assert not torch.equal(x.view(torch.int16), z.view(torch.int16))
            assert 0.9 < float(x.float().std()) < 1.1 and abs(float(x.float().mean())) < 0.1
        assert not torch.equal(a[0], a[1]) and not torch.equal(a[1], a[2])
