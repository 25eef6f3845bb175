"""Shared helpers of the GPU parity tests: run the library, run the oracle on the
same bytes, compare with the stated tolerances.

Tolerances (GPU against the FP64 oracle on the same fp16/bf16 inputs):
  * fp16: O max-abs <= 4e-3 and mean-abs <= 5e-4; lse max-abs <= 1e-4.
  * bf16: the stated O numbers are below bf16's own rounding floor (one bf16 ulp
    on [2, 4) is 1.6e-2), so the bound is derived from the arithmetic the path
    performs.  Rounding the probabilities to bf16 before the P V product moves
    each p by at most u = 2^-8 of itself, which moves O_id by at most
    u * sum_j p_ij |v_jd| / l_i = u * A_id, where A is the oracle run on |V|
    with the same weights; rounding O to bf16 adds at most one ulp.  So
    element-wise |gpu - oracle| <= 4e-3 + ulp_bf16(oracle) + 2^-8 * A, and in
    the mean <= 5e-4 + mean|rn_bf16(oracle) - oracle|.  The stated-tolerance
    figures are still computed and returned.
  * no NaN or Inf anywhere; outputs are NaN-filled before the call so an
    unwritten element fails.

When the environment variable ECA_PARITY_LOG names a file, every comparison that
is given a name appends its measured errors there as one JSON line
(tests/parity_report.py turns the file into a table).
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle
from exact_causal_attention_gb300 import inputs

O_MAX_ABS = 4e-3
O_MEAN_ABS = 5e-4
LSE_MAX_ABS = 1e-4


def run_gpu(q, k, v, causal, scale, stream=None):
    """q, k, v: CPU fp16/bf16 tensors.  Returns (o, lse) as float64 numpy arrays."""
    import exact_causal_attention_gb300 as eca

    dq, dk, dv = (x.cuda() for x in (q, k, v))
    o = torch.full_like(dq, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=dq.device)
    eca.attn_fwd_into(dq, dk, dv, o, lse, causal=causal, scale=scale, stream=stream)
    torch.cuda.synchronize()
    assert eca.device_status() == 0
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def _vbits(v, abs_v):
    b = inputs.bits(v)
    return (b & np.uint16(0x7FFF)) if abs_v else b  # clearing the sign bit is |v|, exactly


def oracle_full(q, k, v, dtype, causal, scale, abs_v=False):
    return oracle.attention_from_bits(inputs.bits(q), inputs.bits(k), _vbits(v, abs_v), dtype, causal, scale)


def oracle_rows(q, k, v, dtype, causal, scale, rows, abs_v=False):
    return oracle.attention_from_bits(inputs.bits(q), inputs.bits(k), _vbits(v, abs_v), dtype, causal, scale,
                                      rows=rows)


def p_rounding_term(q, k, v, dtype, causal, scale, rows=None):
    """A = the oracle's output on |V| (same weights), for the bf16 bound; None for fp16."""
    if dtype != "bf16":
        return None
    if rows is None:
        return oracle_full(q, k, v, dtype, causal, scale, abs_v=True)[0]
    return oracle_rows(q, k, v, dtype, causal, scale, rows, abs_v=True)[0]


def bf16_ulp(x):
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def round_bf16(x):
    t = torch.from_numpy(np.asarray(x, dtype=np.float64))
    return t.to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


def record(name, stats):
    """Append one named comparison to the parity log, if one is configured."""
    path = os.environ.get("ECA_PARITY_LOG")
    if not path or name is None:
        return
    with open(path, "a") as f:
        f.write(json.dumps({"name": name, **stats}) + "\n")


def compare(o_gpu, lse_gpu, o_ref, lse_ref, dtype, p_term=None, name=None, rows="all"):
    """Assert the tolerances; return a dict of the measured errors (logged under `name`).

    `rows` says which rows were compared ("all", or a count of sampled rows)."""
    assert np.isfinite(o_gpu).all(), "non-finite or unwritten O"
    assert np.isfinite(lse_gpu).all(), "non-finite or unwritten lse"
    err = np.abs(o_gpu - o_ref)
    lerr = np.abs(lse_gpu - lse_ref)
    stats = {"dtype": dtype, "rows": rows, "elements": int(err.size),
             "o_max_abs": float(err.max()), "o_mean_abs": float(err.mean()),
             "lse_max_abs": float(lerr.max())}
    stats["meets_stated_o_tolerance"] = bool(stats["o_max_abs"] <= O_MAX_ABS and stats["o_mean_abs"] <= O_MEAN_ABS)
    stats["meets_stated_lse_tolerance"] = bool(stats["lse_max_abs"] <= LSE_MAX_ABS)
    if dtype != "fp16":
        # bf16's own rounding floor, measured on the oracle: rn_bf16(oracle) against the oracle.
        floor = np.abs(round_bf16(o_ref) - o_ref)
        stats["bf16_floor_max"] = float(floor.max())
        stats["bf16_floor_mean"] = float(floor.mean())
        assert p_term is not None, "bf16 comparison needs the oracle's output on |V|"
        floor_bound = O_MAX_ABS + bf16_ulp(o_ref)
        stats["floor_bound_without_p_term_met"] = bool((err <= floor_bound).all())
        stats["excess_over_floor_bound_without_p_term"] = float((err - floor_bound).max())
        bound = floor_bound + 2.0 ** -8 * p_term
        stats["excess_over_derived_bound"] = float((err - bound).max())
        stats["mean_bound"] = O_MEAN_ABS + stats["bf16_floor_mean"]
    record(name, stats)
    assert stats["meets_stated_lse_tolerance"], stats
    if dtype == "fp16":
        assert stats["meets_stated_o_tolerance"], stats
    else:
        assert stats["excess_over_derived_bound"] <= 0, stats
        assert stats["o_mean_abs"] <= stats["mean_bound"], stats
    return stats


def sample_rows(B, H, N, count, seed):
    """(bh, i) pairs: tile edges and ends of a few heads, plus seeded random rows."""
    rng = np.random.default_rng(seed)
    edges = sorted({i for i in (0, 1, 63, 126, 127, 128, 129, 255, 256, 257, N // 2, N - 129, N - 128,
                                N - 2, N - 1) if 0 <= i < N})
    heads = sorted({0, B * H - 1, int(rng.integers(0, B * H))})
    rows = [(bh, i) for bh in heads for i in edges]
    while len(rows) < count:
        rows.append((int(rng.integers(0, B * H)), int(rng.integers(0, N))))
    return rows
