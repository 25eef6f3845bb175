"""Seeded random shapes through every entry point of the attention forward, each
compared with the FP64 oracle on every row.

The shapes are drawn so that, across the draws, every way the kernel forms its
units appears (key-halves units for few heads, pairs of query tiles for many,
head pairs for grouped heads, key segments for the split path), with ragged and
tiny lengths, both head dimensions, both 16-bit types, causal and not.  Sizes stay
small enough for the oracle to finish in seconds.
"""
import math

import numpy as np
import pytest
import torch

from exact_causal_attention_gb300 import inputs

from helpers import compare, oracle_full, p_rounding_term

pytestmark = pytest.mark.gpu


def draw(seed):
    rng = np.random.default_rng(seed)
    D = int(rng.choice([64, 128]))
    dtype = str(rng.choice(["fp16", "bf16"]))
    causal = bool(rng.random() < 0.7)
    N = int(rng.choice([int(rng.integers(1, 130)), int(rng.integers(130, 700)), int(rng.integers(700, 2100))]))
    Hkv = int(rng.choice([1, 2, 3, 4]))
    g = int(rng.choice([1, 1, 2, 3, 4]))
    B = int(rng.integers(1, 4))
    if rng.random() < 0.45:  # many heads: pair (or head-pair) units even at short lengths
        B, Hkv, g = 4, int(rng.choice([20, 40])), int(rng.choice([1, 2]))
        N = min(N, 1100)
    mode = str(rng.choice(["plain", "plain", "gqa", "split"]))
    if mode == "split":
        g = 1
    splits = int(rng.integers(2, 9))
    qk_std = float(rng.choice([1.0, 1.5, 3.0]))
    return dict(B=B, H=Hkv * g, Hkv=Hkv, N=N, D=D, dtype=dtype, causal=causal, mode=mode, splits=splits,
                qk_std=qk_std)


@pytest.mark.parametrize("seed", range(40))
def test_random_shape_matches_oracle(cuda_lib, seed):
    eca = cuda_lib
    c = draw(7000 + seed)
    B, H, Hkv, N, D, dtype = c["B"], c["H"], c["Hkv"], c["N"], c["D"], c["dtype"]
    q, _, _ = inputs.make_qkv(B, H, N, D, dtype, seed=9000 + seed, qk_std=c["qk_std"])
    _, k, v = inputs.make_qkv(B, Hkv, N, D, dtype, seed=9500 + seed, qk_std=c["qk_std"])
    scale = 1.0 / math.sqrt(D)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o = torch.full_like(dq, float("nan"))
    lse = torch.full((B, H, N), float("nan"), device="cuda")
    if c["mode"] == "split":
        need = eca.splitkv_workspace_bytes(B, H, N, D, c["splits"])
        ws = torch.full((need + 256,), 0xFF, dtype=torch.uint8, device="cuda")
        off = (-ws.data_ptr()) % 256
        eca.attn_fwd_splitkv(dq, dk, dv, o, lse, kv_splits=c["splits"], workspace=ws[off:off + need],
                             causal=c["causal"], scale=scale)
    elif c["mode"] == "gqa" or Hkv != H:
        eca.attn_fwd_gqa(dq, dk, dv, causal=c["causal"], scale=scale, o=o, lse=lse)
    else:
        eca.attn_fwd_into(dq, dk, dv, o, lse, causal=c["causal"], scale=scale)
    torch.cuda.synchronize()
    assert eca.device_status() == 0, c
    ro, rl = oracle_full(q, k, v, dtype, c["causal"], scale)
    compare(o.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, dtype,
            p_rounding_term(q, k, v, dtype, c["causal"], scale), name=f"fuzz_{seed}")
