"""GPU parity of grouped key/value heads (GQA, MQA) against the FP64 oracle: query
head h reads key/value head floor(h / g), g = H / Hkv ("CUDA KV Cache：分页存储与
长上下文 Decode 极致优化", section 3.3)."""
import math

import numpy as np
import pytest
import torch

from exact_causal_attention_gb300 import inputs

from helpers import compare, oracle_full, p_rounding_term

pytestmark = pytest.mark.gpu


def make(B, H, Hkv, N, D, dtype, seed):
    q, _, _ = inputs.make_qkv(B, H, N, D, dtype, seed=seed, qk_std=1.5)
    _, k, v = inputs.make_qkv(B, Hkv, N, D, dtype, seed=seed + 1, qk_std=1.5)
    return q, k, v


def run(q, k, v, causal, scale):
    import exact_causal_attention_gb300 as eca

    dq, dk, dv = (x.cuda() for x in (q, k, v))
    B, H, N, D = q.shape
    o = torch.full_like(dq, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    eca.attn_fwd_gqa(dq, dk, dv, causal=causal, scale=scale, o=o, lse=lse)
    torch.cuda.synchronize()
    assert eca.device_status() == 0
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


CASES = [
    # B, H, Hkv, N, D, dtype, causal
    (1, 8, 2, 1000, 128, "fp16", True),
    (2, 4, 1, 300, 64, "bf16", False),
    (1, 32, 8, 2048, 128, "fp16", True),
    (1, 6, 3, 129, 64, "fp16", True),
    (2, 4, 4, 257, 128, "bf16", True),
    (1, 6, 2, 500, 128, "fp16", True),  # three heads per group: consecutive-tile units, not head pairs
]


@pytest.mark.parametrize("B,H,Hkv,N,D,dtype,causal", CASES)
def test_gqa_matches_oracle(cuda_lib, B, H, Hkv, N, D, dtype, causal):
    q, k, v = make(B, H, Hkv, N, D, dtype, seed=3000 + H + Hkv + N)
    scale = 1.0 / math.sqrt(D)
    o, lse = run(q, k, v, causal, scale)
    ro, rl = oracle_full(q, k, v, dtype, causal, scale)
    compare(o, lse, ro, rl, dtype, p_rounding_term(q, k, v, dtype, causal, scale),
            name=f"gqa_b{B}_h{H}_hkv{Hkv}_n{N}_d{D}_{dtype}_{'causal' if causal else 'noncausal'}")


def test_gqa_equals_mha_on_expanded_heads(cuda_lib):
    # Copying each K/V head g times (what the page warns against doing physically)
    # must give bit-identical results through the one-to-one path.
    B, H, Hkv, N, D = 2, 8, 2, 700, 128
    q, k, v = make(B, H, Hkv, N, D, "fp16", seed=91)
    o, lse = run(q, k, v, True, 0.09)
    g = H // Hkv
    ke, ve = k.repeat_interleave(g, dim=1).contiguous(), v.repeat_interleave(g, dim=1).contiguous()
    from helpers import run_gpu

    oe, lsee = run_gpu(q, ke, ve, True, 0.09)
    assert np.array_equal(o, oe) and np.array_equal(lse, lsee)


@pytest.mark.parametrize("H,Hkv", [(80, 40), (160, 40), (120, 40)])
def test_gqa_with_units_taken_dynamically_all_rows(cuda_lib, H, Hkv):
    # K and V of 84 MB (more than the 64 MiB below which one group is used): units
    # are grouped by heads (whole groups of query heads sharing a K/V head) and
    # handed out from a global counter; groups of 2 and 4 heads make head-pair units,
    # groups of 3 consecutive-tile units.  Every row is compared with the oracle.
    B, N, D = 2, 2048, 128
    q, k, v = make(B, H, Hkv, N, D, "fp16", seed=4400 + H)
    scale = 1.0 / math.sqrt(D)
    o, lse = run(q, k, v, True, scale)
    ro, rl = oracle_full(q, k, v, "fp16", True, scale)
    compare(o, lse, ro, rl, "fp16", name=f"gqa_dynamic_b{B}_h{H}_hkv{Hkv}_n{N}_d{D}_fp16_causal")


def test_gqa_with_units_taken_dynamically(cuda_lib):
    # K and V of 134 MB at a long length: every row is written, sampled rows match
    # the oracle, and a repeat launch is bit-identical.
    from helpers import oracle_rows, sample_rows

    B, H, Hkv, N, D = 2, 32, 8, 16384, 128
    q, k, v = make(B, H, Hkv, N, D, "fp16", seed=4343)
    scale = 1.0 / math.sqrt(D)
    o, lse = run(q, k, v, True, scale)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    rows = sample_rows(B, H, N, 160, seed=12)
    ro, rl = oracle_rows(q, k, v, "fp16", True, scale, rows)
    bh = np.array([r[0] for r in rows])
    i = np.array([r[1] for r in rows])
    compare(o.reshape(B * H, N, D)[bh, i], lse.reshape(B * H, N)[bh, i], ro, rl, "fp16",
            name="gqa_dynamic_b2_h32_hkv8_n16384_d128_fp16_causal", rows=len(rows))
    o2, lse2 = run(q, k, v, True, scale)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
