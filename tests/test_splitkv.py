"""GPU parity of the key-split path (segments merged by the second kernel) against
the FP64 oracle; the merge law is section 6.4 of "CUDA KV Cache：分页存储与长上下文
Decode 极致优化".  The workspace is filled with NaN bytes before each call: its
contents on entry must not matter."""
import math

import numpy as np
import pytest
import torch

from exact_causal_attention_gb300 import inputs

from helpers import compare, oracle_full, oracle_rows, p_rounding_term, sample_rows

pytestmark = pytest.mark.gpu


def run_split(q, k, v, causal, scale, splits):
    import exact_causal_attention_gb300 as eca

    dq, dk, dv = (x.cuda() for x in (q, k, v))
    B, H, N, D = q.shape
    o = torch.full_like(dq, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    need = eca.splitkv_workspace_bytes(B, H, N, D, splits)
    assert need > 0
    ws = torch.full((need + 256,), 0xFF, dtype=torch.uint8, device="cuda")
    off = (-ws.data_ptr()) % 256
    eca.attn_fwd_splitkv(dq, dk, dv, o, lse, kv_splits=splits, workspace=ws[off:off + need], causal=causal,
                         scale=scale)
    torch.cuda.synchronize()
    assert eca.device_status() == 0
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


CASES = [
    # B, H, N, D, dtype, causal, splits
    (1, 2, 256, 64, "fp16", True, 2),
    (1, 2, 1000, 128, "bf16", True, 3),
    (1, 4, 2048, 128, "fp16", False, 4),
    (2, 1, 129, 64, "fp16", True, 2),
    (1, 1, 1, 64, "fp16", True, 4),
    (1, 2, 3000, 64, "bf16", False, 64),
    (1, 3, 1536, 128, "fp16", True, 5),
    (1, 2, 2560, 128, "fp16", True, 20),  # rows see 1 to 20 segments: several merge batches
]


@pytest.mark.parametrize("B,H,N,D,dtype,causal,splits", CASES)
def test_splitkv_matches_oracle(cuda_lib, B, H, N, D, dtype, causal, splits):
    q, k, v = inputs.make_qkv(B, H, N, D, dtype, seed=2000 + N + splits, qk_std=1.5)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_split(q, k, v, causal, scale, splits)
    ro, rl = oracle_full(q, k, v, dtype, causal, scale)
    compare(o, lse, ro, rl, dtype, p_rounding_term(q, k, v, dtype, causal, scale),
            name=f"split{splits}_b{B}_h{H}_n{N}_d{D}_{dtype}_{'causal' if causal else 'noncausal'}")


def test_splitkv_agrees_with_unsplit_path(cuda_lib):
    from helpers import run_gpu

    q, k, v = inputs.make_qkv(1, 4, 1500, 128, "fp16", seed=77)
    o1, l1 = run_gpu(q, k, v, True, 0.088)
    for splits in (1, 2, 7):
        o2, l2 = run_split(q, k, v, True, 0.088, splits)
        assert np.abs(o2 - o1).max() <= 2e-3
        assert np.abs(l2 - l1).max() <= 2e-5


def test_splitkv_long_sequence_few_heads_sampled(cuda_lib):
    import exact_causal_attention_gb300 as eca

    B, H, N, D = 1, 2, 8192, 128
    q, k, v = inputs.make_qkv(B, H, N, D, "fp16", seed=31)
    assert 1 <= eca.splitkv_default_splits(B, H, N, D) <= 64
    splits = 4
    o, lse = run_split(q, k, v, True, 1.0 / math.sqrt(D), splits)
    rows = sample_rows(B, H, N, 200, seed=5)
    ro, rl = oracle_rows(q, k, v, "fp16", True, 1.0 / math.sqrt(D), rows)
    bh = np.array([r[0] for r in rows])
    i = np.array([r[1] for r in rows])
    compare(o.reshape(B * H, N, D)[bh, i], lse.reshape(B * H, N)[bh, i], ro, rl, "fp16",
            name=f"split{splits}_b{B}_h{H}_n{N}_d{D}_fp16_causal", rows=len(rows))
    assert np.isfinite(o).all() and np.isfinite(lse).all()


def test_splitkv_with_units_taken_dynamically_all_rows(cuda_lib):
    # K and V of 84 MB (more than 64 MiB): head-grouped units from the launch's
    # counter, with a split on top; every row against the oracle.
    B, H, N, D, splits = 2, 80, 2048, 128, 3
    q, k, v = inputs.make_qkv(B, H, N, D, "fp16", seed=4243)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_split(q, k, v, True, scale, splits)
    ro, rl = oracle_full(q, k, v, "fp16", True, scale)
    compare(o, lse, ro, rl, "fp16", name=f"split{splits}_dynamic_b{B}_h{H}_n{N}_d{D}_fp16_causal")


def test_splitkv_with_units_taken_dynamically(cuda_lib):
    # K and V of 268 MB: the kernel groups heads and hands units out from a global
    # counter; with a split on top.  Every row is written (the outputs start as
    # NaN), sampled rows match the oracle, the unsplit launch agrees, and a second
    # launch (the counters reset themselves) gives bit-identical results.
    B, H, N, D = 4, 16, 8192, 128
    q, k, v = inputs.make_qkv(B, H, N, D, "fp16", seed=4242)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_split(q, k, v, True, scale, 3)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    rows = sample_rows(B, H, N, 160, seed=11)
    ro, rl = oracle_rows(q, k, v, "fp16", True, scale, rows)
    bh = np.array([r[0] for r in rows])
    i = np.array([r[1] for r in rows])
    compare(o.reshape(B * H, N, D)[bh, i], lse.reshape(B * H, N)[bh, i], ro, rl, "fp16",
            name="split3_dynamic_b4_h16_n8192_d128_fp16_causal", rows=len(rows))
    o2, lse2 = run_split(q, k, v, True, scale, 3)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    from helpers import run_gpu

    o1, l1 = run_gpu(q, k, v, True, scale)
    assert np.isfinite(o1).all()
    assert np.abs(o1 - o).max() <= 2e-3 and np.abs(l1 - lse).max() <= 2e-5
