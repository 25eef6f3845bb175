"""GPU parity: the CUDA path through the C ABI against the FP64 oracle.

Same seeded inputs on both sides (exact fp16/bf16 bytes); outputs NaN-filled
before every call (the coverage trap of section 3.4 of the lpnh.cn "Softmax
kernels V1-V9" page); tolerances in tests/helpers.py.
"""
import math

import numpy as np
import pytest
import torch

from exact_causal_attention_gb300 import inputs

from helpers import compare, oracle_full, p_rounding_term, record, run_gpu

pytestmark = pytest.mark.gpu

@pytest.mark.parametrize("name", list(inputs.WORKLOADS))
def test_workload_all_rows(cuda_lib, name):
    """Every row of every workload, the N = 8192 one (the only one whose units are taken
    from the launch's counter in head groups) included, against the oracle."""
    w = inputs.WORKLOADS[name]
    q, k, v = inputs.workload_qkv(w)
    o, lse = run_gpu(q, k, v, w.causal, w.scale)
    ro, rl = oracle_full(q, k, v, w.dtype, w.causal, w.scale)
    stats = compare(o, lse, ro, rl, w.dtype, p_rounding_term(q, k, v, w.dtype, w.causal, w.scale), name=name)
    print(name, stats)


EDGE_N = [1, 2, 127, 128, 129, 255, 256, 257, 383, 513, 1000]


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N", EDGE_N)
def test_edge_lengths(cuda_lib, N, causal, D, dtype):
    B, H = (2, 3) if N < 300 else (1, 2)
    q, k, v = inputs.make_qkv(B, H, N, D, dtype, seed=1000 + N + D, qk_std=1.5)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_gpu(q, k, v, causal, scale)
    ro, rl = oracle_full(q, k, v, dtype, causal, scale)
    compare(o, lse, ro, rl, dtype, p_rounding_term(q, k, v, dtype, causal, scale))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N", [1, 127, 129, 257, 513, 1000])
def test_edge_lengths_with_many_heads(cuda_lib, N, causal, D, dtype):
    """Enough heads that the launch has at least as many pair units as SMs, so the
    kernel keeps two query tiles per unit (few heads, as in test_edge_lengths, give
    key-halves units: one query tile whose key tiles the CTA's two slots share)."""
    B, H = 4, 40
    q, k, v = inputs.make_qkv(B, H, N, D, dtype, seed=5000 + N + D, qk_std=1.5)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_gpu(q, k, v, causal, scale)
    ro, rl = oracle_full(q, k, v, dtype, causal, scale)
    compare(o, lse, ro, rl, dtype, p_rounding_term(q, k, v, dtype, causal, scale))


@pytest.mark.parametrize("causal", [True, False])
def test_zero_queries_give_prefix_mean_at_full_size(cuda_lib, causal):
    # Q = 0: every visible score is 0, so O_i is the mean of the visible v_j and
    # lse_i = ln(count): a closed form that needs no oracle at any size.
    B, H, N, D = 1, 4, 8192, 128
    _, _, v = inputs.make_qkv(B, H, N, D, "fp16", seed=77)
    q = torch.zeros_like(v)
    k = torch.randn(v.shape, generator=torch.Generator().manual_seed(78)).to(torch.float16)
    o, lse = run_gpu(q, k, v, causal, 1.0 / math.sqrt(D))
    vd = v.double().numpy()
    if causal:
        ref = np.cumsum(vd, axis=2) / np.arange(1, N + 1)[None, None, :, None]
        ref_l = np.log(np.arange(1, N + 1, dtype=np.float64))[None, None, :]
    else:
        ref = np.broadcast_to(vd.mean(axis=2, keepdims=True), vd.shape)
        ref_l = np.full((1, 1, N), math.log(N))
    assert np.abs(o - ref).max() <= 2e-3
    assert np.abs(lse - ref_l).max() <= 1e-4


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_values_all_ones_give_ones(cuda_lib, dtype):
    # rows of softmax sum to one: V = 1 gives O = 1 up to rounding of P.
    B, H, N, D = 2, 4, 2000, 64
    q, k, _ = inputs.make_qkv(B, H, N, D, dtype, seed=5, qk_std=3.0)
    v = torch.ones_like(q)
    o, _ = run_gpu(q, k, v, True, 0.125)
    tol = 4e-3 if dtype == "fp16" else 1.6e-2
    assert np.abs(o - 1.0).max() <= tol


def test_key_shift_invariance_through_the_abi(cuda_lib):
    # Integer-valued inputs so k + u is exact in fp16: O unchanged, lse shifted by scale*q.u.
    B, H, N, D = 1, 2, 1000, 64
    g = torch.Generator().manual_seed(11)
    q = torch.randint(-2, 3, (B, H, N, D), generator=g).to(torch.float16)
    k = torch.randint(-2, 3, (B, H, N, D), generator=g).to(torch.float16)
    v = torch.randn((B, H, N, D), generator=g).to(torch.float16)
    u = torch.randint(-3, 4, (D,), generator=g).to(torch.float16)
    scale = 0.125
    o1, l1 = run_gpu(q, k, v, True, scale)
    o2, l2 = run_gpu(q, k + u, v, True, scale)
    shift = scale * (q.double() @ u.double()).numpy()
    assert np.abs(o2 - o1).max() <= 2e-3
    assert np.abs((l2 - l1) - shift).max() <= 1e-4


def test_heads_independent_and_deterministic(cuda_lib):
    B, H, N, D = 2, 3, 700, 128
    q, k, v = inputs.make_qkv(B, H, N, D, "fp16", seed=21)
    o, lse = run_gpu(q, k, v, True, 0.09)
    o2, lse2 = run_gpu(q, k, v, True, 0.09)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    for b, h in [(0, 0), (1, 2), (0, 1)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        os_, ls_ = run_gpu(q[sl].contiguous(), k[sl].contiguous(), v[sl].contiguous(), True, 0.09)
        assert np.array_equal(os_[0, 0], o[b, h]) and np.array_equal(ls_[0, 0], lse[b, h])


def test_lse_null_and_side_stream(cuda_lib):
    import exact_causal_attention_gb300 as eca

    q, k, v = (x.cuda() for x in inputs.make_qkv(1, 2, 300, 64, "bf16", seed=31))
    o_ref, _ = eca.attn_fwd(q, k, v, causal=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o = torch.full_like(q, float("nan"))
        eca.attn_fwd_into(q, k, v, o, None, causal=True, stream=s)
    s.synchronize()
    assert torch.equal(o, o_ref)


def test_rejections_on_device(cuda_lib):
    import exact_causal_attention_gb300 as eca

    x = torch.zeros(1, 1, 64, 64 + 8, dtype=torch.float16, device="cuda")
    q = x[..., 1:65]  # not contiguous
    with pytest.raises(ValueError):
        eca.attn_fwd(q, q, q)
    flat = torch.zeros(1 + 64 * 64, dtype=torch.float16, device="cuda")
    mis = flat[1:].view(1, 1, 64, 64)  # 2-byte offset
    with pytest.raises(eca.AttnError) as e:
        eca.attn_fwd(mis, mis, mis)
    assert e.value.status == -2
    d96 = torch.zeros(1, 1, 64, 96, dtype=torch.float16, device="cuda")
    with pytest.raises(eca.AttnError) as e:
        eca.attn_fwd(d96, d96, d96)
    assert e.value.status == -3


def test_binding_fast_path_declines_bad_outputs(cuda_lib):
    """attn_fwd_into's quick check passes anything unusual to the full checks, which
    raise; a valid call gives the same bytes on the default and an explicit stream."""
    import exact_causal_attention_gb300 as eca

    g = torch.Generator(device="cuda").manual_seed(5)
    q, k, v = (torch.randn(1, 2, 256, 64, device="cuda", generator=g).half() for _ in range(3))
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 256, device="cuda")
    with pytest.raises(ValueError):
        eca.attn_fwd_into(q, k, v, torch.empty_like(q, dtype=torch.bfloat16), lse)
    with pytest.raises(ValueError):
        eca.attn_fwd_into(q, k, v, o, torch.empty(1, 2, 256, device="cuda", dtype=torch.float16))
    with pytest.raises(ValueError):
        eca.attn_fwd_into(q, k, v, o, torch.empty(1, 2, 255, device="cuda"))
    with pytest.raises(TypeError):
        eca.attn_fwd_into(q, k.float(), v, o, lse)
    eca.attn_fwd_into(q, k, v, o, lse)
    s = torch.cuda.Stream()
    o2, lse2 = torch.full_like(o, float("nan")), torch.full_like(lse, float("nan"))
    torch.cuda.synchronize()
    eca.attn_fwd_into(q, k, v, o2, lse2, stream=s)
    s.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("x_row", [-60.0, -6.0, 34.0])
def test_rows_far_from_the_first_reference(cuda_lib, D, x_row):
    """Every key equal, so each causal row's scores are one value x_row (in units of
    scale * log2 e): the output is the running mean of V and lse = s + ln(i + 1).
    The first key tile's reference then sits 64 above the row (p would underflow
    in 16 bits unless the tile's own max replaces it), 10 above (kept: p ~ 2^-10),
    or 30 below (p would overflow, so the max replaces it)."""
    B, H, N = 1, 2, 384
    scale = 1.0 / math.sqrt(D)
    u = torch.ones(D)
    a = x_row / (scale * D * math.log2(math.e))  # q = a u, k = u: s = a D scale
    q = (a * u).expand(B, H, N, D).contiguous().half()
    k = u.expand(B, H, N, D).contiguous().half()
    g = torch.Generator().manual_seed(9)
    v = torch.randn(B, H, N, D, generator=g).half()
    o, lse = run_gpu(q, k, v, True, scale)
    ro, rl = oracle_full(q, k, v, "fp16", True, scale)
    compare(o, lse, ro, rl, "fp16")
    prefix = np.cumsum(v.double().numpy(), axis=2) / np.arange(1, N + 1)[None, None, :, None]
    assert np.abs(o - prefix).max() <= 4e-3


def _rank_one_scores(x_keys, N, D, scale, v_means, seed):
    """q_i = (1, 0, ..., 0) for every row and k_j = (b_j, 0, ..., 0), so the score of key j
    is scale * b_j for every query row: in the kernel's base-2 units x_j = scale log2(e) b_j.
    b_j is x_keys[j] / (scale log2 e) rounded to fp16 (the oracle reads the rounded value).
    V rows are N(mean, 1) with the mean of key j's group."""
    c = scale * math.log2(math.e)
    b = torch.tensor(np.asarray(x_keys) / c, dtype=torch.float64)
    q = torch.zeros(1, 2, N, D, dtype=torch.float64)
    q[..., 0] = 1.0
    k = torch.zeros(1, 2, N, D, dtype=torch.float64)
    k[..., 0] = b
    g = torch.Generator().manual_seed(seed)
    v = torch.randn(1, 2, N, D, generator=g, dtype=torch.float64) + torch.tensor(v_means)[None, None, :, None]
    return tuple(x.to(torch.float32).to(torch.float16) for x in (q, k, v))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("first", ["below_one", "above_one"])
def test_guessed_reference_with_subnormal_probabilities(cuda_lib, D, first):
    """Rows whose later keys would have p in fp16's subnormal range under a guessed
    reference.  Under the fixed assignment (K and V well under 64 MiB) a unit whose
    first key tile is unmasked starts from a guessed reference of 4 (base-2 units).
    Every row sees the same scores: keys 0-127 (the first key tile of every query tile
    past the first) sit 14.9 below the guess (sum of p about 2^-7.9: the guess must be
    rejected, or l would stay near 2^-8) or 6.5 below it (sum of p about 1.4: the guess
    may be kept, l >= 1); every later key sits where, against the guess, p would be
    1.4..5.4 times 2^-24, deep in the subnormal range, rounded by 7-29% in one
    direction.  V rows of the first tile have mean -1 and the later ones +1, so a
    biased weight of the later keys moves O.  With l near 2^-8 that bias reaches about
    1e-2; with l >= 1 it stays below 1e-4 beyond the output's own rounding, as with
    the row max as reference."""
    N = 2048
    scale = 1.0 / math.sqrt(D)
    rng = np.random.default_rng(D)
    guess = 4.0
    offset = -14.9 if first == "below_one" else -6.5
    x_first = guess + offset + rng.uniform(-0.5, 0.5, 128)
    late_p = np.array([1.4, 2.4, 3.4, 4.4, 5.4]) * 2.0 ** -24
    x_late = guess + np.log2(late_p)[np.arange(N - 128) % 5]
    means = [-1.0] * 128 + [1.0] * (N - 128)
    q, k, v = _rank_one_scores(np.concatenate([x_first, x_late]), N, D, scale, means, seed=D + 17)
    o, lse = run_gpu(q, k, v, True, scale)
    ro, rl = oracle_full(q, k, v, "fp16", True, scale)
    # l >= 1 bounds the subnormal rounding by 2^-25 per key relative to l, so beyond the
    # rounding of O itself to fp16 (half an fp16 ulp of the result) only the ordinary
    # rounding of P to fp16 is left (about 3e-4 here, in rows with few keys); with l near
    # 2^-8 the excess would be about 1e-2 and the mean error about 5e-3.
    a = np.abs(ro)
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(a, 2.0 ** -14))) - 11)
    excess = float((np.abs(o - ro) - half_ulp).max())
    stats = compare(o, lse, ro, rl, "fp16")
    record(f"guessed_reference_{first}_d{D}", {**stats, "excess_over_output_rounding": excess})
    assert excess <= 1e-3, {**stats, "excess_over_output_rounding": excess}


@pytest.mark.parametrize("causal,dtype", [(False, "fp16"), (True, "bf16"), (False, "bf16")])
def test_counter_units_other_masks_and_types(cuda_lib, causal, dtype):
    """Launches whose K and V exceed 64 MiB take their units from the launch's counter in
    head groups.  The workloads cover that path causal and in fp16 only; here it runs
    non-causal and in bf16 too (B=2 H=32 N=4096 D=128: K and V 128 MiB), every row
    against the oracle."""
    B, H, N, D = 2, 32, 4096, 128
    q, k, v = inputs.make_qkv(B, H, N, D, dtype, seed=7100 + int(causal) + (dtype == "bf16") * 2)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_gpu(q, k, v, causal, scale)
    ro, rl = oracle_full(q, k, v, dtype, causal, scale)
    compare(o, lse, ro, rl, dtype, p_rounding_term(q, k, v, dtype, causal, scale),
            name=f"counter_units_b2_h32_n4096_d128_{dtype}_{'causal' if causal else 'noncausal'}")


@pytest.mark.parametrize("causal", [True, False])
def test_counter_units_d64_ragged(cuda_lib, causal):
    """The counter path with D = 64 and a ragged length (B=4 H=32 N=4000: K and V
    131 MB), every row against the oracle."""
    B, H, N, D = 4, 32, 4000, 64
    q, k, v = inputs.make_qkv(B, H, N, D, "fp16", seed=7200 + int(causal))
    scale = 1.0 / math.sqrt(D)
    o, lse = run_gpu(q, k, v, causal, scale)
    ro, rl = oracle_full(q, k, v, "fp16", causal, scale)
    compare(o, lse, ro, rl, "fp16", None,
            name=f"counter_units_b4_h32_n4000_d64_fp16_{'causal' if causal else 'noncausal'}")


@pytest.mark.parametrize("dtype,causal", [("fp16", True), ("bf16", False)])
def test_tensors_past_4_gib(cuda_lib, dtype, causal):
    """q, k, v and o of 2^31 elements each (4 GiB: B=128 H=128 N=1024 D=128), so element
    offsets pass 2^31 and byte offsets 2^32; the units come from the launch's counter in head
    groups.  Every element is written and finite; whole slices at the start, the middle and
    the end are compared with the oracle on every row."""
    import exact_causal_attention_gb300 as eca

    B, H, N, D = 128, 128, 1024, 128
    scale = 1.0 / math.sqrt(D)
    q, k, v = inputs.make_qkv_device(B, H, N, D, dtype, seed=1400 + causal, device="cuda")
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    eca.attn_fwd_into(q, k, v, o, lse, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert eca.device_status() == 0
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
    for bh in (0, B * H // 2 + 17, B * H - 1):
        b, h = divmod(bh, H)
        qs, ks, vs = (x[b, h][None, None].cpu() for x in (q, k, v))
        ro, rl = oracle_full(qs, ks, vs, dtype, causal, scale)
        compare(o[b, h][None, None].double().cpu().numpy(), lse[b, h][None, None].double().cpu().numpy(), ro, rl,
                dtype, p_rounding_term(qs, ks, vs, dtype, causal, scale),
                name=f"{'causal' if causal else 'noncausal'}_b128_h128_n1024_d128_{dtype}_slice{bh}")
    del q, k, v, o, lse
    torch.cuda.empty_cache()
