"""Pins of the FP64 oracle to facts fixed by the pages and by the mathematics.

None of these re-types the oracle's formula: each checks a closed form, a
hand-derived worked example, an invariant of softmax attention, a second
algorithm (the online recurrence against the two-pass definition) or an
independent library routine.  The definition pinned is section 1 of "CUDA
FlashAttention：从在线 Softmax 到长序列 IO 极限"; the recurrence is its section 4;
the test inputs follow section 3.3 of the lpnh.cn "Softmax kernels V1-V9" page
(zero rows, a constant added to a whole row, fixed seeds, ragged lengths).
"""
import math

import numpy as np
import pytest

import oracle
from oracle import pyref

pytestmark = pytest.mark.filterwarnings("ignore")


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ---------------------------------------------------------------- decoders

def test_decode_fp16_matches_numpy_on_every_pattern():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(pats, "fp16")
    ref = pats.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_decode_bf16_matches_truncated_binary32_on_every_pattern():
    pats = np.arange(65536, dtype=np.uint32)
    got = oracle.decode(pats.astype(np.uint16), "bf16")
    ref = (pats << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


# ------------------------------------------------------- closed forms

@pytest.mark.parametrize("mode", ["two_pass", "online"])
@pytest.mark.parametrize("causal", [True, False])
def test_single_key_returns_v0(mode, causal):
    q, k, v = rnd((2, 3, 1, 8), 1), rnd((2, 3, 1, 8), 2), rnd((2, 3, 1, 8), 3)
    o, lse = oracle.attention(q, k, v, causal, 0.37, mode=mode, tile=1)
    assert np.array_equal(o, v)
    s00 = 0.37 * np.einsum("bhnd,bhnd->bhn", q, k)
    np.testing.assert_allclose(lse, s00, rtol=0, atol=1e-14)


@pytest.mark.parametrize("mode", ["two_pass", "online"])
def test_causal_row0_is_v0(mode):
    q, k, v = rnd((1, 2, 37, 16), 4), rnd((1, 2, 37, 16), 5), rnd((1, 2, 37, 16), 6)
    o, _ = oracle.attention(q, k, v, True, 0.25, mode=mode, tile=8)
    assert np.array_equal(o[:, :, 0, :], v[:, :, 0, :])


@pytest.mark.parametrize("mode", ["two_pass", "online"])
def test_zero_queries_give_prefix_mean(mode):
    B, H, N, D = 1, 2, 50, 8
    q = np.zeros((B, H, N, D))
    k, v = rnd((B, H, N, D), 7), rnd((B, H, N, D), 8)
    o, lse = oracle.attention(q, k, v, True, 0.125, mode=mode, tile=7)
    prefix = np.cumsum(v, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    np.testing.assert_allclose(o, prefix, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(np.arange(1, N + 1)), (B, H, N)),
                               rtol=0, atol=1e-13)
    o, lse = oracle.attention(q, k, v, False, 0.125, mode=mode, tile=7)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape),
                               rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, math.log(N), rtol=0, atol=1e-13)


def _two_key_case():
    # Hand-derived worked example, scale 1, D = 2:
    #   q0 = (0, 5), q1 = (ln 3, 0); k0 = (1, 0), k1 = (0, 1); v0 = (4, 0), v1 = (0, 8).
    # Scores: s00 = 0, s01 = 5, s10 = ln 3, s11 = 0.
    q = np.array([[[[0.0, 5.0], [math.log(3.0), 0.0]]]])
    k = np.array([[[[1.0, 0.0], [0.0, 1.0]]]])
    v = np.array([[[[4.0, 0.0], [0.0, 8.0]]]])
    return q, k, v


@pytest.mark.parametrize("mode", ["two_pass", "online"])
def test_two_key_worked_example(mode):
    q, k, v = _two_key_case()
    # causal: row 0 sees only key 0 -> v0, lse = s00 = 0.
    # row 1: weights e^{ln3} : e^0 = 3 : 1 -> (3/4) v0 + (1/4) v1 = (3, 2), lse = ln 4.
    o, lse = oracle.attention(q, k, v, True, 1.0, mode=mode, tile=1)
    np.testing.assert_allclose(o[0, 0], [[4.0, 0.0], [3.0, 2.0]], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], [0.0, math.log(4.0)], rtol=0, atol=1e-14)
    # non-causal row 0: weights 1 : e^5 -> (4, 8 e^5) / (1 + e^5), lse = ln(1 + e^5).
    o, lse = oracle.attention(q, k, v, False, 1.0, mode=mode, tile=1)
    e5 = math.exp(5.0)
    np.testing.assert_allclose(o[0, 0, 0], [4.0 / (1 + e5), 8.0 * e5 / (1 + e5)], rtol=1e-14)
    np.testing.assert_allclose(lse[0, 0, 0], math.log1p(e5), rtol=1e-14)
    np.testing.assert_allclose(o[0, 0, 1], [3.0, 2.0], rtol=1e-14)
    # the scale multiplies the scores: scale 1/2 with doubled queries is the same problem.
    o2, lse2 = oracle.attention(2 * q, k, v, False, 0.5, mode=mode, tile=2)
    np.testing.assert_allclose(o2, o, rtol=1e-14)
    np.testing.assert_allclose(lse2, lse, rtol=1e-14)


@pytest.mark.parametrize("causal", [True, False])
def test_one_hot_hard_attention_and_mask_direction(causal):
    # q_i = lam * e_{pi(i)}, k_j = e_j: only key pi(i) scores lam*scale = 60, all others 0.
    N, D = 12, 12
    pi = np.random.default_rng(9).permutation(N)
    q = np.zeros((1, 1, N, D))
    q[0, 0, np.arange(N), pi] = 240.0
    k = np.eye(N)[None, None]
    v = rnd((1, 1, N, D), 10)
    o, lse = oracle.attention(q, k, v, causal, 0.25)
    for i in range(N):
        if not causal or pi[i] <= i:
            np.testing.assert_allclose(o[0, 0, i], v[0, 0, pi[i]], rtol=0, atol=1e-20 + 1e-12)
            assert abs(lse[0, 0, i] - 60.0) < 1e-12
        else:  # the preferred key is in the future: every visible key scores 0 -> prefix mean
            np.testing.assert_allclose(o[0, 0, i], v[0, 0, : i + 1].mean(axis=0), rtol=0, atol=1e-13)
            np.testing.assert_allclose(lse[0, 0, i], math.log(i + 1), rtol=0, atol=1e-13)


# ----------------------------------------------------------- invariants

@pytest.mark.parametrize("causal", [True, False])
def test_key_shift_invariance(causal):
    # adding u to every key adds scale*q_i.u to every score of row i (a constant per row):
    # O is unchanged and lse moves by that constant (lpnh.cn page, section 3.3).
    B, H, N, D = 2, 2, 33, 16
    q, k, v = rnd((B, H, N, D), 11), rnd((B, H, N, D), 12), rnd((B, H, N, D), 13)
    u = rnd((D,), 14, 3.0)
    o, lse = oracle.attention(q, k, v, causal, 0.3)
    o2, lse2 = oracle.attention(q, k + u, v, causal, 0.3)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2 - lse, 0.3 * q @ u, rtol=0, atol=1e-11)


@pytest.mark.parametrize("causal", [True, False])
def test_value_ones_rows_sum_to_one(causal):
    q, k = rnd((1, 3, 40, 8), 15, 4.0), rnd((1, 3, 40, 8), 16, 4.0)
    o, _ = oracle.attention(q, k, np.ones((1, 3, 40, 8)), causal, 0.5)
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-14)


def test_causal_output_ignores_future_keys():
    B, H, N, D = 1, 2, 30, 8
    q, k, v = rnd((B, H, N, D), 17), rnd((B, H, N, D), 18), rnd((B, H, N, D), 19)
    o, lse = oracle.attention(q, k, v, True, 0.4)
    for cut in (0, 7, 29):
        k2, v2 = k.copy(), v.copy()
        k2[:, :, cut + 1:] = rnd(k2[:, :, cut + 1:].shape, 20 + cut, 9.0)
        v2[:, :, cut + 1:] = rnd(v2[:, :, cut + 1:].shape, 40 + cut, 9.0)
        o2, lse2 = oracle.attention(q, k2, v2, True, 0.4)
        assert np.array_equal(o2[:, :, : cut + 1], o[:, :, : cut + 1])
        assert np.array_equal(lse2[:, :, : cut + 1], lse[:, :, : cut + 1])


def test_noncausal_key_permutation_invariance():
    B, H, N, D = 1, 2, 21, 8
    q, k, v = rnd((B, H, N, D), 21), rnd((B, H, N, D), 22), rnd((B, H, N, D), 23)
    perm = np.random.default_rng(24).permutation(N)
    o, lse = oracle.attention(q, k, v, False, 0.4)
    o2, lse2 = oracle.attention(q, k[:, :, perm], v[:, :, perm], False, 0.4)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-13)


def test_heads_and_batches_are_independent():
    B, H, N, D = 2, 3, 19, 8
    q, k, v = rnd((B, H, N, D), 25), rnd((B, H, N, D), 26), rnd((B, H, N, D), 27)
    o, lse = oracle.attention(q, k, v, True, 0.3)
    for b in range(B):
        for h in range(H):
            sl = (slice(b, b + 1), slice(h, h + 1))
            o1, l1 = oracle.attention(q[sl], k[sl], v[sl], True, 0.3)
            assert np.array_equal(o1[0, 0], o[b, h])
            assert np.array_equal(l1[0, 0], lse[b, h])


@pytest.mark.parametrize("mode", ["two_pass", "online"])
def test_huge_scores_need_max_subtraction(mode):
    # scores of order 1e4: without subtracting the row max, exp overflows to inf.
    B, H, N, D = 1, 1, 24, 4
    q, k, v = rnd((B, H, N, D), 28, 100.0), rnd((B, H, N, D), 29, 100.0), rnd((B, H, N, D), 30)
    o, lse = oracle.attention(q, k, v, True, 1.0, mode=mode, tile=5)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    # the largest score dominates by >> 40 nats except on near ties: check against argmax picks
    s = np.einsum("id,jd->ij", q[0, 0], k[0, 0])
    for i in range(N):
        row = s[i, : i + 1]
        top = np.sort(row)[-2:] if i > 0 else np.array([-np.inf, row[0]])
        if top[1] - top[0] > 50:
            np.testing.assert_allclose(o[0, 0, i], v[0, 0, int(np.argmax(row))], rtol=0, atol=1e-15)
            np.testing.assert_allclose(lse[0, 0, i], row.max(), rtol=1e-15)


# ------------------------------------------- second algorithm and brute force

@pytest.mark.parametrize("seed", range(6))
def test_online_equals_two_pass_and_fsum_on_tiny_inputs(seed):
    rng = np.random.default_rng(100 + seed)
    N, D = int(rng.integers(1, 10)), int(rng.integers(1, 5))
    q, k, v = (rng.standard_normal((1, 2, N, D)) * 2 for _ in range(3))
    scale = float(rng.uniform(0.2, 1.5))
    for causal in (True, False):
        ref_o, ref_l = pyref.attention(q.tolist(), k.tolist(), v.tolist(), causal, scale)
        ref_o, ref_l = np.array(ref_o), np.array(ref_l)
        o2, l2 = oracle.attention(q, k, v, causal, scale, mode="two_pass")
        np.testing.assert_allclose(o2, ref_o, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(l2, ref_l, rtol=1e-12, atol=1e-13)
        for tile in range(1, N + 1):
            o1, l1 = oracle.attention(q, k, v, causal, scale, mode="online", tile=tile)
            np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(l1, l2, rtol=1e-12, atol=1e-13)


def test_rows_entry_matches_full_forward():
    B, H, N, D = 2, 2, 40, 8
    q, k, v = rnd((B, H, N, D), 31), rnd((B, H, N, D), 32), rnd((B, H, N, D), 33)
    o, lse = oracle.attention(q, k, v, True, 0.3)
    rows = [(0, 0), (3, 39), (1, 17), (2, 5)]
    ro, rl = oracle.attention_rows(q, k, v, True, 0.3, rows)
    for r, (bh, i) in enumerate(rows):
        assert np.array_equal(ro[r], o.reshape(B * H, N, D)[bh, i])
        assert rl[r] == lse.reshape(B * H, N)[bh, i]


def test_oracle_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.attention(np.zeros((1, 1, 2, 2)), np.zeros((1, 1, 3, 2)), np.zeros((1, 1, 2, 2)), True, 1.0)
    with pytest.raises(ValueError):
        oracle.attention(np.zeros((1, 1, 2, 2)), np.zeros((1, 1, 2, 2)), np.zeros((1, 1, 2, 2)), True, 1.0,
                         mode="online", tile=0)
    with pytest.raises(ValueError):
        oracle.attention_rows(np.zeros((1, 1, 2, 2)), np.zeros((1, 1, 2, 2)), np.zeros((1, 1, 2, 2)), True,
                              1.0, [(0, 2)])


# ---------------------------------------------------------------- grouped heads

@pytest.mark.parametrize("H,Hkv", [(4, 1), (4, 2), (6, 3), (8, 8)])
@pytest.mark.parametrize("mode", ["two_pass", "online"])
def test_grouped_heads_equal_expanded_heads(H, Hkv, mode):
    # The decode page's section 3.3: copying each key/value head g = H / Hkv times
    # (repeat_interleave) turns grouped attention into ordinary attention; the
    # oracle's head map h -> h // g must give exactly that result.
    B, N, D = 2, 21, 8
    q = rnd((B, H, N, D), 50 + H)
    k, v = rnd((B, Hkv, N, D), 60 + Hkv), rnd((B, Hkv, N, D), 70 + Hkv)
    g = H // Hkv
    ke, ve = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)
    for causal in (True, False):
        o, lse = oracle.attention(q, k, v, causal, 0.3, mode=mode, tile=4)
        oe, lsee = oracle.attention(q, ke, ve, causal, 0.3, mode=mode, tile=4)
        assert np.array_equal(o, oe) and np.array_equal(lse, lsee)


def test_grouped_heads_rows_entry_and_errors():
    B, H, Hkv, N, D = 1, 4, 2, 30, 8
    q, k, v = rnd((B, H, N, D), 80), rnd((B, Hkv, N, D), 81), rnd((B, Hkv, N, D), 82)
    o, lse = oracle.attention(q, k, v, True, 0.3)
    rows = [(0, 0), (3, 29), (1, 7), (2, 15)]
    ro, rl = oracle.attention_rows(q, k, v, True, 0.3, rows)
    for r, (bh, i) in enumerate(rows):
        assert np.array_equal(ro[r], o.reshape(B * H, N, D)[bh, i])
    with pytest.raises(ValueError):
        oracle.attention(q, rnd((B, 3, N, D), 1), rnd((B, 3, N, D), 2), True, 0.3)  # 3 does not divide 4
