"""Pins of the paged-cache helpers of the oracle: the address rule of section 2 of
"CUDA KV Cache：分页存储与长上下文 Decode 极致优化" (p = block_table[b, t // T],
offset t % T) against a contiguous cache, and the decode reference against the
plain attention definition on the gathered sequence."""
import math

import numpy as np
import pytest

import oracle


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_identity_table_reads_pages_in_order():
    P, T, Hkv, D = 6, 4, 2, 3
    cache = rnd((P, 2, T, Hkv, D), 1)
    table = np.arange(P)[None, :]
    (k, v), = oracle.gather_paged(cache, table, [P * T], T)
    # contiguous cache [P*T, Hkv, D] read straight through
    np.testing.assert_array_equal(k, cache[:, 0].reshape(P * T, Hkv, D).transpose(1, 0, 2))
    np.testing.assert_array_equal(v, cache[:, 1].reshape(P * T, Hkv, D).transpose(1, 0, 2))


def test_permuted_pages_give_the_same_logical_sequence():
    P, T, Hkv, D, L = 10, 4, 1, 2, 27
    dense_k, dense_v = rnd((L, Hkv, D), 2), rnd((L, Hkv, D), 3)
    perm = np.random.default_rng(4).permutation(P)
    cache = np.full((P, 2, T, Hkv, D), np.nan)
    for t in range(L):
        cache[perm[t // T], 0, t % T] = dense_k[t]
        cache[perm[t // T], 1, t % T] = dense_v[t]
    (k, v), = oracle.gather_paged(cache, perm[None, :], [L], T)
    np.testing.assert_array_equal(k, dense_k.transpose(1, 0, 2))
    np.testing.assert_array_equal(v, dense_v.transpose(1, 0, 2))
    assert not np.isnan(k).any()  # never reads past the length (the rest of the last page is NaN)


def test_decode_equals_softmax_over_the_context():
    B, Hq, Hkv, D, T, P = 2, 4, 2, 8, 4, 12
    cache = rnd((P, 2, T, Hkv, D), 5)
    table = np.array([np.random.default_rng(6).permutation(P)[:6], np.random.default_rng(7).permutation(P)[:6]])
    lengths = [13, 1]
    q = rnd((B, Hq, D), 8)
    o, lse = oracle.decode_paged(q, cache, table, lengths, T, 0.35)
    for b, (k, v) in enumerate(oracle.gather_paged(cache, table, lengths, T)):
        for h in range(Hq):
            kh, vh = k[h // (Hq // Hkv)], v[h // (Hq // Hkv)]
            s = 0.35 * kh @ q[b, h]
            w = np.exp(s - s.max())
            np.testing.assert_allclose(o[b, h], (w / w.sum()) @ vh, rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(lse[b, h], s.max() + math.log(w.sum()), rtol=1e-13)
    # a single token: O is that token's value, lse its score
    np.testing.assert_allclose(o[1], np.repeat(cache[table[1, 0], 1, 0], Hq // Hkv, axis=0), rtol=0, atol=0)


def test_empty_request_gives_zero_and_minus_infinity():
    cache = rnd((2, 2, 4, 1, 2), 9)
    o, lse = oracle.decode_paged(rnd((1, 1, 2), 10), cache, np.array([[0, 1]]), [0], 4, 1.0)
    assert np.all(o == 0.0) and np.all(lse == -np.inf)
