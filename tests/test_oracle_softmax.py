"""Pins of the FP64 row-softmax oracle (oracle/softmax_ref.cpp) to facts fixed by
the page "Softmax kernels V1-V9" (lpnh.cn) and by the mathematics: its section 3.3
test inputs (an all-zero row, a special last element, a constant added to a whole
row, seeded random rows, odd lengths), closed forms, and the online form of
sections 4.4-4.6 against the two-pass definition and a pure-Python fsum leg."""
import math

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def rnd(shape, seed, lo=-10.0, hi=10.0):
    return np.random.default_rng(seed).uniform(lo, hi, shape)


MODES = [("two_pass", 1), ("online", 1), ("online", 7), ("online", 64)]


@pytest.mark.parametrize("mode,tile", MODES)
def test_zero_row_is_uniform(mode, tile):
    for N in (1, 2, 257, 1000):
        y = oracle.softmax(np.zeros((3, N)), mode=mode, tile=tile)
        np.testing.assert_allclose(y, 1.0 / N, rtol=1e-15, atol=0)


@pytest.mark.parametrize("mode,tile", MODES)
def test_special_last_element_closed_form(mode, tile):
    # zeros with the last entry a: y_last = e^a / (N - 1 + e^a), the others 1 / (N - 1 + e^a)
    N = 129
    for a in (-30.0, -1.0, 0.5, 7.0, 80.0):
        x = np.zeros((1, N))
        x[0, -1] = a
        y = oracle.softmax(x, mode=mode, tile=tile)
        den = N - 1 + math.exp(a)
        np.testing.assert_allclose(y[0, :-1], 1.0 / den, rtol=1e-14, atol=0)
        np.testing.assert_allclose(y[0, -1], math.exp(a) / den, rtol=1e-14, atol=0)


@pytest.mark.parametrize("mode,tile", MODES)
def test_constant_added_to_a_row_changes_nothing(mode, tile):
    x = rnd((5, 300), 1)
    c = rnd((5, 1), 2, -1000.0, 1000.0)
    np.testing.assert_allclose(oracle.softmax(x + c, mode=mode, tile=tile), oracle.softmax(x, mode=mode, tile=tile),
                               rtol=1e-12, atol=1e-16)


def test_rows_sum_to_one_and_order_is_kept():
    x = rnd((7, 1001), 3)
    y = oracle.softmax(x)
    np.testing.assert_allclose(y.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert np.array_equal(np.argsort(x, axis=1, kind="stable"), np.argsort(y, axis=1, kind="stable"))
    # ratios follow the differences: y_a / y_b = exp(x_a - x_b)
    np.testing.assert_allclose(y[:, 3] / y[:, 10], np.exp(x[:, 3] - x[:, 10]), rtol=1e-12)


def test_huge_inputs_need_max_subtraction():
    x = rnd((4, 64), 4, 1e4, 2e4)
    y = oracle.softmax(x)
    assert np.isfinite(y).all()
    np.testing.assert_allclose(y.sum(axis=1), 1.0, rtol=0, atol=1e-13)


@pytest.mark.parametrize("tile", [1, 3, 4])
def test_minus_infinity_entries_and_empty_chunks(tile):
    # the first chunks are entirely -inf: merging an empty state (-inf, 0) must not make NaN
    x = np.array([[-np.inf, -np.inf, -np.inf, -np.inf, 1.0, 2.0, -np.inf, 0.0]])
    finite = np.array([1.0, 2.0, 0.0])
    ref = np.exp(finite - 2.0) / np.exp(finite - 2.0).sum()
    for mode in ("two_pass", "online"):
        y = oracle.softmax(x, mode=mode, tile=tile)
        assert np.isfinite(y).all()
        np.testing.assert_allclose(y[0, [4, 5, 7]], ref, rtol=1e-15)
        assert np.all(y[0, [0, 1, 2, 3, 6]] == 0.0)
    assert np.all(oracle.softmax(np.full((1, 5), -np.inf)) == 0.0)


@pytest.mark.parametrize("seed", range(5))
def test_online_equals_two_pass_and_fsum(seed):
    rng = np.random.default_rng(200 + seed)
    M, N = int(rng.integers(1, 4)), int(rng.integers(1, 40))
    x = rng.uniform(-10, 10, (M, N))
    ref = np.array([[math.exp(v - max(r)) / math.fsum(math.exp(w - max(r)) for w in r) for v in r]
                    for r in x.tolist()])
    y2 = oracle.softmax(x, mode="two_pass")
    np.testing.assert_allclose(y2, ref, rtol=1e-13, atol=1e-300)
    for tile in range(1, N + 1):
        np.testing.assert_allclose(oracle.softmax(x, mode="online", tile=tile), y2, rtol=1e-13, atol=1e-300)


def test_rows_are_independent():
    x = rnd((6, 77), 9)
    y = oracle.softmax(x)
    for r in range(6):
        assert np.array_equal(oracle.softmax(x[r:r + 1])[0], y[r])


def test_softmax_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.softmax(np.zeros(5))
    with pytest.raises(ValueError):
        oracle.softmax(np.zeros((2, 3)), mode="online", tile=0)
