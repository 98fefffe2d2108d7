"""Pins for the oracle's row softmax: closed forms, invariants and an
independent library softmax."""
import math

import numpy as np
import pytest


def f16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16)


def test_constant_rows_are_uniform(oracle_lib):
    for N in (1, 3, 64, 1000):
        X = f16(np.full((4, N), 2.5) + np.arange(4)[:, None])
        _, Y64 = oracle_lib.softmax(X, want_f64=True)
        np.testing.assert_allclose(Y64, 1.0 / N, rtol=1e-14)


def test_two_entries_follow_the_logistic(oracle_lib):
    X = f16([[1.5, -0.75], [0.0, 3.0], [-2.0, -2.0]])
    _, Y64 = oracle_lib.softmax(X, want_f64=True)
    for i, (a, b) in enumerate(X.astype(np.float64)):
        p = 1.0 / (1.0 + math.exp(b - a))
        np.testing.assert_allclose(Y64[i], [p, 1 - p], rtol=1e-14)


def test_shift_invariance_and_rows_sum_to_one(oracle_lib):
    rng = np.random.default_rng(1)
    X = f16(np.round(rng.normal(0, 3, size=(20, 77)) * 4) / 4)  # quarters: x + 8 is exact in fp16
    _, a = oracle_lib.softmax(X, want_f64=True)
    _, b = oracle_lib.softmax(f16(X.astype(np.float64) + 8.0), want_f64=True)  # exact shift in fp16 here
    assert np.array_equal(f16(X.astype(np.float64) + 8.0).astype(np.float64) - 8.0, X.astype(np.float64))
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-16)
    np.testing.assert_allclose(a.sum(axis=1), 1.0, rtol=1e-14)


def test_large_values_need_the_max_shift(oracle_lib):
    X = f16([[60000.0, 59968.0, -60000.0, 0.0]])  # binary16 spacing is 32 here: both exact
    _, Y64 = oracle_lib.softmax(X, want_f64=True)
    d = 60000.0 - 59968.0
    assert X[0, 1] == 59968.0
    np.testing.assert_allclose(Y64[0, :2], [1.0 / (1.0 + math.exp(-d)), 1.0 / (1.0 + math.exp(d))], rtol=1e-12)
    assert Y64[0, 2] == 0.0 and Y64[0, 3] == 0.0
    # the largest entry last and first: the maximum must cover every entry
    for row in ([-60000.0, 0.0, 60000.0], [60000.0, 0.0, -60000.0]):
        _, Y64 = oracle_lib.softmax(f16([row]), want_f64=True)
        assert np.array_equal(Y64[0], [1.0 if v == 60000.0 else 0.0 for v in row])


def test_minus_infinity_entries_get_zero(oracle_lib):
    X = f16([[-np.inf, 0.0, -np.inf, 0.0], [-np.inf] * 4])
    Y, Y64 = oracle_lib.softmax(X, want_f64=True)
    assert np.array_equal(Y64[0], [0.0, 0.5, 0.0, 0.5])
    assert np.isnan(Y64[1]).all()


def test_matches_a_library_softmax(oracle_lib):
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(2)
    for M, N in [(5, 1), (7, 33), (16, 4096), (3, 32768)]:
        X = f16(rng.normal(0, 4, size=(M, N)))
        Y, Y64 = oracle_lib.softmax(X, want_f64=True)
        ref = scipy_special.softmax(X.astype(np.float64), axis=1)
        np.testing.assert_allclose(Y64, ref, rtol=1e-12, atol=1e-300)
        assert np.array_equal(Y.view(np.uint16), ref.astype(np.float16).view(np.uint16))


def test_row_ranges(oracle_lib):
    X = f16(np.random.default_rng(3).normal(0, 1, size=(9, 50)))
    full = oracle_lib.softmax(X)
    part = oracle_lib.softmax(X, rows=(3, 4))
    assert np.array_equal(part.view(np.uint16), full[3:7].view(np.uint16))
    with pytest.raises(RuntimeError):
        oracle_lib.softmax(X, rows=(8, 2))
