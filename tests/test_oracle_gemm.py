"""Pins for the oracle's GEMM and epilogue against things other than itself:
closed forms (identity, permutation, rank-1), exact rational brute force on tiny
shapes, numpy's fp64 matrix product, textbook values of the normal CDF, and
the GELU odd-part identity."""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16)


def rand16(rng, shape, lo=-1.0, hi=1.0):
    return f16(rng.uniform(lo, hi, size=shape))


# ---------------------------------------------------------------- GELU ----

def _golden_pairs(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(tuple(float(t) for t in line.split()))
    return rows


def test_gelu_textbook_values(oracle_lib):
    for x, y in _golden_pairs("gelu_normal_cdf.txt"):
        assert oracle_lib.gelu(x) == pytest.approx(y, rel=1e-13, abs=1e-15), x


def test_gelu_odd_part_identity(oracle_lib):
    # x*Phi(x) - (-x)*Phi(-x) = x*(Phi(x) + 1 - Phi(x)) = x
    for x in np.linspace(-8, 8, 161):
        assert oracle_lib.gelu(x) - oracle_lib.gelu(-x) == pytest.approx(x, abs=1e-14)


def test_gelu_tails(oracle_lib):
    assert oracle_lib.gelu(0.0) == 0.0
    assert oracle_lib.gelu(10.0) == 10.0            # Phi(10) rounds to 1 in fp64
    assert abs(oracle_lib.gelu(-10.0)) < 1e-20      # -10 * Phi(-10) ~ -7.6e-23


# ---------------------------------------------------------------- GEMM ----

def test_identity_left_and_right(oracle_lib):
    rng = np.random.default_rng(0)
    for M, N, K in [(5, 7, 4), (33, 17, 40), (64, 64, 64)]:
        I = f16(np.eye(K))
        B = rand16(rng, (K, N))
        assert np.array_equal(oracle_lib.gemm(I, B).view(np.uint16), B.view(np.uint16))
        A = rand16(rng, (M, K))
        assert np.array_equal(oracle_lib.gemm(A, I).view(np.uint16), A.view(np.uint16))


def test_permutations(oracle_lib):
    rng = np.random.default_rng(1)
    M, K, N = 19, 23, 29
    A = rand16(rng, (M, K))
    B = rand16(rng, (K, N))
    # B = column permutation matrix: (A P)[:, j] = A[:, p[j]]
    p = rng.permutation(K)
    P = np.zeros((K, K)); P[p, np.arange(K)] = 1
    assert np.array_equal(oracle_lib.gemm(A, f16(P)).view(np.uint16), A[:, p].view(np.uint16))
    # A = row permutation matrix: (Q B)[i, :] = B[q[i], :]
    q = rng.permutation(K)
    Q = np.zeros((K, K)); Q[np.arange(K), q] = 1
    assert np.array_equal(oracle_lib.gemm(f16(Q), B).view(np.uint16), B[q, :].view(np.uint16))


def test_rank1_closed_form(oracle_lib):
    # A[i,k] = u_i, B[k,j] = v_j  =>  C[i,j] = K * u_i * v_j (exact: powers of two / small ints)
    u = np.array([1, -2, 0.5, 3, -0.25, 4, 1.5])
    v = np.array([2, -1, 0.125, 6, -3, 0.75, 1, 5, -0.5])
    for K in (1, 3, 64, 257):
        A = f16(np.repeat(u[:, None], K, axis=1))
        B = f16(np.repeat(v[None, :], K, axis=0))
        C = oracle_lib.gemm(A, B)
        exact = K * np.outer(u, v)          # exact in fp64; rounded once to binary16
        assert np.array_equal(C.view(np.uint16), exact.astype(np.float16).view(np.uint16))


def test_non_square_orientation(oracle_lib):
    # transposed operands or swapped indices change the answer on these shapes
    A = f16([[1, 2, 3], [4, 5, 6]])          # 2 x 3
    B = f16([[1, 0], [0, 2], [1, 1]])        # 3 x 2
    C = oracle_lib.gemm(A, B).astype(np.float64)
    assert np.array_equal(C, np.array([[4, 7], [10, 16]], dtype=np.float64))


def _exact_ref(A, B, bias):
    """C[i,j] as an exact rational, the sum written out term by term."""
    M, K = A.shape
    N = B.shape[1]
    out = np.empty((M, N), dtype=np.float64)
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            for k in range(K):
                s += Fraction(float(A[i, k])) * Fraction(float(B[k, j]))
            if bias is not None:
                s += Fraction(float(bias[j]))
            out[i, j] = float(s)  # exact: the sums here need far fewer than 53 bits
    return out


def test_brute_force_tiny(oracle_lib):
    vals = [-2.0, -1.0, -0.5, 0.0, 0.5, 1.0, 2.0]
    rng = np.random.default_rng(7)
    n_cases = 0
    for M, N, K in itertools.product((1, 2, 3), repeat=3):
        for _ in range(12):
            A = f16(rng.choice(vals, size=(M, K)))
            B = f16(rng.choice(vals, size=(K, N)))
            bias = f16(rng.choice(vals, size=(N,))) if rng.random() < 0.5 else None
            ref = _exact_ref(A, B, bias)
            C = oracle_lib.gemm(A, B, bias).astype(np.float64)
            assert np.array_equal(C, ref), (M, N, K)
            n_cases += 1
    # exhaustive over every 1x1x2 pair of value pairs
    for a0, a1, b0, b1 in itertools.product(vals, repeat=4):
        A = f16([[a0, a1]]); B = f16([[b0], [b1]])
        assert float(oracle_lib.gemm(A, B)[0, 0]) == a0 * b0 + a1 * b1
        n_cases += 1
    assert n_cases > 2000


def test_against_numpy_fp64_matmul(oracle_lib):
    rng = np.random.default_rng(3)
    for M, N, K in [(1, 1, 1), (17, 300, 5), (64, 65, 130), (200, 33, 299), (3, 128, 1024)]:
        A = rand16(rng, (M, K))
        B = rand16(rng, (K, N))
        bias = rand16(rng, (N,), -0.1, 0.1)
        ref64 = A.astype(np.float64) @ B.astype(np.float64) + bias.astype(np.float64)[None, :]
        C, C64 = oracle_lib.gemm(A, B, bias, want_f64=True)
        np.testing.assert_allclose(C64, ref64, rtol=1e-12, atol=1e-12)
        # the output is the fp64 value rounded once to binary16 (numpy's rounding)
        assert np.array_equal(C.view(np.uint16), ref64.astype(np.float16).view(np.uint16))


def test_bias_is_per_column_and_gelu_after_bias(oracle_lib):
    M, K, N = 3, 4, 5
    A = f16(np.zeros((M, K)))
    B = f16(np.ones((K, N)))
    bias = f16([0.5, -1.0, 2.0, 0.0, -3.0])
    C = oracle_lib.gemm(A, B, bias).astype(np.float64)
    assert np.array_equal(C, np.repeat(bias.astype(np.float64)[None, :], M, axis=0))
    # GELU applied to (A@B + bias), not to A@B alone: A@B = 1, bias = -1 -> GELU(0) = 0
    A1 = f16(np.full((2, 1), 1.0)); B1 = f16(np.full((1, 3), 1.0))
    b1 = f16([-1.0, 0.0, 1.0])
    C1, C64 = oracle_lib.gemm(A1, B1, b1, gelu=True, want_f64=True)
    for j, x in enumerate((0.0, 1.0, 2.0)):
        assert C64[0, j] == pytest.approx(x * 0.5 * (1 + math.erf(x / math.sqrt(2))), abs=1e-15)
    assert float(C1[0, 0]) == 0.0
    assert float(C1[0, 1]) == float(f16(0.841344746068543))
    assert float(C1[0, 2]) == float(f16(1.954499736103642))


def test_single_rounding_from_fp64(oracle_lib):
    # 1 + 2^-11 + 2^-30: above the binary16 midpoint 1 + 2^-11, so the single
    # rounding goes up to 1 + 2^-10; rounding through fp32 first would lose
    # 2^-30, land on the tie and go down to 1.
    A = f16([[1.0, 2.0 ** -11, 2.0 ** -15]])
    B = f16([[1.0], [1.0], [2.0 ** -15]])
    assert float(A[0, 2]) == 2.0 ** -15 and float(B[2, 0]) == 2.0 ** -15
    C = oracle_lib.gemm(A, B)
    assert int(C.view(np.uint16)[0, 0]) == 0x3C01


def test_overflow_and_special_values(oracle_lib):
    A = f16([[256.0, 256.0]])
    B = f16([[256.0], [0.0]])
    assert math.isinf(float(oracle_lib.gemm(A, B)[0, 0]))
    A = f16([[np.inf, 1.0]])
    B = f16([[0.0], [1.0]])
    assert math.isnan(float(oracle_lib.gemm(A, B)[0, 0]))   # inf * 0 is NaN


def test_empty_dimensions(oracle_lib):
    bias = f16([0.5, -1.0, 2.0])
    # K = 0: the empty sum is 0, so C = epi(bias)
    A = np.zeros((4, 0), dtype=np.float16)
    B = np.zeros((0, 3), dtype=np.float16)
    C = oracle_lib.gemm(A, B, bias).astype(np.float64)
    assert np.array_equal(C, np.repeat(bias.astype(np.float64)[None, :], 4, axis=0))
    Cg = oracle_lib.gemm(A, B, bias, gelu=True)
    assert float(Cg[0, 0]) == float(f16(0.5 * 0.691462461274013))
    assert oracle_lib.gemm(np.zeros((0, 5), np.float16), np.zeros((5, 3), np.float16)).shape == (0, 3)
    assert oracle_lib.gemm(np.zeros((2, 5), np.float16), np.zeros((5, 0), np.float16)).shape == (2, 0)


def test_rows_and_samples_agree_with_full(oracle_lib):
    rng = np.random.default_rng(11)
    M, N, K = 37, 41, 53
    A = rand16(rng, (M, K)); B = rand16(rng, (K, N)); bias = rand16(rng, (N,), -0.1, 0.1)
    full = oracle_lib.gemm(A, B, bias, gelu=True)
    part = oracle_lib.gemm(A, B, bias, gelu=True, rows=(10, 7))
    assert np.array_equal(part.view(np.uint16), full[10:17].view(np.uint16))
    ii = rng.integers(0, M, 300); jj = rng.integers(0, N, 300)
    s = oracle_lib.gemm_sampled(A, B, bias, True, ii, jj)
    assert np.array_equal(s.view(np.uint16), full[ii, jj].view(np.uint16))


def test_threads_do_not_change_result(oracle_lib):
    rng = np.random.default_rng(5)
    A = rand16(rng, (64, 200)); B = rand16(rng, (200, 96))
    c1 = oracle_lib.gemm(A, B, threads=1)
    c4 = oracle_lib.gemm(A, B, threads=4)
    assert np.array_equal(c1.view(np.uint16), c4.view(np.uint16))


def test_bad_arguments_rejected(oracle_lib):
    with pytest.raises(ValueError):
        oracle_lib.gemm(np.zeros((2, 3), np.float16), np.zeros((4, 2), np.float16))
    with pytest.raises(RuntimeError):
        oracle_lib.gemm_sampled(np.zeros((2, 3), np.float16), np.zeros((3, 2), np.float16), None,
                                False, [2], [0])
