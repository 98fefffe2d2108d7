"""Pins for the oracle's weight-only 4-bit GEMM: nibble decoding against
numpy's two's-complement int8 shifts, dequantisation against numpy's fp64
product rounded by numpy, hand-packed bytes, per-group scale indexing, a
rank-1 closed form, and agreement with the (separately pinned) fp16 GEMM on
the dequantised weights."""
import numpy as np
import pytest


def f16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16)


def pack(q):
    """q (K x N ints in [-8, 7]) -> N x K/2 bytes, low nibble = even k."""
    u = (np.asarray(q, dtype=np.int64).T & 0xF).astype(np.uint8)
    return np.ascontiguousarray(u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)


def test_int4_decode_exhaustive(oracle_lib):
    for b in range(256):
        lo = int(np.right_shift(np.array((b << 4) & 0xFF, dtype=np.uint8).view(np.int8), 4))
        hi = int(np.right_shift(np.array(b, dtype=np.uint8).view(np.int8), 4))
        assert oracle_lib.int4_value(b, False) == lo, b
        assert oracle_lib.int4_value(b, True) == hi, b


def test_hand_packed_bytes(oracle_lib):
    # column n=0: 0x21 -> k0=1, k1=2; 0xF8 -> k2=-8, k3=-1
    # column n=1: 0x7F -> k0=-1, k1=7; 0x80 -> k2=0, k3=-8
    Bq = np.array([[0x21, 0xF8], [0x7F, 0x80]], dtype=np.uint8)
    s = f16([[1.0, 0.5]])
    W = oracle_lib.dequant_w4(Bq, s, group=128).astype(np.float64)
    assert np.array_equal(W, [[1.0, -0.5], [2.0, 3.5], [-8.0, 0.0], [-1.0, -4.0]])


def test_dequant_matches_numpy_rounding(oracle_lib):
    rng = np.random.default_rng(0)
    K, N, G = 300, 64, 128
    q = rng.integers(-8, 8, size=(K, N))
    s = f16(rng.uniform(-0.05, 0.05, size=((K + G - 1) // G, N)))
    W = oracle_lib.dequant_w4(pack(q), s, group=G)
    ref = (q.astype(np.float64) * s.astype(np.float64)[np.arange(K) // G, :]).astype(np.float16)
    assert np.array_equal(W.view(np.uint16), ref.view(np.uint16))


def test_group_boundaries(oracle_lib):
    K, N, G = 256, 4, 128
    q = np.ones((K, N), dtype=np.int64)
    s = f16([[1.0] * N, [4.0] * N])
    W = oracle_lib.dequant_w4(pack(q), s, group=G).astype(np.float64)
    assert np.all(W[:128] == 1.0) and np.all(W[128:] == 4.0)


def test_rank1_closed_form(oracle_lib):
    # A rows constant u_i, all weights q = 3 with scale 2^-3: C[i,j] = K * u_i * 3/8
    K, N, M = 512, 32, 5
    u = np.array([1.0, -2.0, 0.5, 4.0, -0.25])
    A = f16(np.repeat(u[:, None], K, axis=1))
    Bq = pack(np.full((K, N), 3))
    s = f16(np.full((K // 128, N), 0.125))
    C = oracle_lib.gemm_w4(A, Bq, s, group=128)
    assert np.array_equal(C.view(np.uint16), (K * 3 * 0.125 * np.outer(u, np.ones(N))).astype(np.float16).view(np.uint16))


def test_agrees_with_fp16_gemm_on_dequantised_weights(oracle_lib):
    rng = np.random.default_rng(2)
    M, K, N = 7, 384, 48
    A = f16(rng.uniform(-1, 1, size=(M, K)))
    q = rng.integers(-8, 8, size=(K, N))
    s = f16(rng.uniform(0.002, 0.006, size=(K // 128, N)))
    bias = f16(rng.uniform(-0.1, 0.1, size=N))
    W = oracle_lib.dequant_w4(pack(q), s)
    for gelu in (False, True):
        got = oracle_lib.gemm_w4(A, pack(q), s, bias, gelu=gelu)
        ref = oracle_lib.gemm(A, W, bias, gelu=gelu)
        assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))
    # and the product itself against numpy in fp64 on the numpy-dequantised weights
    W64 = q.astype(np.float64) * s.astype(np.float64)[np.arange(K) // 128, :]
    _, C64 = oracle_lib.gemm_w4(A, pack(q), s, want_f64=True)
    np.testing.assert_allclose(C64, A.astype(np.float64) @ W64.astype(np.float16).astype(np.float64), rtol=1e-12,
                               atol=1e-12)


def test_bad_shapes_rejected(oracle_lib):
    with pytest.raises(ValueError):
        oracle_lib.gemm_w4(f16(np.zeros((2, 128))), np.zeros((16, 32), np.uint8), f16(np.zeros((1, 16))))


# ---------------------------------------------------------------- FP4 (E2M1) weights

def _e2m1_table():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "e2m1_values.txt")
    vals = {}
    for line in open(path):
        line = line.split("#")[0].strip()
        if line:
            code, v = line.split()
            vals[int(code, 16)] = float(v)
    assert sorted(vals) == list(range(16))
    return vals


def test_e2m1_decode_exhaustive_against_the_table(oracle_lib):
    table = _e2m1_table()
    for b in range(256):
        lo, hi = oracle_lib.e2m1_value(b, False), oracle_lib.e2m1_value(b, True)
        assert lo == table[b & 0xF] and np.signbit(lo) == np.signbit(table[b & 0xF]), (b, lo)
        assert hi == table[b >> 4] and np.signbit(hi) == np.signbit(table[b >> 4]), (b, hi)


def test_e2m1_invariants(oracle_lib):
    mags = [oracle_lib.e2m1_value(c, False) for c in range(8)]
    assert all(a < b for a, b in zip(mags, mags[1:]))          # codes 0..7 ordered by magnitude
    for c in range(8):
        assert oracle_lib.e2m1_value(c | 8, False) == -mags[c]  # bit 3 is the sign
        assert float(np.float16(mags[c])) == mags[c]           # every value exact in binary16
    # consecutive codes of one binade differ by half a unit of that binade
    assert [mags[3] - mags[2], mags[5] - mags[4], mags[7] - mags[6]] == [0.5, 1.0, 2.0]


def test_fp4_hand_packed_bytes(oracle_lib):
    # column n=0: 0x72 -> k0 = code 2 (1.0), k1 = code 7 (6.0); 0x9F -> k2 = -6.0, k3 = -0.5
    # column n=1: 0x0B -> k0 = -1.5, k1 = 0.0;  0x45 -> k2 = 3.0,  k3 = 2.0
    Bq = np.array([[0x72, 0x9F], [0x0B, 0x45]], dtype=np.uint8)
    s = f16([[1.0, 0.25]])
    W = oracle_lib.dequant_w4(Bq, s, group=128, fmt=1).astype(np.float64)
    assert np.array_equal(W, [[1.0, -0.375], [6.0, 0.0], [-6.0, 0.75], [-0.5, 0.5]])


def _pack_codes(codes):
    """codes (K x N ints in 0..15) -> N x K/2 bytes, low nibble = even k."""
    u = np.asarray(codes, dtype=np.uint8).T
    return np.ascontiguousarray(u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)


def test_fp4_dequant_matches_numpy_rounding(oracle_lib):
    table = _e2m1_table()
    rng = np.random.default_rng(5)
    K, N, G = 384, 40, 128
    codes = rng.integers(0, 16, size=(K, N))
    s = f16(rng.uniform(0.001, 3.0, size=(K // G, N)))
    W = oracle_lib.dequant_w4(_pack_codes(codes), s, group=G, fmt=1)
    vals = np.vectorize(table.get)(codes).astype(np.float64)
    ref = (vals * np.repeat(s.astype(np.float64), G, axis=0)).astype(np.float16)  # numpy's rounding
    assert np.array_equal(W.view(np.uint16), ref.view(np.uint16))


def test_fp4_gemm_matches_numpy(oracle_lib):
    table = _e2m1_table()
    rng = np.random.default_rng(6)
    M, K, N, G = 7, 256, 24, 128
    A = f16(rng.standard_normal((M, K)))
    codes = rng.integers(0, 16, size=(K, N))
    s = f16(rng.uniform(0.01, 0.1, size=(K // G, N)))
    bias = f16(rng.standard_normal(N) * 0.1)
    W = (np.vectorize(table.get)(codes) * np.repeat(s.astype(np.float64), G, axis=0)).astype(np.float16)
    ref = (A.astype(np.float64) @ W.astype(np.float64) + bias.astype(np.float64)).astype(np.float16)
    got = oracle_lib.gemm_w4(A, _pack_codes(codes), s, bias, fmt=1)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))
