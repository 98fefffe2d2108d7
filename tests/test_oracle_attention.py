"""Pins for the oracle's attention forward (S = Q K^T / sqrt(d), row softmax,
O = P V, optional causal mask), against closed forms, invariants and an
independent library softmax, none of which reuse the oracle's code."""
import math

import numpy as np
import pytest


def f16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16)


def rand_qkv(seed, B, S, H, D, scale=1.0):
    rng = np.random.default_rng(seed)
    return [f16(scale * rng.standard_normal((B, S, H, D))) for _ in range(3)]


def test_equal_scores_average_the_visible_values(oracle_lib):
    # every key identical -> every visible score equal -> O is the plain mean of the visible V rows
    B, S, H, D = 2, 9, 3, 8
    Q, _, V = rand_qkv(1, B, S, H, D)
    K = np.broadcast_to(f16(np.linspace(-1, 1, D)), (B, S, H, D)).copy()
    v = V.astype(np.float64)
    for causal in (False, True):
        _, O64 = oracle_lib.attention(Q, K, V, causal=causal, want_f64=True)
        for s in range(S):
            n = s + 1 if causal else S
            np.testing.assert_allclose(O64[:, s], v[:, :n].mean(axis=1), rtol=1e-12, atol=1e-12)


def test_dominant_key_selects_its_value_even_for_huge_scores(oracle_lib):
    # scores of order 1e4 overflow exp() unless the row maximum is taken out first
    B, S, H, D = 1, 6, 2, 4
    Q = np.zeros((B, S, H, D)); K = np.zeros((B, S, H, D))
    Q[..., 0] = 200.0
    K[:, 3, :, 0] = 200.0      # key 3 scores 200*200/2 = 2e4, every other key 0
    V = f16(np.random.default_rng(2).standard_normal((B, S, H, D)))
    O, O64 = oracle_lib.attention(f16(Q), f16(K), V, want_f64=True)
    assert np.isfinite(O64).all()
    for s in range(S):
        np.testing.assert_array_equal(O64[:, s], V[:, 3].astype(np.float64))


def test_causal_first_query_sees_only_the_first_key(oracle_lib):
    Q, K, V = rand_qkv(3, 2, 7, 2, 16)
    O = oracle_lib.attention(Q, K, V, causal=True)
    np.testing.assert_array_equal(O[:, 0].view(np.uint16), V[:, 0].view(np.uint16))


def test_causal_row_is_attention_over_its_prefix(oracle_lib):
    B, S, H, D = 1, 8, 2, 8
    Q, K, V = rand_qkv(4, B, S, H, D)
    _, full = oracle_lib.attention(Q, K, V, causal=True, want_f64=True)
    for s in range(S):
        _, pre = oracle_lib.attention(Q[:, :s + 1], K[:, :s + 1], V[:, :s + 1], causal=False, want_f64=True)
        np.testing.assert_allclose(full[:, s], pre[:, s], rtol=1e-13, atol=1e-15)


def test_non_causal_is_invariant_to_key_order(oracle_lib):
    B, S, H, D = 1, 11, 2, 8
    Q, K, V = rand_qkv(5, B, S, H, D)
    perm = np.random.default_rng(6).permutation(S)
    _, a = oracle_lib.attention(Q, K, V, want_f64=True)
    _, b = oracle_lib.attention(Q, K[:, perm], V[:, perm], want_f64=True)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-15)


def test_two_keys_follow_the_logistic_closed_form(oracle_lib):
    for D in (4, 16, 64):
        _two_keys(oracle_lib, D)


def _two_keys(oracle_lib, D):
    # two keys: p0 = 1 / (1 + exp(-(s0 - s1))) with s = q.k / sqrt(D) (pins the scale)
    q = np.zeros(D); q[0] = 1.5
    k0 = np.zeros(D); k0[0] = 2.0
    k1 = np.zeros(D); k1[0] = -1.0
    Q = f16(q[None, None, None, :].repeat(2, axis=1))
    K = f16(np.stack([k0, k1])[None, :, None, :])
    V = f16(np.array([[1.0] * D, [-3.0] * D])[None, :, None, :])
    _, O64 = oracle_lib.attention(Q, K, V, want_f64=True)
    ds = (1.5 * 2.0 - 1.5 * -1.0) / math.sqrt(D)
    p0 = 1.0 / (1.0 + math.exp(-ds))
    np.testing.assert_allclose(O64[0, 0, 0], p0 * 1.0 + (1 - p0) * -3.0, rtol=1e-14)


def test_matches_a_library_softmax(oracle_lib):
    scipy_special = pytest.importorskip("scipy.special")
    for seed, (B, S, H, D) in enumerate([(1, 33, 2, 16), (2, 17, 3, 64), (1, 64, 1, 128)]):
        Q, K, V = rand_qkv(10 + seed, B, S, H, D)
        for causal in (False, True):
            _, O64 = oracle_lib.attention(Q, K, V, causal=causal, want_f64=True)
            s = np.einsum("bshd,bthd->bhst", Q.astype(np.float64), K.astype(np.float64)) / np.sqrt(D)
            if causal:
                s = np.where(np.tril(np.ones((S, S), dtype=bool)), s, -np.inf)
            o = np.einsum("bhst,bthd->bshd", scipy_special.softmax(s, axis=-1), V.astype(np.float64))
            np.testing.assert_allclose(O64, o, rtol=1e-11, atol=1e-12)


def test_selected_rows_match_the_full_result(oracle_lib):
    B, S, H, D = 2, 10, 3, 8
    Q, K, V = rand_qkv(7, B, S, H, D)
    full = oracle_lib.attention(Q, K, V, causal=True)
    rows = np.array([0, 5, 31, B * S * H - 1])
    part = oracle_lib.attention(Q, K, V, causal=True, rows=rows)
    flat = full.reshape(-1, D)
    np.testing.assert_array_equal(part.view(np.uint16), flat[rows].view(np.uint16))


def test_bad_shapes_rejected(oracle_lib):
    Q, K, V = rand_qkv(8, 1, 4, 1, 8)
    with pytest.raises(ValueError):
        oracle_lib.attention(Q, K[:, :3], V)
    with pytest.raises(RuntimeError):
        oracle_lib.attention(Q, K, V, rows=[4])
