"""Pins of the oracle's softmax attention against closed forms and invariants."""

import numpy as np
import pytest

from oracle import attention as A


def test_single_key_returns_its_value():
    rng = np.random.default_rng(0)
    q, k, v = rng.normal(size=4), rng.normal(size=(1, 4)), rng.normal(size=(1, 4))
    assert np.array_equal(A.attend(q, k, v), v[0])


def test_zero_query_is_the_mean_of_values():
    rng = np.random.default_rng(1)
    K, V = rng.normal(size=(7, 8)), rng.normal(size=(7, 8))
    np.testing.assert_allclose(A.attend(np.zeros(8), K, V), V.mean(axis=0), rtol=0, atol=1e-15)


def test_two_keys_closed_form_scale_is_inverse_sqrt_d():
    # d = 4 so the scale is 1/2; logits 0 and ln 3 -> weights 1/4 and 3/4.
    q = np.array([2 * np.log(3.0), 0, 0, 0])
    K = np.array([[0.0, 5, -1, 2], [1.0, 5, -1, 2]]) * np.array([1, 0, 0, 0])
    V = np.array([[4.0, 0, 0, 0], [0.0, 8, 0, 0]])
    np.testing.assert_allclose(A.attention_weights(q, K), [0.25, 0.75], rtol=1e-15)
    np.testing.assert_allclose(A.attend(q, K, V), [1.0, 6.0, 0, 0], rtol=1e-15, atol=1e-15)


def test_permuting_cached_entries_does_not_change_output():
    rng = np.random.default_rng(2)
    q, K, V = rng.normal(size=16), rng.normal(size=(33, 16)), rng.normal(size=(33, 16))
    perm = rng.permutation(33)
    np.testing.assert_allclose(A.attend(q, K[perm], V[perm]), A.attend(q, K, V), rtol=1e-13)


def test_logit_shift_invariance_and_large_logits():
    # Adding the same logit to every key changes nothing, even when the logits are far
    # beyond exp's range (the max-subtraction keeps it finite).
    rng = np.random.default_rng(3)
    q = rng.normal(size=8)
    K, V = rng.normal(size=(9, 8)), rng.normal(size=(9, 8))
    shift = 1000.0 * q / (q @ q) * np.sqrt(8)  # q . shift / sqrt(8) = 1000 for every key
    np.testing.assert_allclose(A.attend(q, K + shift, V), A.attend(q, K, V), rtol=1e-10)


def test_masked_route_equals_subset_route():
    rng = np.random.default_rng(4)
    q, K, V = rng.normal(size=8), rng.normal(size=(20, 8)), rng.normal(size=(20, 8))
    vis = rng.random(20) < 0.4
    vis[3] = True
    np.testing.assert_allclose(A.attend_masked(q, K, V, vis), A.attend(q, K[vis], V[vis]),
                               rtol=1e-13)


def test_group_attention_is_per_head():
    rng = np.random.default_rng(5)
    qs, K, V = rng.normal(size=(4, 8)), rng.normal(size=(10, 8)), rng.normal(size=(10, 8))
    out = A.attend_group(qs, K, V)
    for g in range(4):
        np.testing.assert_allclose(out[g], A.attend(qs[g], K, V), rtol=1e-15)


def test_causal_prefill_closed_forms_and_second_route():
    rng = np.random.default_rng(5)
    L, d = 23, 8
    Q, K, V = rng.standard_normal((3, L, d))
    O = A.causal_prefill(Q, K, V)
    # row 0 sees only key 0
    np.testing.assert_allclose(O[0], V[0], rtol=0, atol=1e-15)
    # identical keys: uniform weights, so row i is the running mean of V[0..i]
    Kc = np.tile(K[0], (L, 1))
    cum = np.cumsum(V, axis=0) / np.arange(1, L + 1)[:, None]
    np.testing.assert_allclose(A.causal_prefill(Q, Kc, V), cum, rtol=1e-12, atol=1e-13)
    # keys and values after row i do not reach row i
    K2, V2 = K.copy(), V.copy()
    K2[12:] += 5.0
    V2[12:] -= 3.0
    np.testing.assert_array_equal(A.causal_prefill(Q, K2, V2)[:12], O[:12])
    # a second route: full attention with the future masked to -inf
    for i in (0, 7, L - 1):
        vis = np.arange(L) <= i
        np.testing.assert_allclose(O[i], A.attend_masked(Q[i], K, V, vis), rtol=1e-12, atol=1e-14)


def test_log_sum_exp_hand_worked_rows():
    # d = 4 (scale 1/2), q = (2, 0, 0, 0) and k_j = (x_j, ...) give logits x_j:
    # x = (0, ln 2, ln 5) -> row 0: ln 1, row 1: ln (1 + 2) = ln 3, row 2: ln (1 + 2 + 5) = ln 8.
    x = np.array([0.0, np.log(2.0), np.log(5.0)])
    Q = np.tile(np.array([2.0, 0, 0, 0]), (3, 1))
    K = np.zeros((3, 4))
    K[:, 0] = x
    K[:, 1:] = 7.0  # orthogonal to q: no effect
    np.testing.assert_allclose(A.causal_lse(Q, K), np.log([1.0, 3.0, 8.0]), rtol=0, atol=1e-15)


def test_lse_of_zero_queries_is_log_of_row_length():
    rng = np.random.default_rng(11)
    K = rng.normal(size=(9, 8)) * 5
    np.testing.assert_allclose(A.causal_lse(np.zeros((9, 8)), K), np.log(np.arange(1, 10)),
                               rtol=0, atol=1e-14)


def test_lse_normalises_the_attention_weights_and_matches_scipy():
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(12)
    L, d = 40, 16
    Q, K = rng.normal(size=(L, d)) * 3, rng.normal(size=(L, d)) * 3
    lse = A.causal_lse(Q, K)
    for i in (0, 1, 17, L - 1):
        logits = K[: i + 1] @ Q[i] / np.sqrt(d)
        np.testing.assert_allclose(np.exp(logits - lse[i]), A.attention_weights(Q[i], K[: i + 1]),
                                   rtol=1e-12)
        np.testing.assert_allclose(lse[i], scipy_special.logsumexp(logits), rtol=1e-14)
    # -inf logits add nothing; huge logits stay finite
    assert A.log_sum_exp([-np.inf, 0.0]) == 0.0
    np.testing.assert_allclose(A.log_sum_exp([1000.0, 1000.0]), 1000.0 + np.log(2.0), rtol=1e-15)
