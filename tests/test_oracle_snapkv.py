"""Pins of the SnapKV oracle: votes, pooling, top-k and selection.

Each pin is something other than the oracle's own code: hand-worked examples
(tests/golden), closed forms (harmonic sums for uniform attention), invariants
(every softmax row sums to 1) and brute force over all subsets on tiny inputs.
"""

import itertools
from fractions import Fraction

import numpy as np
import pytest

from conftest import fracs, read_golden
from oracle import attention as A
from oracle import snapkv as S


def test_votes_hand_worked_example():
    g = read_golden("votes_hand.txt")[0]
    d, L, W = int(g["d"][0]), int(g["prompt_len"][0]), int(g["window"][0])
    qs = [[float(x) for x in row[1:]] for row in g["_all"]["q"]]
    assert [int(row[0]) for row in g["_all"]["q"]] == list(range(W))
    q = np.array(qs)[None]
    K = np.zeros((L, d))
    K[:, 0] = np.log([float(x) for x in g["key_logs"]])
    want = fracs(g["votes_num"], g["votes_den"])
    got = S.window_votes(q, K)
    np.testing.assert_allclose(got, [float(x) for x in want], rtol=1e-14)


@pytest.mark.parametrize("G,Wq,L", [(1, 4, 9), (3, 5, 12), (2, 12, 12)])
def test_votes_zero_query_harmonic_closed_form(G, Wq, L):
    # q = 0: row at position p spreads 1/(p+1) over keys 0..p.
    votes = S.window_votes(np.zeros((G, Wq, 6)), np.random.default_rng(0).normal(size=(L, 6)))
    want = [sum(Fraction(G, p + 1) for p in range(L - Wq, L) if p >= j) for j in range(L)]
    np.testing.assert_allclose(votes, [float(x) for x in want], rtol=1e-14)


def test_votes_sum_to_number_of_rows_and_are_additive_over_heads():
    rng = np.random.default_rng(1)
    q, K = rng.normal(size=(3, 7, 16)), rng.normal(size=(40, 16)) * 2
    v = S.window_votes(q, K)
    assert abs(v.sum() - 21) < 1e-12
    parts = sum(S.window_votes(q[g:g + 1], K) for g in range(3))
    np.testing.assert_allclose(v, parts, rtol=1e-13)
    assert (v >= 0).all()


def test_votes_window_causality():
    # Keys inside the window are seen only by window rows at or after them: the last
    # key gets its whole vote from the last window row.
    rng = np.random.default_rng(2)
    q, K = rng.normal(size=(1, 4, 8)), rng.normal(size=(10, 8))
    v = S.window_votes(q, K)
    p_last = A.attention_weights(q[0, 3], K)
    assert abs(v[9] - p_last[9]) < 1e-15


def _golden_pool_cases():
    return read_golden("pool_topk_hand.txt")


@pytest.mark.parametrize("case", _golden_pool_cases(), ids=lambda c: c["name"])
def test_pool_and_topk_hand_examples(case):
    v = np.array([float(x) for x in case["v"]])
    u = S.max_pool_1d(v, int(case["kernel"][0]))
    np.testing.assert_array_equal(u, [float(x) for x in case["u"]])
    keep = S.top_k_lowest_index(u, int(case["k"][0]))
    np.testing.assert_array_equal(keep, [int(x) for x in case["keep"]])


def test_pool_kernel_one_is_identity_and_huge_kernel_is_global_max():
    rng = np.random.default_rng(3)
    v = rng.random(11)
    np.testing.assert_array_equal(S.max_pool_1d(v, 1), v)
    np.testing.assert_array_equal(S.max_pool_1d(v, 21), np.full(11, v.max()))
    with pytest.raises(ValueError):
        S.max_pool_1d(v, 4)


def test_topk_brute_force_all_subsets_with_ties():
    # For every small vector with heavy ties, the returned set is the unique k-subset
    # whose every member precedes every non-member in the order (larger u first,
    # then lower position).
    rng = np.random.default_rng(4)
    for trial in range(300):
        n = int(rng.integers(1, 8))
        u = rng.integers(0, 3, size=n).astype(float)
        k = int(rng.integers(0, n + 1))

        def before(a, b):
            return u[a] > u[b] or (u[a] == u[b] and a < b)

        valid = [set(c) for c in itertools.combinations(range(n), k)
                 if all(before(a, b) for a in c for b in range(n) if b not in c)]
        assert len(valid) == 1
        got = S.top_k_lowest_index(u, k)
        assert set(got.tolist()) == valid[0]
        assert list(got) == sorted(got)


def test_select_positions_window_budget_and_identity():
    rng = np.random.default_rng(5)
    votes = rng.random(100)
    pos = S.select_positions(votes, 100, 8, 7, 30)
    assert len(pos) == 30
    assert list(pos[-8:]) == list(range(92, 100))
    assert list(pos[:22]) == sorted(pos[:22]) and pos[21] < 92
    assert list(S.select_positions(votes, 100, 8, 7, 100)) == list(range(100))
    assert list(S.select_positions(votes, 100, 8, 7, 500)) == list(range(100))
    assert list(S.select_positions(votes, 6, 8, 7, 3)) == list(range(6))
    assert list(S.select_positions(votes, 100, 8, 7, 8)) == list(range(92, 100))
    with pytest.raises(ValueError):
        S.select_positions(votes, 100, 8, 7, 7)


def test_budget_at_least_prompt_reproduces_full_attention_exactly():
    rng = np.random.default_rng(6)
    L, d = 48, 16
    q_win = rng.normal(size=(2, 8, d))
    K, V = rng.normal(size=(L, d)), rng.normal(size=(L, d))
    pos, Kc, Vc, _ = S.compress_unit(q_win, K, V, 8, 7, L)
    q = rng.normal(size=d)
    assert np.array_equal(A.attend(q, Kc, Vc), A.attend(q, K, V))


def test_group_mapping_query_head_to_kv_head():
    # Hq = 4, Hkv = 2: query heads 2, 3 belong to KV head 1.  A query that aims at a
    # planted key is placed only in head 3; that key must win the vote of KV head 1.
    rng = np.random.default_rng(7)
    B, Hq, Hkv, L, W, d = 1, 4, 2, 64, 4, 16
    Q = rng.normal(size=(B, Hq, W, d)) * 0.1
    K = rng.normal(size=(B, Hkv, L, d)) * 0.1
    V = rng.normal(size=(B, Hkv, L, d))
    aim = rng.normal(size=d)
    Q[0, 3] += 4 * aim
    K[0, 1, 17] += 4 * aim
    res = S.compress(Q, K, V, W, 1, W + 1)
    pos1, _, _, votes1 = res[0][1]
    assert pos1[0] == 17 and votes1[:L - W].argmax() == 17
    pos0, _, _, votes0 = res[0][0]
    assert votes0[17] < 0.5 * votes1[17]


def test_avg_pool_hand_examples():
    # a single spike spreads evenly over the kernel; at the edges the divisor stays P
    v = np.array([0, 0, 0, 7, 0, 0, 0, 0, 0], dtype=float)
    np.testing.assert_allclose(S.avg_pool_1d(v, 3), [0, 0, 7 / 3, 7 / 3, 7 / 3, 0, 0, 0, 0],
                               rtol=0, atol=1e-15)
    np.testing.assert_allclose(S.avg_pool_1d(np.ones(5), 3), [2 / 3, 1, 1, 1, 2 / 3],
                               rtol=0, atol=1e-15)
    np.testing.assert_array_equal(S.avg_pool_1d(v, 1), v)
    with pytest.raises(ValueError):
        S.avg_pool_1d(v, 2)


@pytest.mark.parametrize("kernel", [1, 3, 7, 9])
def test_avg_pool_is_a_same_length_box_convolution(kernel):
    # zero-padded moving average == numpy's 'same' convolution with a box of 1/P
    rng = np.random.default_rng(kernel)
    v = rng.random(40)
    ref = np.convolve(v, np.full(kernel, 1.0 / kernel), mode="same")
    np.testing.assert_allclose(S.avg_pool_1d(v, kernel), ref, rtol=1e-14, atol=1e-15)


def test_select_positions_with_average_pooling():
    # 12 candidates + a window of 2, one pick: an isolated spike wins under max pooling,
    # the centre of a dense cluster under average pooling
    votes = np.zeros(14)
    votes[2] = 1.0                       # spike
    votes[7:10] = [0.6, 0.6, 0.6]        # cluster
    u = S.avg_pool_1d(votes[:12], 3)
    assert u[8] == pytest.approx(0.6) and u[2] == pytest.approx(1 / 3) and u[7] == pytest.approx(0.4)
    assert list(S.select_positions(votes, 14, 2, 3, 3, pool="max")) == [1, 12, 13]
    assert list(S.select_positions(votes, 14, 2, 3, 3, pool="avg")) == [8, 12, 13]
    with pytest.raises(ValueError):
        S.select_positions(votes, 14, 2, 3, 3, pool="median")


def test_votes_from_true_lse_equal_window_votes():
    # A second route to steps 1-2: with each row's own log-sum-exp the terms are the rows'
    # softmax weights (GQA group of 3, window 5, prefix 12).
    rng = np.random.default_rng(21)
    G, Wq, L, d = 3, 5, 17, 8
    q_unit = rng.normal(size=(G, Wq, d)) * 2
    K = rng.normal(size=(L, d)) * 2
    lse = np.full((G, L), np.nan)
    for g in range(G):
        Qfull = np.zeros((L, d))
        Qfull[L - Wq:] = q_unit[g]
        lse[g, L - Wq:] = A.causal_lse(Qfull, K)[L - Wq:]
    np.testing.assert_allclose(S.votes_from_lse(q_unit, K, lse), S.window_votes(q_unit, K),
                               rtol=1e-13)


def test_votes_from_shifted_lse_scale_per_row():
    # lse + c on one row scales that row's contribution by e^-c; a non-finite lse drops it.
    rng = np.random.default_rng(22)
    G, Wq, L, d = 2, 3, 9, 4
    q_unit = rng.normal(size=(G, Wq, d))
    K = rng.normal(size=(L, d))
    lse = rng.normal(size=(G, L))
    base = S.votes_from_lse(q_unit, K, lse)
    one_row = np.zeros((G, Wq, d))
    one_row[1, 2] = q_unit[1, 2]
    masked = np.full((G, L), -np.inf)
    masked[1, L - 1] = lse[1, L - 1]
    row_only = S.votes_from_lse(one_row, K, masked)
    assert np.all(row_only > 0)                # only row (1, 2) at position L-1 adds
    shifted = lse.copy()
    shifted[1, L - 1] += np.log(4.0)
    np.testing.assert_allclose(S.votes_from_lse(q_unit, K, shifted), base - 0.75 * row_only,
                               rtol=1e-12)
    dropped = lse.copy()
    dropped[1, L - 1] = np.inf
    np.testing.assert_allclose(S.votes_from_lse(q_unit, K, dropped), base - row_only, rtol=1e-12,
                               atol=1e-15)
