"""Pins of the H2O oracle: a hand-worked eviction sequence, the no-eviction and
no-heavy-hitter special cases (full attention and sliding-window attention, computed by
a second route over the whole history), and invariants."""

import numpy as np

from conftest import fracs, read_golden
from oracle import attention as A
from oracle import h2o as H


def test_hand_worked_eviction_sequence():
    g = read_golden("h2o_hand.txt")[0]
    L, nh, nr, d = int(g["prompt_len"][0]), int(g["n_heavy"][0]), int(g["n_recent"][0]), 4
    Q = np.zeros((1, L, d))
    K = np.zeros((L, d))
    V = np.arange(L * d, dtype=float).reshape(L, d)
    st = H.prefill(Q, K, V, nh, nr)
    assert sorted(st.pos[st.live()].tolist()) == [int(x) for x in g["prefill_keep"]]
    want = fracs(g["prefill_scores_num"], g["prefill_scores_den"])
    live = st.live()
    order = np.argsort(st.pos[live])
    np.testing.assert_allclose(st.score[live][order], [float(x) for x in want], rtol=1e-14)
    for t, _, evict in g["steps"]:
        q = np.zeros((1, d))
        k = np.zeros(d)
        if t == 4:
            q[0, 0] = 2 * np.log(3.0)
            k[0] = 1.0
        out, ev, _ = H.step(st, q, k, np.full(d, float(t)), t, nr)
        assert ev == evict
    live = st.live()
    order = np.argsort(st.pos[live])
    assert st.pos[live][order].tolist() == [int(x) for x in g["final_scores_pos"]]
    want = fracs(g["final_scores_num"], g["final_scores_den"])
    np.testing.assert_allclose(st.score[live][order], [float(x) for x in want], rtol=1e-14)


def _history(rng, L, steps, d, G):
    Qp = rng.normal(size=(G, L, d))
    K = rng.normal(size=(L + steps, d))
    V = rng.normal(size=(L + steps, d))
    qs = rng.normal(size=(steps, G, d))
    return Qp, K, V, qs


def test_no_eviction_when_budget_covers_everything_equals_full_attention():
    rng = np.random.default_rng(0)
    L, steps, d, G = 12, 10, 8, 2
    Qp, K, V, qs = _history(rng, L, steps, d, G)
    st = H.prefill(Qp, K[:L], V[:L], 20, 5)
    for s in range(steps):
        t = L + s
        out, ev, _ = H.step(st, qs[s], K[t], V[t], t, 5)
        assert ev == -1
        for g in range(G):
            np.testing.assert_allclose(out[g], A.attend(qs[s, g], K[:t + 1], V[:t + 1]),
                                       rtol=1e-12)


def test_zero_heavy_hitters_is_sliding_window_attention():
    rng = np.random.default_rng(1)
    L, steps, d, G, nr = 16, 12, 8, 1, 5
    Qp, K, V, qs = _history(rng, L, steps, d, G)
    st = H.prefill(Qp, K[:L], V[:L], 0, nr)
    for s in range(steps):
        t = L + s
        out, ev, _ = H.step(st, qs[s], K[t], V[t], t, nr)
        assert ev == t - nr
        vis = np.zeros(t + 1, dtype=bool)
        vis[t - nr:] = True
        np.testing.assert_allclose(out[0], A.attend_masked(qs[s, 0], K[:t + 1], V[:t + 1], vis),
                                   rtol=1e-12)


def test_invariants_recent_kept_budget_constant_scores_grow_by_group_size():
    rng = np.random.default_rng(2)
    L, steps, d, G, nh, nr = 40, 30, 8, 3, 6, 4
    Qp, K, V, qs = _history(rng, L, steps, d, G)
    st = H.prefill(Qp, K[:L], V[:L], nh, nr)
    assert len(st.live()) == nh + nr
    for s in range(steps):
        t = L + s
        before = st.score.copy()
        f = st.free_slot
        out, ev, cand = H.step(st, qs[s], K[t], V[t], t, nr)
        gained = st.score - before
        gained[f] = st.score[f]
        assert abs(gained.sum() - G) < 1e-12
        live_pos = set(st.pos[st.live()].tolist())
        assert set(range(t - nr + 1, t + 1)) <= live_pos
        assert len(live_pos) == nh + nr
        assert ev <= t - nr
        assert ev not in live_pos
        # the victim had the smallest score among the evictable entries
        assert min(c[2] for c in cand) == [c[2] for c in cand if c[1] == ev][0]


def test_exact_score_tie_evicts_the_higher_position():
    d = 4
    Q = np.zeros((1, 4, d))
    K = np.zeros((4, d))
    V = np.zeros((4, d))
    st = H.prefill(Q, K, V, 2, 1)
    # prompt scores with q = 0: [25/12, 13/12, 7/12, 1/4]; kept: top-2 of {0, 1, 2} ->
    # 0, 1, plus the recent position 3.  Set all three scores equal.
    live = st.live()
    st.score[live] = 1.0
    out, ev, cand = H.step(st, np.zeros((1, d)), np.zeros(d), np.zeros(d), 4, 1)
    # uniform 1/4 added to all four live entries: 0, 1, 3 tie at 5/4; evictable are
    # positions <= 3 -> {0, 1, 3}; the higher position (3) is evicted.
    assert ev == 3
