"""Pins of the StreamingLLM oracle: slot formula, full attention before the cache fills,
and equality with full-history attention masked to sinks + recent (a second route)."""

import numpy as np

from oracle import attention as A
from oracle import streaming as S


def test_slot_formula_examples():
    got = [S.slot_of(t, 4, 3) for t in range(10)]
    assert got == [0, 1, 2, 3, 4, 5, 6, 4, 5, 6]
    assert [S.slot_of(t, 0, 3) for t in range(5)] == [0, 1, 2, 0, 1]


def _stream(rng, T, d, G):
    return rng.normal(size=(T, G, d)), rng.normal(size=(T, d)), rng.normal(size=(T, d))


def test_ring_equals_masked_full_history():
    rng = np.random.default_rng(0)
    Sn, R, T, d, G = 4, 7, 40, 8, 2
    qs, K, V = _stream(rng, T, d, G)
    c = S.SinkCache(Sn, R, d)
    for t in range(T):
        c.append(t, K[t], V[t])
        out = c.attend(qs[t], t)
        vis = np.zeros(t + 1, dtype=bool)
        vis[:Sn] = True
        vis[max(0, t - R + 1):] = True
        for g in range(G):
            want = A.attend_masked(qs[t, g], K[:t + 1], V[:t + 1], vis)
            np.testing.assert_allclose(out[g], want, rtol=1e-12)
        if t + 1 <= Sn + R:
            for g in range(G):
                np.testing.assert_allclose(out[g], A.attend(qs[t, g], K[:t + 1], V[:t + 1]),
                                           rtol=1e-12)
        # sinks are never overwritten; the ring holds exactly the last R tokens
        assert c.pos[:min(Sn, t + 1)].tolist() == list(range(min(Sn, t + 1)))
        if t >= Sn + R:
            assert sorted(c.pos[Sn:].tolist()) == list(range(t - R + 1, t + 1))
        assert sorted(S.visible_positions(t, Sn, R).tolist()) == sorted(c.pos[:c.n_live(t)].tolist())


def test_no_sinks_is_plain_window_attention():
    rng = np.random.default_rng(1)
    R, T, d = 5, 20, 8
    qs, K, V = _stream(rng, T, d, 1)
    c = S.SinkCache(0, R, d)
    for t in range(T):
        c.append(t, K[t], V[t])
        lo = max(0, t - R + 1)
        np.testing.assert_allclose(c.attend(qs[t], t)[0], A.attend(qs[t, 0], K[lo:t + 1], V[lo:t + 1]),
                                   rtol=1e-12)
