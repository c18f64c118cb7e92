"""H2O heavy-hitter + recent-window KV eviction in fp64 (oracle; test infrastructure only).

Follows the H2O article (abeam.tech, 2026-06-24):

* 用語解説 "attention score" / "heavy hitter": a token's importance is the attention it
  has received, summed over the steps so far (a local statistic, only past steps);
* 何を残すのか ("what is kept"): heavy hitters (largest cumulative score) and the
  recent tokens;
* 処理の流れ ("processing flow"): at every decode step the new query's attention over
  the cache updates each cached token's cumulative score; when the cache would exceed
  its budget, everything except the heavy hitters and the recent window is evicted.

Readings taken where the article is silent (it gives no formulas): the cumulative score
starts from the causal column sums of the prompt's own attention; the prompt is cut
to the top ``n_heavy`` scores before the last ``n_recent`` positions plus those
``n_recent`` positions; each step appends the new token, attends over every live
entry (the new one included), adds each entry's probability (summed over the G query
heads of a KV head) to its score, and when the live count exceeds
``n_heavy + n_recent`` evicts one entry: the smallest score among positions
<= t - n_recent, the higher position on exact ties.
"""

import numpy as np

from .attention import attention_weights
from .snapkv import select_positions, window_votes


class H2OState:
    """Cache of one KV head: ``slots = n_heavy + n_recent + 1`` rows.

    ``n_used`` rows hold live tokens after a step; ``free_slot`` is where the next
    token goes.  Until the cache has filled, live rows are 0..n_used-1 and
    free_slot == n_used.
    """

    def __init__(self, slots, d):
        self.slots = slots
        self.k = np.zeros((slots, d))
        self.v = np.zeros((slots, d))
        self.score = np.zeros(slots)
        self.pos = np.full(slots, -1, dtype=np.int64)
        self.n_used = 0
        self.free_slot = 0

    def live(self):
        """Slots holding a token: every occupied slot except the free one."""
        return np.array([s for s in range(self.slots)
                         if self.pos[s] >= 0 and s != self.free_slot], dtype=np.int64)


def prefill(q_unit, K, V, n_heavy, n_recent):
    """Initial H2O cache of one KV head from the prompt.

    q_unit [G, L, d] are all prompt queries of the group; K, V [L, d].  The initial
    cumulative score of position j is the causal column sum of the prompt attention
    (``window_votes`` with every prompt row as a query).  Kept: top ``n_heavy`` scores
    among positions < L - n_recent (lower position first on ties) plus the last
    ``n_recent`` positions, or everything when L <= n_heavy + n_recent.
    """
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    L, d = K.shape
    scores = window_votes(q_unit, K)
    keep = select_positions(scores, L, n_recent, 1, n_heavy + n_recent)
    st = H2OState(n_heavy + n_recent + 1, d)
    n = keep.shape[0]
    st.k[:n] = K[keep]
    st.v[:n] = V[keep]
    st.score[:n] = scores[keep]
    st.pos[:n] = keep
    st.n_used = n
    st.free_slot = n
    return st


def step(st, qs, k_new, v_new, t, n_recent, evict_override=None):
    """One decode step at position t for one KV head; mutates ``st``.

    qs [G, d] are the G query heads of the group.  Returns (out [G, d], evicted
    position or -1, the eviction candidates as (slot, pos, score) tuples).

    ``evict_override`` (a slot) lets a lockstep test follow an equally valid eviction
    (an exact or within-tolerance tie) chosen elsewhere; the test first checks that it
    is a valid choice.
    """
    qs = np.asarray(qs, dtype=np.float64)
    f = st.free_slot
    st.k[f] = np.asarray(k_new, dtype=np.float64)
    st.v[f] = np.asarray(v_new, dtype=np.float64)
    st.pos[f] = t
    st.score[f] = 0.0
    # every occupied slot is live during the step, the new token included
    live = np.array([s for s in range(st.slots) if st.pos[s] >= 0], dtype=np.int64)
    count = live.shape[0]
    outs = []
    added = np.zeros(st.slots)
    for q in qs:
        p = attention_weights(q, st.k[live])
        outs.append(p @ st.v[live])
        added[live] += p
    st.score += added
    if count == st.slots:
        cand = [(int(s), int(st.pos[s]), float(st.score[s])) for s in live
                if st.pos[s] <= t - n_recent]
        if evict_override is None:
            # smallest score; among equal scores the higher position goes
            victim = min(cand, key=lambda c: (c[2], -c[1]))[0]
        else:
            victim = int(evict_override)
        evicted = int(st.pos[victim])
        st.free_slot = victim
        st.n_used = st.slots - 1
        return np.stack(outs), evicted, cand
    st.n_used = count
    st.free_slot = count
    return np.stack(outs), -1, []
