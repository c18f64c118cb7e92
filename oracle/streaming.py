"""StreamingLLM sink + recent ring cache in fp64 (oracle; test infrastructure only).

Follows the StreamingLLM article (abeam.tech, 2026-07-02):

* キャッシュ構造 ("cache structure"): the first few tokens (about 4 suffice in many
  models) stay in the cache for good as attention sinks; besides them only a window of
  the most recent tokens is kept, so the cache has a fixed size;
* 推論の流れ ("inference flow"): each new token's KV is added to the recent region,
  the oldest recent token is dropped once the window is full, sink tokens are never
  dropped, and attention reads only the sink and recent tokens.

Readings taken where the article is silent: the new token is written before attending, so it
attends to itself; before the cache has filled, attention covers all t + 1 tokens;
the recent region is a ring: token t >= S goes to slot S + (t - S) mod R.
Position re-indexing inside the cache (a RoPE detail) is not part of this path: keys
arrive already position-encoded.
"""

import numpy as np

from .attention import attend_group


def slot_of(t, n_sink, n_recent):
    """Cache slot of token t: its own index while t < S, then the ring S + (t - S) mod R."""
    if t < n_sink:
        return t
    return n_sink + (t - n_sink) % n_recent


class SinkCache:
    """One KV head's cache of S sink slots followed by R ring slots."""

    def __init__(self, n_sink, n_recent, d):
        self.S = n_sink
        self.R = n_recent
        self.k = np.zeros((n_sink + n_recent, d))
        self.v = np.zeros((n_sink + n_recent, d))
        self.pos = np.full(n_sink + n_recent, -1, dtype=np.int64)

    def append(self, t, k_new, v_new):
        """Write token t's key/value into its slot (evicting the ring's oldest token)."""
        s = slot_of(t, self.S, self.R)
        self.k[s] = np.asarray(k_new, dtype=np.float64)
        self.v[s] = np.asarray(v_new, dtype=np.float64)
        self.pos[s] = t
        return s

    def n_live(self, t):
        """Entries attended at step t: min(t + 1, S + R)."""
        return min(t + 1, self.S + self.R)

    def attend(self, qs, t):
        """Attention of the query heads qs [G, d] over the live slots after token t."""
        n = self.n_live(t)
        return attend_group(qs, self.k[:n], self.v[:n])


def visible_positions(t, n_sink, n_recent):
    """The token positions a StreamingLLM query at step t attends to: the sinks
    0..S-1 and the last R tokens t-R+1..t (all of 0..t before the cache fills)."""
    if t + 1 <= n_sink + n_recent:
        return np.arange(t + 1)
    return np.concatenate([np.arange(n_sink), np.arange(t - n_recent + 1, t + 1)])
