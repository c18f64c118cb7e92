"""SnapKV prompt-KV compression in fp64 (oracle; test infrastructure only).

Follows the SnapKV article (abeam.tech, 2026-07-18), section 処理の流れ
("processing flow"):

1. the observation-window queries at the end of the prompt attend to the prefix keys,
   per head (step 1);
2. per head, the window queries' attention weights on each prefix position are summed:
   the "vote" (step 2);
3. a 1D pooling clusters neighbouring important positions (step 3);
4. a top-k picks the prefix positions to keep (step 3), and the selected prefix KV is
   concatenated with the window's own KV into the compact cache (step 4);

and section 推論方法 ("inference"): the compression runs once right after the prompt
is processed, and decoding then reads only the compact cache.

Readings taken where the article is silent (it names the steps but gives no formulas):
softmax over every key a window row may see (prefix plus the causal part of the
window), scale 1/sqrt(d), plain sum over window rows, selection per KV head with the
vote summed over the G query heads of the group, max-pool with odd kernel P, stride 1,
same length, truncated at the ends and run over the prefix candidates only (the
average-pool variant: window sum over P with zeros past the ends), top-k
ties resolved towards the lower position, budget counting the window, kept prefix
positions in ascending order followed by the window, budget >= prompt length keeping
everything.
"""

import numpy as np

from .attention import attention_weights


def window_votes(q_unit, K):
    """Vote v_j of every prompt position j for one KV head (steps 1 and 2).

    q_unit: [G, Wq, d] -- the last Wq prompt queries of the G query heads that share
            this KV head; row r of every head sits at absolute position L - Wq + r.
    K:      [L, d]     -- the prompt keys of this KV head.
    Row (g, r) sees keys 0..L-Wq+r (everything before it and itself); its softmax
    weights are added into v.  Returns v [L] in fp64.

    With Wq = L this is the causal column sum over the whole prompt that H2O uses as
    the initial cumulative score.
    """
    q_unit = np.asarray(q_unit, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    G, Wq, _ = q_unit.shape
    L = K.shape[0]
    if Wq > L:
        raise ValueError("more window queries than prompt positions")
    v = np.zeros(L, dtype=np.float64)
    for g in range(G):
        for r in range(Wq):
            pos = L - Wq + r
            p = attention_weights(q_unit[g, r], K[: pos + 1])
            v[: pos + 1] += p
    return v


def votes_from_lse(q_unit, K, lse_unit):
    """Steps 1 and 2 with each window row's softmax normaliser given: row (g, r) at
    position i = L - Wq + r adds exp(q . k_j / sqrt(d) - lse_unit[g, i]) to v_j for every
    key j <= i.  With lse_unit the rows' own log-sum-exp (attention.causal_lse) each
    term is the row's softmax weight and v equals window_votes; another lse scales each
    row's contribution by exp(true lse - given lse).  A non-finite entry makes its row
    add nothing.

    q_unit: [G, Wq, d]; K: [L, d]; lse_unit: [G, L] (positions L-Wq..L-1 are read).
    Returns v [L] in fp64.
    """
    q_unit = np.asarray(q_unit, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    lse_unit = np.asarray(lse_unit, dtype=np.float64)
    G, Wq, d = q_unit.shape
    L = K.shape[0]
    if Wq > L:
        raise ValueError("more window queries than prompt positions")
    v = np.zeros(L, dtype=np.float64)
    for g in range(G):
        for r in range(Wq):
            pos = L - Wq + r
            lse = lse_unit[g, pos]
            if not np.isfinite(lse):
                continue
            v[: pos + 1] += np.exp(K[: pos + 1] @ q_unit[g, r] / np.sqrt(d) - lse)
    return v


def max_pool_1d(v, kernel):
    """Step 3: u_j = max of v over the positions within (kernel-1)/2 of j.

    Stride 1 and same length; windows are cut at both ends of ``v`` (equivalent to
    padding with -inf), so an edge position pools over fewer neighbours.
    """
    if kernel < 1 or kernel % 2 == 0:
        raise ValueError("pool kernel must be odd and >= 1")
    v = np.asarray(v, dtype=np.float64)
    n = v.shape[0]
    h = (kernel - 1) // 2
    u = np.empty(n, dtype=np.float64)
    for j in range(n):
        u[j] = v[max(0, j - h): min(n, j + h + 1)].max()
    return u


def avg_pool_1d(v, kernel):
    """Step 3, the average-pooling variant: u_j = (1/kernel) * sum of v over the positions
    within (kernel-1)/2 of j, with zeros beyond both ends of ``v`` (the divisor stays the
    kernel size at the edges).  Stride 1 and same length.
    """
    if kernel < 1 or kernel % 2 == 0:
        raise ValueError("pool kernel must be odd and >= 1")
    v = np.asarray(v, dtype=np.float64)
    n = v.shape[0]
    h = (kernel - 1) // 2
    u = np.empty(n, dtype=np.float64)
    for j in range(n):
        u[j] = v[max(0, j - h): min(n, j + h + 1)].sum() / kernel
    return u


def top_k_lowest_index(u, k):
    """Step 3 top-k: the k positions with the largest u; equal u -> lower position first.

    Returns the chosen positions in ascending order (int64).
    """
    u = np.asarray(u, dtype=np.float64)
    if k <= 0:
        return np.zeros(0, dtype=np.int64)
    if k >= u.shape[0]:
        return np.arange(u.shape[0], dtype=np.int64)
    idx = np.arange(u.shape[0])
    # lexsort sorts by the last key first: primary key -u (descending u), then index.
    order = np.lexsort((idx, -u))
    return np.sort(order[:k]).astype(np.int64)


def select_positions(votes, prompt_len, keep_window, pool_kernel, budget, pool="max"):
    """Positions kept for one KV head: pooled top-(budget - keep_window) of the prefix,
    ascending, followed by the last ``keep_window`` prompt positions (step 4).  ``pool``
    is "max" (max_pool_1d) or "avg" (avg_pool_1d).

    budget >= prompt_len (or keep_window >= prompt_len) keeps every position.
    """
    L, W = prompt_len, keep_window
    if budget >= L or W >= L:
        return np.arange(L, dtype=np.int64)
    if budget < W:
        raise ValueError("budget smaller than the kept window")
    prefix = np.asarray(votes, dtype=np.float64)[: L - W]
    pooled = pool_1d(prefix, pool_kernel, pool)
    chosen = top_k_lowest_index(pooled, budget - W)
    return np.concatenate([chosen, np.arange(L - W, L, dtype=np.int64)])


def pool_1d(v, kernel, pool="max"):
    """Step 3 with the chosen pooling: "max" or "avg"."""
    if pool == "max":
        return max_pool_1d(v, kernel)
    if pool == "avg":
        return avg_pool_1d(v, kernel)
    raise ValueError("pool must be 'max' or 'avg'")


def compress_unit(q_unit, K, V, window, pool_kernel, budget, pool="max"):
    """Whole SnapKV compression of one KV head.

    Returns (positions [n], K_c [n, d], V_c [n, d], votes [L]) with n = min(budget, L).
    """
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    L = K.shape[0]
    votes = window_votes(q_unit, K)
    pos = select_positions(votes, L, window, pool_kernel, budget, pool)
    return pos, K[pos], V[pos], votes


def compress(Q_win, K, V, window, pool_kernel, budget, pool="max"):
    """SnapKV over a batch: Q_win [B, Hq, W, d], K/V [B, Hkv, L, d].

    Query head h belongs to KV head h // (Hq // Hkv).  Returns per-(b, kv-head) lists
    of positions, compact K, compact V and votes.
    """
    Q_win = np.asarray(Q_win, dtype=np.float64)
    B, Hq, W, _ = Q_win.shape
    _, Hkv, _, _ = K.shape
    if Hq % Hkv:
        raise ValueError("query heads must be a multiple of KV heads")
    G = Hq // Hkv
    out = []
    for b in range(B):
        row = []
        for h in range(Hkv):
            row.append(compress_unit(Q_win[b, h * G:(h + 1) * G], K[b, h], V[b, h],
                                     window, pool_kernel, budget, pool))
        out.append(row)
    return out
