"""Softmax attention in fp64 (oracle; test infrastructure only).

The three articles all rest on ordinary scaled dot-product attention of a decode
query over cached keys/values; the SnapKV and H2O articles use the uncompressed
cache ("All KV", "full cache") as their quality baseline.  The scale is 1/sqrt(d)
and the softmax is taken over exactly the keys the query may see.
"""

import numpy as np


def softmax(logits):
    """Softmax of a 1-D fp64 vector; -inf entries get probability 0.

    Written out: subtract the maximum finite logit, exponentiate, divide by the sum.
    """
    x = np.asarray(logits, dtype=np.float64)
    finite = np.isfinite(x)
    if not finite.any():
        raise ValueError("softmax over an empty key set")
    m = x[finite].max()
    e = np.where(finite, np.exp(x - m), 0.0)
    return e / e.sum()


def attention_weights(q, K):
    """Probabilities p_j = softmax_j(q . k_j / sqrt(d)) of one query over keys K [n, d]."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    d = q.shape[-1]
    return softmax(K @ q / np.sqrt(d))


def attend(q, K, V):
    """o = sum_j p_j v_j for one query q [d] over keys K [n, d] and values V [n, d]."""
    p = attention_weights(q, K)
    return p @ np.asarray(V, dtype=np.float64)


def attend_group(qs, K, V):
    """Attention of G query heads qs [G, d] that share one KV head (GQA); returns [G, d]."""
    return np.stack([attend(q, K, V) for q in np.asarray(qs, dtype=np.float64)])


def attend_masked(q, K, V, visible):
    """Full attention over all keys with the invisible ones masked to -inf.

    This is a second route to the same quantity as ``attend(q, K[visible], V[visible])``;
    the StreamingLLM and H2O pins compare the two routes.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    d = q.shape[-1]
    logits = np.where(np.asarray(visible, dtype=bool), K @ q / np.sqrt(d), -np.inf)
    return softmax(logits) @ np.asarray(V, dtype=np.float64)


def causal_prefill(Q, K, V):
    """Prompt self-attention with the causal mask: row i of Q [L, d] attends to the keys
    and values 0..i.  Returns O [L, d] in fp64 (one row at a time, written out)."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    L = Q.shape[0]
    O = np.empty((L, V.shape[1]), dtype=np.float64)
    for i in range(L):
        O[i] = attend(Q[i], K[: i + 1], V[: i + 1])
    return O


def log_sum_exp(logits):
    """ln sum_j exp(x_j) of a 1-D fp64 vector (-inf entries add nothing): the logarithm of
    the softmax normaliser, so that softmax(x)_j = exp(x_j - log_sum_exp(x)).  Written out
    with the maximum finite logit taken out first."""
    x = np.asarray(logits, dtype=np.float64)
    finite = np.isfinite(x)
    if not finite.any():
        raise ValueError("log-sum-exp over an empty key set")
    m = x[finite].max()
    return m + np.log(np.where(finite, np.exp(x - m), 0.0).sum())


def causal_lse(Q, K):
    """Row log-sum-exp of the prompt's causal attention: lse_i = ln sum_{j <= i}
    exp(q_i . k_j / sqrt(d)) for Q [L, d], K [L, d].  Returns [L] in fp64, one row at a
    time."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    d = Q.shape[-1]
    return np.array([log_sum_exp(K[: i + 1] @ Q[i] / np.sqrt(d)) for i in range(Q.shape[0])])
