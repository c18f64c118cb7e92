"""GPU parity of snapkv_prefill_attention (causal prompt self-attention with the SnapKV
votes as a by-product) against the oracle's causal attention and window votes, and of
snapkv_select (steps 3-4 from those votes) against snapkv_compress."""

import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import snapkv as OS
from parity import assert_outputs_close, assert_votes_close, f64

pytestmark = pytest.mark.gpu

CASES = [  # name, Ly, B, Hq, Hkv, D, L, W
    ("gqa2-d128-ragged-L300", 1, 1, 4, 2, 128, 300, 32),
    ("mha-d64-L700", 1, 1, 2, 2, 64, 700, 16),
    ("one-tile-L128", 1, 2, 2, 1, 128, 128, 8),
    ("window-spans-two-tiles", 1, 1, 2, 1, 128, 400, 160),
    ("gqa4-d128-2layers-L520", 2, 1, 8, 2, 128, 520, 32),
    ("gqa8-one-kv-head-L260", 1, 1, 8, 1, 128, 260, 16),
    ("gqa3-d64-odd-group-L333", 1, 1, 6, 2, 64, 333, 24),
    ("window-is-whole-prompt-L96", 1, 1, 2, 1, 64, 96, 96),
]


def inputs(case, seed):
    _, Ly, B, Hq, Hkv, D, L, W = case
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((Ly, B, Hq, L, D), generator=g).to(torch.bfloat16)
    k = torch.randn((Ly, B, Hkv, L, D), generator=g).to(torch.bfloat16)
    v = torch.randn((Ly, B, Hkv, L, D), generator=g).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_prefill_attention_and_votes_match_oracle(kvc, case):
    _, Ly, B, Hq, Hkv, D, L, W = case
    G = Hq // Hkv
    q, k, v = inputs(case, seed=L + Hq)
    dev = torch.device("cuda")
    out, votes = kvc.snapkv_prefill_attention(q.to(dev), k.to(dev), v.to(dev), window=W)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    oh, qh, kh, vh = f64(out), f64(q), f64(k), f64(v)
    vg = votes.cpu().numpy()
    for ly in range(Ly):
        for b in range(B):
            for h in range(Hkv):
                for g in range(G):
                    hq = h * G + g
                    ref = OA.causal_prefill(qh[ly, b, hq], kh[ly, b, h], vh[ly, b, h])
                    assert_outputs_close(oh[ly, b, hq], ref, "output (%d,%d,%d)" % (ly, b, hq))
                q_win = qh[ly, b, h * G:(h + 1) * G, L - W:]
                assert_votes_close(vg[ly, b, h], OS.window_votes(q_win, kh[ly, b, h]),
                                   "votes (%d,%d,%d)" % (ly, b, h))


def test_prefill_without_votes_and_select_from_votes(kvc):
    # the output alone, then selection from prefill votes == snapkv_compress's selection
    Ly, B, Hq, Hkv, D, L, W, P, Kb = 1, 2, 8, 2, 128, 1000, 32, 7, 256
    q, k, v = inputs(("sel", Ly, B, Hq, Hkv, D, L, W), seed=41)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out_a, none = kvc.snapkv_prefill_attention(qd, kd, vd)
    out_b, votes = kvc.snapkv_prefill_attention(qd, kd, vd, window=W)
    torch.cuda.synchronize()
    assert none is None and kvc.kvc_device_status() == 0
    # rows outside the window tiles are computed identically with or without votes
    assert torch.equal(out_a[..., :768, :], out_b[..., :768, :])
    sel = kvc.snapkv_select(votes, kd, vd, keep_window=W, pool_kernel=P, budget=Kb)
    ref = kvc.snapkv_compress(qd[:, :, :, L - W:].contiguous(), kd, vd, keep_window=W,
                              pool_kernel=P, budget=Kb, want_votes=True)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    rel = ((votes - ref["votes"]).abs() / (ref["votes"].abs() + 1e-9)).max().item()
    assert rel < 1e-5, rel
    pooled_gap = 0
    for b in range(B):
        for h in range(Hkv):
            a, r = sel["pos"][0, b, h].cpu().numpy(), ref["pos"][0, b, h].cpu().numpy()
            if not np.array_equal(a, r):  # only swaps at the selection boundary
                pooled = OS.max_pool_1d(ref["votes"][0, b, h, :L - W].double().cpu().numpy(), P)
                boundary = np.sort(pooled)[::-1][Kb - W - 1]
                for j in set(a.tolist()) ^ set(r.tolist()):
                    assert abs(pooled[j] - boundary) <= 1e-4 * abs(boundary)
                pooled_gap += 1
            idx = torch.as_tensor(a, dtype=torch.long)
            assert torch.equal(sel["k"][0, b, h].cpu(), k[0, b, h, idx])
    assert pooled_gap <= 1


def test_prefill_full_size_mistral_sampled(kvc):
    """The bench's prefill launch (two layers of the Mistral-7B-shaped prompt: batch 2, 32
    query / 8 KV heads, D 128, L 16384, window 32): sampled output rows against the
    oracle's attention of that row over keys 0..row, and the votes of sampled KV heads
    against the oracle's window votes; then selection from those votes against
    snapkv_compress on the same prompt."""
    import workloads as W
    w = W.MISTRAL
    Ly = 2
    dev = torch.device("cuda")
    x = W.snapkv_prompt(w, W.seed_of(2, 7), dev, layers=Ly, full_queries=True)
    Qf, K, V = x["Q_full"], x["K"], x["V"]
    L, Wn, G = w.prompt_len, w.window, w.q_heads // w.kv_heads
    out, votes = kvc.snapkv_prefill_attention(Qf, K, V, window=Wn)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    rng = np.random.default_rng(11)
    rows = [0, 1, 127, 128, 4095, L - Wn - 1, L - Wn, L - 1] + [int(r) for r in rng.integers(0, L, 8)]
    for i, row in enumerate(rows):
        ly, b, hq = i % Ly, (i // 2) % w.batch, int(rng.integers(w.q_heads))
        h = hq // G
        ref = OA.attend(f64(Qf[ly, b, hq, row]), f64(K[ly, b, h, :row + 1]), f64(V[ly, b, h, :row + 1]))
        assert_outputs_close(out[ly, b, hq, row].float().cpu().numpy(), ref,
                             "output (%d,%d,%d) row %d" % (ly, b, hq, row))
    for (ly, b, h) in [(0, 0, 0), (Ly - 1, w.batch - 1, w.kv_heads - 1), (1, 0, 5)]:
        ref = OS.window_votes(f64(Qf[ly, b, h * G:(h + 1) * G, L - Wn:]), f64(K[ly, b, h]))
        assert_votes_close(votes[ly, b, h].cpu().numpy(), ref, "votes (%d,%d,%d)" % (ly, b, h))
    kw = dict(keep_window=Wn, pool_kernel=w.pool_kernel, budget=w.budget)
    sel = kvc.snapkv_select(votes, K, V, **kw)
    ref = kvc.snapkv_compress(x["Q_win"], K, V, want_votes=True, **kw)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    rel = ((votes - ref["votes"]).abs() / (ref["votes"].abs() + 1e-9)).max().item()
    assert rel < 1e-5, rel
    # the kept sets may differ only by swaps at the selection boundary (the two routes'
    # votes differ by rounding)
    differ = (sel["pos"] != ref["pos"]).any(dim=-1).nonzero().tolist()
    assert len(differ) <= 16, len(differ)
    kp = w.budget - Wn
    for (ly, b, h) in differ:
        a, r = sel["pos"][ly, b, h].cpu().numpy(), ref["pos"][ly, b, h].cpu().numpy()
        pooled = OS.max_pool_1d(ref["votes"][ly, b, h, :L - Wn].double().cpu().numpy(), w.pool_kernel)
        boundary = np.sort(pooled)[::-1][kp - 1]
        for j in set(a[:kp].tolist()) ^ set(r[:kp].tolist()):
            assert abs(pooled[j] - boundary) <= 1e-4 * abs(boundary), (ly, b, h, j)
