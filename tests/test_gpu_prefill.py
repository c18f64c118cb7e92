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
