"""GPU parity of snapkv_compress on seeded random shapes: head dim, head grouping (any G
up to 8), prompt length (1 to 20000 tokens, so every selection path and window-vote
kernel is reached), window, pool kernel, max or average pooling and budget (from keeping
only the window to keeping everything) are drawn from a fixed list of seeds, and every
call is checked against the fp64 oracle with the shared parity rules: votes within 1e-5
relative, kept sets identical up to swaps inside the tie band, window positions appended
in order, and the compact cache holding exactly the rows at the reported positions."""

import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from oracle import snapkv as OS
from parity import assert_votes_close, check_selected_set, f64

pytestmark = pytest.mark.gpu

SEEDS = list(range(101, 117))


def draw_shape(seed):
    """(name, batch, layers, Hq, Hkv, D, L, W, P, budget, pool_avg) for one seed."""
    r = np.random.RandomState(seed)
    D = int(r.choice([64, 128]))
    Hkv = int(r.choice([1, 2]))
    G = int(r.randint(1, 9))
    L = int(np.exp(r.uniform(0.0, np.log(20000.0))))
    L = max(L, 1)
    Wn = int(r.randint(1, min(L, 64) + 1))
    P = int(r.choice([1, 3, 5, 7, 9, 15]))
    avg = bool(r.rand() < 0.3)
    mode = r.rand()
    if mode < 0.1:
        Kb = L + int(r.randint(0, 4))              # keep everything
    elif mode < 0.2:
        Kb = Wn                                    # keep only the window
    else:
        Kb = Wn + int(r.randint(1, max(2, L - Wn + 1)))
    B = int(r.choice([1, 2]))
    name = "seed%d-D%d-G%d-Hkv%d-L%d-W%d-P%d-%s-Kb%d" % (seed, D, G, Hkv, L, Wn, P,
                                                       "avg" if avg else "max", Kb)
    return (name, B, 1, G * Hkv, Hkv, D, L, Wn, P, Kb, avg)


SHAPES = [draw_shape(s) for s in SEEDS]


@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
def test_random_shape_matches_oracle(kvc, shape):
    name, B, Ly, Hq, Hkv, D, L, Wn, P, Kb, avg = shape
    w = dataclasses.replace(W.TINY, name=name, batch=B, layers=Ly, q_heads=Hq, kv_heads=Hkv,
                            head_dim=D, prompt_len=L, window=Wn, pool_kernel=P, budget=Kb,
                            spans_per_head=max(1, min(4, (L - Wn) // 8)), span_len=1)
    x = W.snapkv_prompt(w, 7, "cpu")
    G = Hq // Hkv
    dev = torch.device("cuda")
    Q, K, V = (x[n].to(dev) for n in ("Q_win", "K", "V"))
    identity = Kb >= L or Wn >= L
    n_keep = L if identity else Kb
    res = kvc.snapkv_compress(Q, K, V, keep_window=Wn, pool_kernel=P, budget=Kb,
                              cap=n_keep + 3, want_votes=not identity, pool_avg=avg)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    Qh, Kh = f64(x["Q_win"]), f64(x["K"])
    pos = res["pos"].cpu().numpy()
    nv = res["n_valid"].cpu().numpy()
    kc, vc = res["k"].cpu(), res["v"].cpu()
    k = Kb - Wn
    swaps = 0
    for b in range(B):
        for h in range(Hkv):
            assert nv[0, b, h] == n_keep
            p = pos[0, b, h]
            assert (p[n_keep:] == -1).all()
            got = p[:n_keep]
            if identity:
                assert list(got) == list(range(L))
            else:
                votes_ref = OS.window_votes(Qh[0, b, h * G:(h + 1) * G], Kh[0, b, h])
                assert_votes_close(res["votes"][0, b, h].cpu().numpy(), votes_ref,
                                   "%s votes (%d,%d)" % (name, b, h))
                assert list(got[k:]) == list(range(L - Wn, L))
                if k > 0:
                    pooled = OS.pool_1d(votes_ref[:L - Wn], P, "avg" if avg else "max")
                    swaps += check_selected_set(got[:k], OS.top_k_lowest_index(pooled, k),
                                                pooled, k, "%s unit (%d,%d)" % (name, b, h))
            idx = torch.as_tensor(got, dtype=torch.long)
            assert torch.equal(kc[0, b, h, :n_keep], x["K"][0, b, h, idx])
            assert torch.equal(vc[0, b, h, :n_keep], x["V"][0, b, h, idx])
    assert swaps <= max(1, B * Hkv // 4)
