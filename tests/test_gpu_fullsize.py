"""Full-size SnapKV parity on the Mistral-7B-shaped workload (batch 2, 32 layers, 32 query
/ 8 KV heads, head dim 128, 16384-token prompt, window 32, pool 7, budget 1024), called
the way the bench calls it: all 32 layers in one snapkv_compress call (512 units over the
persistent grid, several jobs per CTA group), then compressed_decode_attn with the fused
append over the compact caches.  The fp64 oracle checks sampled units one by one.

A moderate case with many more jobs than CTA groups (256 units of 2048 keys) is checked
in full: it covers the interleaving of one job's pass 2 with the next job's pass 1 and
the statistics exchange across rounds, which the small cases of test_gpu_snapkv never
reach."""

import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as OA
from oracle import snapkv as OS
from parity import assert_outputs_close, assert_votes_close, check_selected_set, f64

pytestmark = pytest.mark.gpu


def sample_units(Ly, B, H, n, seed):
    rng = np.random.default_rng(seed)
    units = {(0, 0, 0), (Ly - 1, B - 1, H - 1)}
    while len(units) < n:
        units.add((int(rng.integers(Ly)), int(rng.integers(B)), int(rng.integers(H))))
    return sorted(units)


def check_units(w, x, res, units):
    """Votes, kept set and gathered rows of the given units against the oracle."""
    L, Wn, P, Kb = w.prompt_len, w.window, w.pool_kernel, w.budget
    G = w.q_heads // w.kv_heads
    k = Kb - Wn
    swaps = 0
    for (ly, b, h) in units:
        what = "unit (%d,%d,%d)" % (ly, b, h)
        q = f64(x["Q_win"][ly, b, h * G:(h + 1) * G])
        K = f64(x["K"][ly, b, h])
        votes_ref = OS.window_votes(q, K)
        assert_votes_close(res["votes"][ly, b, h].cpu().numpy(), votes_ref, "votes " + what)
        assert int(res["n_valid"][ly, b, h]) == Kb
        got = res["pos"][ly, b, h].cpu().numpy()
        assert (got[Kb:] == -1).all()
        got = got[:Kb]
        assert list(got[k:]) == list(range(L - Wn, L))
        pooled = OS.max_pool_1d(votes_ref[:L - Wn], P)
        swaps += check_selected_set(got[:k], OS.top_k_lowest_index(pooled, k), pooled, k, what)
        idx = torch.as_tensor(got, dtype=torch.long, device=x["K"].device)
        assert torch.equal(res["k"][ly, b, h, :Kb], x["K"][ly, b, h, idx]), what
        assert torch.equal(res["v"][ly, b, h, :Kb], x["V"][ly, b, h, idx]), what
    return swaps


def test_mistral_full_size_compress_and_decode_sampled(kvc):
    w = W.MISTRAL
    dev = torch.device("cuda")
    x = W.snapkv_prompt(w, W.seed_of(2, 0), dev)
    L, Kb = w.prompt_len, w.budget
    cap = Kb + 256
    res = kvc.snapkv_compress(x["Q_win"], x["K"], x["V"], keep_window=w.window,
                              pool_kernel=w.pool_kernel, budget=Kb, cap=cap, want_votes=True)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    units = sample_units(w.layers, w.batch, w.kv_heads, 6, seed=3)
    assert check_units(w, x, res, units) <= 1

    # two decode steps with the fused append, planned with the exact row bound
    G = w.q_heads // w.kv_heads
    kc, vc, pos, nv = res["k"], res["v"], res["pos"], res["n_valid"]
    out = torch.empty((w.layers, w.batch, w.q_heads, w.head_dim), dtype=torch.bfloat16,
                      device=dev)
    for s in range(2):
        q, kn, vn = W.decode_token(w, s, W.seed_of(2, 100), dev)
        kvc.compressed_decode_attn(q, kc, vc, n_valid=nv, n_uniform=Kb + s + 1, k_new=kn,
                                   v_new=vn, pos=pos, new_pos=L + s, out=out)
        torch.cuda.synchronize()
        assert kvc.kvc_device_status() == 0
        assert int(nv.min()) == int(nv.max()) == Kb + s + 1
        for (ly, b, h) in units:
            n = Kb + s + 1
            assert int(pos[ly, b, h, n - 1]) == L + s
            assert torch.equal(kc[ly, b, h, n - 1], kn[ly, b, h])
            ref = OA.attend_group(f64(q[ly, b, h * G:(h + 1) * G]), f64(kc[ly, b, h, :n]),
                                  f64(vc[ly, b, h, :n]))
            assert_outputs_close(out[ly, b, h * G:(h + 1) * G].float().cpu().numpy(), ref,
                                 "decode step %d unit (%d,%d,%d)" % (s, ly, b, h))


def test_many_rounds_per_cta_group_all_units(kvc):
    # 256 units of 2048 keys: each CTA group runs several jobs in sequence
    w = dataclasses.replace(W.MISTRAL, name="many-rounds", layers=8, batch=4, prompt_len=2048,
                            budget=256)
    dev = torch.device("cuda")
    x = W.snapkv_prompt(w, 29, dev)
    res = kvc.snapkv_compress(x["Q_win"], x["K"], x["V"], keep_window=w.window,
                              pool_kernel=w.pool_kernel, budget=w.budget, cap=w.budget,
                              want_votes=True)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    units = [(ly, b, h) for ly in range(w.layers) for b in range(w.batch)
             for h in range(w.kv_heads)]
    assert check_units(w, x, res, units) <= len(units) // 4
