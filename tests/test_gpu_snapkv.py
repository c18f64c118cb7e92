"""GPU parity of snapkv_compress (window votes, pool + top-k, gather) against the fp64
oracle on seeded inputs: sizes that span several 128-key tiles, ragged tails, GQA, two
row tiles, the multi-CTA statistics exchange, the degenerate budgets, and shapes served
by each window-vote kernel (single-pass for jobs of up to 64 rows with enough keys, two
passes for 128-row jobs)."""

import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from oracle import snapkv as OS
from parity import assert_votes_close, check_selected_set, f64

pytestmark = pytest.mark.gpu

# name, batch, layers, Hq, Hkv, D, L, W, P, budget
CASES = [
    ("tiny-config", 1, 1, 4, 4, 64, 512, 8, 7, 64),
    ("gqa4-d128-ragged-L1000", 2, 1, 8, 2, 128, 1000, 32, 7, 256),
    ("gqa8-two-row-tiles", 1, 1, 8, 1, 128, 700, 24, 5, 100),
    ("mha-d128-2layers", 1, 2, 2, 2, 128, 2048, 32, 7, 512),
    ("pool1-budget-equals-window", 1, 1, 2, 2, 64, 300, 16, 1, 16),
    ("budget-at-least-prompt", 1, 1, 2, 2, 64, 200, 8, 7, 256),
    ("window-is-whole-prompt", 1, 1, 2, 2, 64, 6, 6, 7, 4),
    ("long-unit-group-exchange", 1, 1, 4, 1, 128, 8192, 32, 7, 1024),
    ("tiny-prompt-one-tile", 1, 1, 4, 2, 128, 40, 8, 3, 20),
    # pool 7 with the keys in registers: 16-byte vote loads plus a tail of n % 4 = 2, and
    # an odd prompt length whose vote rows are mostly misaligned (4-byte loads)
    ("window30-vector-tail", 1, 1, 8, 2, 128, 1000, 30, 7, 200),
    ("odd-length-L1023", 1, 1, 4, 4, 64, 1023, 16, 7, 128),
    # single-pass window votes with a group exchange: 32 rows (one statistics chunk, two
    # vote sets), 64 rows and 48 rows (a ragged 16-row chunk)
    ("mha-rows32-L20000-exchange", 1, 1, 4, 4, 128, 20000, 32, 7, 1024),
    ("gqa2-rows64-L4096-exchange", 1, 1, 4, 2, 128, 4096, 32, 7, 256),
    ("gqa3-rows48-L3000-exchange", 1, 1, 6, 2, 64, 3000, 16, 5, 200),
    # 128 window rows against 80000 keys: the two-pass window-vote kernel (as for every
    # job of 128 rows)
    ("two-pass-kernel-L80000", 1, 1, 4, 1, 128, 80000, 32, 7, 1024),
]


def make_inputs(case, seed):
    name, B, Ly, Hq, Hkv, D, L, Wn, P, Kb = case
    w = dataclasses.replace(W.TINY, name=name, batch=B, layers=Ly, q_heads=Hq, kv_heads=Hkv,
                            head_dim=D, prompt_len=L, window=Wn, pool_kernel=P, budget=Kb,
                            spans_per_head=max(1, min(4, (L - Wn) // 8)), span_len=1)
    x = W.snapkv_prompt(w, seed, "cpu")
    return w, x


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_snapkv_compress_matches_oracle(kvc, case):
    w, x = make_inputs(case, seed=17)
    L, Wn, P, Kb = w.prompt_len, w.window, w.pool_kernel, w.budget
    G = w.q_heads // w.kv_heads
    dev = torch.device("cuda")
    Q, K, V = (x[n].to(dev) for n in ("Q_win", "K", "V"))
    identity = Kb >= L or Wn >= L
    n_keep = L if identity else Kb
    cap = n_keep + 5
    res = kvc.snapkv_compress(Q, K, V, keep_window=Wn, pool_kernel=P, budget=Kb, cap=cap,
                              want_votes=not identity)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    Qh, Kh, Vh = f64(x["Q_win"]), f64(x["K"]), f64(x["V"])
    pos = res["pos"].cpu().numpy()
    nv = res["n_valid"].cpu().numpy()
    kc = res["k"].cpu()
    vc = res["v"].cpu()
    swaps = 0
    for ly in range(w.layers):
        for b in range(w.batch):
            for h in range(w.kv_heads):
                assert nv[ly, b, h] == n_keep
                p = pos[ly, b, h]
                assert (p[n_keep:] == -1).all()
                got = p[:n_keep]
                if identity:
                    assert list(got) == list(range(L))
                else:
                    votes_ref = OS.window_votes(Qh[ly, b, h * G:(h + 1) * G], Kh[ly, b, h])
                    assert_votes_close(res["votes"][ly, b, h].cpu().numpy(), votes_ref,
                                       "votes unit (%d,%d,%d)" % (ly, b, h))
                    k = Kb - Wn
                    assert list(got[k:]) == list(range(L - Wn, L))
                    if k > 0:
                        pooled = OS.max_pool_1d(votes_ref[:L - Wn], P)
                        ref_sel = OS.top_k_lowest_index(pooled, k)
                        swaps += check_selected_set(got[:k], ref_sel, pooled, k,
                                                    "unit (%d,%d,%d)" % (ly, b, h))
                # the compact cache holds exactly the rows at the reported positions
                idx = torch.as_tensor(got, dtype=torch.long)
                assert torch.equal(kc[ly, b, h, :n_keep], x["K"][ly, b, h, idx])
                assert torch.equal(vc[ly, b, h, :n_keep], x["V"][ly, b, h, idx])
    assert swaps <= max(1, w.layers * w.batch * w.kv_heads // 4)


def test_planted_keys_are_kept_on_the_tiny_workload(kvc):
    """Sanity (not parity): on the tiny workload every planted key position survives."""
    x = W.snapkv_prompt(W.TINY, W.seed_of(1), "cuda")
    res = kvc.snapkv_compress(x["Q_win"], x["K"], x["V"], keep_window=W.TINY.window,
                              pool_kernel=W.TINY.pool_kernel, budget=W.TINY.budget)
    pos = res["pos"].cpu().numpy()
    planted = x["planted"].cpu().numpy()
    kept = sum(len(set(planted[0, 0, h]) & set(pos[0, 0, h])) for h in range(4))
    assert kept >= 0.9 * planted.size


def test_repeated_calls_are_bit_identical(kvc):
    case = CASES[1]
    w, x = make_inputs(case, seed=5)
    dev = torch.device("cuda")
    Q, K, V = (x[n].to(dev) for n in ("Q_win", "K", "V"))
    a = kvc.snapkv_compress(Q, K, V, keep_window=w.window, pool_kernel=w.pool_kernel,
                            budget=w.budget, want_votes=True)
    a = {k: v.clone() for k, v in a.items()}
    b = kvc.snapkv_compress(Q, K, V, keep_window=w.window, pool_kernel=w.pool_kernel,
                            budget=w.budget, want_votes=True)
    for key in ("k", "v", "pos", "n_valid", "votes"):
        assert torch.equal(a[key], b[key]), key


def test_argument_errors_launch_nothing(kvc):
    dev = torch.device("cuda")
    q = torch.zeros((1, 1, 4, 8, 64), dtype=torch.bfloat16, device=dev)
    k = torch.zeros((1, 1, 4, 64, 64), dtype=torch.bfloat16, device=dev)
    with pytest.raises(kvc.KVCError) as e:
        kvc.snapkv_compress(q, k, k, keep_window=8, pool_kernel=4, budget=16)  # even kernel
    assert e.value.code == 2
    with pytest.raises(kvc.KVCError) as e:
        kvc.snapkv_compress(q, k, k, keep_window=16, pool_kernel=3, budget=12)  # budget < window
    assert e.value.code == 4
    with pytest.raises(kvc.KVCError) as e:
        kvc.snapkv_compress(q, k, k, keep_window=8, pool_kernel=3, budget=16, cap=10)  # cap < budget
    assert e.value.code == 4
    q3 = torch.zeros((1, 1, 3, 8, 64), dtype=torch.bfloat16, device=dev)  # 3 q heads, 4 kv heads
    with pytest.raises(kvc.KVCError) as e:
        kvc.snapkv_compress(q3, k, k, keep_window=8, pool_kernel=3, budget=16)
    assert e.value.code == 2
    with pytest.raises(TypeError):
        kvc.snapkv_compress(q.float(), k, k, keep_window=8, pool_kernel=3, budget=16)


def test_multiple_budgets_same_prompt(kvc):
    """Budgets 64, 256, 1024 and 2048 on one prompt (GQA-4, D 128, L 4096): every call
    matches the oracle, and without boundary swaps each smaller budget's picks are a
    subset of the larger one's (top-k sets nest)."""
    case = ("budgets-gqa4-L4096", 1, 1, 8, 2, 128, 4096, 32, 7, 64)
    w, x = make_inputs(case, seed=23)
    L, Wn, P = w.prompt_len, w.window, w.pool_kernel
    G = w.q_heads // w.kv_heads
    dev = torch.device("cuda")
    Q, K, V = (x[n].to(dev) for n in ("Q_win", "K", "V"))
    Qh, Kh = f64(x["Q_win"]), f64(x["K"])
    pooled = [OS.max_pool_1d(OS.window_votes(Qh[0, 0, h * G:(h + 1) * G], Kh[0, 0, h])[:L - Wn], P)
              for h in range(w.kv_heads)]
    picks = {}
    swaps = 0
    for Kb in (64, 256, 1024, 2048):
        res = kvc.snapkv_compress(Q, K, V, keep_window=Wn, pool_kernel=P, budget=Kb, cap=Kb)
        torch.cuda.synchronize()
        assert kvc.kvc_device_status() == 0
        pos = res["pos"].cpu().numpy()
        k = Kb - Wn
        for h in range(w.kv_heads):
            got = pos[0, 0, h]
            assert list(got[k:]) == list(range(L - Wn, L))
            s = check_selected_set(got[:k], OS.top_k_lowest_index(pooled[h], k), pooled[h], k,
                                   "budget %d head %d" % (Kb, h))
            swaps += s
            picks[(Kb, h)] = (set(got[:k].tolist()), s)
            idx = torch.as_tensor(got, dtype=torch.long)
            assert torch.equal(res["k"][0, 0, h].cpu(), x["K"][0, 0, h, idx])
    assert swaps <= 2
    for h in range(w.kv_heads):
        for small, big in ((64, 256), (256, 1024), (1024, 2048)):
            (a, sa), (b, sb) = picks[(small, h)], picks[(big, h)]
            if sa == 0 and sb == 0:
                assert a <= b


AVG_CASES = [  # the three pooling paths: kernel 7 in shared memory, chunked, direct
    ("avg-gqa4-d128-ragged-L1000", 2, 1, 8, 2, 128, 1000, 32, 7, 256),
    ("avg-gqa8-kernel5-chunked", 1, 1, 8, 1, 128, 700, 24, 5, 100),
    ("avg-wide-kernel-direct", 1, 1, 2, 2, 64, 5000, 8, 4097, 64),
    ("avg-long-unit-group-exchange", 1, 1, 4, 1, 128, 8192, 32, 7, 1024),
    ("avg-odd-length-L1023", 1, 1, 4, 4, 64, 1023, 16, 7, 128),
]


@pytest.mark.parametrize("case", AVG_CASES, ids=[c[0] for c in AVG_CASES])
def test_snapkv_average_pool_matches_oracle(kvc, case):
    w, x = make_inputs(case, seed=29)
    L, Wn, P, Kb = w.prompt_len, w.window, w.pool_kernel, w.budget
    G = w.q_heads // w.kv_heads
    dev = torch.device("cuda")
    Q, K, V = (x[n].to(dev) for n in ("Q_win", "K", "V"))
    res = kvc.snapkv_compress(Q, K, V, keep_window=Wn, pool_kernel=P, budget=Kb, cap=Kb,
                              want_votes=True, pool_avg=True)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    Qh, Kh = f64(x["Q_win"]), f64(x["K"])
    pos = res["pos"].cpu().numpy()
    k = Kb - Wn
    swaps = 0
    for b in range(w.batch):
        for h in range(w.kv_heads):
            votes_ref = OS.window_votes(Qh[0, b, h * G:(h + 1) * G], Kh[0, b, h])
            assert_votes_close(res["votes"][0, b, h].cpu().numpy(), votes_ref)
            pooled = OS.avg_pool_1d(votes_ref[:L - Wn], P)
            got = pos[0, b, h]
            assert list(got[k:]) == list(range(L - Wn, L))
            swaps += check_selected_set(got[:k], OS.top_k_lowest_index(pooled, k), pooled, k,
                                        "avg unit (%d,%d)" % (b, h))
            idx = torch.as_tensor(got, dtype=torch.long)
            assert torch.equal(res["k"][0, b, h].cpu(), x["K"][0, b, h, idx])
    assert swaps <= max(1, w.batch * w.kv_heads // 4)


@pytest.mark.parametrize("case", [CASES[1], CASES[5]], ids=["gqa4-d128-ragged", "keep-all"])
def test_value_rows_from_pinned_host_memory(kvc, case):
    """V left in page-locked host memory: the gather reads the kept rows over the host
    link and the compact cache is bit-identical to the one from a device-resident V."""
    w, x = make_inputs(case, seed=31)
    L, Wn, P, Kb = w.prompt_len, w.window, w.pool_kernel, w.budget
    dev = torch.device("cuda")
    Q, K, V = (x[n].to(dev) for n in ("Q_win", "K", "V"))
    hV = x["V"].contiguous().pin_memory()
    kw = dict(keep_window=Wn, pool_kernel=P, budget=Kb)
    a = kvc.snapkv_compress(Q, K, V, **kw)
    b = kvc.snapkv_compress(Q, K, hV, **kw)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    for name in ("k", "v", "pos", "n_valid"):
        assert torch.equal(a[name], b[name]), name
    # pageable host memory is refused before anything is launched
    with pytest.raises(Exception):
        kvc.snapkv_compress(Q, K, x["V"], **kw)


def test_more_units_than_a_grid_dimension_holds(kvc):
    """70000 units (beyond the 65535 a grid's y or z dimension takes): every unit is
    compressed; sampled units against the oracle, and the last unit's rows gathered."""
    Ly, B, Hq, Hkv, D, L, Wn, P, Kb = 1, 70000, 1, 1, 64, 64, 8, 3, 16
    g = torch.Generator().manual_seed(70000)
    dev = torch.device("cuda")
    Q = torch.randn((Ly, B, Hq, Wn, D), generator=g).to(torch.bfloat16).to(dev)
    K = torch.randn((Ly, B, Hkv, L, D), generator=g).to(torch.bfloat16).to(dev)
    V = torch.randn((Ly, B, Hkv, L, D), generator=g).to(torch.bfloat16).to(dev)
    res = kvc.snapkv_compress(Q, K, V, keep_window=Wn, pool_kernel=P, budget=Kb, want_votes=True)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    assert (res["n_valid"] == Kb).all()
    for b in (0, 12345, 65535, 65536, B - 1):
        votes_ref = OS.window_votes(f64(Q[0, b]), f64(K[0, b, 0]))
        assert_votes_close(res["votes"][0, b, 0].cpu().numpy(), votes_ref, "votes unit %d" % b)
        pooled = OS.max_pool_1d(votes_ref[:L - Wn], P)
        got = res["pos"][0, b, 0].cpu().numpy()
        assert list(got[Kb - Wn:]) == list(range(L - Wn, L))
        check_selected_set(got[:Kb - Wn], OS.top_k_lowest_index(pooled, Kb - Wn), pooled, Kb - Wn,
                           "unit %d" % b)
        idx = torch.as_tensor(got, dtype=torch.long, device=dev)
        assert torch.equal(res["k"][0, b, 0], K[0, b, 0, idx])
        assert torch.equal(res["v"][0, b, 0], V[0, b, 0, idx])
