"""GPU parity on seeded random shapes, against the fp64 oracle with the shared parity
rules.

* snapkv_compress: head dim, head grouping (any G up to 8), prompt length (1 to 20000
  tokens, so every selection path and window-vote kernel is reached), window, pool
  kernel, max or average pooling and budget (from keeping only the window to keeping
  everything): votes within 1e-5 relative, kept sets identical up to swaps inside the tie
  band, window positions appended in order, the compact cache holding exactly the rows
  at the reported positions.
* snapkv_votes_from_lse: head dim, grouping, prompt length and voting rows (from one
  query to every prompt query), given each row's log-sum-exp shifted by up to 0.5 and
  NaN at every position the kernel must not read: votes within 1e-5 relative.
* compressed_decode_attn with the fused append: layers, batch, KV heads, grouping, head
  dim, capacity and ragged row counts: appended rows, row counts and outputs (2e-2
  absolute + 1e-2 relative).
* H2O: head dim, grouping, prompt length, heavy and recent budgets (either may be small,
  the heavy one zero) and enough decode steps that decode-appended tokens become eviction
  candidates, in lockstep with the oracle (prefill cut and scores, then every step's
  output, evicted position, live set and cumulative scores), whichever of the one-CTA and
  split step kernels the shape gets.
* prefill_attention_lse: head dim, grouping and prompt length (1 to 1500 tokens): every
  row's log-sum-exp (2e-5 absolute) and the attention output of sampled heads.
* StreamingLLM: sink count (0 = plain window attention), ring size, grouping and head dim,
  streamed past the ring at least twice: the attention after every append against the
  oracle's sink + ring cache on sampled steps (every step until the ring first wraps),
  and the final slot positions."""

import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as OA
from oracle import snapkv as OS
from oracle import streaming as OSt
from parity import assert_outputs_close, assert_votes_close, check_selected_set, f64
from test_gpu_h2o_sink import run_h2o_lockstep

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


def draw_vote_shape(seed):
    """(name, batch, layers, Hq, Hkv, D, L, Wq) for one seed; G * Wq * L stays small
    enough for the oracle."""
    r = np.random.RandomState(seed)
    D = int(r.choice([64, 128]))
    Hkv = int(r.choice([1, 2]))
    G = int(r.randint(1, 9))
    L = max(1, int(np.exp(r.uniform(0.0, np.log(2500.0)))))
    if r.rand() < 0.25:
        Wq = L                                     # every prompt query votes (H2O)
    else:
        Wq = int(r.randint(1, min(L, 96) + 1))
    while G * Wq * L > 4_000_000 and Wq > 1:
        Wq //= 2
    B = int(r.choice([1, 2]))
    name = "seed%d-D%d-G%d-Hkv%d-L%d-Wq%d" % (seed, D, G, Hkv, L, Wq)
    return (name, B, 1, G * Hkv, Hkv, D, L, Wq)


VOTE_SHAPES = [draw_vote_shape(s) for s in range(201, 213)]


@pytest.mark.parametrize("shape", VOTE_SHAPES, ids=[s[0] for s in VOTE_SHAPES])
def test_random_shape_votes_from_lse(kvc, shape):
    name, B, Ly, Hq, Hkv, D, L, Wq = shape
    G = Hq // Hkv
    g = torch.Generator().manual_seed(L * 31 + Wq)
    q = torch.randn((Ly, B, Hq, Wq, D), generator=g).to(torch.bfloat16)
    k = torch.randn((Ly, B, Hkv, L, D), generator=g).to(torch.bfloat16)
    qh, kh = f64(q), f64(k)
    rng = np.random.default_rng(L + Wq)
    lse = np.full((Ly, B, Hq, L), np.nan)          # positions before the window: never read
    for b in range(B):
        for hq in range(Hq):
            for r in range(Wq):
                pos = L - Wq + r
                lse[0, b, hq, pos] = (OA.log_sum_exp(kh[0, b, hq // G, :pos + 1] @ qh[0, b, hq, r]
                                                     / np.sqrt(D)) + rng.uniform(-0.5, 0.5))
    dev = torch.device("cuda")
    lse_d = torch.as_tensor(lse, dtype=torch.float32).to(dev)
    votes = kvc.snapkv_votes_from_lse(q.to(dev), k.to(dev), lse_d)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    vg = votes.cpu().numpy()
    lse32 = lse_d.double().cpu().numpy()            # the normalisers the kernel was given
    for b in range(B):
        for h in range(Hkv):
            ref = OS.votes_from_lse(qh[0, b, h * G:(h + 1) * G], kh[0, b, h],
                                    lse32[0, b, h * G:(h + 1) * G])
            assert_votes_close(vg[0, b, h], ref, "%s votes (%d,%d)" % (name, b, h))


def draw_decode_shape(seed):
    """(name, layers, batch, Hq, Hkv, D, cap) for one seed."""
    r = np.random.RandomState(seed)
    D = int(r.choice([64, 128]))
    Hkv = int(r.randint(1, 9))
    G = int(r.randint(1, 9))
    Ly = int(r.choice([1, 2]))
    B = int(r.randint(1, 5))
    cap = max(2, int(np.exp(r.uniform(np.log(2.0), np.log(3000.0)))))
    name = "seed%d-Ly%d-B%d-G%d-Hkv%d-D%d-cap%d" % (seed, Ly, B, G, Hkv, D, cap)
    return (name, Ly, B, G * Hkv, Hkv, D, cap)


DECODE_SHAPES = [draw_decode_shape(s) for s in range(301, 313)]


@pytest.mark.parametrize("shape", DECODE_SHAPES, ids=[s[0] for s in DECODE_SHAPES])
def test_random_shape_decode_with_append(kvc, shape):
    name, Ly, B, Hq, Hkv, D, cap = shape
    G = Hq // Hkv
    g = torch.Generator().manual_seed(cap * 13 + Hq)
    q = torch.randn((Ly, B, Hq, D), generator=g).to(torch.bfloat16)
    kc = torch.randn((Ly, B, Hkv, cap, D), generator=g).to(torch.bfloat16)
    vc = torch.randn((Ly, B, Hkv, cap, D), generator=g).to(torch.bfloat16)
    kn = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16)
    vn = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16)
    n0 = torch.randint(0, cap, (Ly, B, Hkv), generator=g, dtype=torch.int32)
    n0.view(-1)[0] = cap - 1                        # a unit the append fills
    dev = torch.device("cuda")
    kcd, vcd, nd = kc.to(dev), vc.to(dev), n0.to(dev)
    out = kvc.compressed_decode_attn(q.to(dev), kcd, vcd, n_valid=nd, k_new=kn.to(dev),
                                     v_new=vn.to(dev))
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    kc2, vc2 = kc.clone(), vc.clone()
    for idx in np.ndindex(*n0.shape):
        kc2[idx + (int(n0[idx]),)] = kn[idx]
        vc2[idx + (int(n0[idx]),)] = vn[idx]
    assert torch.equal(nd.cpu(), n0 + 1)
    assert torch.equal(kcd.cpu(), kc2) and torch.equal(vcd.cpu(), vc2)
    qh, kh, vh = f64(q), f64(kc2), f64(vc2)
    ref = np.zeros_like(qh)
    for ly in range(Ly):
        for b in range(B):
            for h in range(Hkv):
                m = int(n0[ly, b, h]) + 1
                ref[ly, b, h * G:(h + 1) * G] = OA.attend_group(qh[ly, b, h * G:(h + 1) * G],
                                                                kh[ly, b, h, :m], vh[ly, b, h, :m])
    assert_outputs_close(f64(out), ref, name)


def draw_h2o_shape(seed):
    """(name, layers, batch, Hq, Hkv, D, L, n_heavy, n_recent, steps) for one seed."""
    r = np.random.RandomState(seed)
    D = int(r.choice([64, 128]))
    Hkv = int(r.choice([1, 2]))
    G = int(r.randint(1, 9))
    B = int(r.choice([1, 2]))
    n_heavy = int(r.randint(1, 200))
    if seed % 4 == 1:
        n_heavy = 0                                # recent window only: a sliding window
    n_recent = int(r.randint(1, 40))
    L = int(r.randint(max(1, n_heavy + n_recent - 8), n_heavy + n_recent + 400))
    steps = n_recent + int(r.randint(2, 10))
    name = "seed%d-D%d-G%d-Hkv%d-B%d-L%d-heavy%d-recent%d-steps%d" % (seed, D, G, Hkv, B, L,
                                                                     n_heavy, n_recent, steps)
    return (name, 1, B, G * Hkv, Hkv, D, L, n_heavy, n_recent, steps)


H2O_SHAPES = [draw_h2o_shape(s) for s in range(401, 409)]


@pytest.mark.parametrize("shape", H2O_SHAPES, ids=[s[0] for s in H2O_SHAPES])
def test_random_shape_h2o_lockstep(kvc, shape):
    name, Ly, B, Hq, Hkv, D, L, n_heavy, n_recent, steps = shape
    swaps = run_h2o_lockstep(kvc, Ly, B, Hq, Hkv, D, L, n_heavy, n_recent, steps,
                             seed=L + 7 * n_heavy + n_recent)
    assert swaps <= 2


def draw_sink_shape(seed):
    """(name, batch, Hq, Hkv, D, n_sink, ring, stream length) for one seed."""
    r = np.random.RandomState(seed)
    D = int(r.choice([64, 128]))
    Hkv = int(r.choice([1, 2, 3]))
    G = int(r.randint(1, 9))
    B = int(r.choice([1, 2]))
    S = int(r.randint(0, 9))
    R = max(1, int(np.exp(r.uniform(0.0, np.log(300.0)))))
    T = S + 2 * R + int(r.randint(1, 40))
    name = "seed%d-D%d-G%d-Hkv%d-B%d-sinks%d-ring%d-T%d" % (seed, D, G, Hkv, B, S, R, T)
    return (name, B, G * Hkv, Hkv, D, S, R, T)


SINK_SHAPES = [draw_sink_shape(s) for s in range(501, 507)]


@pytest.mark.parametrize("shape", SINK_SHAPES, ids=[s[0] for s in SINK_SHAPES])
def test_random_shape_sink_ring(kvc, shape):
    name, B, Hq, Hkv, D, S, R, T = shape
    G = Hq // Hkv
    dev = torch.device("cuda")
    kc = torch.zeros((1, B, Hkv, S + R, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    pos = torch.full((1, B, Hkv, S + R), -1, dtype=torch.int32, device=dev)
    caches = {(b, h): OSt.SinkCache(S, R, D) for b in range(B) for h in range(Hkv)}
    g = torch.Generator().manual_seed(S * 1000 + R)
    for t in range(T):
        q = torch.randn((1, B, Hq, D), generator=g).to(torch.bfloat16)
        k = torch.randn((1, B, Hkv, D), generator=g).to(torch.bfloat16)
        v = torch.randn((1, B, Hkv, D), generator=g).to(torch.bfloat16)
        kvc.sink_window_append(k.to(dev), v.to(dev), kc, vc, t, n_sink=S, n_recent=R, pos=pos)
        out = kvc.compressed_decode_attn(q.to(dev), kc, vc, n_uniform=min(t + 1, S + R))
        kh, vh = f64(k), f64(v)
        for (b, h), c in caches.items():
            c.append(t, kh[0, b, h], vh[0, b, h])
        if t <= S + R + 2 or t % 5 == 0 or t == T - 1:
            outh, qh = f64(out), f64(q)
            for (b, h), c in caches.items():
                ref = c.attend(qh[0, b, h * G:(h + 1) * G], t)
                assert_outputs_close(outh[0, b, h * G:(h + 1) * G], ref, "%s step %d" % (name, t))
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    p = pos.cpu().numpy()
    for b in range(B):
        for h in range(Hkv):
            assert sorted(p[0, b, h].tolist()) == sorted(OSt.visible_positions(T - 1, S, R).tolist())


def draw_prefill_shape(seed):
    """(name, batch, Hq, Hkv, D, L) for one seed."""
    r = np.random.RandomState(seed)
    D = int(r.choice([64, 128]))
    Hkv = int(r.choice([1, 2]))
    G = int(r.randint(1, 5))
    B = int(r.choice([1, 2]))
    if seed % 2:                                   # several key tiles, ragged last one
        L = int(r.randint(129, 1501))
    else:
        L = max(1, int(np.exp(r.uniform(0.0, np.log(1500.0)))))
    name = "seed%d-D%d-G%d-Hkv%d-B%d-L%d" % (seed, D, G, Hkv, B, L)
    return (name, B, G * Hkv, Hkv, D, L)


PREFILL_SHAPES = [draw_prefill_shape(s) for s in range(601, 607)]


@pytest.mark.parametrize("shape", PREFILL_SHAPES, ids=[s[0] for s in PREFILL_SHAPES])
def test_random_shape_prefill_lse(kvc, shape):
    name, B, Hq, Hkv, D, L = shape
    G = Hq // Hkv
    g = torch.Generator().manual_seed(L * 7 + Hq)
    q = torch.randn((1, B, Hq, L, D), generator=g).to(torch.bfloat16)
    k = torch.randn((1, B, Hkv, L, D), generator=g).to(torch.bfloat16)
    v = torch.randn((1, B, Hkv, L, D), generator=g).to(torch.bfloat16)
    dev = torch.device("cuda")
    out, lse = kvc.prefill_attention_lse(q.to(dev), k.to(dev), v.to(dev))
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    qh, kh, vh = f64(q), f64(k), f64(v)
    lg = lse.double().cpu().numpy()
    for b in range(B):
        for hq in range(Hq):
            h = hq // G
            err = np.abs(lg[0, b, hq] - OA.causal_lse(qh[0, b, hq], kh[0, b, h])).max()
            assert err <= 2e-5, (name, b, hq, err)
            if hq % G == 0:  # one query head of each group
                ref = OA.causal_prefill(qh[0, b, hq], kh[0, b, h], vh[0, b, h])
                assert_outputs_close(f64(out[0, b, hq]), ref, "%s output (%d,%d)" % (name, b, hq))
