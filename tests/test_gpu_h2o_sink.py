"""GPU parity of H2O (prefill scores and cut, then decode steps with score accumulation
and eviction, in lockstep with the oracle) and of the StreamingLLM sink + ring cache."""

import numpy as np
import pytest
import torch

import workloads as W
from oracle import h2o as OH
from oracle import streaming as OSt
from parity import BAND, assert_outputs_close, assert_votes_close, check_selected_set, f64

pytestmark = pytest.mark.gpu


def run_h2o_lockstep(kvc, Ly, B, Hq, Hkv, D, L, n_heavy, n_recent, steps, seed):
    g = torch.Generator().manual_seed(seed)
    Q = torch.randn((Ly, B, Hq, L, D), generator=g).to(torch.bfloat16)
    K = torch.randn((Ly, B, Hkv, L, D), generator=g).to(torch.bfloat16)
    V = torch.randn((Ly, B, Hkv, L, D), generator=g).to(torch.bfloat16)
    dev = torch.device("cuda")
    st = kvc.h2o_prefill(Q.to(dev), K.to(dev), V.to(dev), n_heavy=n_heavy, n_recent=n_recent)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    G = Hq // Hkv
    Qh, Kh, Vh = f64(Q), f64(K), f64(V)
    units = [(ly, b, h) for ly in range(Ly) for b in range(B) for h in range(Hkv)]
    ref = {}
    swaps = 0
    pos = st.pos.cpu().numpy()
    score = st.score.cpu().numpy()
    for (ly, b, h) in units:
        o = OH.prefill(Qh[ly, b, h * G:(h + 1) * G], Kh[ly, b, h], Vh[ly, b, h], n_heavy, n_recent)
        n_keep = min(L, n_heavy + n_recent)
        gp = pos[ly, b, h, :n_keep]
        assert (pos[ly, b, h, n_keep:] == -1).all()
        if L > n_heavy + n_recent:
            from oracle.snapkv import window_votes
            full = window_votes(Qh[ly, b, h * G:(h + 1) * G], Kh[ly, b, h])
            assert list(gp[n_heavy:]) == list(range(L - n_recent, L))
            if n_heavy:
                swaps += check_selected_set(gp[:n_heavy], np.sort(o.pos[:n_heavy]),
                                            full[:L - n_recent], n_heavy)
            if set(gp) != set(o.pos[:n_keep].tolist()):
                # follow the GPU's equally valid cut: rebuild the oracle state from it
                o = OH.H2OState(n_heavy + n_recent + 1, D)
                o.k[:n_keep], o.v[:n_keep] = Kh[ly, b, h, gp], Vh[ly, b, h, gp]
                o.score[:n_keep], o.pos[:n_keep] = full[gp], gp
                o.n_used = o.free_slot = n_keep
        # scores of the kept entries (slot order may differ: compare by position)
        ref_by_pos = {int(p): s for p, s in zip(o.pos[:o.n_used], o.score[:o.n_used])}
        assert_votes_close(score[ly, b, h, :n_keep], [ref_by_pos[int(p)] for p in gp],
                           "prefill scores")
        ref[(ly, b, h)] = o
    for s in range(steps):
        t = L + s
        q = torch.randn((Ly, B, Hq, D), generator=g).to(torch.bfloat16)
        kn = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16)
        vn = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16)
        out, ev = kvc.h2o_decode_step(q.to(dev), kn.to(dev), vn.to(dev), st, t)
        torch.cuda.synchronize()
        assert kvc.kvc_device_status() == 0
        outh, evh = f64(out), ev.cpu().numpy()
        gpu_pos = st.pos.cpu().numpy()
        for (ly, b, h) in units:
            o = ref[(ly, b, h)]
            qh = f64(q)[ly, b, h * G:(h + 1) * G]
            # run the oracle step; if the GPU evicted a different entry, it must be an
            # equally valid choice (score within the band of the minimum), then follow it
            snap = (o.k.copy(), o.v.copy(), o.score.copy(), o.pos.copy(), o.n_used, o.free_slot)
            ro, rev, cand = OH.step(o, qh, f64(kn)[ly, b, h], f64(vn)[ly, b, h], t, n_recent)
            assert_outputs_close(outh[ly, b, h * G:(h + 1) * G], ro, "h2o step %d" % s)
            if int(evh[ly, b, h]) != rev:
                best = min(c[2] for c in cand)
                gsel = [c for c in cand if c[1] == int(evh[ly, b, h])]
                assert gsel and abs(gsel[0][2] - best) <= BAND * abs(best), (
                    "step %d unit %s: evicted %d, oracle %d" % (t, (ly, b, h), evh[ly, b, h], rev))
                o.k, o.v, o.score, o.pos, o.n_used, o.free_slot = snap
                o.k, o.v, o.score, o.pos = (a.copy() for a in (o.k, o.v, o.score, o.pos))
                OH.step(o, qh, f64(kn)[ly, b, h], f64(vn)[ly, b, h], t, n_recent,
                        evict_override=gsel[0][0])
                swaps += 1
            assert set(gpu_pos[ly, b, h][gpu_pos[ly, b, h] >= 0].tolist()) - {int(evh[ly, b, h])} \
                == set(o.pos[o.live()].tolist())
    return swaps


def test_h2o_tiny_workload_lockstep(kvc):
    w = W.TINY
    swaps = run_h2o_lockstep(kvc, 1, 1, 4, 4, 64, w.prompt_len, w.n_heavy, w.n_recent,
                             w.decode_steps, seed=W.seed_of(1, 2))
    assert swaps <= 4


def test_h2o_gqa_ragged_lockstep(kvc):
    swaps = run_h2o_lockstep(kvc, 1, 2, 8, 2, 128, 300, 20, 12, 24, seed=3)
    assert swaps <= 4


def test_h2o_no_eviction_until_full(kvc):
    # prompt shorter than the budget: the cache first fills, then starts evicting
    run_h2o_lockstep(kvc, 1, 1, 2, 2, 64, 10, 8, 4, 10, seed=4)


def test_sink_ring_tiny_workload(kvc):
    w = W.TINY
    S, R, D = w.n_sink, w.ring, w.head_dim
    Ly, B, Hkv, Hq = 1, 1, w.kv_heads, w.q_heads
    dev = torch.device("cuda")
    kc = torch.zeros((Ly, B, Hkv, S + R, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    pos = torch.full((Ly, B, Hkv, S + R), -1, dtype=torch.int32, device=dev)
    caches = [OSt.SinkCache(S, R, D) for _ in range(Hkv)]
    seed = W.seed_of(1, 3)
    for t in range(w.stream_len):
        q, k, v = W.stream_token(w, t, seed, "cpu")
        kvc.sink_window_append(k.to(dev), v.to(dev), kc, vc, t, n_sink=S, n_recent=R, pos=pos)
        n = min(t + 1, S + R)
        out = kvc.compressed_decode_attn(q.to(dev), kc, vc, n_uniform=n)
        if t % 7 == 0 or t < S + R + 3 or t == w.stream_len - 1:
            outh = f64(out)
            for h in range(Hkv):
                caches[h].append(t, f64(k)[0, 0, h], f64(v)[0, 0, h])
                ref = caches[h].attend(f64(q)[0, 0, h:h + 1], t)
                assert_outputs_close(outh[0, 0, h:h + 1], ref, "sink step %d" % t)
        else:
            for h in range(Hkv):
                caches[h].append(t, f64(k)[0, 0, h], f64(v)[0, 0, h])
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    p = pos.cpu().numpy()[0, 0, 0]
    assert list(p[:S]) == list(range(S))
    assert sorted(p[S:]) == list(range(w.stream_len - R, w.stream_len))
