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


def check_prefill_unit(q, K, V, gpu_pos, gpu_score, n_heavy, n_recent):
    """One unit's prefill cut and scores against the oracle (fp64 q [G,L,D], K, V [L,D]).
    Returns (oracle state that follows the GPU's cut, number of in-band swaps)."""
    L, D = K.shape
    o = OH.prefill(q, K, V, n_heavy, n_recent)
    n_keep = min(L, n_heavy + n_recent)
    gp = gpu_pos[:n_keep]
    assert (gpu_pos[n_keep:] == -1).all()
    swaps = 0
    if L > n_heavy + n_recent:
        from oracle.snapkv import window_votes
        full = window_votes(q, K)
        assert list(gp[n_heavy:]) == list(range(L - n_recent, L))
        if n_heavy:
            swaps += check_selected_set(gp[:n_heavy], np.sort(o.pos[:n_heavy]), full[:L - n_recent],
                                        n_heavy)
        if set(gp) != set(o.pos[:n_keep].tolist()):
            # follow the GPU's equally valid cut: rebuild the oracle state from it
            o = OH.H2OState(n_heavy + n_recent + 1, D)
            o.k[:n_keep], o.v[:n_keep] = K[gp], V[gp]
            o.score[:n_keep], o.pos[:n_keep] = full[gp], gp
            o.n_used = o.free_slot = n_keep
    # scores of the kept entries (slot order may differ: compare by position)
    ref_by_pos = {int(p): s for p, s in zip(o.pos[:o.n_used], o.score[:o.n_used])}
    assert_votes_close(gpu_score[:n_keep], [ref_by_pos[int(p)] for p in gp], "prefill scores")
    return o, swaps


def check_step_unit(o, q, k_new, v_new, t, n_recent, gpu_out, gpu_evicted, gpu_pos, what,
                    gpu_score=None):
    """One unit's decode step against the oracle state o (advanced in place).  If the GPU
    evicted a different entry, it must be an equally valid choice (score within the band
    of the minimum); the oracle then follows it.  With gpu_score (the unit's per-slot
    cumulative scores after the step) every live entry's score is compared, by position,
    with the oracle's at the vote tolerance.  Returns the number of such swaps."""
    snap = (o.k.copy(), o.v.copy(), o.score.copy(), o.pos.copy(), o.n_used, o.free_slot)
    ro, rev, cand = OH.step(o, q, k_new, v_new, t, n_recent)
    assert_outputs_close(gpu_out, ro, what)
    swaps = 0
    if int(gpu_evicted) != rev:
        best = min(c[2] for c in cand)
        gsel = [c for c in cand if c[1] == int(gpu_evicted)]
        assert gsel and abs(gsel[0][2] - best) <= BAND * abs(best), (
            "%s: evicted %d, oracle %d" % (what, gpu_evicted, rev))
        o.k, o.v, o.score, o.pos, o.n_used, o.free_slot = snap
        o.k, o.v, o.score, o.pos = (a.copy() for a in (o.k, o.v, o.score, o.pos))
        OH.step(o, q, k_new, v_new, t, n_recent, evict_override=gsel[0][0])
        swaps = 1
    assert set(gpu_pos[gpu_pos >= 0].tolist()) - {int(gpu_evicted)} == set(o.pos[o.live()].tolist())
    if gpu_score is not None:
        live = o.live()
        by_pos = {int(p): float(s) for p, s in zip(gpu_pos, gpu_score)
                  if p >= 0 and int(p) != int(gpu_evicted)}
        assert_votes_close([by_pos[int(p)] for p in o.pos[live]], o.score[live],
                           what + " cumulative scores")
    return swaps


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
        ref[(ly, b, h)], sw = check_prefill_unit(Qh[ly, b, h * G:(h + 1) * G], Kh[ly, b, h],
                                                 Vh[ly, b, h], pos[ly, b, h], score[ly, b, h],
                                                 n_heavy, n_recent)
        swaps += sw
    for s in range(steps):
        t = L + s
        q = torch.randn((Ly, B, Hq, D), generator=g).to(torch.bfloat16)
        kn = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16)
        vn = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16)
        out, ev = kvc.h2o_decode_step(q.to(dev), kn.to(dev), vn.to(dev), st, t)
        torch.cuda.synchronize()
        assert kvc.kvc_device_status() == 0
        outh, evh = f64(out), ev.cpu().numpy()
        gpu_pos, gpu_score = st.pos.cpu().numpy(), st.score.cpu().numpy()
        qh, knh, vnh = f64(q), f64(kn), f64(vn)
        for (ly, b, h) in units:
            swaps += check_step_unit(ref[(ly, b, h)], qh[ly, b, h * G:(h + 1) * G], knh[ly, b, h],
                                     vnh[ly, b, h], t, n_recent, outh[ly, b, h * G:(h + 1) * G],
                                     evh[ly, b, h], gpu_pos[ly, b, h],
                                     "h2o step %d unit %s" % (t, (ly, b, h)),
                                     gpu_score[ly, b, h])
    return swaps


def test_h2o_tiny_workload_lockstep(kvc):
    # 16 steps past the workload's 32, so that the first decode-appended tokens leave the
    # recent window and become eviction candidates with scores accumulated on the GPU.
    # The workload's 4 units are few: the step splits each over several CTAs (more CTAs
    # than units)
    w = W.TINY
    assert kvc.h2o_step_ctas_per_unit(1, 1, 4, 4, 64, w.n_heavy, w.n_recent) > 1
    swaps = run_h2o_lockstep(kvc, 1, 1, 4, 4, 64, w.prompt_len, w.n_heavy, w.n_recent,
                             w.decode_steps + 16, seed=W.seed_of(1, 2))
    assert swaps <= 4


def test_h2o_gqa_ragged_lockstep(kvc):
    swaps = run_h2o_lockstep(kvc, 1, 2, 8, 2, 128, 300, 20, 12, 24, seed=3)
    assert swaps <= 4


@pytest.mark.parametrize("G", [1, 2, 3, 4, 6, 7, 8], ids=lambda g: "G%d" % g)
def test_h2o_every_head_group_lockstep(kvc, G):
    # two KV heads of G query heads each; the recent window of 6 is passed after six
    # steps, so decode-appended tokens become eviction candidates
    swaps = run_h2o_lockstep(kvc, 1, 1, 2 * G, 2, 64, 150, 12, 6, 14, seed=40 + G)
    assert swaps <= 2


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


@pytest.mark.parametrize("n_sink", [0, 1, 2, 8], ids=lambda s: "sinks%d" % s)
def test_sink_count_sweep_gqa(kvc, n_sink):
    """Plain window attention (no sinks) and other sink counts: fill, wrap and stream
    past the ring several times, GQA with two query heads per KV head, every step
    checked against the oracle's sink + ring cache."""
    S, R, D, Ly, B, Hkv, G = n_sink, 20, 128, 1, 2, 2, 2
    T = S + 3 * R + 5
    dev = torch.device("cuda")
    kc = torch.zeros((Ly, B, Hkv, S + R, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    pos = torch.full((Ly, B, Hkv, S + R), -1, dtype=torch.int32, device=dev)
    caches = {(b, h): OSt.SinkCache(S, R, D) for b in range(B) for h in range(Hkv)}
    g = torch.Generator().manual_seed(100 + n_sink)
    for t in range(T):
        q = torch.randn((Ly, B, Hkv * G, D), generator=g).to(torch.bfloat16)
        k = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16)
        v = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16)
        kvc.sink_window_append(k.to(dev), v.to(dev), kc, vc, t, n_sink=S, n_recent=R, pos=pos)
        out = kvc.compressed_decode_attn(q.to(dev), kc, vc, n_uniform=min(t + 1, S + R))
        outh, qh = f64(out), f64(q)
        for (b, h), c in caches.items():
            c.append(t, f64(k)[0, b, h], f64(v)[0, b, h])
            ref = c.attend(qh[0, b, h * G:(h + 1) * G], t)
            assert_outputs_close(outh[0, b, h * G:(h + 1) * G], ref, "sinks %d step %d" % (S, t))
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    p = pos.cpu().numpy()[0, 1, 1]
    assert sorted(p.tolist()) == sorted(OSt.visible_positions(T - 1, S, R).tolist())


def test_h2o_step_plans(kvc):
    # one CTA per unit for the OPT-shaped workload (65536 units), several for few units,
    # the split step for logits beyond one CTA's shared memory, 0 out of range
    assert kvc.h2o_step_ctas_per_unit(32, 64, 32, 32, 128, 204, 204) == 1
    assert kvc.h2o_step_ctas_per_unit(8, 1, 32, 32, 128, 13107, 13107) > 1
    assert kvc.h2o_step_ctas_per_unit(256, 64, 32, 8, 128, 13107, 13107) > 1  # G 4: too wide
    assert kvc.h2o_step_ctas_per_unit(1, 1, 36, 4, 128, 8, 8) == 0          # G 9
    assert kvc.h2o_step_ctas_per_unit(1, 1, 4, 4, 128, 8, 0) == 0           # no recent window


@pytest.mark.parametrize("G", [1, 4], ids=["G1-few-units", "G4-logits-exceed-one-cta"])
def test_h2o_split_step_budget_20pct_of_131072(kvc, G):
    """The H2O step on a cache of 20% of a 131072-token context (13107 heavy + 13107
    recent), built directly (a prefill of that prompt is far beyond the oracle), for two
    KV heads: the step splits each unit's cache over several CTAs (few units; at G = 4
    the logits would not fit one CTA's shared memory either).  Three steps in lockstep
    with the oracle: outputs, evicted positions and every live entry's score."""
    Ly, B, Hkv, D = 1, 1, 2, 128
    n_heavy = n_recent = 13107
    S = n_heavy + n_recent + 1
    t0 = 131072
    g = torch.Generator().manual_seed(500 + G)
    dev = torch.device("cuda")
    st = kvc.H2OState(Ly, B, Hkv, D, n_heavy, n_recent, dev)
    k = torch.randn((Ly, B, Hkv, S, D), generator=g).to(torch.bfloat16)
    v = torch.randn((Ly, B, Hkv, S, D), generator=g).to(torch.bfloat16)
    score = (1.0 + 99.0 * torch.rand((Ly, B, Hkv, S), generator=g)).float()
    pos = torch.full((Ly, B, Hkv, S), -1, dtype=torch.int32)
    refs = {}
    for h in range(Hkv):
        heavy = torch.randperm(t0 - n_recent, generator=g)[:n_heavy]
        recent = torch.arange(t0 - n_recent, t0, dtype=torch.int64)
        allpos = torch.cat([heavy, recent])[torch.randperm(S - 1, generator=g)]
        pos[0, 0, h, :S - 1] = allpos.int()
        score[0, 0, h, S - 1] = 0.0
        o = OH.H2OState(S, D)
        o.k[:], o.v[:] = f64(k[0, 0, h]), f64(v[0, 0, h])
        o.score[:], o.pos[:] = f64(score[0, 0, h]), pos[0, 0, h].numpy()
        o.n_used = o.free_slot = S - 1
        refs[h] = o
    st.k.copy_(k)
    st.v.copy_(v)
    st.score.copy_(score)
    st.pos.copy_(pos)
    st.n_used.fill_(S - 1)
    st.free_slot.fill_(S - 1)
    swaps = 0
    for s in range(3):
        t = t0 + s
        q = torch.randn((Ly, B, Hkv * G, D), generator=g).to(torch.bfloat16)
        kn = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16)
        vn = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16)
        out, ev = kvc.h2o_decode_step(q.to(dev), kn.to(dev), vn.to(dev), st, t)
        torch.cuda.synchronize()
        assert kvc.kvc_device_status() == 0
        outh, evh = f64(out), ev.cpu().numpy()
        gpos, gscore = st.pos.cpu().numpy(), st.score.cpu().numpy()
        for h in range(Hkv):
            swaps += check_step_unit(refs[h], f64(q[0, 0, h * G:(h + 1) * G]), f64(kn[0, 0, h]),
                                     f64(vn[0, 0, h]), t, n_recent, outh[0, 0, h * G:(h + 1) * G],
                                     evh[0, 0, h], gpos[0, 0, h], "split step %d head %d" % (t, h),
                                     gscore[0, 0, h])
    assert swaps <= 1
