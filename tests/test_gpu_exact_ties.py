"""Exact tie rules on the GPU, compared bit for bit with the oracle (no tolerance band).

* SnapKV top-k (SnapKV article, 処理の流れ step 3): among equal pooled votes the lower
  position is kept.  Max-pooling turns a vote peak into a plateau of exactly equal
  values, so ties at the k-th boundary are the normal case, not a rare one.  The votes
  here are multiples of 1/4 below 3, so every pooled value (a maximum, or a window sum
  of such multiples, which fp32 forms exactly) is exact in fp32 and in fp64: the
  oracle's fp64 selection is then the only correct answer, and the GPU's must equal it.
  Each case runs one of the selection kernels' radix paths: pool 7 (or 1) with the
  candidates in registers; pool 7 (or 1) over more than 16384 candidates in chunks of 16384 (each chunk's
  local top-k, then their merge; the plateaus straddle the chunk boundaries); keys in
  shared memory (other pool sizes, or chunks whose candidates exceed the merge's 8192);
  keys in global memory (more than 49152 candidates); unaligned vote rows take the
  scalar staging path.
* H2O eviction (H2O article, 処理の流れ): among exactly equal smallest cumulative
  scores the entry with the higher position is evicted (the lower position is kept).
  The planted state has several evictable entries with the same score whose keys are
  identical (or whose query is zero), so their probabilities and new scores stay
  exactly equal on both sides; they sit in slots that different threads and warps of
  the step kernel scan.
"""

import numpy as np
import pytest
import torch

from oracle import h2o as OH
from oracle import snapkv as OS
from parity import assert_outputs_close, assert_votes_close, f64

pytestmark = pytest.mark.gpu

# (name, candidates n = L - W, window W, pool kernel, prefix picks k, average pooling)
SELECT_CASES = [
    ("registers-max7", 4096, 32, 7, 600, False),
    ("registers-max7-16384", 16384, 32, 7, 2400, False),
    ("registers-avg7", 4096, 32, 7, 480, True),
    ("shared-max5", 3000, 16, 5, 300, False),
    ("registers-max1", 5000, 8, 1, 700, False),
    ("chunked-max1-40000", 40000, 8, 1, 2000, False),
    ("shared-max1-20000", 20000, 8, 1, 5000, False),
    ("shared-max7-20000", 20000, 32, 7, 5000, False),
    ("chunked-max7-20000", 20000, 32, 7, 3000, False),
    ("chunked-avg7-40000", 40000, 32, 7, 992, True),
    ("chunked-max7-short-last-chunk", 16884, 32, 7, 4000, False),
    ("chunked-unaligned-avg7-33001", 33001, 32, 7, 1500, True),
    ("shared-avg5", 3000, 16, 5, 300, True),
    ("global-max7-60000", 60000, 32, 7, 9000, False),
    ("global-avg3-60000", 60000, 32, 3, 992, True),
    ("unaligned-rows-max7", 1001, 32, 7, 140, False),
]


@pytest.mark.parametrize("case", SELECT_CASES, ids=[c[0] for c in SELECT_CASES])
def test_snapkv_select_plateau_ties_bit_exact(kvc, case):
    name, n, W, P, k, avg = case
    L = n + W
    Ly, B, Hkv, D = 1, 2, 2, 64
    g = torch.Generator().manual_seed(sum(map(ord, name)))
    # skewed towards small values, so the boundary sits below a run of larger ones
    votes = (torch.rand((Ly, B, Hkv, L), generator=g) ** 6 * 12).floor() * 0.25
    K = torch.randn((Ly, B, Hkv, L, D), generator=g).to(torch.bfloat16)
    V = torch.randn((Ly, B, Hkv, L, D), generator=g).to(torch.bfloat16)
    dev = torch.device("cuda")
    res = kvc.snapkv_select(votes.to(dev), K.to(dev), V.to(dev), keep_window=W, pool_kernel=P,
                            budget=k + W, pool_avg=avg)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    pos = res["pos"].cpu().numpy()
    kc, vc = res["k"].cpu(), res["v"].cpu()
    vh = votes.numpy().astype(np.float64)
    for ly in range(Ly):
        for b in range(B):
            for h in range(Hkv):
                pooled = OS.pool_1d(vh[ly, b, h, :n], P, "avg" if avg else "max")
                # larger values are kept whole, and the boundary value is shared by more
                # candidates than the top-k takes
                kth = np.sort(pooled)[::-1][k - 1]
                above = int((pooled > kth).sum())
                assert above > 0 and int((pooled == kth).sum()) > k - above, "no tie at the boundary"
                want = OS.select_positions(vh[ly, b, h], L, W, P, k + W, "avg" if avg else "max")
                got = pos[ly, b, h]
                assert got.tolist() == want.tolist(), (
                    "unit %s: kept sets differ at %s" % ((ly, b, h), sorted(set(got) ^ set(want))))
                assert torch.equal(kc[ly, b, h], K[ly, b, h, got])
                assert torch.equal(vc[ly, b, h], V[ly, b, h, got])


# tied slots of the planted H2O state (read by different threads and warps of the step
# kernel: 256 threads, slot s is scanned by thread s % 256) and which of them holds the
# highest position
TIE_SLOTS = [0, 37, 130, 256]


@pytest.mark.parametrize("zero_query", [False, True], ids=["equal-keys", "zero-query"])
@pytest.mark.parametrize("top", range(len(TIE_SLOTS)), ids=["top-slot%d" % s for s in TIE_SLOTS])
def test_h2o_equal_scores_evict_higher_position(kvc, top, zero_query):
    Ly, B, Hkv, G, D = 1, 1, 2, 2, 128
    n_heavy, n_recent = 300, 20
    S = n_heavy + n_recent + 1
    t = 1000
    g = torch.Generator().manual_seed(77 + top + 10 * zero_query)
    dev = torch.device("cuda")
    st = kvc.H2OState(Ly, B, Hkv, D, n_heavy, n_recent, dev)
    k = torch.randn((Ly, B, Hkv, S, D), generator=g).to(torch.bfloat16)
    v = torch.randn((Ly, B, Hkv, S, D), generator=g).to(torch.bfloat16)
    score = (10.0 + 10.0 * torch.rand((Ly, B, Hkv, S), generator=g)).float()
    pos = torch.full((Ly, B, Hkv, S), -1, dtype=torch.int32)
    q = torch.randn((Ly, B, Hkv * G, D), generator=g).to(torch.bfloat16)
    if zero_query:
        q.zero_()
    kn = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16)
    vn = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16)
    want = {}
    for h in range(Hkv):
        # 300 heavy-hitter positions below t - n_recent, then the 19 most recent, in a
        # shuffled slot order; the last slot is free
        heavy = torch.randperm(t - n_recent, generator=g)[:S - 20].sort().values
        recent = torch.arange(t - n_recent + 1, t, dtype=torch.int64)
        allpos = torch.cat([heavy, recent])
        allpos = allpos[torch.randperm(S - 1, generator=g)]
        # the tied slots hold heavy positions, the chosen one the highest of them
        tied = sorted(heavy[torch.randperm(heavy.numel(), generator=g)[:len(TIE_SLOTS)]].tolist())
        order = [s for s in TIE_SLOTS if s != TIE_SLOTS[top]] + [TIE_SLOTS[top]]
        for s, p in zip(order, tied):
            j = int((allpos == p).nonzero()[0])
            allpos[j], allpos[s] = allpos[s].clone(), p
        pos[0, 0, h, :S - 1] = allpos.int()
        for s in TIE_SLOTS:
            score[0, 0, h, s] = 2.0
            k[0, 0, h, s] = k[0, 0, h, TIE_SLOTS[0]]
        # recent entries may score lower than the tie: they are never candidates
        rec = (pos[0, 0, h] > t - n_recent).nonzero().flatten()
        score[0, 0, h, rec] = 0.5
        score[0, 0, h, S - 1] = 0.0
        want[h] = tied[-1]
    st.k.copy_(k)
    st.v.copy_(v)
    st.score.copy_(score)
    st.pos.copy_(pos)
    st.n_used.fill_(S - 1)
    st.free_slot.fill_(S - 1)
    out, ev = kvc.h2o_decode_step(q.to(dev), kn.to(dev), vn.to(dev), st, t)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    ev = ev.cpu().numpy()
    gscore, gpos = st.score.cpu().numpy(), st.pos.cpu().numpy()
    for h in range(Hkv):
        o = OH.H2OState(S, D)
        o.k[:], o.v[:] = f64(k[0, 0, h]), f64(v[0, 0, h])
        o.score[:], o.pos[:] = f64(score[0, 0, h]), pos[0, 0, h].numpy()
        o.n_used = o.free_slot = S - 1
        ro, rev, _ = OH.step(o, f64(q[0, 0, h * G:(h + 1) * G]), f64(kn[0, 0, h]), f64(vn[0, 0, h]),
                             t, n_recent)
        assert rev == want[h], "oracle evicted %d, expected %d" % (rev, want[h])
        assert int(ev[0, 0, h]) == rev, "GPU evicted %d, oracle %d" % (ev[0, 0, h], rev)
        assert_outputs_close(f64(out[0, 0, h * G:(h + 1) * G]), ro, "h2o tie step head %d" % h)
        live = o.live()
        by_pos = {int(p): float(s) for p, s in zip(gpos[0, 0, h], gscore[0, 0, h]) if p >= 0}
        assert_votes_close([by_pos[int(p)] for p in o.pos[live]], o.score[live], "tie scores")
        # the other tied entries are still cached, with scores exactly equal to each other
        rest = [by_pos[p] for p in o.pos[live] if p in set(int(x) for x in gpos[0, 0, h, TIE_SLOTS])]
        assert len(rest) == len(TIE_SLOTS) - 1 and len(set(rest)) == 1
