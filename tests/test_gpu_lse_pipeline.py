"""GPU parity of the log-sum-exp route to the scores: prefill_attention_lse (the prompt's
causal attention that also returns each row's log-sum-exp), snapkv_votes_from_lse (the
SnapKV votes, or H2O's initial scores, from those normalisers in one pass over the keys)
and h2o_prefill_from_votes, against the oracle's causal_lse, votes_from_lse and
window_votes and against the direct routes (snapkv_compress, h2o_prefill)."""

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as OA
from oracle import snapkv as OS
from parity import assert_outputs_close, assert_votes_close, check_selected_set, f64

pytestmark = pytest.mark.gpu

# absolute tolerance of a row's log-sum-exp: ln of an fp32 sum of at most a few thousand
# positive terms (relative rounding well below 1e-5) plus the ex2/lg2 approximations
LSE_ATOL = 2e-5

PREFILL_CASES = [  # name, Ly, B, Hq, Hkv, D, L
    ("gqa2-d128-ragged-L300", 1, 1, 4, 2, 128, 300),
    ("mha-d64-L700", 1, 1, 2, 2, 64, 700),
    ("one-tile-L128", 1, 2, 2, 1, 128, 128),
    ("gqa3-d64-L333", 1, 1, 6, 2, 64, 333),
    ("single-row-L1", 1, 1, 2, 1, 128, 1),
]


def prompt(Ly, B, Hq, Hkv, D, L, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((Ly, B, Hq, L, D), generator=g).to(torch.bfloat16)
    k = torch.randn((Ly, B, Hkv, L, D), generator=g).to(torch.bfloat16)
    v = torch.randn((Ly, B, Hkv, L, D), generator=g).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("case", PREFILL_CASES, ids=[c[0] for c in PREFILL_CASES])
def test_prefill_lse_matches_oracle(kvc, case):
    _, Ly, B, Hq, Hkv, D, L = case
    G = Hq // Hkv
    q, k, v = prompt(Ly, B, Hq, Hkv, D, L, seed=3 * L + Hq)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out, lse = kvc.prefill_attention_lse(qd, kd, vd)
    plain, _ = kvc.snapkv_prefill_attention(qd, kd, vd)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    assert torch.equal(out, plain)  # the same attention; the lse is an extra output
    qh, kh, vh, lg = f64(q), f64(k), f64(v), lse.double().cpu().numpy()
    for ly in range(Ly):
        for b in range(B):
            for hq in range(Hq):
                h = hq // G
                ref = OA.causal_lse(qh[ly, b, hq], kh[ly, b, h])
                err = np.abs(lg[ly, b, hq] - ref).max()
                assert err <= LSE_ATOL, ("lse", ly, b, hq, err)
                if hq == 0:
                    o = OA.causal_prefill(qh[ly, b, hq], kh[ly, b, h], vh[ly, b, h])
                    assert_outputs_close(f64(out[ly, b, hq]), o)


VOTE_CASES = [  # name, Ly, B, Hq, Hkv, D, L, Wq
    ("snapkv-gqa4-w32-L1000", 1, 1, 8, 2, 128, 1000, 32),        # 128 rows: one row tile
    ("snapkv-mha-w32-d64-ragged-L333", 1, 2, 2, 2, 64, 333, 32),   # 32 rows, many buffers
    ("gqa3-w48-wrapping-tiles-L520", 1, 1, 6, 2, 128, 520, 48),    # 144 rows: a tile spans two heads
    ("gqa8-w16-L260", 1, 1, 8, 1, 128, 260, 16),
    ("window-spans-tiles-L400-w160", 1, 1, 2, 1, 64, 400, 160),
    ("h2o-whole-prompt-L300", 1, 1, 2, 2, 128, 300, 300),          # Wq = L, 3 row tiles
    ("h2o-gqa2-whole-prompt-L260", 2, 1, 4, 2, 64, 260, 260),
    ("one-query-L1", 1, 1, 2, 1, 128, 1, 1),
]


def true_lse(qh, kh, G):
    """Oracle log-sum-exp of every prompt row, [Ly,B,Hq,L] fp64."""
    Ly, B, Hq, L, _ = qh.shape
    out = np.empty((Ly, B, Hq, L))
    for ly in range(Ly):
        for b in range(B):
            for hq in range(Hq):
                out[ly, b, hq] = OA.causal_lse(qh[ly, b, hq], kh[ly, b, hq // G])
    return out


@pytest.mark.parametrize("case", VOTE_CASES, ids=[c[0] for c in VOTE_CASES])
def test_votes_from_lse_match_oracle(kvc, case):
    """The vote kernel against the oracle's votes_from_lse with a perturbed lse (each row
    offset by up to 0.5: any row read with the wrong normaliser shows), then with the
    rows' true lse against window_votes."""
    _, Ly, B, Hq, Hkv, D, L, Wq = case
    G = Hq // Hkv
    q, k, _ = prompt(Ly, B, Hq, Hkv, D, L, seed=L + 7 * Wq + Hq)
    dev = torch.device("cuda")
    qh, kh = f64(q), f64(k)
    q_win = q[:, :, :, L - Wq:].contiguous()
    lse = true_lse(qh, kh, G)
    rng = np.random.default_rng(L + Wq)
    shifted = lse + rng.uniform(-0.5, 0.5, size=lse.shape)
    for lse_in, route in ((shifted, "perturbed"), (lse, "true")):
        lse_d = torch.as_tensor(lse_in, dtype=torch.float32).to(dev)
        votes = kvc.snapkv_votes_from_lse(q_win.to(dev), k.to(dev), lse_d)
        torch.cuda.synchronize()
        assert kvc.kvc_device_status() == 0
        vg = votes.cpu().numpy()
        lse32 = lse_d.double().cpu().numpy()  # the normalisers the kernel was given
        for ly in range(Ly):
            for b in range(B):
                for h in range(Hkv):
                    qu = qh[ly, b, h * G:(h + 1) * G, L - Wq:]
                    ref = OS.votes_from_lse(qu, kh[ly, b, h], lse32[ly, b, h * G:(h + 1) * G])
                    assert_votes_close(vg[ly, b, h], ref, "%s votes (%d,%d,%d)" % (route, ly, b, h))
                    if route == "true":
                        assert_votes_close(vg[ly, b, h], OS.window_votes(qu, kh[ly, b, h]),
                                           "window votes (%d,%d,%d)" % (ly, b, h))


def test_votes_from_lse_drop_rows_with_non_finite_lse(kvc):
    Ly, B, Hq, Hkv, D, L, Wq = 1, 1, 4, 1, 128, 200, 40
    G = Hq // Hkv
    q, k, _ = prompt(Ly, B, Hq, Hkv, D, L, seed=5)
    qh, kh = f64(q), f64(k)
    lse = true_lse(qh, kh, G)
    lse[0, 0, 1, L - Wq + 3] = np.inf
    lse[0, 0, 2, L - 1] = -np.inf
    lse[0, 0, 3, L - Wq] = np.nan
    dev = torch.device("cuda")
    lse_d = torch.as_tensor(lse, dtype=torch.float32).to(dev)
    votes = kvc.snapkv_votes_from_lse(q[:, :, :, L - Wq:].contiguous().to(dev), k.to(dev), lse_d)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    ref = OS.votes_from_lse(qh[0, 0, :, L - Wq:], kh[0, 0, 0], lse_d.double().cpu().numpy()[0, 0])
    assert np.isfinite(votes.cpu().numpy()).all()
    assert_votes_close(votes[0, 0, 0].cpu().numpy(), ref)


def test_lse_pipeline_equals_direct_routes(kvc):
    """prefill_attention_lse -> snapkv_votes_from_lse -> snapkv_select against
    snapkv_compress, and with every query voting -> h2o_prefill_from_votes against
    h2o_prefill, on one prompt (GQA 4, L 1500)."""
    Ly, B, Hq, Hkv, D, L, Wq, P, Kb = 1, 2, 8, 2, 128, 1500, 32, 7, 256
    q, k, v = prompt(Ly, B, Hq, Hkv, D, L, seed=77)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    _, lse = kvc.prefill_attention_lse(qd, kd, vd)
    q_win = qd[:, :, :, L - Wq:].contiguous()
    votes = kvc.snapkv_votes_from_lse(q_win, kd, lse)
    kw = dict(keep_window=Wq, pool_kernel=P, budget=Kb)
    sel = kvc.snapkv_select(votes, kd, vd, **kw)
    ref = kvc.snapkv_compress(q_win, kd, vd, want_votes=True, **kw)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    qh, kh = f64(q), f64(k)
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hkv):
            ov = OS.window_votes(qh[0, b, h * G:(h + 1) * G, L - Wq:], kh[0, b, h])
            assert_votes_close(votes[0, b, h].cpu().numpy(), ov, "pipeline votes (%d,%d)" % (b, h))
            pooled = OS.max_pool_1d(ov[:L - Wq], P)
            check_selected_set(sel["pos"][0, b, h, :Kb - Wq].cpu().numpy(),
                               ref["pos"][0, b, h, :Kb - Wq].cpu().numpy(), pooled, Kb - Wq)
    # H2O: every prompt query votes
    n_heavy, n_recent = 100, 60
    scores = kvc.snapkv_votes_from_lse(qd, kd, lse)
    st = kvc.h2o_prefill_from_votes(scores, kd, vd, n_q_heads=Hq, n_heavy=n_heavy,
                                    n_recent=n_recent)
    st_ref = kvc.h2o_prefill(qd, kd, vd, n_heavy=n_heavy, n_recent=n_recent)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    n_keep = n_heavy + n_recent
    assert torch.equal(st.n_used, st_ref.n_used)
    for b in range(B):
        for h in range(Hkv):
            full = OS.window_votes(qh[0, b, h * G:(h + 1) * G], kh[0, b, h])
            assert_votes_close(scores[0, b, h].cpu().numpy(), full, "h2o scores (%d,%d)" % (b, h))
            gp = st.pos[0, b, h, :n_keep].cpu().numpy()
            assert list(gp[n_heavy:]) == list(range(L - n_recent, L))
            check_selected_set(gp[:n_heavy], st_ref.pos[0, b, h, :n_heavy].cpu().numpy(),
                               full[:L - n_recent], n_heavy)
            assert_votes_close(st.score[0, b, h, :n_keep].cpu().numpy(), full[gp],
                               "h2o kept scores (%d,%d)" % (b, h))
            assert torch.equal(st.k[0, b, h, :n_keep].cpu(), k[0, b, h, torch.as_tensor(gp).long()])


def test_lse_route_full_size_mistral_and_opt_sampled(kvc):
    """The bench's launches: two layers of the Mistral-7B-shaped prompt (batch 2, 32 query
    / 8 KV heads, L 16384, window 32) and one layer of the OPT-6.7B-shaped H2O prompt
    (batch 64, 32 heads, L 2048, every query voting), through prefill_attention_lse and
    snapkv_votes_from_lse; sampled units against the oracle's window votes."""
    dev = torch.device("cuda")
    w = W.MISTRAL
    x = W.snapkv_prompt(w, W.seed_of(2, 9), dev, layers=2, full_queries=True)
    _, lse = kvc.prefill_attention_lse(x["Q_full"], x["K"], x["V"])
    votes = kvc.snapkv_votes_from_lse(x["Q_win"], x["K"], lse)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    G = w.q_heads // w.kv_heads
    for (ly, b, h) in [(0, 0, 0), (1, 1, 7), (1, 0, 3)]:
        ref = OS.window_votes(f64(x["Q_win"][ly, b, h * G:(h + 1) * G]), f64(x["K"][ly, b, h]))
        assert_votes_close(votes[ly, b, h].cpu().numpy(), ref, "mistral votes (%d,%d,%d)" % (ly, b, h))
    del x, lse, votes
    w = W.H2O_OPT
    Q, K, V = W.h2o_prompt_layer(w, 0, W.seed_of(4, 3), dev)
    _, lse = kvc.prefill_attention_lse(Q[None], K[None], V[None])
    scores = kvc.snapkv_votes_from_lse(Q[None], K[None], lse)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    for (b, h) in [(0, 0), (63, 31), (17, 5)]:
        ref = OS.window_votes(f64(Q[b, h:h + 1]), f64(K[b, h]))
        assert_votes_close(scores[0, b, h].cpu().numpy(), ref, "opt scores (%d,%d)" % (b, h))


def test_lse_route_argument_errors_launch_nothing(kvc):
    """The C entry points check their arguments before any launch: NULL pointers, sizes out
    of range and misaligned bases return their codes and leave the device status clear."""
    import ctypes

    from attention_score_kv_snapkv_gb300._binding import H2OParams, SnapKVParams
    lib = kvc.lib()
    dev = torch.device("cuda")
    q = torch.zeros((1, 1, 2, 64, 64), dtype=torch.bfloat16, device=dev)
    k = torch.zeros((1, 1, 1, 64, 64), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((1, 1, 2, 64), dtype=torch.float32, device=dev)
    votes = torch.zeros((1, 1, 1, 64), dtype=torch.float32, device=dev)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    p = SnapKVParams(1, 1, 2, 1, 64, 64, 8, 0, 1, 1, 1, 0)
    assert lib.snapkv_votes_from_lse(ctypes.byref(p), P(q), P(k), None, P(votes), None) == 1
    assert lib.snapkv_votes_from_lse(ctypes.byref(p), P(q), P(k), P(lse), None, None) == 1
    assert lib.snapkv_votes_from_lse(None, P(q), P(k), P(lse), P(votes), None) == 1
    bad = SnapKVParams(1, 1, 2, 1, 64, 64, 65, 0, 1, 1, 1, 0)  # n_query > prompt_len
    assert lib.snapkv_votes_from_lse(ctypes.byref(bad), P(q), P(k), P(lse), P(votes), None) == 2
    bad = SnapKVParams(1, 1, 2, 1, 96, 64, 8, 0, 1, 1, 1, 0)  # head_dim 96
    assert lib.snapkv_votes_from_lse(ctypes.byref(bad), P(q), P(k), P(lse), P(votes), None) == 2
    off = ctypes.c_void_p(q.data_ptr() + 2)  # not 16-byte aligned
    assert lib.snapkv_votes_from_lse(ctypes.byref(p), off, P(k), P(lse), P(votes), None) == 3
    out = torch.empty_like(q)
    assert lib.prefill_attention_lse(ctypes.byref(p), P(q), P(k), P(k), P(out), None, None) == 1
    hp = H2OParams(1, 1, 2, 1, 64, 8, 8)
    st = kvc.H2OState(1, 1, 1, 64, 8, 8, dev)
    sc = st.c_struct()
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=dev)
    assert lib.h2o_prefill_from_votes(ctypes.byref(hp), 64, None, P(k), P(k), ctypes.byref(sc),
                                      P(ws), ws.numel(), None) == 1
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0


def test_votes_from_lse_long_context_sampled(kvc):
    """One layer of the long-context prompt (32 MHA heads, L = 131072, window 32): the
    window rows' log-sum-exp from the oracle (fp64, every head), then the vote kernel
    against the oracle's window votes for sampled heads."""
    dev = torch.device("cuda")
    w = W.LONG
    x = W.snapkv_prompt(w, W.seed_of(3, 5), dev, layers=1)
    Qw, K = x["Q_win"], x["K"]
    L, Wn, H, D = w.prompt_len, w.window, w.kv_heads, w.head_dim
    lse = np.full((1, 1, w.q_heads, L), np.nan)
    for h in range(H):
        qh, kh = f64(Qw[0, 0, h]), f64(K[0, 0, h])
        logits = qh @ kh.T / np.sqrt(D)                      # [Wn, L]
        for r in range(Wn):
            lse[0, 0, h, L - Wn + r] = OA.log_sum_exp(logits[r, :L - Wn + r + 1])
    votes = kvc.snapkv_votes_from_lse(Qw, K, torch.as_tensor(lse, dtype=torch.float32).to(dev))
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    for h in (0, 17, H - 1):
        ref = OS.window_votes(f64(Qw[0, 0, h:h + 1]), f64(K[0, 0, h]))
        assert_votes_close(votes[0, 0, h].cpu().numpy(), ref, "long-context votes (head %d)" % h)
