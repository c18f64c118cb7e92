"""Full-size parity of the other three workloads, at the shapes the bench measures, checked
by the fp64 oracle on sampled units:

* long context: batch 1, 8 layers, 32 MHA heads, head dim 128, 131072-token prompt,
  window 32, pool 7, budget 1024 (one compression call), then two fused-append decode
  steps over the 1024-row caches;
* H2O on OPT-6.7B shapes: batch 64, 32 MHA heads, 2048-token prompt, 204 heavy + 204
  recent; two layers prefilled layer by layer through a one-layer view of the state (as
  the bench does), then decode steps of both layers in lockstep with the oracle;
* StreamingLLM on Llama-2-13B shapes: batch 16, 40 layers, 40 MHA heads, 4 sinks + a
  2044-token ring.  The ring keeps only the last 2044 tokens, so appending the sinks
  and then tokens 63488..65535 leaves the cache the full 65536-token stream ends with;
  the test streams through the first fill and wrap-around, then through that tail.
"""

import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as OA
from oracle import streaming as OSt
from parity import assert_outputs_close, f64
from test_gpu_fullsize import check_units, sample_units
from test_gpu_h2o_sink import check_prefill_unit, check_step_unit

pytestmark = pytest.mark.gpu


def test_long_context_full_size_sampled(kvc):
    w = W.LONG
    dev = torch.device("cuda")
    x = W.snapkv_prompt(w, W.seed_of(3), dev)
    L, Kb = w.prompt_len, w.budget
    cap = Kb + 2
    res = kvc.snapkv_compress(x["Q_win"], x["K"], x["V"], keep_window=w.window,
                              pool_kernel=w.pool_kernel, budget=Kb, cap=cap, want_votes=True)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    units = sample_units(w.layers, w.batch, w.kv_heads, 3, seed=5)
    assert check_units(w, x, res, units) <= 1
    # every planted span of a sampled unit lies in its kept set
    for (ly, b, h) in units:
        kept = set(res["pos"][ly, b, h, :Kb].cpu().tolist())
        planted = x["planted"][ly, b, h].cpu().tolist()
        assert set(planted) <= kept, "unit %s lost planted positions" % ((ly, b, h),)
    kc, vc, pos, nv = res["k"], res["v"], res["pos"], res["n_valid"]
    out = torch.empty((w.layers, w.batch, w.q_heads, w.head_dim), dtype=torch.bfloat16, device=dev)
    for s in range(2):
        q, kn, vn = W.decode_token(w, s, W.seed_of(3, 100), dev)
        kvc.compressed_decode_attn(q, kc, vc, n_valid=nv, n_uniform=Kb + s + 1, k_new=kn,
                                   v_new=vn, pos=pos, new_pos=L + s, out=out)
        torch.cuda.synchronize()
        assert kvc.kvc_device_status() == 0
        n = Kb + s + 1
        for (ly, b, h) in units:
            assert int(pos[ly, b, h, n - 1]) == L + s
            ref = OA.attend_group(f64(q[ly, b, h:h + 1]), f64(kc[ly, b, h, :n]), f64(vc[ly, b, h, :n]))
            assert_outputs_close(out[ly, b, h:h + 1].float().cpu().numpy(), ref,
                                 "decode step %d unit %s" % (s, (ly, b, h)))
    del x, res, kc, vc
    torch.cuda.empty_cache()


@pytest.mark.parametrize("budget", [(204, 204), (409, 409), (204, 4)],
                         ids=["20pct-of-prompt", "20pct-of-total", "recent4"])
def test_h2o_full_shape_sampled_lockstep(kvc, budget):
    # the budget read as 20% of the prompt (204 + 204) and as 20% of the total length
    # 4096 (409 + 409); with a recent window of 4 the decode-appended tokens become
    # eviction candidates after four steps
    w = dataclasses.replace(W.H2O_OPT, n_heavy=budget[0], n_recent=budget[1])
    Ly, steps = 2, max(6, budget[1] + 6)
    dev = torch.device("cuda")
    st = kvc.H2OState(Ly, w.batch, w.kv_heads, w.head_dim, w.n_heavy, w.n_recent, dev)
    units = sample_units(Ly, w.batch, w.kv_heads, 4, seed=7)
    inputs = {}
    for l in range(Ly):
        Q, K, V = W.h2o_prompt_layer(w, l, W.seed_of(4), dev)
        kvc.h2o_prefill(Q[None], K[None], V[None], n_heavy=w.n_heavy, n_recent=w.n_recent,
                        state=st.layer(l))
        for (ly, b, h) in units:
            if ly == l:
                inputs[(ly, b, h)] = (f64(Q[b, h:h + 1]), f64(K[b, h]), f64(V[b, h]))
        del Q, K, V
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    pos, score = st.pos.cpu().numpy(), st.score.cpu().numpy()
    ref, swaps = {}, 0
    for u in units:
        ly, b, h = u
        ref[u], sw = check_prefill_unit(*inputs[u], pos[ly, b, h], score[ly, b, h], w.n_heavy,
                                        w.n_recent)
        swaps += sw
    for s in range(steps):
        t = w.prompt_len + s
        q, kn, vn = W.decode_token(w, s, W.seed_of(4, 100), dev, layers=Ly)
        out, ev = kvc.h2o_decode_step(q, kn, vn, st, t)
        torch.cuda.synchronize()
        assert kvc.kvc_device_status() == 0
        gpu_pos, gpu_score = st.pos.cpu().numpy(), st.score.cpu().numpy()
        for u in units:
            ly, b, h = u
            swaps += check_step_unit(ref[u], f64(q[ly, b, h:h + 1]), f64(kn[ly, b, h]),
                                     f64(vn[ly, b, h]), t, w.n_recent,
                                     f64(out[ly, b, h:h + 1]), int(ev[ly, b, h]),
                                     gpu_pos[ly, b, h], "h2o step %d unit %s" % (t, u),
                                     gpu_score[ly, b, h])
    assert swaps <= 2
    del st
    torch.cuda.empty_cache()


def test_streaming_full_shape_fill_wrap_and_stream_end(kvc):
    w = W.STREAM
    S, R, D = w.n_sink, w.ring, w.head_dim
    Ly, B, H = w.layers, w.batch, w.kv_heads
    dev = torch.device("cuda")
    kc = torch.zeros((Ly, B, H, S + R, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    pos = torch.full((Ly, B, H, S + R), -1, dtype=torch.int32, device=dev)
    out = torch.empty((Ly, B, w.q_heads, D), dtype=torch.bfloat16, device=dev)
    units = sample_units(Ly, B, H, 4, seed=11)
    caches = {u: OSt.SinkCache(S, R, D) for u in units}
    seed = W.seed_of(5)
    first = list(range(S + R + 40))                    # fill, then wrap the ring
    tail = list(range(w.stream_len - (S + R), w.stream_len))  # the stream's last 2048 tokens
    check_at = {S + R - 1, S + R, S + R + 39, w.stream_len - 1}
    for t in first + tail:
        q, k, v = W.stream_token(w, t, seed, dev)
        kvc.sink_window_append(k, v, kc, vc, t, n_sink=S, n_recent=R, pos=pos)
        for u in units:
            caches[u].append(t, f64(k[u]), f64(v[u]))
        if t in check_at:
            n = min(t + 1, S + R)
            kvc.compressed_decode_attn(q, kc, vc, n_uniform=n, out=out)
            torch.cuda.synchronize()
            assert kvc.kvc_device_status() == 0
            for u in units:
                ly, b, h = u
                ref = caches[u].attend(f64(q[ly, b, h:h + 1]), t)
                assert_outputs_close(f64(out[ly, b, h:h + 1]), ref, "sink step %d unit %s" % (t, u))
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    # the cache holds the sinks and the stream's last R tokens, with their positions
    t_end = w.stream_len - 1
    want = OSt.visible_positions(t_end, S, R)
    for u in units:
        p = pos[u].cpu().numpy()
        assert list(p[:S]) == list(range(S))
        assert sorted(p[S:].tolist()) == list(want[S:])
        assert sorted(caches[u].pos.tolist()) == sorted(want.tolist())
    del kc, vc
    torch.cuda.empty_cache()
