"""Seeded synthetic inputs for the KV-cache compression path.

This module is shared by the CUDA path's tests/benchmark and by the oracle's tests;
it holds no arithmetic of the methods themselves: only random draws, the planting of
hot keys, and the shapes of the five workloads.  All values are bf16 (the dtype the
path consumes); the oracle receives the same tensors converted to float64.

The articles measure on model/dataset workloads (needle retrieval, LongBench, PG-19,
OPT inside FlexGen).  None of those is available here; these inputs stand in for
them with the same shapes: K/V ~ N(0, 1), queries ~ N(0, 1), and "hot" keys planted
by adding 3x the mean window query of their KV head so that the window votes have
real structure to find.
"""

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    layers: int
    q_heads: int
    kv_heads: int
    head_dim: int
    prompt_len: int = 0
    window: int = 0          # SnapKV observation window W (queries scored and kept)
    pool_kernel: int = 1     # SnapKV max-pool kernel P
    budget: int = 0          # SnapKV budget incl. the window
    decode_steps: int = 0
    spans_per_head: int = 0  # planted hot spans per (layer, batch, kv-head)
    span_len: int = 0
    n_heavy: int = 0         # H2O
    n_recent: int = 0        # H2O recent window
    n_sink: int = 0          # StreamingLLM sink tokens
    ring: int = 0            # StreamingLLM recent ring size
    sink_key_scale: float = 1.0
    stream_len: int = 0


# The five workloads (tiny check, Mistral-7B-shaped, long context, H2O on OPT-6.7B
# shapes, StreamingLLM on Llama-2-13B shapes).
TINY = Workload("tiny-mha4-d64-L512", batch=1, layers=1, q_heads=4, kv_heads=4, head_dim=64,
                prompt_len=512, window=8, pool_kernel=7, budget=64, decode_steps=32,
                spans_per_head=8, span_len=1, n_heavy=32, n_recent=32, n_sink=4, ring=60,
                stream_len=544)
MISTRAL = Workload("mistral7b-b2-L16384-gqa32x8-d128-kb1024", batch=2, layers=32, q_heads=32,
                   kv_heads=8, head_dim=128, prompt_len=16384, window=32, pool_kernel=7,
                   budget=1024, decode_steps=256, spans_per_head=10, span_len=16)
LONG = Workload("longctx-b1-L131072-mha32-d128-kb1024", batch=1, layers=8, q_heads=32,
                kv_heads=32, head_dim=128, prompt_len=131072, window=32, pool_kernel=7,
                budget=1024, decode_steps=128, spans_per_head=1, span_len=64)
H2O_OPT = Workload("h2o-opt6.7b-b64-mha32-d128-prompt2048-gen2048", batch=64, layers=32,
                   q_heads=32, kv_heads=32, head_dim=128, prompt_len=2048, decode_steps=2048,
                   n_heavy=204, n_recent=204)
STREAM = Workload("streamingllm-llama2-13b-b16-mha40-d128-s4-r2044", batch=16, layers=40,
                  q_heads=40, kv_heads=40, head_dim=128, n_sink=4, ring=2044,
                  sink_key_scale=4.0, stream_len=65536)

WORKLOADS = {1: TINY, 2: MISTRAL, 3: LONG, 4: H2O_OPT, 5: STREAM}


def seed_of(config_no, salt=0):
    return 1000 + config_no + 7919 * salt


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn_bf16(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def plant_hot_keys(K, Q_win, positions, group):
    """Add 3 * q_bar to the keys at ``positions`` of every (layer, batch, kv-head).

    q_bar is the mean of the bf16 window queries of the G query heads of that KV head
    over all window rows, taken in fp32 and rounded to bf16; the sum is taken in fp32
    and rounded to bf16.  K: [Ly, B, Hkv, L, d]; Q_win: [Ly, B, Hq, W, d];
    positions: int64 [Ly, B, Hkv, n] (in place on K).
    """
    Ly, B, Hkv, L, d = K.shape
    qbar = Q_win.float().reshape(Ly, B, Hkv, group * Q_win.shape[3], d).mean(dim=3)
    qbar = qbar.to(torch.bfloat16).float()                      # [Ly, B, Hkv, d]
    idx = positions.to(K.device).unsqueeze(-1).expand(*positions.shape, d)
    rows = torch.gather(K, 3, idx).float() + 3.0 * qbar.unsqueeze(3)
    K.scatter_(3, idx, rows.to(torch.bfloat16))


def hot_positions(w, gen, device):
    """Planted positions per (layer, batch, kv-head): [Ly, B, Hkv, spans*span_len].

    Spans never overlap and never touch the observation window: span s of a head
    lives in its own 2*span_len block of the prefix, at a random offset in it.
    """
    Ly, B, H = w.layers, w.batch, w.kv_heads
    n_cand = w.prompt_len - w.window
    if n_cand < w.span_len or w.spans_per_head == 0:
        return torch.zeros((Ly, B, H, 0), dtype=torch.int64, device=device)
    if w.span_len == 1:
        keys = torch.rand((Ly * B * H, n_cand), generator=gen, device=device)
        n = min(w.spans_per_head, n_cand)
        pos = keys.argsort(dim=1)[:, :n].sort(dim=1).values
        return pos.reshape(Ly, B, H, n)
    block = 2 * w.span_len
    n_blocks = n_cand // block
    spans = min(w.spans_per_head, n_blocks)
    keys = torch.rand((Ly * B * H, n_blocks), generator=gen, device=device)
    blocks = keys.argsort(dim=1)[:, :spans].sort(dim=1).values
    off = torch.randint(0, w.span_len + 1, blocks.shape, generator=gen, device=device)
    start = blocks * block + off                                 # [units, spans]
    pos = start.unsqueeze(-1) + torch.arange(w.span_len, device=device)
    return pos.reshape(Ly, B, H, spans * w.span_len)


def snapkv_prompt(w, seed, device, layers=None, full_queries=False):
    """Prompt tensors of a SnapKV workload.

    Returns dict with Q_win [Ly, B, Hq, W, d], K, V [Ly, B, Hkv, L, d] (bf16) and the
    planted positions.  With ``full_queries`` also Q_full [Ly, B, Hq, L, d], whose last
    W rows are Q_win (used by the tiny workload's H2O prefill).
    """
    Ly = w.layers if layers is None else layers
    gen = _gen(device, seed)
    B, Hq, Hkv, L, d, W = w.batch, w.q_heads, w.kv_heads, w.prompt_len, w.head_dim, w.window
    if full_queries:
        Q_full = randn_bf16((Ly, B, Hq, L, d), gen, device)
        Q_win = Q_full[:, :, :, L - W:, :].contiguous()
    else:
        Q_full = None
        Q_win = randn_bf16((Ly, B, Hq, W, d), gen, device)
    K = randn_bf16((Ly, B, Hkv, L, d), gen, device)
    V = randn_bf16((Ly, B, Hkv, L, d), gen, device)
    wl = dataclasses.replace(w, layers=Ly)
    pos = hot_positions(wl, gen, device)
    plant_hot_keys(K, Q_win, pos, Hq // Hkv)
    out = dict(Q_win=Q_win, K=K, V=V, planted=pos)
    if full_queries:
        out["Q_full"] = Q_full
    return out


def decode_token(w, step, seed, device, layers=None):
    """Fresh decode-step inputs: q [Ly, B, Hq, d], k_new/v_new [Ly, B, Hkv, d] ~ N(0, 1)."""
    Ly = w.layers if layers is None else layers
    gen = _gen(device, seed * 1000003 + step)
    q = randn_bf16((Ly, w.batch, w.q_heads, w.head_dim), gen, device)
    k = randn_bf16((Ly, w.batch, w.kv_heads, w.head_dim), gen, device)
    v = randn_bf16((Ly, w.batch, w.kv_heads, w.head_dim), gen, device)
    return q, k, v


def h2o_prompt_layer(w, layer, seed, device, batch=None):
    """One layer of an H2O prompt: Q [B, Hq, L, d], K, V [B, Hkv, L, d] ~ N(0, 1).

    Generated one layer at a time: all 32 layers of the OPT-6.7B-shaped prompt would
    hold about 100 GB at once.
    """
    B = w.batch if batch is None else batch
    gen = _gen(device, seed * 7 + layer)
    Q = randn_bf16((B, w.q_heads, w.prompt_len, w.head_dim), gen, device)
    K = randn_bf16((B, w.kv_heads, w.prompt_len, w.head_dim), gen, device)
    V = randn_bf16((B, w.kv_heads, w.prompt_len, w.head_dim), gen, device)
    return Q, K, V


def stream_token(w, t, seed, device, layers=None, batch=None):
    """StreamingLLM token t: q [Ly, B, Hq, d], k/v [Ly, B, Hkv, d] ~ N(0, 1); the keys of
    the first ``n_sink`` tokens are scaled by ``sink_key_scale`` (made into sinks)."""
    Ly = w.layers if layers is None else layers
    B = w.batch if batch is None else batch
    gen = _gen(device, seed * 1000003 + t)
    q = randn_bf16((Ly, B, w.q_heads, w.head_dim), gen, device)
    k = torch.randn((Ly, B, w.kv_heads, w.head_dim), generator=gen, device=device)
    if t < w.n_sink:
        k = k * w.sink_key_scale
    k = k.to(torch.bfloat16)
    v = randn_bf16((Ly, B, w.kv_heads, w.head_dim), gen, device)
    return q, k, v
