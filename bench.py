"""Benchmark of the SnapKV hot path on the Mistral-7B-shaped workload.

Workload (synthetic, seeded; the articles' model/dataset workloads are not available):
batch 2, 32 layers, 32 query / 8 KV heads, head dim 128, prompt 16384 bf16 tokens with
1% planted hot spans per head, observation window 32, max-pool 7, budget 1024; then
256 decode steps.  One step = SnapKV compression of all 32 layers (one library call)
followed by 256 decode steps, each one call that appends the step's K/V to the compact
cache of all 32 layers and attends over it.

Printed JSON (rank 0): value = prefix tokens compressed per second (B * L / compression
time); decode_attn = decode-attention HBM GB/s (algorithmic bytes / time) and its
fraction of the measured HBM peak; roofline of the dominant kernel (decode attention)
and of the window-score kernel; e2e through the same API with host buffers; the fp64
oracle as CPU baseline.  --impl reference times the oracle itself.
"""

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefix tokens/s compressed & decode-attn HBM GB/s (% of roofline), 1 GB300"
UNIT = "prefix tokens/s"

# Mistral-7B-shaped workload (--layers / --decode-steps shrink it for profiling only)
B, LY, HQ, HKV, D, L, W, P, KB, STEPS = 2, 32, 32, 8, 128, 16384, 32, 7, 1024, 256
G = HQ // HKV


def set_size(layers, steps):
    global LY, STEPS, CAP, UNITS
    LY, STEPS = layers, steps
    CAP = KB + STEPS
    UNITS = LY * B * HKV


set_size(LY, STEPS)


def compress_bytes():
    """Algorithmic bytes of one compression of all layers: window queries and keys read
    once, fp32 votes written and read once, kept K/V rows read and written, positions."""
    per = (HQ * W * D * 2 + HKV * L * D * 2 + 8 * HKV * (L - W) + 8 * HKV * KB * D + 4 * HKV * KB)
    return per * LY * B


def window_vote_bytes():
    """Algorithmic bytes of the window-score/vote kernel: Q_win and K read once, votes written."""
    return (HQ * W * D * 2 + HKV * L * D * 2 + 4 * HKV * L) * LY * B


def decode_bytes(n):
    """Algorithmic bytes of one decode step over n cached rows per unit (all layers): K and
    V rows read, q read, out written, the appended K/V row written."""
    return LY * B * (4 * HKV * n * D + 4 * HQ * D + 4 * HKV * D)


def decode_traffic(rows_per_launch_avg):
    """dram read + write bytes of one decode launch from the committed ncu capture, scaled
    by the rows attended (traffic grows with them); None if the kernel sources changed
    since the capture."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "decode_kernel_traffic.json")) as f:
            j = json.load(f)
        h = hashlib.sha256()
        for name in ("decode.cu", "kvc_internal.cuh"):
            with open(os.path.join(ROOT, "attention_score_kv_snapkv_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != j["sources_sha256"] or j["units"] != UNITS:
            return None
        return (j["dram_read_bytes"] + j["dram_write_bytes"]) * rows_per_launch_avg / j["rows_per_unit"]
    except Exception:
        return None


def compress_traffic():
    """dram read + write bytes of one compression of all layers (the two-pass window vote,
    then the fused selection and gather: the kernels this workload launches) from the
    committed ncu capture; None if those kernels' sources changed since the capture or
    the layer count differs."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "compress_traffic.json")) as f:
            j = json.load(f)
        h = hashlib.sha256()
        for name in j["sources"]:
            with open(os.path.join(ROOT, "attention_score_kv_snapkv_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != j["sources_sha256"] or j["units"] != UNITS:
            return None
        return sum(k["dram_read_bytes"] + k["dram_write_bytes"] for k in j["kernels"])
    except Exception:
        return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j.get("bf16_tflops", 1897.3)), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, device="cpu"):
    """Element-wise maximum of `values` over all ranks: the slowest rank sets the whole
    job's time.  Unchanged without an initialised process group of more than one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def whole_job_rate(units_per_rank, ms_max, world):
    """Units of all ranks per second, over the slowest rank's time (weak scaling)."""
    return world * units_per_rank / (ms_max / 1e3)


# ------------------------------------------------------------------------------------
# CPU baseline: the fp64 oracle on a bounded sample of the same workload
# ------------------------------------------------------------------------------------

def oracle_sample(units_sampled, decode_units, decode_steps, seed):
    """Times the oracle on `units_sampled` (layer, batch, KV head) units of the workload
    (votes, pool, top-k, gather) and on decode attention for `decode_units` units over
    `decode_steps` steps.  Returns (compress s per unit, decode s per unit-step)."""
    import numpy as np
    import torch

    import workloads as WL
    from oracle import attention as OA
    from oracle import snapkv as OS

    w = WL.MISTRAL
    import dataclasses
    w1 = dataclasses.replace(w, layers=1, batch=1)
    x = WL.snapkv_prompt(w1, seed, "cpu")
    Q = x["Q_win"].float().numpy().astype(np.float64)
    K = x["K"].float().numpy().astype(np.float64)
    V = x["V"].float().numpy().astype(np.float64)
    t0 = time.perf_counter()
    kept = []
    for u in range(units_sampled):
        h = u % HKV
        pos, kc, vc, _ = OS.compress_unit(Q[0, 0, h * G:(h + 1) * G], K[0, 0, h], V[0, 0, h], W, P, KB)
        kept.append((kc, vc))
    t_c = (time.perf_counter() - t0) / units_sampled
    rng = np.random.default_rng(seed)
    t0 = time.perf_counter()
    for u in range(decode_units):
        kc, vc = kept[u % len(kept)]
        kc, vc = kc.copy(), vc.copy()
        for s in range(decode_steps):
            q = rng.standard_normal((G, D))
            kc = np.concatenate([kc, rng.standard_normal((1, D))])
            vc = np.concatenate([vc, rng.standard_normal((1, D))])
            OA.attend_group(q, kc, vc)
    t_d = (time.perf_counter() - t0) / max(1, decode_units * decode_steps)
    return t_c, t_d


def oracle_compress_timed(units, seed, start_at):
    """One all-cores child: builds its prompt, waits for the common start time, then
    compresses `units` units with the oracle.  Returns seconds from the start to its end."""
    import numpy as np

    import dataclasses

    import workloads as WL
    from oracle import snapkv as OS
    w1 = dataclasses.replace(WL.MISTRAL, layers=1, batch=1)
    x = WL.snapkv_prompt(w1, seed, "cpu")
    Q = x["Q_win"].float().numpy().astype(np.float64)
    K = x["K"].float().numpy().astype(np.float64)
    V = x["V"].float().numpy().astype(np.float64)
    time.sleep(max(0.0, start_at - time.time()))
    for u in range(units):
        h = u % HKV
        OS.compress_unit(Q[0, 0, h * G:(h + 1) * G], K[0, 0, h], V[0, 0, h], W, P, KB)
    return time.time() - start_at


def oracle_all_cores(units_per_proc=8):
    """The oracle's compression on every host core at once: one single-threaded child per
    core, each on its own units, all starting together after their imports.  Returns
    (prefix tokens/s scaled to the workload, processes, units) or None."""
    nproc = os.cpu_count() or 1
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    start_at = time.time() + 30.0 + 0.1 * nproc  # after every child has its prompt ready
    code = ("import sys, json; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench.oracle_compress_timed(%d, 2000 + int(sys.argv[1]), %r)))"
            % (ROOT, units_per_proc, start_at))
    procs = [subprocess.Popen([sys.executable, "-c", code, str(i)], stdout=subprocess.PIPE,
                              stderr=subprocess.PIPE, text=True, env=env) for i in range(nproc)]
    ends = []
    for pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0:
            return None
        ends.append(json.loads(out.strip().splitlines()[-1]))
    # every child starts compressing at start_at; the last one to finish bounds the run
    units = nproc * units_per_proc
    return B * L * units / UNITS / max(ends), nproc, units


def cpu_baseline(units_sampled=128, decode_units=8, decode_steps=128):
    """Runs oracle_sample single-threaded in a child process (BLAS pinned to 1 thread), then
    the compression on every host core (oracle_all_cores)."""
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    code = ("import sys, json; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench.oracle_sample(%d, %d, %d, 1002)))"
            % (ROOT, units_sampled, decode_units, decode_steps))
    t0 = time.perf_counter()
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    wall = time.perf_counter() - t0
    if r.returncode != 0:
        return {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle",
                "error": r.stderr.strip().splitlines()[-1] if r.stderr else "failed"}
    t_c, t_d = json.loads(r.stdout.strip().splitlines()[-1])
    compress_s = t_c * UNITS
    decode_s = t_d * UNITS * STEPS
    one = {"value": B * L / compress_s, "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": ("%d of %d (layer,batch,kv-head) units compressed, %d units x %d decode steps; "
                      "scaled by units" % (units_sampled, UNITS, decode_units, decode_steps)),
           "compress_s_full_workload": compress_s, "decode_ms_per_token_full_workload": 1e3 * decode_s / STEPS,
           "sample_wall_s": wall}
    allc = oracle_all_cores()
    if allc is None:
        return one
    rate, nproc, units = allc
    return {"value": rate, "unit": UNIT, "cores": nproc, "kind": "oracle",
            "sample": ("%d single-threaded processes started together, %d units each (%d of %d "
                       "units), scaled by units" % (nproc, units // nproc, units, UNITS)),
            "single_core": one}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    steps, warm = args.steps, args.warmup
    # each step: one oracle unit compression (bounded sample), scaled to the workload
    import numpy as np  # noqa: F401
    times = []
    for i in range(warm + steps):
        t_c, _ = oracle_sample(1, 0, 0, 1002 + i)
        if i >= warm:
            times.append(t_c)
    per_unit = statistics.median(times)
    # the rate of the sample, in the workload's unit: each unit stands for B*L/UNITS prefix
    # tokens of the full workload
    value = B * L / (per_unit * UNITS)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": steps, "warmup": warm,
            # measured: one step is one sampled unit's compression by the oracle
            "ms_per_step": 1e3 * per_unit,
            "step": "1 of the workload's %d (layer,batch,kv-head) units per step (a bounded "
                    "sample); value = that unit's %d prefix tokens / its time" % (UNITS, B * L // UNITS),
            "extrapolated_ms_full_workload": 1e3 * per_unit * UNITS,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": "1 (layer,batch,kv-head) unit per step, scaled by %d units" % UNITS},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_dict():
    full = LY == 32 and STEPS == 256
    return {"workload": "mistral7b-b2-L16384-gqa32x8-d128-w32-p7-kb1024-decode256" if full else
            "PROFILING SUBSET (not a bench line): mistral7b-shaped, %d layers, %d decode steps" % (LY, STEPS),
            "batch": B, "layers": LY, "q_heads": HQ, "kv_heads": HKV, "head_dim": D,
            "prompt_len": L, "window": W, "pool_kernel": P, "budget": KB, "decode_steps": STEPS,
            "l2": "inputs larger than L2 (K/V 4.3 GB, compact caches 0.34 GB)"}


# ------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------

def _events_ms(fn, n, warm):
    """Median-free mean of n timed calls of fn (CUDA events on the current stream)."""
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(n):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n


def measure_long(kvc, WL, dev, hbm_peak):
    """Long-context SnapKV (batch 1, 8 layers, 32 MHA heads, L 131072, budget 1024): one
    compression of all layers, then 128 decode steps with the fused append."""
    import torch
    w = WL.LONG
    x = WL.snapkv_prompt(w, WL.seed_of(3), dev)
    Ly, Bb, H, Dd, Ll, Wn, Kb, S = w.layers, w.batch, w.kv_heads, w.head_dim, w.prompt_len, \
        w.window, w.budget, w.decode_steps
    cap = Kb + S
    kc = torch.empty((Ly, Bb, H, cap, Dd), dtype=torch.bfloat16, device=dev)
    vc, pos = torch.empty_like(kc), torch.empty((Ly, Bb, H, cap), dtype=torch.int32, device=dev)
    nv = torch.empty((Ly, Bb, H), dtype=torch.int32, device=dev)

    def compress():
        kvc.snapkv_compress(x["Q_win"], x["K"], x["V"], keep_window=Wn, pool_kernel=w.pool_kernel,
                            budget=Kb, cap=cap, k_out=kc, v_out=vc, pos_out=pos, n_valid_out=nv)

    c_ms = _events_ms(compress, 5, 3)
    per = (w.q_heads * Wn * Dd * 2 + H * Ll * Dd * 2 + 8 * H * (Ll - Wn) + 8 * H * Kb * Dd + 4 * H * Kb)
    c_bytes = per * Ly * Bb
    dec = [WL.decode_token(w, s, WL.seed_of(3, 100), dev) for s in range(8)]
    out = torch.empty((Ly, Bb, w.q_heads, Dd), dtype=torch.bfloat16, device=dev)

    def steps():
        for s in range(S):
            q, kn, vn = dec[s % 8]
            kvc.compressed_decode_attn(q, kc, vc, n_valid=nv, n_uniform=Kb + s + 1, k_new=kn,
                                       v_new=vn, pos=pos, new_pos=Ll + s, out=out)

    def timed(fn):
        compress()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / S

    d_eager = timed(steps)  # (also allocates the cached workspace before the capture)
    # the 128 calls captured once as a CUDA graph, as the headline decode is
    compress()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        steps()
    torch.cuda.synchronize()
    d_ms = timed(graph.replay)
    d_bytes = sum(Ly * Bb * (4 * H * (Kb + s + 1) * Dd + 4 * w.q_heads * Dd + 4 * H * Dd)
                  for s in range(S)) / S
    # The same compression from the window rows' log-sum-exp, which a prefill through
    # prefill_attention_lse would return; here the harness forms it (fp32, one layer at a
    # time) because a prefill of this prompt takes seconds.  Timed: the vote pass and the
    # selection only.
    lse = torch.full((Ly, Bb, w.q_heads, Ll), float("nan"), dtype=torch.float32, device=dev)
    G = w.q_heads // H
    rows = torch.arange(Ll - Wn, Ll, device=dev)
    keys = torch.arange(Ll, device=dev)
    for l in range(Ly):
        for b in range(Bb):
            qf = x["Q_win"][l, b].float().view(H, G * Wn, Dd)
            sc = torch.matmul(qf, x["K"][l, b].float().transpose(1, 2)) / math.sqrt(Dd)
            sc = sc.view(H, G, Wn, Ll).masked_fill(keys.view(1, 1, 1, Ll) > rows.view(1, 1, Wn, 1),
                                                    float("-inf"))
            lse[l, b, :, Ll - Wn:] = torch.logsumexp(sc, dim=-1).view(w.q_heads, Wn)
            del qf, sc
    votes = torch.empty((Ly, Bb, H, Ll), dtype=torch.float32, device=dev)
    v_ms = _events_ms(lambda: kvc.snapkv_votes_from_lse(x["Q_win"], x["K"], lse, votes_out=votes), 5, 3)
    s_ms = _events_ms(lambda: kvc.snapkv_select(votes, x["K"], x["V"], keep_window=Wn,
                                                pool_kernel=w.pool_kernel, budget=Kb, cap=cap), 5, 3)
    v_bytes = Ly * Bb * (H * Ll * Dd * 2 + w.q_heads * Wn * Dd * 2 + w.q_heads * Wn * 4 + H * Ll * 4)
    status = kvc.kvc_device_status()
    del x, kc, vc, graph, lse, votes
    torch.cuda.empty_cache()
    return {"workload": w.name, "compress_ms": c_ms, "prefix_tokens_per_s": Bb * Ll / (c_ms / 1e3),
            "compress_GBps": c_bytes / (c_ms / 1e3) / 1e9,
            "compress_frac_of_hbm_peak": c_bytes / (c_ms / 1e3) / 1e9 / hbm_peak,
            "decode_ms_per_step": d_ms, "decode_GBps": d_bytes / (d_ms / 1e3) / 1e9,
            "decode_frac_of_hbm_peak": d_bytes / (d_ms / 1e3) / 1e9 / hbm_peak,
            "decode_launch": "one call per step for all layers; the 128 calls replayed as a CUDA graph",
            "decode_eager_ms_per_step": d_eager,
            "votes_from_lse_ms": v_ms, "votes_from_lse_GBps": v_bytes / (v_ms / 1e3) / 1e9,
            "votes_from_lse_frac_of_hbm_peak": v_bytes / (v_ms / 1e3) / 1e9 / hbm_peak,
            "compress_from_lse_ms": v_ms + s_ms,
            "compress_from_lse_prefix_tokens_per_s": Bb * Ll / ((v_ms + s_ms) / 1e3),
            "device_status": status}


def measure_h2o(kvc, WL, dev, hbm_peak, steps=64, n_heavy=None, n_recent=None):
    """H2O on OPT-6.7B shapes (batch 64, 32 layers, 32 MHA heads, prompt 2048, 204 heavy +
    204 recent, or the given budget): layer-by-layer prefill (scores + cut), then decode
    steps of all layers."""
    import dataclasses

    import torch
    w = WL.H2O_OPT
    if n_heavy is not None:
        w = dataclasses.replace(w, n_heavy=n_heavy, n_recent=n_recent)
    Ly, Bb, H, Dd = w.layers, w.batch, w.kv_heads, w.head_dim
    st = kvc.H2OState(Ly, Bb, H, Dd, w.n_heavy, w.n_recent, dev)
    pre_ms = []
    for l in range(Ly):
        Q, K, V = WL.h2o_prompt_layer(w, l, WL.seed_of(4), dev)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        kvc.h2o_prefill(Q[None], K[None], V[None], n_heavy=w.n_heavy, n_recent=w.n_recent,
                        state=st.layer(l))
        b.record()
        torch.cuda.synchronize()
        pre_ms.append(a.elapsed_time(b))
        del Q, K, V
    torch.cuda.empty_cache()
    toks = [WL.decode_token(w, s, WL.seed_of(4, 100), dev) for s in range(4)]
    out = torch.empty((Ly, Bb, w.q_heads, Dd), dtype=torch.bfloat16, device=dev)
    ev = torch.empty((Ly, Bb, H), dtype=torch.int32, device=dev)
    t0 = w.prompt_len
    for s in range(4):  # warm-up steps
        q, kn, vn = toks[s]
        kvc.h2o_decode_step(q, kn, vn, st, t0 + s, out=out, evicted=ev)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for s in range(steps):
        q, kn, vn = toks[s % 4]
        kvc.h2o_decode_step(q, kn, vn, st, t0 + 4 + s, out=out, evicted=ev)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    n = w.n_heavy + w.n_recent + 1
    step_bytes = Ly * Bb * H * (n * (4 * Dd + 12) + 4 * (w.q_heads // H) * Dd + 4 * Dd)
    status = kvc.kvc_device_status()
    del st
    torch.cuda.empty_cache()
    # causal Q.K^T flops of the prefill scores (half the square) per layer
    pre_flops = 2.0 * Bb * w.q_heads * w.prompt_len * w.prompt_len / 2 * Dd
    return {"workload": w.name, "n_heavy": w.n_heavy, "n_recent": w.n_recent,
            "prefill_ms_per_layer": statistics.median(pre_ms),
            "prefill_causal_qk_TFLOPs": pre_flops / (statistics.median(pre_ms) / 1e3) / 1e12,
            "step_ms": ms, "step_GBps": step_bytes / (ms / 1e3) / 1e9,
            "step_frac_of_hbm_peak": step_bytes / (ms / 1e3) / 1e9 / hbm_peak,
            "steps_timed": steps, "device_status": status}


def h2o_built_state(kvc, dev, layers, heads, head_dim, n_heavy, n_recent, t0, seed):
    """An H2O cache of every slot filled (random K/V, scores, distinct positions with the
    last n_recent positions recent), built directly: a prefill of a prompt that long would
    only be timed here, not needed."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    S = n_heavy + n_recent + 1
    st = kvc.H2OState(layers, 1, heads, head_dim, n_heavy, n_recent, dev)
    st.k.copy_(torch.randn(st.k.shape, generator=g, device=dev).to(torch.bfloat16))
    st.v.copy_(torch.randn(st.v.shape, generator=g, device=dev).to(torch.bfloat16))
    st.score.copy_(1.0 + 99.0 * torch.rand(st.score.shape, generator=g, device=dev))
    heavy = torch.randperm(t0 - n_recent, generator=g, device=dev)[:n_heavy]
    recent = torch.arange(t0 - n_recent, t0, device=dev)
    pos = torch.cat([heavy, recent, torch.tensor([-1], device=dev)]).to(torch.int32)
    st.pos.copy_(pos.expand(st.pos.shape))
    st.n_used.fill_(S - 1)
    st.free_slot.fill_(S - 1)
    return st


def measure_h2o_long_budget(kvc, WL, dev, hbm_peak, steps=32):
    """H2O steps with a budget of 20% of a 131072-token context (13107 heavy + 13107
    recent) on the long-context shapes (batch 1, 8 layers, 32 heads, D 128): 256 units of
    26215 slots, too few units for one CTA each to fill the GPU, so the step splits every
    unit's cache over several CTAs."""
    import torch
    w = WL.LONG
    nh = nr = w.prompt_len // 10
    t0 = w.prompt_len
    st = h2o_built_state(kvc, dev, w.layers, w.kv_heads, w.head_dim, nh, nr, t0, 31)
    g = torch.Generator(device=dev)
    g.manual_seed(32)
    q = torch.randn((w.layers, 1, w.q_heads, w.head_dim), generator=g, device=dev).to(torch.bfloat16)
    kn = torch.randn((w.layers, 1, w.kv_heads, w.head_dim), generator=g, device=dev).to(torch.bfloat16)
    vn = torch.randn_like(kn)
    out = torch.empty_like(q)
    ev = torch.empty((w.layers, 1, w.kv_heads), dtype=torch.int32, device=dev)
    for s in range(4):
        kvc.h2o_decode_step(q, kn, vn, st, t0 + s, out=out, evicted=ev)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for s in range(steps):
        kvc.h2o_decode_step(q, kn, vn, st, t0 + 4 + s, out=out, evicted=ev)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    n = nh + nr + 1
    units = w.layers * w.kv_heads
    step_bytes = units * (n * (4 * w.head_dim + 12) + 8 * w.head_dim)
    status = kvc.kvc_device_status()
    del st
    torch.cuda.empty_cache()
    return {"workload": "h2o budget 20%% of %d tokens (%d heavy + %d recent), %d layers x %d heads, "
                        "batch 1, D %d" % (t0, nh, nr, w.layers, w.kv_heads, w.head_dim),
            "units": units, "slots_per_unit": n, "step_ms": ms,
            "step_GBps": step_bytes / (ms / 1e3) / 1e9,
            "step_frac_of_hbm_peak": step_bytes / (ms / 1e3) / 1e9 / hbm_peak,
            "steps_timed": steps, "device_status": status}


def measure_budget(kvc, Q, K, V, budget, hbm_peak, reps=5):
    """Compression of the headline prompt at another budget (the cache holds exactly the
    budget): CUDA-event time per call after two warm-up calls."""
    import torch
    Ly, Bb, Hkv, Ll, Dd = K.shape
    for _ in range(2):
        res = kvc.snapkv_compress(Q, K, V, keep_window=W, pool_kernel=P, budget=budget, cap=budget)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        kvc.snapkv_compress(Q, K, V, keep_window=W, pool_kernel=P, budget=budget, cap=budget,
                            k_out=res["k"], v_out=res["v"], pos_out=res["pos"],
                            n_valid_out=res["n_valid"])
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps
    per = (Q.shape[2] * W * Dd * 2 + Hkv * Ll * Dd * 2 + 8 * Hkv * (Ll - W)
           + 8 * Hkv * budget * Dd + 4 * Hkv * budget)
    byts = Ly * Bb * per
    status = kvc.kvc_device_status()
    del res
    torch.cuda.empty_cache()
    return {"budget": budget, "compress_ms": ms, "prefix_tokens_per_s": Bb * Ll / (ms / 1e3),
            "compress_frac_of_hbm_peak": byts / (ms / 1e3) / 1e9 / hbm_peak,
            "device_status": status}


def measure_pool(kvc, Q, K, V, planted, pool_kernel, pool_avg, reps=5):
    """Pooling ablation on the headline prompt: max-pool, average pool or none (kernel 1).
    Reports the compression time and the share of the planted hot-span positions that
    the selection keeps (a synthetic stand-in for the retrieval ablation)."""
    import torch
    Ly, Bb, Hkv, Ll, Dd = K.shape
    kw = dict(keep_window=W, pool_kernel=pool_kernel, budget=KB, cap=KB, pool_avg=pool_avg)
    res = kvc.snapkv_compress(Q, K, V, **kw)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        kvc.snapkv_compress(Q, K, V, k_out=res["k"], v_out=res["v"], pos_out=res["pos"],
                            n_valid_out=res["n_valid"], **kw)
    b.record()
    torch.cuda.synchronize()
    kept = torch.zeros((Ly, Bb, Hkv, Ll), dtype=torch.bool, device=K.device)
    kept.scatter_(3, res["pos"].long().clamp(min=0), True)
    recall = kept.gather(3, planted).float().mean().item() if planted.numel() else None
    status = kvc.kvc_device_status()
    del res, kept
    torch.cuda.empty_cache()
    return {"pool": "none" if pool_kernel == 1 else ("avg" if pool_avg else "max"),
            "pool_kernel": pool_kernel, "compress_ms": a.elapsed_time(b) / reps,
            "planted_positions_kept": recall, "device_status": status}


def measure_prefill(kvc, WL, dev, tf_peak, layers=2, reps=3):
    """Prompt self-attention with the votes as a by-product, on `layers` layers of the
    Mistral-7B-shaped prompt (full 16384-token causal attention): the plain prefill, the
    prefill with votes, selection from those votes, and the alternative of the plain
    prefill followed by snapkv_compress."""
    import torch
    w = WL.MISTRAL
    x = WL.snapkv_prompt(w, WL.seed_of(2, 7), dev, layers=layers, full_queries=True)
    Qf, K, V, Qw = x["Q_full"], x["K"], x["V"], x["Q_win"]
    out = torch.empty_like(Qf)
    votes = torch.empty((layers, w.batch, w.kv_heads, w.prompt_len), dtype=torch.float32, device=dev)

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    kw = dict(keep_window=w.window, pool_kernel=w.pool_kernel, budget=w.budget, cap=w.budget)
    t_plain = timed(lambda: kvc.snapkv_prefill_attention(Qf, K, V, out=out))
    t_votes = timed(lambda: kvc.snapkv_prefill_attention(Qf, K, V, window=w.window, out=out,
                                                         votes_out=votes))
    t_select = timed(lambda: kvc.snapkv_select(votes, K, V, **kw))
    t_compress = timed(lambda: kvc.snapkv_compress(Qw, K, V, **kw))
    status = kvc.kvc_device_status()
    # causal attention work: Q.K^T and P.V over the lower triangle (incl. diagonal)
    L = w.prompt_len
    flop = layers * w.batch * w.q_heads * 2 * 2 * w.head_dim * (L * (L + 1) / 2)
    del x, Qf, K, V, Qw, out, votes
    torch.cuda.empty_cache()
    return {"workload": "mistral7b-b2-L16384-gqa32x8-d128, %d layers" % layers,
            "prefill_ms_per_layer": t_plain / layers,
            "prefill_TFLOPs": flop / (t_plain / 1e3) / 1e12,
            "prefill_frac_of_bf16_peak": flop / (t_plain / 1e3) / 1e12 / tf_peak,
            "prefill_with_votes_ms_per_layer": t_votes / layers,
            "select_from_votes_ms_per_layer": t_select / layers,
            "separate_compress_ms_per_layer": t_compress / layers,
            "fused_path_ms_per_layer": (t_votes + t_select) / layers,
            "unfused_path_ms_per_layer": (t_plain + t_compress) / layers,
            "device_status": status}


def measure_lse_route(kvc, WL, dev, tf_peak, hbm_peak, reps=3):
    """The scores through the rows' log-sum-exp: prefill_attention_lse, then
    snapkv_votes_from_lse (one pass over the keys) and the selection, against the plain
    prefill followed by the direct route (snapkv_compress / h2o_prefill).  SnapKV on all
    32 layers of the Mistral-7B-shaped prompt (the headline's compression workload, with
    every prompt query for the prefill); H2O on one layer of the OPT-6.7B-shaped prompt
    (every query votes)."""
    import torch

    def timed(fn, n=reps):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    w = WL.MISTRAL
    layers = w.layers
    x = WL.snapkv_prompt(w, WL.seed_of(2, 7), dev, layers=layers, full_queries=True)
    Qf, K, V, Qw = x["Q_full"], x["K"], x["V"], x["Q_win"]
    out = torch.empty_like(Qf)
    lse = torch.empty(Qf.shape[:4], dtype=torch.float32, device=dev)
    votes = torch.empty((layers, w.batch, w.kv_heads, w.prompt_len), dtype=torch.float32, device=dev)
    kw = dict(keep_window=w.window, pool_kernel=w.pool_kernel, budget=w.budget, cap=w.budget)
    kvc.prefill_attention_lse(Qf, K, V, out=out, lse_out=lse)
    torch.cuda.synchronize()
    time.sleep(1.0)  # the compressions are timed away from the power draw of the prefill
    t_vfl = timed(lambda: kvc.snapkv_votes_from_lse(Qw, K, lse, votes_out=votes), 10)
    t_select = timed(lambda: kvc.snapkv_select(votes, K, V, **kw), 10)
    t_compress = timed(lambda: kvc.snapkv_compress(Qw, K, V, **kw), 10)
    t_plain = timed(lambda: kvc.snapkv_prefill_attention(Qf, K, V, out=out), 1)
    t_lse = timed(lambda: kvc.prefill_attention_lse(Qf, K, V, out=out, lse_out=lse), 1)
    L, Wn = w.prompt_len, w.window
    # algorithmic bytes of the vote pass: K once, the window queries, their lse, the votes
    vfl_bytes = layers * w.batch * (w.kv_heads * L * w.head_dim * 2 + w.q_heads * Wn * w.head_dim * 2
                                    + w.q_heads * Wn * 4 + w.kv_heads * L * 4)
    snap = {"workload": "mistral7b-b2-L16384-gqa32x8-d128, %d layers" % layers,
            "prefill_ms": t_plain, "prefill_lse_ms": t_lse,
            "votes_from_lse_ms": t_vfl,
            "votes_from_lse_GBps": vfl_bytes / (t_vfl / 1e3) / 1e9,
            "votes_from_lse_frac_of_hbm_peak": vfl_bytes / (t_vfl / 1e3) / 1e9 / hbm_peak,
            "select_ms": t_select,
            "compress_from_lse_ms": t_vfl + t_select,
            "compress_from_lse_prefix_tokens_per_s": w.batch * L / ((t_vfl + t_select) / 1e3),
            "compress_direct_ms": t_compress,
            "compress_direct_prefix_tokens_per_s": w.batch * L / (t_compress / 1e3),
            "lse_route_ms": t_lse + t_vfl + t_select,
            "direct_route_ms": t_plain + t_compress}
    del x, Qf, K, V, Qw, out, lse, votes
    torch.cuda.empty_cache()

    w = WL.H2O_OPT
    Q, K, V = WL.h2o_prompt_layer(w, 0, WL.seed_of(4), dev)
    Q, K, V = Q[None], K[None], V[None]
    out = torch.empty_like(Q)
    lse = torch.empty(Q.shape[:4], dtype=torch.float32, device=dev)
    scores = torch.empty((1, w.batch, w.kv_heads, w.prompt_len), dtype=torch.float32, device=dev)
    st = kvc.H2OState(1, w.batch, w.kv_heads, w.head_dim, w.n_heavy, w.n_recent, dev)
    hk = dict(n_heavy=w.n_heavy, n_recent=w.n_recent, state=st)
    time.sleep(1.0)
    t_plain = timed(lambda: kvc.snapkv_prefill_attention(Q, K, V, out=out))
    t_lse = timed(lambda: kvc.prefill_attention_lse(Q, K, V, out=out, lse_out=lse))
    t_vfl = timed(lambda: kvc.snapkv_votes_from_lse(Q, K, lse, votes_out=scores))
    t_cut = timed(lambda: kvc.h2o_prefill_from_votes(scores, K, V, n_q_heads=w.q_heads, **hk))
    t_direct = timed(lambda: kvc.h2o_prefill(Q, K, V, **hk))
    status = kvc.kvc_device_status()
    Lp = w.prompt_len
    qk_flops = 2.0 * w.batch * w.q_heads * Lp * (Lp + 1) / 2 * w.head_dim
    h2o = {"workload": w.name + ", 1 layer",
           "prefill_ms": t_plain, "prefill_lse_ms": t_lse,
           "scores_from_lse_ms": t_vfl,
           "scores_from_lse_causal_qk_TFLOPs": qk_flops / (t_vfl / 1e3) / 1e12,
           "scores_from_lse_frac_of_bf16_peak": qk_flops / (t_vfl / 1e3) / 1e12 / tf_peak,
           "cut_from_scores_ms": t_cut,
           "h2o_prefill_direct_ms": t_direct,
           "lse_route_ms": t_lse + t_vfl + t_cut,
           "direct_route_ms": t_plain + t_direct}
    del Q, K, V, out, lse, scores, st
    torch.cuda.empty_cache()
    return {"snapkv": snap, "h2o": h2o, "device_status": status}


def measure_stream(kvc, WL, dev, hbm_peak, steps=256, n_sink=None, ring=None):
    """StreamingLLM on Llama-2-13B shapes (batch 16, 40 layers, 40 MHA heads, 4 sinks +
    2044-token ring, or the given sink count and ring): fill the cache, then steady-state
    steps of append + attention."""
    import dataclasses

    import torch
    w = WL.STREAM
    if n_sink is not None:
        w = dataclasses.replace(w, n_sink=n_sink, ring=ring)
    Ly, Bb, H, Dd, S, R = w.layers, w.batch, w.kv_heads, w.head_dim, w.n_sink, w.ring
    kc = torch.zeros((Ly, Bb, H, S + R, Dd), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    pos = torch.full((Ly, Bb, H, S + R), -1, dtype=torch.int32, device=dev)
    toks = [WL.stream_token(w, t, WL.seed_of(5), dev) for t in range(8)]
    for t in range(S + R):
        _, k, v = toks[t % 8]
        kvc.sink_window_append(k, v, kc, vc, t, n_sink=S, n_recent=R, pos=pos)
    out = torch.empty((Ly, Bb, w.q_heads, Dd), dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()
    t0 = S + R

    def step(t):
        q, k, v = toks[t % 8]
        kvc.sink_window_append(k, v, kc, vc, t, n_sink=S, n_recent=R, pos=pos)
        kvc.compressed_decode_attn(q, kc, vc, n_uniform=S + R, out=out)

    for t in range(t0, t0 + 4):
        step(t)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(steps):
        step(t0 + 4 + i)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    step_bytes = Ly * Bb * (4 * H * (S + R) * Dd + 4 * w.q_heads * Dd + 4 * H * Dd + 4 * H)
    status = kvc.kvc_device_status()
    del kc, vc
    torch.cuda.empty_cache()
    return {"workload": w.name, "n_sink": S, "ring": R, "step_ms": ms,
            "step_GBps": step_bytes / (ms / 1e3) / 1e9,
            "step_frac_of_hbm_peak": step_bytes / (ms / 1e3) / 1e9 / hbm_peak,
            "steps_timed": steps, "launches_per_step": 2, "device_status": status}


def run_host_link(args):
    """Host-link rates behind the end-to-end number (printed as one JSON line): 2 GiB
    from pinned host memory to the device over 1, 2, 4 and 8 streams, the same as 64 MB
    copies on one stream, and 2 GiB device to pinned host (best of three, CUDA events);
    then the library's gather reading 128 MiB of V rows in place from pinned host memory
    (SM loads over the link, checked against the rows)."""
    import torch

    n = 2 * 1024 ** 3
    h = torch.empty(n, dtype=torch.uint8).pin_memory()
    d = torch.empty(n, dtype=torch.uint8, device="cuda")
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    cur = torch.cuda.current_stream()

    def best(fn):
        ms = []
        for _ in range(3):
            torch.cuda.synchronize()
            a, b = ev(), ev()
            a.record(cur)
            fn()
            b.record(cur)
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        return n / (min(ms) / 1e3) / 1e9

    res = {"bytes": n}
    for ns in (1, 2, 4, 8):
        ss = [torch.cuda.Stream() for _ in range(ns)]
        chunk = n // ns

        def h2d():
            for i, st in enumerate(ss):
                st.wait_stream(cur)
                with torch.cuda.stream(st):
                    d[i * chunk:(i + 1) * chunk].copy_(h[i * chunk:(i + 1) * chunk], non_blocking=True)
            for st in ss:
                cur.wait_stream(st)
        res["h2d_GBps_streams%d" % ns] = best(h2d)

    def h2d_chunks():
        c = 64 * 1024 ** 2
        for i in range(0, n, c):
            d[i:i + c].copy_(h[i:i + c], non_blocking=True)
    res["h2d_GBps_64MB_copies_one_stream"] = best(h2d_chunks)
    res["d2h_GBps"] = best(lambda: h.copy_(d, non_blocking=True))
    del h, d
    # SM loads over the same link: the library's gather reading a pinned host V in place
    # (snapkv_select with a budget covering the prompt keeps every row: 8 units x 65536
    # rows x 256 B of V from the host, K from the device)
    import attention_score_kv_snapkv_gb300 as kvc
    L = 65536
    kd = torch.randn((1, 1, 8, L, 128), device="cuda").to(torch.bfloat16)
    vh = torch.empty((1, 1, 8, L, 128), dtype=torch.bfloat16).pin_memory()
    vh.copy_(kd.cpu())
    vd = vh.to("cuda")
    votes = torch.zeros((1, 1, 8, L), dtype=torch.float32, device="cuda")
    vbytes = vh.numel() * vh.element_size()

    def gather_rate(v):
        ms = []
        for _ in range(4):
            torch.cuda.synchronize()
            a, b = ev(), ev()
            a.record(cur)
            r = kvc.snapkv_select(votes, kd, v, keep_window=32, pool_kernel=7, budget=L)
            b.record(cur)
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        assert torch.equal(r["v"], vd), "gathered rows differ from the input rows"
        return min(ms[1:])

    t_host, t_dev = gather_rate(vh), gather_rate(vd)
    res["gather_v_bytes"] = vbytes
    res["gather_host_v_ms"] = t_host
    res["gather_device_v_ms"] = t_dev
    res["gather_host_v_GBps"] = vbytes / (t_host / 1e3) / 1e9
    res["device_status"] = kvc.kvc_device_status()
    print(json.dumps({"host_link": res}), flush=True)
    return 0


def run_profile_driver(args):
    """Short fixed workloads for ncu captures (no timing printed):
    h2o-split: four H2O steps of one layer with a cache of 20% of a 131072-token context
            (32 units of 26215 slots: the split step);
    decode: four launches of the 32-layer Mistral-shaped decode at n = 1100 on the
            compact caches (the prompt is freed before the launches);
    aux:    two layers of the H2O (OPT-6.7B) shape, prefill + 4 steps, then two layers
            of the StreamingLLM (Llama-2-13B) shape, fill + 4 steady-state steps;
    long:   three compressions of two layers of the long-context shape (L = 131072);
    prefill: three prefill attentions with votes on one layer, batch 1 of the
            Mistral-7B-shaped prompt (32 query heads, 8 KV heads, L = 16384, D = 128);
    lse:    the log-sum-exp route: one prefill_attention_lse and three
            snapkv_votes_from_lse on four layers of the Mistral-7B-shaped prompt, then the
            same on one layer of the OPT-6.7B-shaped H2O prompt at batch 16 (every query
            votes)."""
    import torch

    import attention_score_kv_snapkv_gb300 as kvc
    import workloads as WL

    dev = torch.device("cuda")
    if args.profile == "long":
        w = WL.LONG
        x = WL.snapkv_prompt(w, 5, dev, layers=2)
        for _ in range(3):
            kvc.snapkv_compress(x["Q_win"], x["K"], x["V"], keep_window=w.window,
                                pool_kernel=w.pool_kernel, budget=w.budget, cap=w.budget)
    elif args.profile == "prefill":
        import dataclasses
        w = dataclasses.replace(WL.MISTRAL, batch=1)
        x = WL.snapkv_prompt(w, 5, dev, layers=1, full_queries=True)
        out = torch.empty_like(x["Q_full"])
        votes = torch.empty((1, 1, w.kv_heads, w.prompt_len), dtype=torch.float32, device=dev)
        for _ in range(3):
            kvc.snapkv_prefill_attention(x["Q_full"], x["K"], x["V"], window=w.window, out=out,
                                         votes_out=votes)
    elif args.profile == "lse":
        import dataclasses
        w = WL.MISTRAL
        x = WL.snapkv_prompt(w, 5, dev, layers=4, full_queries=True)
        out, lse = kvc.prefill_attention_lse(x["Q_full"], x["K"], x["V"])
        votes = torch.empty((4, w.batch, w.kv_heads, w.prompt_len), dtype=torch.float32, device=dev)
        for _ in range(3):
            kvc.snapkv_votes_from_lse(x["Q_win"], x["K"], lse, votes_out=votes)
        torch.cuda.synchronize()
        del x, out, lse, votes
        torch.cuda.empty_cache()
        w = dataclasses.replace(WL.H2O_OPT, batch=16)
        Q, K, V = WL.h2o_prompt_layer(w, 0, WL.seed_of(4), dev)
        out, lse = kvc.prefill_attention_lse(Q[None], K[None], V[None])
        del out
        for _ in range(3):
            kvc.snapkv_votes_from_lse(Q[None], K[None], lse)
    elif args.profile == "h2o-split":
        # one layer of the H2O cache at 20% of a 131072-token context: 32 units of 26215
        # slots, each split over several CTAs; four steps
        w = WL.LONG
        st = h2o_built_state(kvc, dev, 1, w.kv_heads, w.head_dim, w.prompt_len // 10,
                             w.prompt_len // 10, w.prompt_len, 31)
        q, kn, vn = WL.decode_token(w, 0, 5, dev, layers=1)
        for s in range(4):
            kvc.h2o_decode_step(q, kn, vn, st, w.prompt_len + s)
    elif args.profile == "decode":
        w = WL.MISTRAL
        x = WL.snapkv_prompt(w, 5, dev)
        res = kvc.snapkv_compress(x["Q_win"], x["K"], x["V"], keep_window=W, pool_kernel=P,
                                  budget=KB, cap=KB + 256)
        del x
        torch.cuda.empty_cache()
        q, _, _ = WL.decode_token(w, 0, 5, dev)
        out = torch.empty_like(q)
        for _ in range(4):
            kvc.compressed_decode_attn(q, res["k"], res["v"], n_uniform=1100, out=out)
    else:
        w = WL.H2O_OPT
        Ly = 2
        st = kvc.H2OState(Ly, w.batch, w.kv_heads, w.head_dim, w.n_heavy, w.n_recent, dev)
        for l in range(Ly):
            Q, K, V = WL.h2o_prompt_layer(w, l, WL.seed_of(4), dev)
            kvc.h2o_prefill(Q[None], K[None], V[None], n_heavy=w.n_heavy, n_recent=w.n_recent,
                            state=st.layer(l))
            del Q, K, V
        for s in range(4):
            q, kn, vn = WL.decode_token(w, s, WL.seed_of(4, 100), dev, layers=Ly)
            kvc.h2o_decode_step(q, kn, vn, st, w.prompt_len + s)
        torch.cuda.synchronize()
        del st
        torch.cuda.empty_cache()
        w = WL.STREAM
        S, R = w.n_sink, w.ring
        kc = torch.zeros((Ly, w.batch, w.kv_heads, S + R, w.head_dim), dtype=torch.bfloat16, device=dev)
        vc = torch.zeros_like(kc)
        for t in range(S + R + 4):
            q, k, v = WL.stream_token(w, t, WL.seed_of(5), dev, layers=Ly)
            kvc.sink_window_append(k, v, kc, vc, t, n_sink=S, n_recent=R)
            if t >= S + R:
                kvc.compressed_decode_attn(q, kc, vc, n_uniform=S + R)
    torch.cuda.synchronize()
    status = kvc.kvc_device_status()
    if status:
        raise RuntimeError("device status flags %#x" % status)
    return 0


def run_ours(args):
    import torch
    import torch.distributed as dist

    import attention_score_kv_snapkv_gb300 as kvc
    import workloads as WL

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    hbm_peak, tf_peak, peak_kind = peaks()

    w = WL.MISTRAL
    x = WL.snapkv_prompt(w, WL.seed_of(2, rank), dev, layers=LY)
    Q, K, V = x["Q_win"], x["K"], x["V"]
    dec = [WL.decode_token(w, s, WL.seed_of(2, 100 + rank), dev, layers=LY) for s in range(STEPS)]
    kc = torch.empty((LY, B, HKV, CAP, D), dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    pos = torch.empty((LY, B, HKV, CAP), dtype=torch.int32, device=dev)
    nv = torch.empty((LY, B, HKV), dtype=torch.int32, device=dev)
    outs = torch.empty((LY, B, HQ, D), dtype=torch.bfloat16, device=dev)

    def compress():
        kvc.snapkv_compress(Q, K, V, keep_window=W, pool_kernel=P, budget=KB, cap=CAP, k_out=kc,
                            v_out=vc, pos_out=pos, n_valid_out=nv)

    def decode(s):
        # n_uniform: the exact bound on the rows after this step's append (KB + s + 1)
        q, kn, vn = dec[s]
        kvc.compressed_decode_attn(q, kc, vc, n_valid=nv, n_uniform=KB + s + 1, k_new=kn,
                                   v_new=vn, pos=pos, new_pos=L + s, out=outs)

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    # The 256 decode calls of a step are captured once as a CUDA graph (as a serving loop
    # would) and replayed after each compression, so host submission is not timed.
    compress()
    for s_ in range(STEPS):  # eager pass: allocates the cached workspace before capture
        decode(s_)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for s_ in range(STEPS):
            decode(s_)
    torch.cuda.synchronize()

    def step(record):
        e0, e1, e2 = ev(), ev(), ev()
        e0.record(stream)
        compress()
        e1.record(stream)
        graph.replay()
        e2.record(stream)
        if record is not None:
            record.append((e0, e1, e2))

    for _ in range(args.warmup):
        step(None)
    torch.cuda.synchronize()
    status = kvc.kvc_device_status()
    clocks = ClockSampler(dev.index)
    recs = []
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_all0, t_all1 = ev(), ev()
    t_all0.record(stream)
    for _ in range(args.steps):
        step(recs)
    t_all1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if ws > 1:
        dist.barrier()
    status |= kvc.kvc_device_status()
    if status:  # a kernel gave up on a bounded wait: its results and timings are invalid
        raise RuntimeError("device status flags %#x after the timed steps" % status)
    total_ms = t_all0.elapsed_time(t_all1)
    comp_ms = [a.elapsed_time(b) for a, b, c in recs]
    comp_avg = sum(comp_ms) / len(comp_ms)
    dec_avg_step = sum(b.elapsed_time(c) for a, b, c in recs) / len(recs)  # 256 decode calls
    dec_bytes_step = sum(decode_bytes(KB + s + 1) for s in range(STEPS))
    # eager (host-submitted) decode calls, for reference: includes host submission gaps
    compress()
    ea, eb = ev(), ev()
    ea.record(stream)
    for s_ in range(STEPS):
        decode(s_)
    eb.record(stream)
    torch.cuda.synchronize()
    eager_ms_per_token = ea.elapsed_time(eb) / STEPS
    total_ms, comp_avg, dec_avg_step = max_over_ranks([total_ms, comp_avg, dec_avg_step], dev)

    # e2e: the same API with host (pinned) inputs; H2D of Q_win and K and of every decode
    # step's q/k/v, D2H of the final attention output and the cache sizes.  V stays in
    # pinned host memory: the gather reads only the kept rows over the host link.
    e2e = None
    if rank == 0 or ws > 1:
        hQ, hK, hV = (t.cpu().pin_memory() for t in (Q, K, V))
        hdec = [tuple(t.cpu().pin_memory() for t in d) for d in dec]
        hout = torch.empty(outs.shape, dtype=outs.dtype).pin_memory()
        hnv = torch.empty(nv.shape, dtype=nv.dtype).pin_memory()
        dq, dk = torch.empty_like(Q), torch.empty_like(K)
        ddec = [tuple(torch.empty_like(t) for t in d) for d in dec]
        kept_v = LY * B * HKV * KB * D * V.element_size()  # V rows the gather reads from the host
        h2d = sum(t.numel() * t.element_size() for t in (hQ, hK)) + kept_v + \
            sum(t.numel() * t.element_size() for d in hdec for t in d)
        d2h = hout.numel() * hout.element_size() + hnv.numel() * hnv.element_size()

        # the prompt goes over in chunks of layers on a copy stream, and each chunk is
        # compressed as soon as it has landed, so compression overlaps the next copy
        copy_stream = torch.cuda.Stream()
        nch = 4 if LY % 4 == 0 else 1
        cl = LY // nch

        def e2e_step(rec):
            a, b, c = ev(), ev(), ev()
            a.record(stream)
            copy_stream.wait_stream(stream)
            landed = []
            with torch.cuda.stream(copy_stream):
                for ci in range(nch):
                    sl = slice(ci * cl, (ci + 1) * cl)
                    dq[sl].copy_(hQ[sl], non_blocking=True)
                    dk[sl].copy_(hK[sl], non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(copy_stream)
                    landed.append(e)
            for ci in range(nch):
                sl = slice(ci * cl, (ci + 1) * cl)
                stream.wait_event(landed[ci])
                kvc.snapkv_compress(dq[sl], dk[sl], hV[sl], keep_window=W, pool_kernel=P,
                                    budget=KB, cap=CAP, k_out=kc[sl], v_out=vc[sl],
                                    pos_out=pos[sl], n_valid_out=nv[sl])
            hnv.copy_(nv, non_blocking=True)
            b.record(stream)
            for s in range(STEPS):
                for dst, src in zip(ddec[s], hdec[s]):
                    dst.copy_(src, non_blocking=True)
                q, kn, vn = ddec[s]
                kvc.compressed_decode_attn(q, kc, vc, n_valid=nv, k_new=kn, v_new=vn, pos=pos,
                                           new_pos=L + s, out=outs)
            hout.copy_(outs, non_blocking=True)
            c.record(stream)
            if rec is not None:
                rec.append((a, b, c))

        e2e_step(None)
        torch.cuda.synchronize()
        erec = []
        for _ in range(max(1, min(args.steps, 3))):
            e2e_step(erec)
        torch.cuda.synchronize()
        e2e_status = kvc.kvc_device_status()
        if e2e_status:
            raise RuntimeError("device status flags %#x after the end-to-end steps" % e2e_status)
        comp_e2e = statistics.median(a.elapsed_time(b) for a, b, c in erec)
        all_e2e = statistics.median(a.elapsed_time(c) for a, b, c in erec)
        comp_e2e, all_e2e = max_over_ranks([comp_e2e, all_e2e], dev)
        e2e = {"value": whole_job_rate(B * L, comp_e2e, ws), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": all_e2e,
               "note": "prefix tokens / (H2D of Q_win and K + compression, whose gather reads "
                       "the kept V rows from pinned host memory + D2H of n_valid); "
                       "ms_per_step adds 256 decode steps with per-step H2D of q,k,v"}

    dec_gbs = dec_bytes_step / (dec_avg_step / 1e3) / 1e9
    dec_call_ms = dec_avg_step / STEPS
    wv_bytes = window_vote_bytes()
    line = {
        "metric": METRIC,
        "value": whole_job_rate(B * L, comp_avg, ws),
        "unit": UNIT,
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 in, fp32 accumulate",
        "data": "synthetic (seeded N(0,1) bf16, planted hot spans)",
        "config": config_dict(),
        "compress_ms": comp_avg,
        "decode_attn": {"GBps": dec_gbs, "frac_of_hbm_peak": dec_gbs / hbm_peak,
                        "peak_GBps": hbm_peak, "peak_kind": peak_kind,
                        "frac_of_nominal_8TBps": dec_gbs / 8000.0,
                        "ms_per_token_all_layers": dec_call_ms,
                        "launch": "one kernel per decode step covers all %d layers (append fused); "
                                  "the step's 256 calls replayed as a CUDA graph" % LY,
                        "eager_ms_per_token_all_layers": eager_ms_per_token},
        "roofline": {"kernel": "decode_kernel (compressed_decode_attn, %d layers per launch)" % LY,
                     "bound": "hbm", "achieved": dec_gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": dec_gbs / hbm_peak,
                     "traffic": decode_traffic(sum(KB + s + 1 for s in range(STEPS)) / STEPS),
                     "traffic_source": "profiles/decode_kernel_traffic.json (ncu dram bytes of "
                                       "one 32-layer launch at n = 1100, scaled by rows)",
                     "peak_kind": peak_kind + " burst copy"},
        "roofline_compress": {"kernel": "snapkv_compress (window vote + pool/top-k + gather)",
                              "bound": "hbm", "achieved": compress_bytes() / (comp_avg / 1e3) / 1e9,
                              "peak": hbm_peak, "unit": "GB/s",
                              "frac": compress_bytes() / (comp_avg / 1e3) / 1e9 / hbm_peak,
                              "algorithmic_bytes": compress_bytes(),
                              "traffic": compress_traffic(),
                              "traffic_source": "profiles/compress_traffic.json (ncu dram bytes of "
                                                "the launches of one %d-layer compression: the window vote, then the fused "
                                                "selection and gather)" % LY},
        "gpu_launches": args.steps * (3 + STEPS),
        "device_status": status,
        "clocks": clk,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if rank == 0 and not args.no_aux:
        # the other configurations of the hot path, measured after the headline: first
        # larger budgets on the same prompt
        budgets = [measure_budget(kvc, Q, K, V, b, hbm_peak) for b in (1024, 2048, 4096)]
        pools = [measure_pool(kvc, Q, K, V, x["planted"], pk, avg)
                 for pk, avg in ((7, False), (7, True), (1, False))]
        del Q, K, V, x, kc, vc, graph
        torch.cuda.empty_cache()
        line["aux"] = {"mistral_budget_sweep": budgets,
                       "mistral_pool_ablation": pools,
                       "long_context": measure_long(kvc, WL, dev, hbm_peak),
                       "prefill_with_votes": measure_prefill(kvc, WL, dev, tf_peak),
                       "lse_route": measure_lse_route(kvc, WL, dev, tf_peak, hbm_peak),
                       "h2o": measure_h2o(kvc, WL, dev, hbm_peak),
                       # the other reading of the 20% budget: 20% of the total length
                       # (prompt 2048 + 2048 generated), 409 heavy + 409 recent
                       "h2o_budget_total_length": measure_h2o(kvc, WL, dev, hbm_peak, steps=32,
                                                              n_heavy=409, n_recent=409),
                       "h2o_budget_20pct_of_131072": measure_h2o_long_budget(kvc, WL, dev, hbm_peak),
                       "streaming": measure_stream(kvc, WL, dev, hbm_peak),
                       # plain window attention (no sinks) and other sink counts, with the
                       # same 2048-slot cache per head
                       "streaming_sink_sweep": [
                           {k2: v2 for k2, v2 in measure_stream(kvc, WL, dev, hbm_peak, steps=64,
                                                                n_sink=S, ring=2048 - S).items()
                            if k2 in ("n_sink", "ring", "step_ms", "step_GBps",
                                      "step_frac_of_hbm_peak", "device_status")}
                           for S in (0, 1, 2, 4, 8)]}
        # the same compression when the prefill (prefill_attention_lse) supplies each row's
        # log-sum-exp: snapkv_votes_from_lse + snapkv_select (aux.lse_route); a second
        # route, not the headline value, which times snapkv_compress alone
        lr = line["aux"]["lse_route"]["snapkv"]
        line["compress_from_lse"] = {
            "ms": lr["compress_from_lse_ms"],
            "prefix_tokens_per_s": lr["compress_from_lse_prefix_tokens_per_s"],
            "GBps": compress_bytes() / (lr["compress_from_lse_ms"] / 1e3) / 1e9,
            "frac_of_hbm_peak": compress_bytes() / (lr["compress_from_lse_ms"] / 1e3) / 1e9 / hbm_peak,
            "entry_points": "snapkv_votes_from_lse + snapkv_select, given the rows' log-sum-exp"}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-aux", action="store_true",
                    help="skip the long-context, H2O and streaming measurements")
    ap.add_argument("--profile", choices=["decode", "aux", "long", "prefill", "h2d", "h2o-split",
                                          "lse"],
                    default=None,
                    help="run a short fixed workload for an ncu capture instead of the bench "
                         "(h2d: measure the host-link copy rates)")
    ap.add_argument("--layers", type=int, default=32, help="profiling only: fewer layers")
    ap.add_argument("--decode-steps", type=int, default=256, help="profiling only")
    args = ap.parse_args()
    set_size(args.layers, args.decode_steps)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[v] = "1"  # the oracle runs on one core (set before numpy loads)
        return run_reference(args)
    if args.profile == "h2d":
        return run_host_link(args)
    if args.profile:
        return run_profile_driver(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
