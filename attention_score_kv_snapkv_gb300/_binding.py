"""ctypes binding of libkvcompress (include/kvcompress.h).

Argument marshalling only: shapes, dtypes and devices of torch tensors are checked and
turned into the C structs and raw pointers of the ABI; outputs and workspaces are
allocated with torch (PyTorch provides device memory and streams).  Every step of the
path runs in the library's CUDA kernels; there is no fallback: if the library cannot
be built or loaded, the first call raises.
"""

import ctypes
import os
import threading

import torch

from . import build as _build

_lib = None
_lock = threading.Lock()

KVC_OK = 0
STATUS_NAMES = {0: "KVC_OK", 1: "KVC_ERR_NULL", 2: "KVC_ERR_SHAPE", 3: "KVC_ERR_ALIGN",
                4: "KVC_ERR_BUDGET", 5: "KVC_ERR_CUDA", 6: "KVC_ERR_TIMEOUT",
                7: "KVC_ERR_WORKSPACE", 8: "KVC_ERR_UNSUPPORTED"}
DEV_TIMEOUT, DEV_CACHE_FULL, DEV_BAD_STATE = 0x1, 0x2, 0x4


class KVCError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__("%s failed: %s" % (what, lib().kvc_status_string(code).decode()))


class SnapKVParams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "batch", "n_q_heads", "n_kv_heads", "head_dim", "prompt_len", "n_query",
        "keep_window", "pool_kernel", "budget", "cap", "pool_avg")]


class DecodeParams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "batch", "n_q_heads", "n_kv_heads", "head_dim", "cap", "n_uniform", "new_pos")]


class H2OParams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "batch", "n_q_heads", "n_kv_heads", "head_dim", "n_heavy", "n_recent")]


class H2OStateC(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("score", ctypes.c_void_p),
                ("pos", ctypes.c_void_p), ("n_used", ctypes.c_void_p), ("free_slot", ctypes.c_void_p),
                ("scratch", ctypes.c_void_p), ("scratch_bytes", ctypes.c_size_t)]


class SinkParams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "batch", "n_kv_heads", "head_dim", "n_sink", "n_recent")]


_P = ctypes.c_void_p
_SIGS = {
    "kvc_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "kvc_version": (ctypes.c_int, []),
    "kvc_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int, _P]),
    "kvc_set_wait_timeout_ns": (None, [ctypes.c_uint64]),
    "kvc_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint32, _P]),
    "snapkv_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(SnapKVParams)]),
    "snapkv_vote_plan": (ctypes.c_int, [ctypes.POINTER(SnapKVParams), ctypes.c_int32,
                                        ctypes.POINTER(ctypes.c_int64)]),
    "snapkv_compress": (ctypes.c_int, [ctypes.POINTER(SnapKVParams), _P, _P, _P, _P, _P, _P, _P,
                                       _P, _P, _P, ctypes.c_size_t, _P]),
    "snapkv_select": (ctypes.c_int, [ctypes.POINTER(SnapKVParams), _P, _P, _P, _P, _P, _P, _P, _P,
                                     _P, ctypes.c_size_t, _P]),
    "snapkv_prefill_attention": (ctypes.c_int, [ctypes.POINTER(SnapKVParams), _P, _P, _P, _P, _P,
                                                _P]),
    "prefill_attention_lse": (ctypes.c_int, [ctypes.POINTER(SnapKVParams), _P, _P, _P, _P, _P,
                                             _P]),
    "snapkv_votes_from_lse": (ctypes.c_int, [ctypes.POINTER(SnapKVParams), _P, _P, _P, _P, _P]),
    "compressed_decode_attn_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(DecodeParams)]),
    "compressed_decode_attn": (ctypes.c_int, [ctypes.POINTER(DecodeParams), _P, _P, _P, _P, _P, _P,
                                              _P, _P, _P, ctypes.c_size_t, _P]),
    "compressed_decode_attn_noalloc": (ctypes.c_int, [ctypes.POINTER(DecodeParams), _P, _P, _P, _P,
                                                      _P, _P, _P, _P, _P]),
    "h2o_prefill_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(H2OParams), ctypes.c_int32]),
    "h2o_step_scratch_bytes": (ctypes.c_size_t, [ctypes.POINTER(H2OParams)]),
    "h2o_step_ctas_per_unit": (ctypes.c_int32, [ctypes.POINTER(H2OParams)]),
    "h2o_prefill": (ctypes.c_int, [ctypes.POINTER(H2OParams), ctypes.c_int32, _P, _P, _P,
                                   ctypes.POINTER(H2OStateC), _P, ctypes.c_size_t, _P]),
    "h2o_prefill_from_votes": (ctypes.c_int, [ctypes.POINTER(H2OParams), ctypes.c_int32, _P, _P,
                                              _P, ctypes.POINTER(H2OStateC), _P, ctypes.c_size_t,
                                              _P]),
    "h2o_decode_step": (ctypes.c_int, [ctypes.POINTER(H2OParams), _P, _P, _P,
                                       ctypes.POINTER(H2OStateC), ctypes.c_int32, _P, _P, _P]),
    "sink_window_append": (ctypes.c_int, [ctypes.POINTER(SinkParams), _P, _P, _P, _P, _P,
                                          ctypes.c_int64, _P]),
}


def library_path():
    return _build.LIB


def lib():
    """Load (building first if needed) libkvcompress.so and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            handle = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def _check(code, what):
    if code != KVC_OK:
        raise KVCError(code, what)


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    return t


def _need_v(t, shape):
    """v of snapkv_compress: a CUDA tensor, or a page-locked (pinned) CPU tensor whose kept
    rows the gather reads over the host link."""
    if isinstance(t, torch.Tensor) and not t.is_cuda and t.is_pinned():
        if t.dtype != torch.bfloat16:
            raise TypeError("v must be torch.bfloat16, got %s" % t.dtype)
        if not t.is_contiguous() or tuple(t.shape) != tuple(shape):
            raise ValueError("v must be contiguous with shape %s" % (tuple(shape),))
        return t
    return _need(t, "v", torch.bfloat16, shape)


_ws_cache = {}


def workspace(nbytes, device, tag):
    """A zero-initialised device workspace of at least nbytes, reused per (device, tag)."""
    key = (device.index if device.index is not None else torch.cuda.current_device(), tag)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


# ----------------------------------------------------------------------------------
# entry points
# ----------------------------------------------------------------------------------

def kvc_version():
    return lib().kvc_version()


def kvc_device_status(clear=True, stream=None):
    flags = ctypes.c_uint32(0)
    code = lib().kvc_device_status(ctypes.byref(flags), 1 if clear else 0, _stream(stream))
    if code not in (KVC_OK, 6):
        _check(code, "kvc_device_status")
    return flags.value


def kvc_set_wait_timeout_ns(ns):
    lib().kvc_set_wait_timeout_ns(int(ns))


def kvc_selftest_wait_timeout(timeout_us, stream=None):
    return lib().kvc_selftest_wait_timeout(int(timeout_us), _stream(stream))


def snapkv_params(q_win, k, n_query, keep_window, pool_kernel, budget, cap, pool_avg=False):
    Ly, B, Hq, Wq, D = q_win.shape
    Ly2, B2, Hkv, L, D2 = k.shape
    if (Ly, B, D) != (Ly2, B2, D2) or Wq != n_query:
        raise ValueError("q_win %s and k %s disagree" % (tuple(q_win.shape), tuple(k.shape)))
    return SnapKVParams(Ly, B, Hq, Hkv, D, L, n_query, keep_window, pool_kernel, budget, cap,
                        1 if pool_avg else 0)


def snapkv_workspace_bytes(params):
    return lib().snapkv_workspace_bytes(ctypes.byref(params))


def snapkv_vote_plan(n_layers, batch, n_q_heads, n_kv_heads, head_dim, prompt_len, n_query,
                     keep_window, pool_kernel, budget, cap=None, pool_avg=False, num_sms=0):
    """The window-vote plan snapkv_compress uses for these sizes on a GPU with num_sms SMs
    (0: the current device's): a dict with single (1: the single-pass kernel, 0: two
    passes), g (CTAs per job), groups, row_tiles, rows_per_tile and exchange_bytes.  No
    device is needed.  Raises KVCError where snapkv_compress would reject the sizes."""
    cap = budget if cap is None else cap
    p = SnapKVParams(n_layers, batch, n_q_heads, n_kv_heads, head_dim, prompt_len, n_query,
                     keep_window, pool_kernel, budget, cap, 1 if pool_avg else 0)
    out = (ctypes.c_int64 * 6)()
    _check(lib().snapkv_vote_plan(ctypes.byref(p), num_sms, out), "snapkv_vote_plan")
    keys = ("single", "g", "groups", "row_tiles", "rows_per_tile", "exchange_bytes")
    return {k: int(v) for k, v in zip(keys, out)}


def snapkv_compress(q_win, k, v, *, keep_window, pool_kernel, budget, cap=None, k_out=None,
                    v_out=None, pos_out=None, n_valid_out=None, votes_out=None,
                    kept_scores_out=None, want_votes=False, workspace_buf=None, stream=None,
                    pool_avg=False):
    """SnapKV compression of every (layer, batch, KV head): q_win [Ly,B,Hq,W,D] (the last
    W prompt queries), k, v [Ly,B,Hkv,L,D] -> compact cache [Ly,B,Hkv,cap,D], positions,
    n_valid (and the raw votes with want_votes).  v may be a pinned CPU tensor (only the
    kept rows are read, over the host link).  pool_avg selects average pooling instead of
    max pooling.  Returns a dict of the output tensors."""
    bf = torch.bfloat16
    _need(q_win, "q_win", bf)
    _need(k, "k", bf)
    _need_v(v, k.shape)
    Ly, B, Hkv, L, D = k.shape
    n_keep = L if (budget >= L or keep_window >= L) else budget
    cap = n_keep if cap is None else cap
    p = snapkv_params(q_win, k, q_win.shape[3], keep_window, pool_kernel, budget, cap, pool_avg)
    dev = k.device
    if k_out is None:
        k_out = torch.empty((Ly, B, Hkv, cap, D), dtype=bf, device=dev)
    if v_out is None:
        v_out = torch.empty((Ly, B, Hkv, cap, D), dtype=bf, device=dev)
    if pos_out is None:
        pos_out = torch.empty((Ly, B, Hkv, cap), dtype=torch.int32, device=dev)
    if n_valid_out is None:
        n_valid_out = torch.empty((Ly, B, Hkv), dtype=torch.int32, device=dev)
    if votes_out is None and want_votes:
        votes_out = torch.empty((Ly, B, Hkv, L), dtype=torch.float32, device=dev)
    _need(k_out, "k_out", bf, (Ly, B, Hkv, cap, D))
    _need(v_out, "v_out", bf, (Ly, B, Hkv, cap, D))
    _need(pos_out, "pos_out", torch.int32, (Ly, B, Hkv, cap))
    _need(n_valid_out, "n_valid_out", torch.int32, (Ly, B, Hkv))
    if votes_out is not None:
        _need(votes_out, "votes_out", torch.float32, (Ly, B, Hkv, L))
    if kept_scores_out is not None:
        _need(kept_scores_out, "kept_scores_out", torch.float32, (Ly, B, Hkv, cap))
    nbytes = snapkv_workspace_bytes(p)
    ws = workspace(nbytes, dev, "snapkv") if workspace_buf is None else workspace_buf
    code = lib().snapkv_compress(ctypes.byref(p), _ptr(q_win), _ptr(k), _ptr(v), _ptr(k_out),
                                 _ptr(v_out), _ptr(pos_out), _ptr(n_valid_out), _ptr(votes_out),
                                 _ptr(kept_scores_out), _ptr(ws), ws.numel(), _stream(stream))
    _check(code, "snapkv_compress")
    return dict(k=k_out, v=v_out, pos=pos_out, n_valid=n_valid_out, votes=votes_out)


def decode_params(q, k_cache, n_uniform=0, new_pos=0):
    Ly, B, Hq, D = q.shape
    Ly2, B2, Hkv, cap, D2 = k_cache.shape
    if (Ly, B, D) != (Ly2, B2, D2):
        raise ValueError("q %s and cache %s disagree" % (tuple(q.shape), tuple(k_cache.shape)))
    return DecodeParams(Ly, B, Hq, Hkv, D, cap, n_uniform, new_pos)


def snapkv_prefill_attention(q, k, v, *, window=None, out=None, votes_out=None, stream=None):
    """Causal self-attention of the prompt, q [Ly,B,Hq,L,D], k, v [Ly,B,Hkv,L,D] -> out
    [Ly,B,Hq,L,D]; with window = W also the SnapKV votes of the last W rows, fp32
    [Ly,B,Hkv,L].  Returns (out, votes or None)."""
    bf = torch.bfloat16
    _need(q, "q", bf)
    _need(k, "k", bf)
    _need(v, "v", bf, k.shape)
    Ly, B, Hkv, L, D = k.shape
    if q.shape[:2] != k.shape[:2] or q.shape[3:] != k.shape[3:] or q.shape[2] % Hkv:
        raise ValueError("q %s and k %s disagree" % (tuple(q.shape), tuple(k.shape)))
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", bf, q.shape)
    if window is not None and votes_out is None:
        votes_out = torch.empty((Ly, B, Hkv, L), dtype=torch.float32, device=k.device)
    if votes_out is not None:
        _need(votes_out, "votes_out", torch.float32, (Ly, B, Hkv, L))
    p = SnapKVParams(Ly, B, q.shape[2], Hkv, D, L, window or 1, 0, 1, 1, 1, 0)
    code = lib().snapkv_prefill_attention(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                          _ptr(votes_out), _stream(stream))
    _check(code, "snapkv_prefill_attention")
    return out, votes_out


def prefill_attention_lse(q, k, v, *, out=None, lse_out=None, stream=None):
    """Causal self-attention of the prompt, q [Ly,B,Hq,L,D], k, v [Ly,B,Hkv,L,D] -> out
    [Ly,B,Hq,L,D] and each row's log-sum-exp lse [Ly,B,Hq,L] fp32 (natural log of the
    softmax normaliser).  Returns (out, lse)."""
    bf = torch.bfloat16
    _need(q, "q", bf)
    _need(k, "k", bf)
    _need(v, "v", bf, k.shape)
    Ly, B, Hkv, L, D = k.shape
    if q.shape[:2] != k.shape[:2] or q.shape[3:] != k.shape[3:] or q.shape[2] % Hkv:
        raise ValueError("q %s and k %s disagree" % (tuple(q.shape), tuple(k.shape)))
    if out is None:
        out = torch.empty_like(q)
    if lse_out is None:
        lse_out = torch.empty(q.shape[:4], dtype=torch.float32, device=q.device)
    _need(out, "out", bf, q.shape)
    _need(lse_out, "lse_out", torch.float32, tuple(q.shape[:4]))
    p = SnapKVParams(Ly, B, q.shape[2], Hkv, D, L, 1, 0, 1, 1, 1, 0)
    code = lib().prefill_attention_lse(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                       _ptr(lse_out), _stream(stream))
    _check(code, "prefill_attention_lse")
    return out, lse_out


def snapkv_votes_from_lse(q_win, k, lse, *, votes_out=None, stream=None):
    """Votes of the Wq window queries q_win [Ly,B,Hq,Wq,D] over k [Ly,B,Hkv,L,D], given every
    row's log-sum-exp lse [Ly,B,Hq,L] (prefill_attention_lse's): fp32 [Ly,B,Hkv,L], the
    votes snapkv_compress forms (H2O's initial scores when Wq = L)."""
    bf = torch.bfloat16
    _need(q_win, "q_win", bf)
    _need(k, "k", bf)
    Ly, B, Hkv, L, D = k.shape
    Hq, Wq = q_win.shape[2], q_win.shape[3]
    if q_win.shape[:2] != k.shape[:2] or q_win.shape[4] != D or Hq % Hkv or Wq > L:
        raise ValueError("q_win %s and k %s disagree" % (tuple(q_win.shape), tuple(k.shape)))
    _need(lse, "lse", torch.float32, (Ly, B, Hq, L))
    if votes_out is None:
        votes_out = torch.empty((Ly, B, Hkv, L), dtype=torch.float32, device=k.device)
    _need(votes_out, "votes_out", torch.float32, (Ly, B, Hkv, L))
    p = SnapKVParams(Ly, B, Hq, Hkv, D, L, Wq, 0, 1, 1, 1, 0)
    code = lib().snapkv_votes_from_lse(ctypes.byref(p), _ptr(q_win), _ptr(k), _ptr(lse),
                                       _ptr(votes_out), _stream(stream))
    _check(code, "snapkv_votes_from_lse")
    return votes_out


def snapkv_select(votes, k, v, *, keep_window, pool_kernel, budget, cap=None, pool_avg=False,
                  stream=None):
    """Steps 3-4 of snapkv_compress (pool, top-k, gather) from given votes [Ly,B,Hkv,L]
    (e.g. snapkv_prefill_attention's).  Returns the dict snapkv_compress returns, without
    votes."""
    bf = torch.bfloat16
    _need(votes, "votes", torch.float32)
    _need(k, "k", bf)
    _need_v(v, k.shape)
    Ly, B, Hkv, L, D = k.shape
    _need(votes, "votes", torch.float32, (Ly, B, Hkv, L))
    n_keep = L if (budget >= L or keep_window >= L) else budget
    cap = n_keep if cap is None else cap
    p = SnapKVParams(Ly, B, Hkv, Hkv, D, L, 1, keep_window, pool_kernel, budget, cap,
                     1 if pool_avg else 0)
    dev = k.device
    k_out = torch.empty((Ly, B, Hkv, cap, D), dtype=bf, device=dev)
    v_out = torch.empty_like(k_out)
    pos_out = torch.empty((Ly, B, Hkv, cap), dtype=torch.int32, device=dev)
    n_valid_out = torch.empty((Ly, B, Hkv), dtype=torch.int32, device=dev)
    nbytes = snapkv_workspace_bytes(p)
    ws = workspace(nbytes, dev, "snapkv")
    code = lib().snapkv_select(ctypes.byref(p), _ptr(votes), _ptr(k), _ptr(v), _ptr(k_out),
                               _ptr(v_out), _ptr(pos_out), _ptr(n_valid_out), None, _ptr(ws),
                               ws.numel(), _stream(stream))
    _check(code, "snapkv_select")
    return {"k": k_out, "v": v_out, "pos": pos_out, "n_valid": n_valid_out}


def compressed_decode_attn_workspace_bytes(params):
    return lib().compressed_decode_attn_workspace_bytes(ctypes.byref(params))


def compressed_decode_attn(q, k_cache, v_cache, *, n_valid=None, n_uniform=None, k_new=None,
                           v_new=None, pos=None, new_pos=0, out=None, workspace_buf=None,
                           stream=None):
    """One decode step: optional append of (k_new, v_new) at n_valid, then attention of
    q [Ly,B,Hq,D] over the first n rows of the cache [Ly,B,Hkv,cap,D].  With n_valid,
    n_uniform may give an upper bound on the rows after the append (plans less work).
    Returns out."""
    bf = torch.bfloat16
    _need(q, "q", bf)
    _need(k_cache, "k_cache", bf)
    _need(v_cache, "v_cache", bf, k_cache.shape)
    Ly, B, Hkv, cap, D = k_cache.shape
    if n_valid is not None:
        _need(n_valid, "n_valid", torch.int32, (Ly, B, Hkv))
    elif n_uniform is None:
        raise ValueError("give n_valid or n_uniform")
    if k_new is not None:
        _need(k_new, "k_new", bf, (Ly, B, Hkv, D))
        _need(v_new, "v_new", bf, (Ly, B, Hkv, D))
    if pos is not None:
        _need(pos, "pos", torch.int32, (Ly, B, Hkv, cap))
    p = decode_params(q, k_cache, 0 if n_uniform is None else n_uniform, new_pos)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", bf, q.shape)
    nbytes = compressed_decode_attn_workspace_bytes(p)
    ws = workspace(nbytes, q.device, "decode") if workspace_buf is None else workspace_buf
    code = lib().compressed_decode_attn(ctypes.byref(p), _ptr(q), _ptr(k_new), _ptr(v_new),
                                        _ptr(k_cache), _ptr(v_cache), _ptr(pos), _ptr(n_valid),
                                        _ptr(out), _ptr(ws), ws.numel(), _stream(stream))
    _check(code, "compressed_decode_attn")
    return out


def compressed_decode_attn_noalloc(q, k_cache, v_cache, *, n_valid=None, n_uniform=None,
                                   k_new=None, v_new=None, pos=None, new_pos=0, out=None,
                                   stream=None):
    """compressed_decode_attn without a workspace: the library's fixed 8 MiB device
    scratch array holds the split-K partials (for callers that cannot allocate)."""
    bf = torch.bfloat16
    _need(q, "q", bf)
    _need(k_cache, "k_cache", bf)
    _need(v_cache, "v_cache", bf, k_cache.shape)
    Ly, B, Hkv, cap, D = k_cache.shape
    if n_valid is not None:
        _need(n_valid, "n_valid", torch.int32, (Ly, B, Hkv))
    elif n_uniform is None:
        raise ValueError("give n_valid or n_uniform")
    if k_new is not None:
        _need(k_new, "k_new", bf, (Ly, B, Hkv, D))
        _need(v_new, "v_new", bf, (Ly, B, Hkv, D))
    if pos is not None:
        _need(pos, "pos", torch.int32, (Ly, B, Hkv, cap))
    if out is None:
        raise ValueError("out must be given: this entry point allocates nothing")
    _need(out, "out", bf, q.shape)
    p = decode_params(q, k_cache, 0 if n_uniform is None else n_uniform, new_pos)
    code = lib().compressed_decode_attn_noalloc(ctypes.byref(p), _ptr(q), _ptr(k_new),
                                                _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                                _ptr(pos), _ptr(n_valid), _ptr(out),
                                                _stream(stream))
    _check(code, "compressed_decode_attn_noalloc")
    return out


class H2OState:
    """Device state of an H2O cache: k, v [Ly,B,Hkv,S,D] bf16, score [..,S] fp32,
    pos [..,S] int32, n_used and free_slot [Ly,B,Hkv] int32, S = n_heavy + n_recent + 1,
    and the zero-filled scratch of the split step (allocated by the first step that asks
    for it)."""

    def __init__(self, n_layers, batch, n_kv_heads, head_dim, n_heavy, n_recent, device):
        S = n_heavy + n_recent + 1
        shp = (n_layers, batch, n_kv_heads)
        self.n_heavy, self.n_recent, self.slots = n_heavy, n_recent, S
        self.k = torch.zeros(shp + (S, head_dim), dtype=torch.bfloat16, device=device)
        self.v = torch.zeros_like(self.k)
        self.score = torch.zeros(shp + (S,), dtype=torch.float32, device=device)
        self.pos = torch.full(shp + (S,), -1, dtype=torch.int32, device=device)
        self.n_used = torch.zeros(shp, dtype=torch.int32, device=device)
        self.free_slot = torch.zeros(shp, dtype=torch.int32, device=device)
        self.scratch = None

    def c_struct(self):
        sc = self.scratch
        return H2OStateC(self.k.data_ptr(), self.v.data_ptr(), self.score.data_ptr(),
                         self.pos.data_ptr(), self.n_used.data_ptr(), self.free_slot.data_ptr(),
                         None if sc is None else sc.data_ptr(), 0 if sc is None else sc.numel())

    def layer(self, l):
        """A view of layer l alone (the state of a one-layer call, e.g. a layer-by-layer
        prefill); it shares memory (and the scratch) with this state."""
        view = H2OState.__new__(H2OState)
        view.n_heavy, view.n_recent, view.slots = self.n_heavy, self.n_recent, self.slots
        for name in ("k", "v", "score", "pos", "n_used", "free_slot", "scratch"):
            v = getattr(self, name)
            setattr(view, name, v if name == "scratch" else v[l:l + 1])
        return view


def _h2o_params(q, state, Hkv_from):
    Ly, B, Hq, D = q.shape[0], q.shape[1], q.shape[2], q.shape[-1]
    return H2OParams(Ly, B, Hq, Hkv_from, D, state.n_heavy, state.n_recent)


def h2o_prefill(q, k, v, *, n_heavy, n_recent, state=None, workspace_buf=None, stream=None):
    """Initial H2O cache from the prompt: q [Ly,B,Hq,L,D] (all prompt queries), k, v
    [Ly,B,Hkv,L,D].  Returns an H2OState."""
    bf = torch.bfloat16
    _need(q, "q", bf)
    _need(k, "k", bf)
    _need(v, "v", bf, k.shape)
    Ly, B, Hkv, L, D = k.shape
    if q.shape[:2] != k.shape[:2] or q.shape[3] != L or q.shape[4] != D:
        raise ValueError("q %s and k %s disagree" % (tuple(q.shape), tuple(k.shape)))
    if state is None:
        state = H2OState(Ly, B, Hkv, D, n_heavy, n_recent, k.device)
    p = H2OParams(Ly, B, q.shape[2], Hkv, D, n_heavy, n_recent)
    nbytes = lib().h2o_prefill_workspace_bytes(ctypes.byref(p), L)
    ws = workspace(nbytes, k.device, "snapkv") if workspace_buf is None else workspace_buf
    st = state.c_struct()
    code = lib().h2o_prefill(ctypes.byref(p), L, _ptr(q), _ptr(k), _ptr(v), ctypes.byref(st),
                             _ptr(ws), ws.numel(), _stream(stream))
    _check(code, "h2o_prefill")
    return state


def h2o_prefill_from_votes(votes, k, v, *, n_q_heads, n_heavy, n_recent, state=None,
                           workspace_buf=None, stream=None):
    """h2o_prefill from given initial scores votes [Ly,B,Hkv,L] fp32 (e.g.
    snapkv_votes_from_lse over every prompt query); k, v [Ly,B,Hkv,L,D].  Returns an
    H2OState."""
    bf = torch.bfloat16
    _need(k, "k", bf)
    _need(v, "v", bf, k.shape)
    Ly, B, Hkv, L, D = k.shape
    _need(votes, "votes", torch.float32, (Ly, B, Hkv, L))
    if state is None:
        state = H2OState(Ly, B, Hkv, D, n_heavy, n_recent, k.device)
    p = H2OParams(Ly, B, n_q_heads, Hkv, D, n_heavy, n_recent)
    nbytes = lib().h2o_prefill_workspace_bytes(ctypes.byref(p), L)
    ws = workspace(nbytes, k.device, "snapkv") if workspace_buf is None else workspace_buf
    st = state.c_struct()
    code = lib().h2o_prefill_from_votes(ctypes.byref(p), L, _ptr(votes), _ptr(k), _ptr(v),
                                        ctypes.byref(st), _ptr(ws), ws.numel(),
                                        _stream(stream))
    _check(code, "h2o_prefill_from_votes")
    return state


def h2o_step_ctas_per_unit(n_layers, batch, n_q_heads, n_kv_heads, head_dim, n_heavy, n_recent):
    """CTAs per unit of the H2O step on the current device (1: one CTA per unit; more: the
    split step), 0 if the sizes are out of range."""
    p = H2OParams(n_layers, batch, n_q_heads, n_kv_heads, head_dim, n_heavy, n_recent)
    return lib().h2o_step_ctas_per_unit(ctypes.byref(p))


def h2o_decode_step(q, k_new, v_new, state, t, *, out=None, evicted=None, stream=None):
    """One H2O decode step at position t: q [Ly,B,Hq,D], k_new/v_new [Ly,B,Hkv,D].
    Returns (out, evicted positions [Ly,B,Hkv] int32, -1 where nothing was evicted)."""
    bf = torch.bfloat16
    _need(q, "q", bf)
    Ly, B, Hkv = state.n_used.shape
    D = state.k.shape[-1]
    _need(k_new, "k_new", bf, (Ly, B, Hkv, D))
    _need(v_new, "v_new", bf, (Ly, B, Hkv, D))
    if out is None:
        out = torch.empty_like(q)
    if evicted is None:
        evicted = torch.empty((Ly, B, Hkv), dtype=torch.int32, device=q.device)
    _need(out, "out", bf, q.shape)
    _need(evicted, "evicted", torch.int32, (Ly, B, Hkv))
    p = H2OParams(Ly, B, q.shape[2], Hkv, D, state.n_heavy, state.n_recent)
    need = lib().h2o_step_scratch_bytes(ctypes.byref(p))
    if state.scratch is None or state.scratch.numel() < need:
        state.scratch = torch.zeros(max(int(need), 256), dtype=torch.uint8, device=q.device)
    st = state.c_struct()
    code = lib().h2o_decode_step(ctypes.byref(p), _ptr(q), _ptr(k_new), _ptr(v_new),
                                 ctypes.byref(st), int(t), _ptr(out), _ptr(evicted),
                                 _stream(stream))
    _check(code, "h2o_decode_step")
    return out, evicted


def sink_window_append(k_new, v_new, k_cache, v_cache, t, *, n_sink, n_recent, pos=None,
                       stream=None):
    """StreamingLLM append of token t into the sink + ring cache [Ly,B,Hkv,S+R,D]."""
    bf = torch.bfloat16
    _need(k_cache, "k_cache", bf)
    _need(v_cache, "v_cache", bf, k_cache.shape)
    Ly, B, Hkv, rows, D = k_cache.shape
    if rows != n_sink + n_recent:
        raise ValueError("cache rows %d != n_sink + n_recent = %d" % (rows, n_sink + n_recent))
    _need(k_new, "k_new", bf, (Ly, B, Hkv, D))
    _need(v_new, "v_new", bf, (Ly, B, Hkv, D))
    if pos is not None:
        _need(pos, "pos", torch.int32, (Ly, B, Hkv, rows))
    p = SinkParams(Ly, B, Hkv, D, n_sink, n_recent)
    code = lib().sink_window_append(ctypes.byref(p), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                    _ptr(v_cache), _ptr(pos), int(t), _stream(stream))
    _check(code, "sink_window_append")
