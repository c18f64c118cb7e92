"""The C-ABI library builds for sm_103a, loads, and exports every function that
include/kvcompress.h declares.  Only host-side calls are made (no GPU needed)."""

import ctypes
import os
import re
import subprocess

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "kvcompress.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                       src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "return", "sizeof")))


def test_header_declares_the_four_entry_points():
    names = declared_functions()
    for n in ("snapkv_compress", "h2o_decode_step", "sink_window_append",
              "compressed_decode_attn"):
        assert n in names


def test_library_builds_loads_and_exports_every_declared_symbol():
    from attention_score_kv_snapkv_gb300 import build
    path = build.build()
    assert os.path.exists(path)
    lib = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing


def test_host_only_calls():
    from attention_score_kv_snapkv_gb300 import _binding as B
    lib = B.lib()
    assert lib.kvc_version() == 100
    for code, name in B.STATUS_NAMES.items():
        assert lib.kvc_status_string(code).decode().startswith(name)
    assert lib.kvc_status_string(99) == b"unknown kvc_status"
    p = B.SnapKVParams(32, 2, 32, 8, 128, 16384, 32, 32, 7, 1024, 1280)
    ws = lib.snapkv_workspace_bytes(ctypes.byref(p))
    assert ws >= 512 * 16384 * 4          # at least the fp32 votes of every unit
    assert ws % 256 == 0
    bad = B.SnapKVParams(1, 1, 3, 2, 128, 100, 8, 8, 7, 64, 64)  # Hq % Hkv != 0
    assert lib.snapkv_workspace_bytes(ctypes.byref(bad)) == 256
    avg = B.SnapKVParams(32, 2, 32, 8, 128, 16384, 32, 32, 7, 1024, 1280, 1)  # average pool
    assert lib.snapkv_workspace_bytes(ctypes.byref(avg)) == ws
    bad_pool = B.SnapKVParams(32, 2, 32, 8, 128, 16384, 32, 32, 7, 1024, 1280, 2)  # no such mode
    assert lib.snapkv_workspace_bytes(ctypes.byref(bad_pool)) == 256
    d = B.DecodeParams(32, 2, 32, 8, 128, 1280, 0, 0)
    assert lib.compressed_decode_attn_workspace_bytes(ctypes.byref(d)) >= 512 * 4


def test_calls_without_a_gpu_fail_cleanly():
    import torch
    if torch.cuda.is_available():
        return
    from attention_score_kv_snapkv_gb300 import _binding as B
    lib = B.lib()
    p = B.SnapKVParams(1, 1, 4, 4, 64, 512, 8, 8, 7, 64, 64)
    code = lib.snapkv_compress(ctypes.byref(p), None, None, None, None, None, None, None, None,
                               None, None, 0, None)
    assert code == 8  # KVC_ERR_UNSUPPORTED: nothing launched
