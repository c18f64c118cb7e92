"""compressed_decode_attn_noalloc: the decode step for callers that cannot give the
library a device workspace (engines that own all device memory in their own pool and
pass only the step's tensors down; a cudaMalloc mid-step would also synchronise the
device).  Its split-K scratch is the library's fixed 8 MiB device array.

Checks, through the C ABI: two calls in a row agree with compressed_decode_attn (which
takes a caller workspace) within the decode tolerance, with and without the fused
append, and with the fp64 oracle's attention directly; a call that would need more
scratch than the array holds is rejected with KVC_ERR_WORKSPACE, and a call rejected by
an argument check returns its error without disturbing the next call.  The file name sorts last so that a run stopping at its
first failure has run every other test before this one; the tests themselves depend on
no order."""

import ctypes

import pytest
import torch

from oracle import attention as OA
from parity import assert_outputs_close, f64

pytestmark = pytest.mark.gpu


def _inputs(Ly, B, Hq, Hkv, D, cap, seed):
    g = torch.Generator().manual_seed(seed)
    dev = torch.device("cuda")
    q = torch.randn((Ly, B, Hq, D), generator=g).to(torch.bfloat16).to(dev)
    kc = torch.randn((Ly, B, Hkv, cap, D), generator=g).to(torch.bfloat16).to(dev)
    vc = torch.randn((Ly, B, Hkv, cap, D), generator=g).to(torch.bfloat16).to(dev)
    n = torch.randint(1, cap, (Ly, B, Hkv), generator=g, dtype=torch.int32).to(dev)
    return q, kc, vc, n


def _noalloc_call(kvc, q, kc, vc, n, out, k_new=None, v_new=None, pos=None, new_pos=0):
    """Direct C-ABI call of compressed_decode_attn_noalloc (no workspace argument)."""
    from attention_score_kv_snapkv_gb300 import _binding as Bd
    p = Bd.decode_params(q, kc, 0, new_pos)
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return kvc.lib().compressed_decode_attn_noalloc(
        ctypes.byref(p), ptr(q), ptr(k_new), ptr(v_new), ptr(kc), ptr(vc), ptr(pos), ptr(n),
        ptr(out), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("shape", [(1, 2, 32, 8, 128, 1280), (2, 1, 8, 8, 64, 300)],
                         ids=["gqa4-d128-cap1280", "mha-d64-cap300"])
def test_noalloc_matches_workspace_entry_point_twice(kvc, shape):
    q, kc, vc, n = _inputs(*shape, seed=shape[-1])
    Ly, B, Hq, Hkv = shape[:4]
    G = Hq // Hkv
    qh, kh, vh, nh = f64(q), f64(kc), f64(vc), n.cpu().numpy()
    for call in range(2):
        ref = kvc.compressed_decode_attn(q, kc, vc, n_valid=n)
        out = torch.empty_like(q)
        assert _noalloc_call(kvc, q, kc, vc, n, out) == 0
        torch.cuda.synchronize()
        assert_outputs_close(f64(out), f64(ref), "no-alloc call %d" % call)
        # and directly against the oracle's attention over each unit's first n rows
        outh = f64(out)
        for ly in range(Ly):
            for b in range(B):
                for h in range(Hkv):
                    m = int(nh[ly, b, h])
                    want = OA.attend_group(qh[ly, b, h * G:(h + 1) * G], kh[ly, b, h, :m],
                                           vh[ly, b, h, :m])
                    assert_outputs_close(outh[ly, b, h * G:(h + 1) * G], want,
                                         "no-alloc call %d unit %s" % (call, (ly, b, h)))
    assert kvc.kvc_device_status() == 0


def test_noalloc_append_matches_twice(kvc):
    Ly, B, Hq, Hkv, D, cap = 1, 2, 16, 4, 128, 400
    q, kc, vc, n = _inputs(Ly, B, Hq, Hkv, D, cap, seed=9)
    g = torch.Generator().manual_seed(10)
    dev = q.device
    kc2, vc2, n2 = kc.clone(), vc.clone(), n.clone()
    pos1 = torch.full((Ly, B, Hkv, cap), -1, dtype=torch.int32, device=dev)
    pos2 = pos1.clone()
    for call in range(2):
        kn = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16).to(dev)
        vn = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16).to(dev)
        ref = kvc.compressed_decode_attn(q, kc, vc, n_valid=n, k_new=kn, v_new=vn, pos=pos1,
                                         new_pos=100 + call)
        out = torch.empty_like(q)
        assert _noalloc_call(kvc, q, kc2, vc2, n2, out, kn, vn, pos2, 100 + call) == 0
        torch.cuda.synchronize()
        assert_outputs_close(f64(out), f64(ref), "no-alloc append call %d" % call)
        assert torch.equal(n, n2) and torch.equal(pos1, pos2)
        assert torch.equal(kc, kc2) and torch.equal(vc, vc2)
    assert kvc.kvc_device_status() == 0


def test_noalloc_rejects_calls_beyond_the_fixed_scratch(kvc):
    # 512 units x 20 splits x 4 heads x 520 bytes of partials: about 21 MB > 8 MiB
    from attention_score_kv_snapkv_gb300 import _binding as Bd
    p = Bd.DecodeParams(32, 2, 32, 8, 128, 1280, 0, 0)
    assert kvc.lib().compressed_decode_attn_workspace_bytes(ctypes.byref(p)) > (8 << 20)
    code = kvc.lib().compressed_decode_attn_noalloc(ctypes.byref(p), None, None, None, None, None,
                                                    None, None, None, None)
    assert code == 7  # KVC_ERR_WORKSPACE, nothing launched


def test_rejected_call_leaves_the_scratch_alone(kvc):
    # a call rejected by an argument check (a misaligned output) between two good calls
    # returns KVC_ERR_ALIGN, and the next call still matches the workspace entry point
    q, kc, vc, n = _inputs(1, 2, 16, 4, 128, 700, seed=21)
    out = torch.empty_like(q)
    assert _noalloc_call(kvc, q, kc, vc, n, out) == 0
    bad = torch.empty(out.numel() + 8, dtype=out.dtype, device=out.device)[1:1 + out.numel()]
    p_code = _noalloc_call(kvc, q, kc, vc, n, bad.view(out.shape))
    assert p_code == 3  # KVC_ERR_ALIGN
    ref = kvc.compressed_decode_attn(q, kc, vc, n_valid=n)
    assert _noalloc_call(kvc, q, kc, vc, n, out) == 0
    torch.cuda.synchronize()
    assert_outputs_close(f64(out), f64(ref), "no-alloc call after a rejected one")
    assert kvc.kvc_device_status() == 0
