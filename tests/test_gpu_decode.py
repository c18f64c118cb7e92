"""GPU parity of compressed_decode_attn (split-K decode over a compact cache, with and
without the fused append) against fp64 attention of the oracle."""

import numpy as np
import pytest
import torch

from oracle import attention as OA
from parity import assert_outputs_close, f64

pytestmark = pytest.mark.gpu


def rand_cache(Ly, B, Hq, Hkv, D, cap, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((Ly, B, Hq, D), generator=g).to(torch.bfloat16)
    kc = torch.randn((Ly, B, Hkv, cap, D), generator=g).to(torch.bfloat16)
    vc = torch.randn((Ly, B, Hkv, cap, D), generator=g).to(torch.bfloat16)
    return q, kc, vc


def oracle_decode(q, kc, vc, n):
    """q [Ly,B,Hq,D], caches [Ly,B,Hkv,cap,D], n [Ly,B,Hkv] -> [Ly,B,Hq,D] (fp64)."""
    qh, kh, vh = f64(q), f64(kc), f64(vc)
    Ly, B, Hq, D = qh.shape
    Hkv = kh.shape[2]
    G = Hq // Hkv
    out = np.zeros_like(qh)
    for ly in range(Ly):
        for b in range(B):
            for h in range(Hkv):
                m = int(n[ly, b, h])
                if m == 0:
                    continue
                out[ly, b, h * G:(h + 1) * G] = OA.attend_group(qh[ly, b, h * G:(h + 1) * G],
                                                                kh[ly, b, h, :m], vh[ly, b, h, :m])
    return out


SHAPES = [  # Ly, B, Hq, Hkv, D, cap
    (1, 2, 8, 2, 128, 300),
    (2, 1, 4, 4, 64, 129),
    (1, 1, 32, 8, 128, 1280),
    (1, 3, 16, 2, 128, 700),
    (1, 1, 2, 2, 128, 64),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_decode_ragged_n_valid(kvc, shape):
    Ly, B, Hq, Hkv, D, cap = shape
    q, kc, vc = rand_cache(Ly, B, Hq, Hkv, D, cap, seed=cap + Hq)
    g = torch.Generator().manual_seed(7)
    n = torch.randint(0, cap + 1, (Ly, B, Hkv), generator=g, dtype=torch.int32)
    n.view(-1)[0] = cap
    n.view(-1)[-1] = 1 if n.numel() > 1 else cap
    dev = torch.device("cuda")
    out = kvc.compressed_decode_attn(q.to(dev), kc.to(dev), vc.to(dev), n_valid=n.to(dev))
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    assert_outputs_close(f64(out), oracle_decode(q, kc, vc, n.numpy()))


def test_decode_uniform_n_and_zero_rows(kvc):
    q, kc, vc = rand_cache(1, 2, 8, 2, 128, 256, seed=3)
    dev = torch.device("cuda")
    for n in (0, 1, 63, 64, 65, 256):
        out = kvc.compressed_decode_attn(q.to(dev), kc.to(dev), vc.to(dev), n_uniform=n)
        ref = oracle_decode(q, kc, vc, np.full((1, 2, 2), n))
        assert_outputs_close(f64(out), ref, "n=%d" % n)
        if n == 0:
            assert float(out.abs().max()) == 0.0


def test_decode_append_then_attend(kvc):
    Ly, B, Hq, Hkv, D, cap = 1, 2, 8, 2, 128, 200
    q, kc, vc = rand_cache(Ly, B, Hq, Hkv, D, cap, seed=11)
    g = torch.Generator().manual_seed(12)
    kn = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16)
    vn = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16)
    n0 = torch.tensor([[[10, 199], [0, 150]]], dtype=torch.int32)
    dev = torch.device("cuda")
    kcd, vcd, nd = kc.to(dev), vc.to(dev), n0.to(dev)
    pos = torch.full((Ly, B, Hkv, cap), -1, dtype=torch.int32, device=dev)
    out = kvc.compressed_decode_attn(q.to(dev), kcd, vcd, n_valid=nd, k_new=kn.to(dev),
                                     v_new=vn.to(dev), pos=pos, new_pos=12345)
    torch.cuda.synchronize()
    kc2, vc2 = kc.clone(), vc.clone()
    for b in range(B):
        for h in range(Hkv):
            kc2[0, b, h, n0[0, b, h]] = kn[0, b, h]
            vc2[0, b, h, n0[0, b, h]] = vn[0, b, h]
    assert torch.equal(nd.cpu(), n0 + 1)
    assert torch.equal(kcd.cpu(), kc2) and torch.equal(vcd.cpu(), vc2)
    assert int(pos[0, 0, 1, 199]) == 12345
    assert_outputs_close(f64(out), oracle_decode(q, kc2, vc2, (n0 + 1).numpy()))
    # the unit that is now full drops the next token and flags it
    out = kvc.compressed_decode_attn(q.to(dev), kcd, vcd, n_valid=nd, k_new=kn.to(dev),
                                     v_new=vn.to(dev))
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() & kvc.DEV_CACHE_FULL
    assert int(nd[0, 0, 1]) == cap


def test_decode_repeated_calls_reuse_workspace(kvc):
    q, kc, vc = rand_cache(1, 1, 32, 8, 128, 1280, seed=21)
    dev = torch.device("cuda")
    args = (q.to(dev), kc.to(dev), vc.to(dev))
    outs = [kvc.compressed_decode_attn(*args, n_uniform=1100).clone() for _ in range(3)]
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


def test_rows_past_n_are_never_read_into_the_output(kvc):
    # stale cache rows past n (here NaN bit patterns) must not reach the output
    q, kc, vc = rand_cache(1, 2, 8, 2, 128, 300, seed=31)
    n = torch.tensor([[[130, 257]]], dtype=torch.int32).expand(1, 2, 2).contiguous()
    kc2, vc2 = kc.clone(), vc.clone()
    for b in range(2):
        for h in range(2):
            kc2[0, b, h, n[0, b, h]:] = float("nan")
            vc2[0, b, h, n[0, b, h]:] = float("nan")
    dev = torch.device("cuda")
    out = kvc.compressed_decode_attn(q.to(dev), kc2.to(dev), vc2.to(dev), n_valid=n.to(dev))
    assert torch.isfinite(out.float()).all()
    assert_outputs_close(f64(out), oracle_decode(q, kc, vc, n.numpy()))


MANY_TILES = [  # Ly, B, Hq, Hkv, D, cap: units x tile slots well above the resident grid
    (1, 16, 32, 8, 128, 2304),
    (2, 8, 32, 4, 64, 2100),
    (1, 24, 8, 8, 128, 1500),
]


@pytest.mark.parametrize("shape", MANY_TILES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("append", [False, True], ids=["attend", "append"])
def test_decode_many_tiles_per_cta(kvc, shape, append):
    """Each CTA streams several tiles of several units: the shared-memory ring wraps many
    times, units split over CTAs merge through the workspace, and ragged row counts
    (including empty units, empty segments and, with the append, a full unit) mix."""
    Ly, B, Hq, Hkv, D, cap = shape
    q, kc, vc = rand_cache(Ly, B, Hq, Hkv, D, cap, seed=cap + Hkv + (1 if append else 0))
    g = torch.Generator().manual_seed(cap)
    n0 = torch.randint(0, cap + 1, (Ly, B, Hkv), generator=g, dtype=torch.int32)
    flat = n0.view(-1)
    flat[0], flat[1], flat[2], flat[-1] = 0, cap, 1, cap - 1
    flat[3:8] = torch.tensor([128, 129, 127, 0, 2 * 128])
    dev = torch.device("cuda")
    kcd, vcd, nd = kc.to(dev), vc.to(dev), n0.to(dev)
    if append:
        kn = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16)
        vn = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16)
        out = kvc.compressed_decode_attn(q.to(dev), kcd, vcd, n_valid=nd, k_new=kn.to(dev),
                                         v_new=vn.to(dev))
        torch.cuda.synchronize()
        st = kvc.kvc_device_status()
        assert st & kvc.DEV_CACHE_FULL and st & ~kvc.DEV_CACHE_FULL == 0, st
        kc2, vc2, n1 = kc.clone(), vc.clone(), n0.clone()
        for idx in np.ndindex(*n0.shape):
            if int(n0[idx]) < cap:
                kc2[idx + (int(n0[idx]),)] = kn[idx]
                vc2[idx + (int(n0[idx]),)] = vn[idx]
                n1[idx] += 1
        assert torch.equal(nd.cpu(), n1)
        assert torch.equal(kcd.cpu(), kc2) and torch.equal(vcd.cpu(), vc2)
        assert_outputs_close(f64(out), oracle_decode(q, kc2, vc2, n1.numpy()))
    else:
        out = kvc.compressed_decode_attn(q.to(dev), kcd, vcd, n_valid=nd)
        torch.cuda.synchronize()
        assert kvc.kvc_device_status() == 0
        assert_outputs_close(f64(out), oracle_decode(q, kc, vc, n0.numpy()))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 7, 8])
def test_decode_every_head_group_and_dim(kvc, D, G):
    """Every head group G = 1..8 (G = 3, 5, 6, 7 run the next compiled group size with
    zero query rows padding the MMA) and both head dims, with enough units that CTAs
    stream several tiles and units split between CTAs, ragged row counts and the fused
    append."""
    Ly, B, Hkv, cap = 1, 4, 16, 777
    Hq = Hkv * G
    q, kc, vc = rand_cache(Ly, B, Hq, Hkv, D, cap, seed=D * 10 + G)
    g = torch.Generator().manual_seed(D + G)
    n0 = torch.randint(0, cap, (Ly, B, Hkv), generator=g, dtype=torch.int32)
    n0.view(-1)[:3] = torch.tensor([0, 1, cap - 1], dtype=torch.int32)
    kn = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16)
    vn = torch.randn((Ly, B, Hkv, D), generator=g).to(torch.bfloat16)
    dev = torch.device("cuda")
    kcd, vcd, nd = kc.to(dev), vc.to(dev), n0.to(dev)
    out = kvc.compressed_decode_attn(q.to(dev), kcd, vcd, n_valid=nd, k_new=kn.to(dev),
                                     v_new=vn.to(dev))
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    kc2, vc2 = kc.clone(), vc.clone()
    for idx in np.ndindex(*n0.shape):
        kc2[idx + (int(n0[idx]),)] = kn[idx]
        vc2[idx + (int(n0[idx]),)] = vn[idx]
    assert torch.equal(nd.cpu(), n0 + 1)
    assert_outputs_close(f64(out), oracle_decode(q, kc2, vc2, (n0 + 1).numpy()))


def test_decode_rejects_more_than_eight_heads_per_group(kvc):
    dev = torch.device("cuda")
    q = torch.zeros((1, 1, 9, 64), dtype=torch.bfloat16, device=dev)
    kc = torch.zeros((1, 1, 1, 16, 64), dtype=torch.bfloat16, device=dev)
    with pytest.raises(kvc.KVCError) as e:
        kvc.compressed_decode_attn(q, kc, kc, n_uniform=4)
    assert e.value.code == 2  # KVC_ERR_SHAPE
