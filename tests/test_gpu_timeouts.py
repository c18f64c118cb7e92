"""Device-side waits give up after their limit and report KVC_DEV_TIMEOUT; the context
stays usable.  The waits run out on a flag that nothing sets and an mbarrier that
nothing arrives on: no fault, trap or hang is involved."""

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bounded_waits_report_timeout_and_context_survives(kvc):
    code = kvc.kvc_selftest_wait_timeout(2000)   # 2 ms per wait
    assert code == 6                              # KVC_ERR_TIMEOUT: both waits gave up
    assert kvc.kvc_device_status(clear=True) & kvc.DEV_TIMEOUT
    assert kvc.kvc_device_status(clear=True) == 0
    dev = torch.device("cuda")
    q = torch.randn((1, 1, 4, 128), device=dev).to(torch.bfloat16)
    kc = torch.randn((1, 1, 1, 100, 128), device=dev).to(torch.bfloat16)
    out = kvc.compressed_decode_attn(q, kc, kc.clone(), n_uniform=100)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    assert kvc.kvc_device_status() == 0
