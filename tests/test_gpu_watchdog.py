"""Failure detection without a GPU fault: a bounded device wait on an
mbarrier that nothing arrives on gives up, records FA_ERR_DEVICE_TIMEOUT in
the status word and returns; the context stays usable afterwards."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_cleared(fa):
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    assert fa.selftest_wait_timeout(2_000_000) == fa.FA_OK   # ~1 ms of SM cycles
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_ERR_DEVICE_TIMEOUT
    assert fa.device_status() == fa.FA_OK                     # read clears it
    # the context still works
    x = torch.randn(1, 1, 128, 64, device="cuda").to(torch.bfloat16)
    o, lse = fa.forward(x, x, x)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and fa.device_status() == 0
