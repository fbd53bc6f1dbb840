"""Failure detection on the GPU without a fault: every device wait is bounded.
A self-test kernel waits on a barrier nothing signals, with a short limit; the
kernel must record ATTN_ERR_TIMEOUT in the status word and return, and the
context must stay usable."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu

ATTN_ERR_TIMEOUT = 6


@pytest.fixture(scope="module")
def attn():
    import online_softmax_fusion_gb300 as m
    from online_softmax_fusion_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    return m


def test_bounded_wait_reports_timeout_and_context_survives(attn):
    assert attn.device_status() == 0
    t0 = time.time()
    attn.selftest_wait_timeout(200)
    st = attn.device_status()          # synchronises the stream
    dt = time.time() - t0
    assert st == ATTN_ERR_TIMEOUT
    assert 0.15 < dt < 5.0
    assert attn.device_status() == 0  # read-and-clear
    # the context still runs kernels correctly
    q = torch.randn(1, 2, 256, 128, device="cuda").to(torch.bfloat16)
    O, L = attn.prefill(q, q, q, causal=True)
    torch.cuda.synchronize()
    assert torch.isfinite(O.float()).all() and torch.isfinite(L).all()
    assert attn.device_status() == 0


def test_selftest_rejects_bad_limit(attn):
    with pytest.raises(attn.AttnError):
        attn.selftest_wait_timeout(0)
