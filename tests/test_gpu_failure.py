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


@pytest.mark.parametrize("impl", ["tcgen05", "tcgen05_1tile"])
@pytest.mark.parametrize("skip", [0, 3, 15])
def test_prefill_kernel_abort_path(attn, skip, impl):
    """The real tcgen05 prefill (both CTA forms) whose first CTA's producer
    stops before one K/V ring entry (entries K_0, V_0, K_1, ...; that CTA
    streams 8 KV tiles, so 15 is its last entry), with a 100 ms limit on every
    wait. That CTA's MMA warp must give up, record ATTN_ERR_TIMEOUT and wind
    the CTA down (warps leave their waits together, copies in flight land,
    issued products complete, tensor memory is freed); every other CTA's rows
    must be exact, and the next ordinary prefill must match the oracle."""
    from oracle import attention_ref
    from tests.parity import assert_attention_close

    B, H, L, d = 1, 2, 1024, 128
    g = torch.Generator().manual_seed(40 + skip)
    q = torch.randn(B, H, L, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, H, L, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, H, L, d, generator=g).to(torch.bfloat16)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    assert attn.device_status() == 0
    t0 = time.time()
    O, Ls = attn.selftest_prefill_abort(qd, kd, vd, skip, limit_ms=100, causal=True, impl=impl)
    st = attn.device_status()          # synchronises the stream
    dt = time.time() - t0
    assert st == ATTN_ERR_TIMEOUT
    assert 0.05 < dt < 5.0
    assert attn.device_status() == 0
    Or, Lr = attention_ref(q, k, v, scale=d ** -0.5, causal=True)
    # the first CTA owns the heaviest row block of head 0 (rows 768..1023 with
    # two tiles per CTA, 896..1023 with one); every other row was computed by
    # a CTA that ran normally
    first = 768 if impl == "tcgen05" else 896
    assert_attention_close(O[0, 0, :first], Ls[0, 0, :first], Or[0, 0, :first],
                           Lr[0, 0, :first])
    assert_attention_close(O[0, 1], Ls[0, 1], Or[0, 1], Lr[0, 1])
    # the context is intact: an ordinary prefill right after matches the oracle
    O2, L2 = attn.prefill(qd, kd, vd, causal=True)
    assert attn.device_status() == 0
    assert_attention_close(O2, L2, Or, Lr)
