"""attn_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (a runtime that owns all device memory through its own
pool, a token loop that must not block on cudaMalloc/cudaFree, or C code that
only holds the tensors it was given). It keeps the split partials in a fixed
array inside the library instead of caller buffers.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test. It passes both alone in a fresh
process and after the rest of the suite."""
import ctypes

import pytest
import torch

from oracle import decode_ref
from tests.parity import assert_attention_close, assert_o_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    import online_softmax_fusion_gb300 as m
    from online_softmax_fusion_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    return m


def _inputs(B, Hq, Hkv, Lmax, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, d, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(B, Hkv, Lmax, d, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(B, Hkv, Lmax, d, generator=g).to(torch.bfloat16).cuda()
    lens = torch.randint(1, Lmax + 1, (B,), generator=g).to(torch.int32).cuda()
    return q, k, v, lens


def _call_noalloc(lib, q, k, v, lens, S, O, LSE):
    """Straight through the C ABI with plain pointers (LSE may be None)."""
    B, Hq, d = q.shape
    Hkv, Lmax = k.shape[1], k.shape[2]
    st = lib.attn_decode_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(lens.data_ptr()),
        B, Hq, Hkv, Lmax, d, d ** -0.5, S, ctypes.c_void_p(O.data_ptr()),
        None if LSE is None else ctypes.c_void_p(LSE.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_noalloc_matches_workspace_decode_and_oracle(attn):
    lib = attn.lib()
    # calls in a row with different shapes, head dims and split counts; each
    # reuses the array the one before it filled. The last one passes no LSE.
    for (B, Hq, Hkv, Lmax, d, S, seed, want_lse) in [(8, 32, 8, 3000, 128, 0, 1, True),
                                                     (4, 64, 8, 9000, 128, 64, 2, True),
                                                     (3, 16, 2, 700, 64, 3, 5, True),
                                                     (2, 8, 2, 1500, 64, 0, 6, False)]:
        q, k, v, lens = _inputs(B, Hq, Hkv, Lmax, d, seed)
        O_ws, L_ws = attn.decode(q, k, v, lens, num_splits=S)
        O = torch.full((B, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        LSE = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda") \
            if want_lse else None
        assert _call_noalloc(lib, q, k, v, lens, S, O, LSE) == 0
        torch.cuda.synchronize()
        assert attn.device_status() == 0
        # the same partials and combine as the workspace decode: identical output
        assert torch.equal(O, O_ws)
        if want_lse:
            assert torch.equal(LSE, L_ws)
        # and the oracle
        Or, Lr = decode_ref(q.cpu(), k.cpu(), v.cpu(), lens.cpu(), scale=d ** -0.5)
        if want_lse:
            assert_attention_close(O, LSE, Or, Lr)
        else:
            assert_o_close(O, Or, lse_ref=Lr)


def test_noalloc_rejects_sizes_beyond_its_array(attn):
    lib = attn.lib()
    q, k, v, lens = _inputs(2, 8, 2, 256, 128, 3)
    O = torch.empty((2, 8, 128), dtype=torch.bfloat16, device="cuda")
    LSE = torch.empty((2, 8), dtype=torch.float32, device="cuda")
    # B*Hq*S*(d+1) floats beyond 8 Mi: 65535 batch entries x 64 heads x 256 splits
    st = lib.attn_decode_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), None, 65535, 64, 8, 1 << 20, 128, 0.1, 256,
        ctypes.c_void_p(O.data_ptr()), ctypes.c_void_p(LSE.data_ptr()), None)
    assert st == 4  # ATTN_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert attn.device_status() == 0
