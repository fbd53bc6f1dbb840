"""GPU parity of the host-buffer prefill (attn_prefill_host) through the C ABI.

Each chunk is an ordinary prefill launch over a contiguous run of KV-head
units, and every (batch, head, query tile) is computed by the same kernel
arithmetic whatever the launch's extent, so the pipelined result must equal
the device-buffer prefill bit for bit; small cases are also compared with the
fp64 oracle element by element.
"""
import pytest
import torch

import workloads as W
from oracle import attention_ref
from tests.parity import assert_attention_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    import online_softmax_fusion_gb300 as m
    from online_softmax_fusion_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    return m


def _rand(shape, seed, pin=True):
    g = torch.Generator().manual_seed(seed)
    t = torch.randn(*shape, generator=g).to(torch.bfloat16)
    return t.pin_memory() if pin else t


def _device_ref(attn, q, k, v, **kw):
    O, L = attn.prefill(q.cuda(), k.cuda(), v.cuda(), **kw)
    torch.cuda.synchronize()
    return O.cpu(), L.cpu()


CASES = [
    # B, Hq, Hkv, Lq, Lk, d, causal, alibi, chunk_kv_heads
    (2, 8, 2, 200, 200, 128, True, False, 0),
    (2, 8, 2, 200, 200, 128, True, False, 1),     # one KV head per chunk
    (3, 12, 4, 130, 257, 128, True, False, 3),    # ragged: 3 + 1 KV heads per item
    (3, 12, 4, 130, 257, 128, False, False, 5),   # rounded up to 2 whole items: 2 + 1
    (2, 8, 8, 96, 300, 64, True, True, 3),        # MHA, d = 64, ALiBi slope offsets 0, 3, 6
    (4, 16, 2, 64, 64, 128, True, True, 0),       # whole batch items per chunk, ALiBi
    (1, 1, 1, 1, 1, 128, True, False, 0),         # one query, one key
    (1, 4, 2, 300, 150, 128, True, False, 1),     # Lq > Lk: leading rows see no key
    (2, 8, 8, 257, 513, 64, False, True, 3),      # non-causal ALiBi, ragged lengths, d = 64
]


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,d,causal,alibi,chunk", CASES)
def test_host_prefill_equals_device_prefill(attn, B, Hq, Hkv, Lq, Lk, d, causal, alibi, chunk):
    seed = B * 1000 + Hq * 10 + Lq
    q = _rand((B, Hq, Lq, d), seed)
    k = _rand((B, Hkv, Lk, d), seed + 1)
    v = _rand((B, Hkv, Lk, d), seed + 2)
    slopes = W.alibi_slopes(Hq) if alibi else None
    sl = None if slopes is None else slopes.cuda()
    scale = d ** -0.5
    O, L = attn.prefill_host(q, k, v, causal=causal, scale=scale, alibi_slopes=sl,
                             chunk_kv_heads=chunk)
    assert attn.device_status() == 0
    Od, Ld = _device_ref(attn, q, k, v, causal=causal, scale=scale, alibi_slopes=sl)
    assert torch.equal(O, Od)
    assert torch.equal(L, Ld)
    Or, Lr = attention_ref(q, k, v, scale=scale, causal=causal, alibi_slopes=slopes)
    assert_attention_close(O, L, Or, Lr)


def test_host_prefill_options_and_pageable_memory(attn):
    """SoftCap + a sliding window through the options; pageable (not
    page-locked) host tensors give the same result; LSE may be omitted."""
    q = _rand((2, 4, 300, 128), 5, pin=False)
    k = _rand((2, 2, 300, 128), 6, pin=False)
    v = _rand((2, 2, 300, 128), 7, pin=False)
    kw = dict(causal=True, scale=128 ** -0.5, softcap=20.0, window=(100, -1))
    O, L = attn.prefill_host(q, k, v, chunk_kv_heads=1, **kw)
    Od, Ld = _device_ref(attn, q, k, v, **kw)
    assert torch.equal(O, Od) and torch.equal(L, Ld)
    O2, L2 = attn.prefill_host(q, k, v, chunk_kv_heads=1, with_lse=False, **kw)
    assert L2 is None and torch.equal(O2, Od)
    assert attn.device_status() == 0


def test_host_prefill_back_to_back_without_sync(attn):
    """Two calls queued on one stream with no synchronisation between them,
    sharing the workspace: the second waits for the first's read-back."""
    a = [_rand((1, 8, 256, 128), 20 + i) for i in range(3)]
    b = [_rand((1, 8, 256, 128), 30 + i) for i in range(3)]
    ws = attn.prefill_host_workspace(1, 8, 8, 256, 256, 128)
    Oa, La = attn.prefill_host(*a, causal=True, workspace=ws, synchronize=False)
    Ob, Lb = attn.prefill_host(*b, causal=True, workspace=ws, synchronize=False)
    torch.cuda.synchronize()
    for (q, k, v), O, L in ((a, Oa, La), (b, Ob, Lb)):
        Od, Ld = _device_ref(attn, q, k, v, causal=True)
        assert torch.equal(O, Od) and torch.equal(L, Ld)


def test_host_prefill_full_size_causal_mha(attn):
    """The causal MHA workload (B=4, H=32, L=4096, d=128) with automatic
    chunking (8 chunks of 16 KV heads) equals the device prefill."""
    cfg = W.PREFILL_CONFIGS["prefill_mha_causal_4k"]
    inp = W.make_prefill_inputs(cfg, "cuda")
    q, k, v = inp["q"], inp["k"], inp["v"]
    Od, Ld = attn.prefill(q, k, v, causal=True, scale=cfg.scale)
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    O, L = attn.prefill_host(hq, hk, hv, causal=True, scale=cfg.scale)
    assert attn.device_status() == 0
    assert torch.equal(O, Od.cpu())
    assert torch.equal(L, Ld.cpu())
