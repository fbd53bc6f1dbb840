"""GPU parity of the attention backward (dQ, dK, dV) against the fp64 oracle,
through the C ABI. The backward's inputs O and LSE come from this library's
own forward (the chain a training step runs).

Tolerance: P and dS enter the tensor-core products as bf16 (relative rounding
2^-9 each) and the gradients are written as bf16 (another 2^-9), with fp32
accumulation; the comparison is relative to each gradient's largest
magnitude: max-abs <= 2e-2 * max|ref| and mean-abs <= 2e-3 * max|ref|. The
magnitude is floored at 1e-4: where the exact gradient vanishes (one key: P = 1
and dS = dO.v - dO.O = 0 since O = v), the kernel returns the fp32
cancellation of two O(1) dot products, ~1e-7."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention_backward_ref
from tests.parity import to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    import online_softmax_fusion_gb300 as m
    from online_softmax_fusion_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    return m


def _rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


def _close(got, ref, what):
    g = to64(got)
    r = to64(ref)
    assert g.shape == r.shape
    assert np.all(np.isfinite(g)), what
    mag = max(float(np.abs(r).max()), 1e-4)
    err = np.abs(g - r)
    assert err.max() <= 2e-2 * mag, f"{what}: max-abs {err.max():.3e} vs {mag:.3e}"
    assert err.mean() <= 2e-3 * mag, f"{what}: mean-abs {err.mean():.3e} vs {mag:.3e}"


def _impls(d):
    return ["mma_sync"] + (["tcgen05"] if d == 128 else [])


CASES = [
    (1, 2, 2, 128, 128, 128, False, False),
    (2, 4, 2, 200, 200, 128, True, False),     # GQA, ragged, causal
    (1, 4, 1, 130, 130, 64, True, True),       # MQA, d = 64, ALiBi
    (1, 2, 2, 96, 250, 128, True, False),      # Lq < Lk (bottom-right causal)
    (1, 2, 2, 300, 150, 128, True, False),     # Lq > Lk: leading rows see no key
    (1, 8, 2, 256, 256, 128, True, True),      # GQA + ALiBi, tile-aligned
    (2, 2, 2, 70, 330, 128, False, True),      # non-causal ALiBi, key tail inside a 128-key block
    (1, 1, 1, 1, 1, 128, True, False),         # one query, one key
]


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,d,causal,alibi,impl",
                         [c + (i,) for c in CASES for i in _impls(c[5])])
def test_backward_small(attn, B, Hq, Hkv, Lq, Lk, d, causal, alibi, impl):
    q = _rand((B, Hq, Lq, d), 11 + Lq)
    k = _rand((B, Hkv, Lk, d), 12 + Lk)
    v = _rand((B, Hkv, Lk, d), 13 + Lk)
    do = _rand((B, Hq, Lq, d), 14 + Lq)
    slopes = W.alibi_slopes(Hq) if alibi else None
    scale = d ** -0.5
    qc, kc, vc, dc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    sl = None if slopes is None else slopes.cuda()
    O, L = attn.prefill(qc, kc, vc, causal=causal, scale=scale, alibi_slopes=sl)
    dq, dk, dv = attn.backward(qc, kc, vc, O, L, dc, causal=causal, scale=scale, alibi_slopes=sl,
                               impl=impl)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    rq, rk, rv = attention_backward_ref(q, k, v, do, scale=scale, causal=causal,
                                        alibi_slopes=slopes)
    _close(dq, rq, "dQ")
    _close(dk, rk, "dK")
    _close(dv, rv, "dV")


@pytest.mark.parametrize("impl", ["mma_sync", "tcgen05"])
def test_backward_causal_mha_1k(attn, impl):
    """B=1, 8 heads, L=1024 causal (many K/V blocks per row, many Q blocks per
    key block): full comparison."""
    B, H, L, d = 1, 8, 1024, 128
    q = _rand((B, H, L, d), 1)
    k = _rand((B, H, L, d), 2)
    v = _rand((B, H, L, d), 3)
    do = _rand((B, H, L, d), 4)
    qc, kc, vc, dc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    O, Ls = attn.prefill(qc, kc, vc, causal=True)
    dq, dk, dv = attn.backward(qc, kc, vc, O, Ls, dc, causal=True, impl=impl)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    rq, rk, rv = attention_backward_ref(q, k, v, do, scale=d ** -0.5, causal=True)
    _close(dq, rq, "dQ")
    _close(dk, rk, "dK")
    _close(dv, rv, "dV")


def test_backward_tcgen05_matches_mma_sync_at_full_size(attn):
    """The causal MHA workload (B=4, H=32, L=4096, d=128): the two
    implementations agree within the bf16 rounding of their outputs, and a
    sample of rows matches the oracle."""
    cfg = W.PREFILL_CONFIGS["prefill_mha_causal_4k"]
    inp = W.make_prefill_inputs(cfg, "cuda")
    q, k, v = inp["q"], inp["k"], inp["v"]
    g = W.seeded_generator(cfg.seed + 7, "cuda")
    do = W._normal_bf16(q.shape, g, "cuda")
    O, L = attn.prefill(q, k, v, causal=True)
    a = attn.backward(q, k, v, O, L, do, causal=True, impl="tcgen05")
    b = attn.backward(q, k, v, O, L, do, causal=True, impl="mma_sync")
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    for x, y, name in zip(a, b, ("dQ", "dK", "dV")):
        xf, yf = x.float(), y.float()
        mag = yf.abs().max().item()
        assert torch.isfinite(xf).all(), name
        assert (xf - yf).abs().max().item() <= 2e-2 * mag, name
        assert (xf - yf).abs().mean().item() <= 2e-3 * mag, name
    # one head in full against the oracle (batch 1, head 5)
    sl = (slice(1, 2), slice(5, 6))
    rq, rk, rv = attention_backward_ref(q[sl].cpu(), k[sl].cpu(), v[sl].cpu(), do[sl].cpu(),
                                        scale=cfg.scale, causal=True)
    _close(a[0][sl], rq, "dQ")
    _close(a[1][sl], rk, "dK")
    _close(a[2][sl], rv, "dV")
