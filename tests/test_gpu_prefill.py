"""GPU parity of the prefill kernels against the fp64 oracle, through the C ABI.

Every case is compared element by element with the oracle: the small cases,
the full causal MHA workload (every head and row) and the causal GQA + ALiBi
sweep up to L = 8192 in full; at L >= 16384 every head is compared on a seeded
sample of rows plus the first and last 128 (rows are independent, so each is
an exact check of that row).
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention_ref
from tests.parity import assert_attention_close

pytestmark = pytest.mark.gpu

IMPLS = ["tcgen05", "tcgen05_1tile", "mma_sync"]


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


def _run_case(attn, impl, B, Hq, Hkv, Lq, Lk, d, causal, alibi, seed=0, scale=None, qscale=1.0):
    q = _rand((B, Hq, Lq, d), seed, qscale)
    k = _rand((B, Hkv, Lk, d), seed + 1, qscale)
    v = _rand((B, Hkv, Lk, d), seed + 2)
    slopes = W.alibi_slopes(Hq) if alibi else None
    scale = (1.0 / d ** 0.5) if scale is None else scale
    O, L = attn.prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale,
                        alibi_slopes=None if slopes is None else slopes.cuda(), impl=impl)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    Or, Lr = attention_ref(q, k, v, scale=scale, causal=causal, alibi_slopes=slopes)
    assert_attention_close(O, L, Or, Lr)
    return O, L


@pytest.mark.parametrize("impl", IMPLS)
def test_single_head_noncausal_config(attn, impl):
    cfg = W.PREFILL_CONFIGS["single_head_noncausal"]
    inp = W.make_prefill_inputs(cfg, "cpu")
    O, L = attn.prefill(inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda(), causal=False,
                        scale=cfg.scale, impl=impl)
    Or, Lr = attention_ref(inp["q"], inp["k"], inp["v"], scale=cfg.scale)
    assert_attention_close(O, L, Or, Lr)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,d,causal,alibi", [
    (1, 2, 2, 300, 300, 128, False, False),    # ragged tail, several tiles
    (2, 4, 2, 300, 300, 128, True, False),     # GQA, causal, ragged
    (1, 4, 1, 257, 257, 64, True, True),       # d = 64, ALiBi, MQA
    (1, 2, 2, 100, 333, 128, True, False),     # Lq < Lk: bottom-right aligned mask
    (1, 2, 1, 384, 200, 128, True, False),     # Lq > Lk: leading rows see no key
    (1, 2, 2, 1, 1, 128, False, False),        # single query, single key
    (1, 1, 1, 1, 777, 64, True, False),        # one query row against many keys
    (2, 8, 2, 512, 512, 128, True, True),      # GQA + ALiBi + causal, tile-aligned
    (1, 2, 2, 129, 129, 64, False, True),      # non-causal ALiBi (|i - j|)
])
def test_prefill_small_cases(attn, impl, B, Hq, Hkv, Lq, Lk, d, causal, alibi):
    _run_case(attn, impl, B, Hq, Hkv, Lq, Lk, d, causal, alibi, seed=Lq * 7 + Lk)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("Hq,Lq", [(8, 1024), (4, 1000)])
def test_alibi_far_keys_dominate(attn, impl, Hq, Lq):
    """Causal ALiBi where the keys far from the diagonal carry much larger
    scores (K rows scaled x8 below the first 256 keys): scanned diagonal-
    first, later tiles raise the row maximum, so the bound that lets a warp
    skip the exact maximum fails and the reference is repaired mid-row, on
    top of the masked diagonal tile and a ragged tail."""
    d = 128
    q = _rand((1, Hq, Lq, d), 71)
    k = _rand((1, 2, Lq, d), 72)
    v = _rand((1, 2, Lq, d), 73)
    kf = k.float()
    kf[:, :, : Lq - 256] *= 8.0
    k = kf.to(torch.bfloat16)
    slopes = W.alibi_slopes(Hq)
    scale = 1.0 / d ** 0.5
    O, L = attn.prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale,
                        alibi_slopes=slopes.cuda(), impl=impl)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    Or, Lr = attention_ref(q, k, v, scale=scale, causal=True, alibi_slopes=slopes)
    assert_attention_close(O, L, Or, Lr)


@pytest.mark.parametrize("impl", IMPLS)
def test_large_logits_stay_finite(attn, impl):
    """q and K scaled x8 (logits in the hundreds): the repaired online softmax
    stays finite and matches the oracle."""
    _run_case(attn, impl, 1, 2, 2, 256, 256, 128, True, False, seed=99, qscale=8.0)


@pytest.mark.parametrize("impl", IMPLS)
def test_causal_masking_is_exact(attn, impl):
    """Future keys contribute exactly zero weight: overwriting every K/V row
    past the causal frontier with +/-1e4 leaves O and LSE bit-identical."""
    B, H, L, d = 1, 2, 256, 128
    q = _rand((B, H, L, d), 5).cuda()
    k = _rand((B, H, L, d), 6).cuda()
    v = _rand((B, H, L, d), 7).cuda()
    # now square causal problem; perturb keys beyond each row tile's frontier
    Oa, La = attn.prefill(q, k, v, causal=True, impl=impl)
    for cut in (64, 128, 200):
        kp = k.clone()
        vp = v.clone()
        kp[:, :, cut:] = 1e4
        vp[:, :, cut:] = -1e4
        Ob, Lb = attn.prefill(q, kp, vp, causal=True, impl=impl)
        assert torch.equal(Oa[:, :, :cut], Ob[:, :, :cut])
        assert torch.equal(La[:, :, :cut], Lb[:, :, :cut])


def _full_size_check(attn, cfg, impls, rows=None):
    """Runs each implementation on the full workload, then compares every
    query head of every batch entry with the oracle: every row when rows is
    None, else the given rows of every head (rows are independent, so each
    compared row is an exact check of that row)."""
    inp = W.make_prefill_inputs(cfg, "cuda")
    q, k, v, slopes = inp["q"], inp["k"], inp["v"], inp["alibi_slopes"]
    outs = {}
    for impl in impls:
        O, L = attn.prefill(q, k, v, causal=cfg.causal, scale=cfg.scale, alibi_slopes=slopes,
                            impl=impl)
        torch.cuda.synchronize()
        assert attn.device_status() == 0
        if rows is not None:
            idx = torch.from_numpy(rows).cuda()
            O, L = O.index_select(2, idx), L.index_select(2, idx)
        outs[impl] = (O.cpu(), L.cpu())
        del O, L
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    del q, k, v
    G = cfg.Hq // cfg.Hkv
    sl = None if slopes is None else slopes.cpu()
    worst = 0.0
    for b in range(cfg.B):
        for h in range(cfg.Hq):
            kv = h // G
            Or, Lr = attention_ref(qc[b:b + 1, h:h + 1], kc[b:b + 1, kv:kv + 1],
                                   vc[b:b + 1, kv:kv + 1], scale=cfg.scale, causal=cfg.causal,
                                   alibi_slopes=None if sl is None else sl[h:h + 1], rows=rows)
            for impl, (O, L) in outs.items():
                (mx, _), _ = assert_attention_close(O[b, h], L[b, h], Or[0, 0], Lr[0, 0],
                                                    what=f"[{impl}, b={b}, h={h}]")
                worst = max(worst, mx)
    return worst


def test_causal_mha_4k_full_size(attn):
    """Causal MHA at B=4, H=32, L=4096: every head and every row, both
    tensor-core paths, against the oracle."""
    _full_size_check(attn, W.PREFILL_CONFIGS["prefill_mha_causal_4k"], IMPLS)


@pytest.mark.parametrize("L", [512, 1024, 2048, 4096, 8192])
def test_gqa_alibi_sweep_full(attn, L):
    """Causal GQA + ALiBi sweep up to L = 8192: every head, every row."""
    _full_size_check(attn, W.gqa_sweep_config(L), ["tcgen05", "tcgen05_1tile"])


@pytest.mark.parametrize("L", [16384, 32768, 65536])
def test_gqa_alibi_sweep_long_sampled(attn, L):
    """L >= 16384: every head on a seeded sample of 512 rows plus the first
    and last 128 rows."""
    rows = W.sample_rows(L, 512, 128, L).numpy()
    _full_size_check(attn, W.gqa_sweep_config(L), ["tcgen05", "tcgen05_1tile"], rows=rows)


@pytest.mark.skipif("tcgen05" not in IMPLS, reason="single tensor-core path built")
def test_impls_agree_closely(attn):
    """The two tensor-core paths agree with each other far inside the oracle
    tolerance (same inputs, different tilings)."""
    q = _rand((2, 4, 640, 128), 21).cuda()
    k = _rand((2, 2, 640, 128), 22).cuda()
    v = _rand((2, 2, 640, 128), 23).cuda()
    Oa, La = attn.prefill(q, k, v, causal=True, impl="tcgen05")
    Ob, Lb = attn.prefill(q, k, v, causal=True, impl="mma_sync")
    assert (Oa.float() - Ob.float()).abs().max().item() < 2e-2
    assert (La - Lb).abs().max().item() < 1e-4


# ------------------------------------------------------ SoftCap and Window
@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,d,causal,alibi,softcap,window", [
    (1, 2, 2, 300, 300, 128, True, False, 20.0, (-1, -1)),     # softcap, causal, ragged
    (1, 4, 2, 256, 256, 128, False, False, 5.0, (-1, -1)),     # tight cap, non-causal
    (1, 2, 2, 700, 700, 128, True, False, 0.0, (200, -1)),     # sliding window, causal
    (2, 4, 2, 513, 513, 64, False, False, 0.0, (64, 100)),     # two-sided window, d = 64
    (1, 8, 2, 640, 640, 128, True, True, 30.0, (300, -1)),     # softcap + window + ALiBi + GQA
    (1, 2, 2, 100, 400, 128, True, False, 0.0, (50, -1)),      # Lq < Lk with window
    (1, 2, 2, 384, 384, 128, True, False, 0.0, (0, -1)),       # window 0: the diagonal only
])
@pytest.mark.parametrize("impl", ["tcgen05", "tcgen05_1tile"])
def test_prefill_softcap_window(attn, B, Hq, Hkv, Lq, Lk, d, causal, alibi, softcap, window,
                                impl):
    q = _rand((B, Hq, Lq, d), Lq + 1, 2.0)
    k = _rand((B, Hkv, Lk, d), Lk + 2, 2.0)
    v = _rand((B, Hkv, Lk, d), Lk + 3)
    slopes = W.alibi_slopes(Hq) if alibi else None
    scale = d ** -0.5
    O, L = attn.prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale,
                        alibi_slopes=None if slopes is None else slopes.cuda(),
                        softcap=softcap, window=window, impl=impl)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    Or, Lr = attention_ref(q, k, v, scale=scale, causal=causal, alibi_slopes=slopes,
                           softcap=softcap, window_left=window[0], window_right=window[1])
    assert_attention_close(O, L, Or, Lr)


def test_window_long_sequence_sampled(attn):
    """Causal sliding window of 1024 keys over L = 16384 (tiles outside the
    window are skipped): sampled rows against the oracle."""
    L, d, w = 16384, 128, 1024
    q = _rand((1, 4, L, d), 1, 1.0).cuda()
    k = _rand((1, 2, L, d), 2, 1.0).cuda()
    v = _rand((1, 2, L, d), 3, 1.0).cuda()
    O, Ls = attn.prefill(q, k, v, causal=True, window=(w, -1))
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    rows = W.sample_rows(L, 512, 128, 5).numpy()
    idx = torch.from_numpy(rows).cuda()
    for h in range(4):
        Or, Lr = attention_ref(q[:, h:h + 1].cpu(), k[:, h // 2:h // 2 + 1].cpu(),
                               v[:, h // 2:h // 2 + 1].cpu(), scale=d ** -0.5, causal=True,
                               rows=rows, window_left=w)
        assert_attention_close(O[0, h].index_select(0, idx), Ls[0, h].index_select(0, idx),
                               Or[0, 0], Lr[0, 0], what=f"[h={h}]")


def test_softcap_window_unsupported_on_register_tile_kernel(attn):
    q = torch.zeros(1, 1, 128, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(attn.AttnError):
        attn.prefill(q, q, q, impl="mma_sync", softcap=10.0)


# ------------------------------------------------------------ split-KV prefill
@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,causal,alibi,splits", [
    (1, 8, 2, 512, 512, True, True, 2),       # GQA + ALiBi, the short sweep shape
    (1, 8, 2, 512, 512, True, True, 4),
    (2, 4, 4, 300, 300, True, False, 3),      # ragged, MHA
    (1, 4, 2, 100, 700, False, False, 5),     # Lq < Lk, non-causal
    (1, 2, 2, 256, 256, True, False, 8),      # more splits than KV tiles: empty splits
    (1, 2, 1, 384, 130, True, False, 2),      # Lq > Lk: rows that see no key
])
def test_prefill_splitkv(attn, B, Hq, Hkv, Lq, Lk, causal, alibi, splits):
    d = 128
    q = _rand((B, Hq, Lq, d), 31 + Lq)
    k = _rand((B, Hkv, Lk, d), 32 + Lk)
    v = _rand((B, Hkv, Lk, d), 33 + Lk)
    slopes = W.alibi_slopes(Hq) if alibi else None
    scale = d ** -0.5
    sl = None if slopes is None else slopes.cuda()
    O, L = attn.prefill_splitkv(q.cuda(), k.cuda(), v.cuda(), splits, causal=causal, scale=scale,
                                alibi_slopes=sl)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    Or, Lr = attention_ref(q, k, v, scale=scale, causal=causal, alibi_slopes=slopes)
    assert_attention_close(O, L, Or, Lr)
    # the unsplit kernel on the same inputs agrees far inside the tolerance
    O1, L1 = attn.prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale,
                          alibi_slopes=sl)
    torch.cuda.synchronize()
    assert (O.float() - O1.float()).abs().max().item() <= 2e-2
    fin = torch.isfinite(L1)
    assert torch.equal(fin, torch.isfinite(L))
    assert (L[fin] - L1[fin]).abs().max().item() <= 1e-4 if fin.any() else True
