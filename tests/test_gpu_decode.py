"""GPU parity of split-K decode and the log-sum-exp combine against the fp64
oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import combine_ref, decode_ref, decode_split_partials_ref
from tests.parity import assert_attention_close

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


@pytest.mark.parametrize("B,Hq,Hkv,Lmax,d,lens,S", [
    (3, 8, 2, 1000, 128, [1, 63, 1000], 0),      # tiny lengths, auto splits
    (2, 8, 8, 777, 128, [64, 65], 3),             # G = 1, boundaries of a 64-key tile
    (2, 32, 8, 4096, 128, [4096, 1500], 4),       # G = 4 (the varlen workload's grouping)
    (1, 64, 8, 3000, 128, [3000], 64),            # G = 8 with many short splits
    (2, 16, 1, 700, 64, [700, 17], 2),            # G = 16, d = 64
    (1, 32, 1, 500, 128, [500], 1),               # G = 32: two CTAs per KV head
    (2, 4, 4, 5000, 128, [0, 4999], 5),           # an empty sequence
])
def test_decode_small(attn, B, Hq, Hkv, Lmax, d, lens, S):
    q = _rand((B, Hq, d), 1 + B + Hq)
    k = _rand((B, Hkv, Lmax, d), 2 + Lmax)
    v = _rand((B, Hkv, Lmax, d), 3 + Lmax)
    kv_lens = torch.tensor(lens, dtype=torch.int32)
    scale = d ** -0.5
    Op, Lp = attn.decode_splitk(q.cuda(), k.cuda(), v.cuda(), kv_lens.cuda(), scale=scale,
                                num_splits=S)
    Sres = Op.shape[2]
    C = attn.split_len(Lmax, Sres)
    O, L = attn.combine(Op, Lp)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    # partials against the oracle's local reductions
    Opr, Lpr = decode_split_partials_ref(q, k, v, kv_lens, scale=scale, split_len=C,
                                         num_splits=Sres)
    assert_attention_close(Op, Lp, Opr, Lpr)
    # merged result against the unsplit oracle
    Or, Lr = decode_ref(q, k, v, kv_lens, scale=scale)
    assert_attention_close(O, L, Or, Lr)


def test_decode_padding_garbage_is_ignored(attn):
    """K/V rows past kv_len may hold anything (here NaN and huge values)."""
    B, Hq, Hkv, Lmax, d = 2, 8, 2, 300, 128
    q = _rand((B, Hq, d), 41)
    k = _rand((B, Hkv, Lmax, d), 42)
    v = _rand((B, Hkv, Lmax, d), 43)
    lens = torch.tensor([77, 300], dtype=torch.int32)
    kg, vg = k.clone(), v.clone()
    kg[0, :, 77:] = float("nan")
    vg[0, :, 77:] = float("nan")
    kg[0, :, 78] = 3e4
    O, L = attn.decode(q.cuda(), kg.cuda(), vg.cuda(), lens.cuda(), num_splits=2)
    Or, Lr = decode_ref(q, k, v, lens, scale=d ** -0.5)
    assert_attention_close(O, L, Or, Lr)


def test_combine_against_oracle_partials(attn):
    """The combine kernel alone, fed the oracle's own partials, including
    splits with LSE = -inf and a row whose splits are all empty."""
    B, Hq, S, d = 2, 3, 7, 128
    g = np.random.default_rng(7)
    Op = g.standard_normal((B, Hq, S, d))
    Lp = g.standard_normal((B, Hq, S)) * 5
    Lp[0, 1, [0, 3]] = -np.inf
    Lp[1, 2, :] = -np.inf
    O, L = attn.combine(torch.tensor(Op, dtype=torch.float32).cuda(),
                        torch.tensor(Lp, dtype=torch.float32).cuda())
    Or, Lr = combine_ref(Op.astype(np.float32), Lp.astype(np.float32))
    assert_attention_close(O, L, Or, Lr)
    assert torch.all(O[1, 2] == 0)


def _full_size(attn, cfg):
    """The full workload on the GPU, then every (batch entry, KV head) group of
    query heads against the oracle (K/V brought to the host one batch entry at
    a time)."""
    inp = W.make_decode_inputs(cfg, "cuda")
    q, k, v, lens = inp["q"], inp["k"], inp["v"], inp["kv_lens"]
    O, L = attn.decode(q, k, v, lens, scale=cfg.scale, num_splits=cfg.num_splits)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    Oc, Lc, qc, lens_c = O.cpu(), L.cpu(), q.cpu(), lens.cpu()
    for b in range(cfg.B):
        n = int(lens_c[b])
        kb, vb = k[b:b + 1, :, :n].cpu(), v[b:b + 1, :, :n].cpu()
        Or, Lr = decode_ref(qc[b:b + 1], kb, vb, lens_c[b:b + 1], scale=cfg.scale)
        assert_attention_close(Oc[b], Lc[b], Or[0], Lr[0], what=f"[b={b}]")
    return inp


def test_decode_varlen_full_size(attn):
    """Batch 64, 32 query / 8 KV heads, kv_len uniform in [1024, 32768]:
    every batch entry and head against the oracle."""
    _full_size(attn, W.DECODE_CONFIGS["decode_gqa_varlen"])


def test_decode_long_outlier_full_size(attn):
    """Batch 4, 64 query / 8 KV heads, L = 131072 with 1% of K rows x8, 64
    splits: every batch entry and head against the oracle."""
    inp = _full_size(attn, W.DECODE_CONFIGS["decode_long_outlier"])
    # the outlier rows really are there (x8 keys): scores reach well past N(0,1)
    assert float(inp["k"][0, 0].float().abs().max()) > 16.0
