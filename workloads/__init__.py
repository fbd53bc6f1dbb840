"""Seeded synthetic inputs shaped like the attention workloads the pages measure.

This module is shared by the oracle side (tests, CPU baseline) and the CUDA side
(tests, bench). It holds workload shapes and random-number generation only:
none of the attention arithmetic (no scores, softmax, masking or merging) lives
here.

Workload shapes follow the attention variants named in Neptune论文浅读
(gentlecold.top) §9 (Global, Causal, ALiBi, GQA; prefill and decode), the
forward-attention benchmark shape of the Twill review (xllm-io) §七
(batch 4, 32 heads, head dim 128) and the grouped-query decode layout of
CMU 15-779 第 11 讲 §7.1 (query heads stacked per KV head). The pages measure
on no dataset; inputs are i.i.d. normal bf16 values from a fixed seed.

The RMSNorm + MatMul workload takes the LLaMA-2-7B shape of CMU 15-779
第 11 讲 §3.3 (hidden H = output D = 4096) at a small batch and at batch 256.
X is N(0, 1), the RMSNorm weight G is 1 + 0.1 N(0, 1) and W is N(0, 1) / sqrt(H)
(so O has unit scale), all rounded to bf16.

Layout of every tensor (row-major, innermost dimension last):
  prefill  Q [B, Hq, Lq, d], K and V [B, Hkv, Lk, d]
  decode   Q [B, Hq, d],     K and V [B, Hkv, Lk_max, d], kv_lens [B] int32
  rmsnorm  X [B, H], G [H], W [H, D], O [B, D]
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = [
    "PrefillConfig", "DecodeConfig", "PREFILL_CONFIGS", "DECODE_CONFIGS",
    "GQA_SWEEP_LENGTHS", "gqa_sweep_config", "alibi_slopes",
    "make_prefill_inputs", "make_decode_inputs", "seeded_generator",
    "sample_rows", "RmsMatmulConfig", "RMS_MATMUL_CONFIGS", "make_rmsnorm_matmul_inputs",
]


@dataclass(frozen=True)
class PrefillConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    Lq: int
    Lk: int
    d: int
    causal: bool
    alibi: bool = False
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    Lk_max: int
    d: int
    len_lo: int            # kv_len drawn uniformly in [len_lo, len_hi]
    len_hi: int
    num_splits: int = 0    # 0 lets the library choose
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# The five workloads: a single-head check, causal MHA prefill, a causal GQA +
# ALiBi sweep over L, a variable-length GQA decode and a long-context decode
# with outlier keys.
PREFILL_CONFIGS = {
    "single_head_noncausal": PrefillConfig(
        "single_head_noncausal", B=1, Hq=1, Hkv=1, Lq=128, Lk=128, d=64,
        causal=False, seed=1234),
    "prefill_mha_causal_4k": PrefillConfig(
        "prefill_mha_causal_4k", B=4, Hq=32, Hkv=32, Lq=4096, Lk=4096, d=128,
        causal=True, seed=1235),
}

GQA_SWEEP_LENGTHS = (512, 1024, 2048, 4096, 8192, 16384, 32768, 65536)


def gqa_sweep_config(L: int) -> PrefillConfig:
    return PrefillConfig(f"prefill_gqa_alibi_causal_L{L}", B=1, Hq=32, Hkv=8,
                         Lq=L, Lk=L, d=128, causal=True, alibi=True,
                         seed=1236 + L)


for _L in GQA_SWEEP_LENGTHS:
    PREFILL_CONFIGS[gqa_sweep_config(_L).name] = gqa_sweep_config(_L)

DECODE_CONFIGS = {
    "decode_gqa_varlen": DecodeConfig(
        "decode_gqa_varlen", B=64, Hq=32, Hkv=8, Lk_max=32768, d=128,
        len_lo=1024, len_hi=32768, seed=1237),
    "decode_long_outlier": DecodeConfig(
        "decode_long_outlier", B=4, Hq=64, Hkv=8, Lk_max=131072, d=128,
        len_lo=131072, len_hi=131072, num_splits=64, outlier_frac=0.01,
        outlier_scale=8.0, seed=1238),
}


@dataclass(frozen=True)
class RmsMatmulConfig:
    name: str
    B: int
    H: int
    D: int
    seed: int = 0


RMS_MATMUL_CONFIGS = {
    "rmsnorm_matmul_small_ragged": RmsMatmulConfig(
        "rmsnorm_matmul_small_ragged", B=5, H=328, D=200, seed=1300),
    "rmsnorm_matmul_llama7b_b16": RmsMatmulConfig(
        "rmsnorm_matmul_llama7b_b16", B=16, H=4096, D=4096, seed=1301),
    "rmsnorm_matmul_llama7b_b256": RmsMatmulConfig(
        "rmsnorm_matmul_llama7b_b256", B=256, H=4096, D=4096, seed=1302),
}


def seeded_generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def alibi_slopes(Hq: int) -> torch.Tensor:
    """Per-query-head ALiBi slopes 2^(-8h/Hq) for h = 1..Hq (fp32, CPU).

    This is a workload parameter (a fixed geometric sequence), passed to both
    sides as an input.
    """
    h = torch.arange(1, Hq + 1, dtype=torch.float64)
    return torch.pow(2.0, -8.0 * h / Hq).to(torch.float32)


def _normal_bf16(shape, g: torch.Generator, device) -> torch.Tensor:
    return torch.randn(*shape, generator=g, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


def make_prefill_inputs(cfg: PrefillConfig, device="cpu", seed: int | None = None):
    """Q, K, V bf16 i.i.d. N(0, 1); ALiBi slopes when the config uses them."""
    dev = torch.device(device)
    g = seeded_generator(cfg.seed if seed is None else seed, dev)
    q = _normal_bf16((cfg.B, cfg.Hq, cfg.Lq, cfg.d), g, dev)
    k = _normal_bf16((cfg.B, cfg.Hkv, cfg.Lk, cfg.d), g, dev)
    v = _normal_bf16((cfg.B, cfg.Hkv, cfg.Lk, cfg.d), g, dev)
    slopes = alibi_slopes(cfg.Hq).to(dev) if cfg.alibi else None
    return {"q": q, "k": k, "v": v, "alibi_slopes": slopes}


def make_decode_inputs(cfg: DecodeConfig, device="cpu", seed: int | None = None):
    """Q [B,Hq,d], padded K/V [B,Hkv,Lk_max,d] bf16 N(0,1), kv_lens [B] int32.

    kv_len_b is uniform in [len_lo, len_hi]. With outlier_frac > 0, for every
    (b, kv head) exactly round(outlier_frac * kv_len) K rows, chosen without
    replacement, are multiplied by outlier_scale (a power of two, so exact in
    bf16).
    """
    dev = torch.device(device)
    g = seeded_generator(cfg.seed if seed is None else seed, dev)
    q = _normal_bf16((cfg.B, cfg.Hq, cfg.d), g, dev)
    k = _normal_bf16((cfg.B, cfg.Hkv, cfg.Lk_max, cfg.d), g, dev)
    v = _normal_bf16((cfg.B, cfg.Hkv, cfg.Lk_max, cfg.d), g, dev)
    if cfg.len_lo == cfg.len_hi:
        kv_lens = torch.full((cfg.B,), cfg.len_hi, dtype=torch.int32, device=dev)
    else:
        kv_lens = torch.randint(cfg.len_lo, cfg.len_hi + 1, (cfg.B,), generator=g,
                                device=dev, dtype=torch.int64).to(torch.int32)
    if cfg.outlier_frac > 0.0:
        lens = kv_lens.cpu().tolist()
        for b in range(cfg.B):
            n_out = int(round(cfg.outlier_frac * lens[b]))
            for h in range(cfg.Hkv):
                idx = torch.randperm(lens[b], generator=g, device=dev)[:n_out]
                k[b, h, idx] = k[b, h, idx] * cfg.outlier_scale
    return {"q": q, "k": k, "v": v, "kv_lens": kv_lens}


def sample_rows(L: int, n_random: int, n_edge: int, seed: int) -> torch.Tensor:
    """Sorted unique query-row indices: the first and last n_edge rows plus
    n_random rows drawn from a seeded generator (CPU, int64)."""
    g = seeded_generator(seed, "cpu")
    parts = [torch.arange(0, min(n_edge, L)),
             torch.arange(max(0, L - n_edge), L)]
    if n_random > 0:
        parts.append(torch.randint(0, L, (n_random,), generator=g))
    return torch.unique(torch.cat(parts)).to(torch.int64)


def make_rmsnorm_matmul_inputs(cfg: RmsMatmulConfig, device="cpu", seed: int | None = None):
    """X [B, H] ~ N(0, 1), G [H] ~ 1 + 0.1 N(0, 1), W [H, D] ~ N(0, 1) / sqrt(H); bf16."""
    dev = torch.device(device)
    g = seeded_generator(cfg.seed if seed is None else seed, dev)
    x = _normal_bf16((cfg.B, cfg.H), g, dev)
    gw = (1.0 + 0.1 * torch.randn(cfg.H, generator=g, device=dev)).to(torch.bfloat16)
    w = (torch.randn(cfg.H, cfg.D, generator=g, device=dev) / math.sqrt(cfg.H)).to(torch.bfloat16)
    return {"x": x, "g": gw, "w": w}
