"""Parity of the fused RMSNorm + product kernel (through the C ABI) with the
CPU fp64 oracle, on seeded inputs.

Tolerance, derived from the arithmetic: the kernel rounds X ⊙ G to bf16
before the product (relative error <= 2^-9 per term, random in sign, so the
product's error has standard deviation ~ 2^-9 / sqrt(3) times the output
scale s = RMS of the reference output), accumulates in fp32 and rounds O to
bf16 (<= 2^-9 |O|). Hence, element-wise,
    |O - O_ref| <= 2^-8 |O_ref| + 1e-2 s        (about 2x the round-off plus 6 sigma)
and mean |O - O_ref| <= 2e-3 s. The RMS output is an fp32 sum of exact
scaled squares: relative error <= 2e-5.
"""
import math

import numpy as np
import pytest
import torch

import online_softmax_fusion_gb300 as attn
import workloads as W
from oracle import rms_ref, rmsnorm_matmul_ref

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(B, H, D, seed):
    cfg = W.RmsMatmulConfig("t", B=B, H=H, D=D, seed=seed)
    d = W.make_rmsnorm_matmul_inputs(cfg, DEV)
    return d["x"], d["g"], d["w"]


def _check(O, ref, rows=None):
    O = O.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        O = O[rows]
    s = math.sqrt(float(np.mean(ref * ref))) or 1.0
    err = np.abs(O - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-2 * s
    worst = float(np.max(err - bound))
    assert worst <= 0.0, f"max excess {worst:.3e} (scale {s:.3e})"
    assert float(np.mean(err)) <= 2e-3 * s


CASES = [
    # B, H, D, splits, eps
    (5, 328, 200, 0, 0.0),        # ragged everywhere: K tail, feature tail, batch tail
    (1, 64, 8, 1, 0.0),           # smallest: one K step, 8 features
    (16, 512, 256, 1, 1e-5),
    (16, 512, 256, 2, 0.0),
    (16, 512, 256, 4, 0.0),
    (16, 512, 256, 8, 0.0),
    (33, 1024, 384, 4, 1e-6),
    (128, 768, 136, 2, 0.0),
    (256, 512, 256, 0, 0.0),      # largest batch tile
    (300, 256, 128, 2, 0.0),      # two batch tiles of 160
    (7, 136, 520, 2, 0.5),        # K split with uneven ranges (3 K steps over 2 CTAs)
]


@pytest.mark.parametrize("B,H,D,splits,eps", CASES)
def test_parity_small(B, H, D, splits, eps):
    x, g, w = _inputs(B, H, D, seed=B * 7919 + H * 31 + D + splits)
    O, rms = attn.rmsnorm_matmul(x, g, w, eps=eps, splits=splits, with_rms=True)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    ref = rmsnorm_matmul_ref(x.cpu(), g.cpu(), w.cpu(), eps)
    _check(O, ref)
    np.testing.assert_allclose(rms.cpu().numpy(), rms_ref(x.cpu(), eps), rtol=2e-5)


@pytest.mark.parametrize("tile,splits", [(16, 1), (32, 2), (64, 1), (64, 4), (128, 2), (256, 8)])
def test_batch_tiles(tile, splits):
    """Explicit batch tiles: several batch tiles per launch, each with its own
    converter grouping and ring depth."""
    x, g, w = _inputs(200, 768, 264, seed=tile + splits)
    O, rms = attn.rmsnorm_matmul(x, g, w, splits=splits, batch_tile=tile, with_rms=True)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    _check(O, rmsnorm_matmul_ref(x.cpu(), g.cpu(), w.cpu()))
    np.testing.assert_allclose(rms.cpu().numpy(), rms_ref(x.cpu()), rtol=2e-5)


def test_every_split_count_agrees():
    """The cluster reduction: 1, 2, 4 and 8 CTAs per tile give the same O up
    to fp32 summation order (well inside one bf16 ulp)."""
    x, g, w = _inputs(24, 1024, 512, seed=99)
    outs = [attn.rmsnorm_matmul(x, g, w, splits=s)[0].float() for s in (1, 2, 4, 8)]
    for o in outs[1:]:
        assert torch.max(torch.abs(o - outs[0])).item() <= 2.0 ** -7 * max(
            1.0, torch.max(torch.abs(outs[0])).item())


def test_scale_invariance_beyond_fp32_squares():
    """X * 2^100: every square overflows fp32, the repaired sum of squares does
    not; O equals O(X) and RMS scales by 2^100."""
    x, g, w = _inputs(12, 1024, 256, seed=5)
    big = (x.float() * 2.0 ** 100).to(torch.bfloat16)   # exact: a power of two
    assert torch.isinf((big.float() ** 2).sum(dim=1)).all()
    O, rms = attn.rmsnorm_matmul(big, g, w, with_rms=True)
    torch.cuda.synchronize()
    ref = rmsnorm_matmul_ref(x.cpu(), g.cpu(), w.cpu())
    _check(O, ref)
    np.testing.assert_allclose(rms.cpu().numpy().astype(np.float64) / 2.0 ** 100,
                               rms_ref(x.cpu()), rtol=2e-5)


def test_tiny_and_mixed_magnitude_rows():
    """Rows at 2^-60 and rows whose largest entry sits in a late K step (the
    reference exponent grows mid-row and the running sum is repaired)."""
    x, g, w = _inputs(16, 2048, 128, seed=6)
    xf = x.float()
    xf[0:4] *= 2.0 ** -60
    xf[4:8, 1500:] *= 2.0 ** 20
    xf[8:12, :100] *= 2.0 ** -30
    x2 = xf.to(torch.bfloat16)
    for splits in (1, 4):
        O, rms = attn.rmsnorm_matmul(x2, g, w, splits=splits, with_rms=True)
        torch.cuda.synchronize()
        ref = rmsnorm_matmul_ref(x2.cpu(), g.cpu(), w.cpu())
        for rows in (slice(0, 4), slice(4, 8), slice(8, 16)):
            _check(O[rows], ref[rows])
        np.testing.assert_allclose(rms.cpu().numpy(), rms_ref(x2.cpu()), rtol=2e-5)


def test_zero_rows():
    x, g, w = _inputs(20, 256, 128, seed=7)
    x[3] = 0
    x[17] = 0
    O, rms = attn.rmsnorm_matmul(x, g, w, with_rms=True)
    torch.cuda.synchronize()
    assert torch.all(O[3] == 0) and torch.all(O[17] == 0)
    assert rms[3].item() == 0.0 and rms[17].item() == 0.0
    ref = rmsnorm_matmul_ref(x.cpu(), g.cpu(), w.cpu())
    _check(O, ref)
    O2, rms2 = attn.rmsnorm_matmul(x, g, w, eps=1e-4, with_rms=True)
    torch.cuda.synchronize()
    assert torch.all(O2[3] == 0)
    assert rms2[3].item() == pytest.approx(math.sqrt(1e-4), rel=1e-6)


def test_deterministic_repeat():
    x, g, w = _inputs(64, 1024, 512, seed=8)
    a = attn.rmsnorm_matmul(x, g, w)[0]
    b = attn.rmsnorm_matmul(x, g, w)[0]
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["rmsnorm_matmul_llama7b_b16", "rmsnorm_matmul_llama7b_b256"])
def test_full_size_sampled_rows(name):
    """LLaMA-2-7B shape (H = D = 4096) in the launch configuration the bench
    times; the oracle computes a sample of rows in full."""
    cfg = W.RMS_MATMUL_CONFIGS[name]
    d = W.make_rmsnorm_matmul_inputs(cfg, DEV)
    O, rms = attn.rmsnorm_matmul(d["x"], d["g"], d["w"], with_rms=True)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    rows = sorted(set([0, 1, cfg.B - 1] + list(
        np.random.default_rng(11).choice(cfg.B, size=min(cfg.B, 13), replace=False))))
    xs = d["x"].cpu()[rows]
    ref = rmsnorm_matmul_ref(xs, d["g"].cpu(), d["w"].cpu())
    _check(O, ref, rows=rows)
    np.testing.assert_allclose(rms.cpu().numpy()[rows], rms_ref(xs), rtol=2e-5)


# --------------------------------------------- chained (programmatic) launches
@pytest.mark.parametrize("B,H,D", [(16, 4096, 4096), (5, 328, 328), (256, 1024, 1024)])
def test_chained_stack_of_layers(B, H, D):
    """Each call's X is the previous call's output (read after write across
    launches that may overlap): every layer matches the oracle on the exact
    input it was given, and bit for bit the same call launched plainly."""
    x, g, _ = _inputs(B, H, D, 7)
    ws = [_inputs(B, H, D, 20 + i)[2] for i in range(4)]   # square W: O feeds the next X
    outs, rms = [], []
    cur = x
    for w in ws:
        O, R = attn.rmsnorm_matmul(cur, g, w, with_rms=True, chained=True)
        outs.append(O)
        rms.append(R)
        cur = O
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    cur = x
    for w, O, R in zip(ws, outs, rms):
        ref = rmsnorm_matmul_ref(cur, g, w)
        _check(O, ref)
        assert np.allclose(R.cpu().numpy(), rms_ref(cur), rtol=2e-5, atol=0)
        O_plain, R_plain = attn.rmsnorm_matmul(cur, g, w, with_rms=True)
        torch.cuda.synchronize()
        assert torch.equal(O, O_plain) and torch.equal(R, R_plain)
        cur = O


def test_chained_overwrites_the_previous_input():
    """A chained call may start while the call before it still runs; its
    outputs wait for that call, so writing over the previous call's X
    (write after read) leaves the previous result intact."""
    B, H, D = 16, 4096, 4096
    xa, g, w = _inputs(B, H, D, 31)
    xb = _inputs(B, H, D, 32)[0]
    xa_host = xa.cpu()
    Oa = torch.empty((B, D), dtype=torch.bfloat16, device=DEV)
    attn.rmsnorm_matmul(xa, g, w, out=Oa, chained=True)
    attn.rmsnorm_matmul(xb, g, w, out=xa, chained=True)     # writes over xa
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    _check(Oa, rmsnorm_matmul_ref(xa_host, g, w))
    _check(xa[:, :D], rmsnorm_matmul_ref(xb, g, w))


# ------------------------------------------- two-pass form (workspace entry)
TWO_PASS_CASES = [
    # B, H, D, eps
    (5, 328, 200, 0.0),           # ragged everywhere
    (1, 64, 8, 0.0),
    (16, 512, 256, 1e-5),
    (128, 768, 136, 0.0),
    (256, 512, 256, 0.0),
    (300, 256, 128, 0.5),         # two batch tiles
    (256, 4096, 1024, 1e-6),      # the K split of a large hidden size
]


@pytest.mark.parametrize("B,H,D,eps", TWO_PASS_CASES)
def test_two_pass_parity(B, H, D, eps):
    """The conversion pass + product kernel against the oracle; O agrees with
    the fused kernel to one bf16 rounding (same tensor-core operands, the
    per-row scale summed in another order)."""
    x, g, w = _inputs(B, H, D, seed=B * 31 + H + D)
    O, rms = attn.rmsnorm_matmul(x, g, w, eps=eps, with_rms=True, form="two_pass")
    O1, rms1 = attn.rmsnorm_matmul(x, g, w, eps=eps, with_rms=True)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    ref = rmsnorm_matmul_ref(x.cpu(), g.cpu(), w.cpu(), eps)
    _check(O, ref)
    np.testing.assert_allclose(rms.cpu().numpy(), rms_ref(x.cpu(), eps), rtol=2e-5)
    # both are fp32 sums of the same exactly scaled squares, in other orders
    np.testing.assert_allclose(rms.cpu().numpy(), rms1.cpu().numpy(), rtol=1e-5)
    diff = torch.abs(O.float() - O1.float())
    assert torch.all(diff <= 2.0 ** -7 * torch.abs(O1.float()) + 1e-30)


def test_two_pass_extreme_magnitudes_and_zero_rows():
    """Rows at 2^100 (every fp32 square overflows), at 2^-60, all-zero rows,
    with and without eps, through the conversion pass."""
    x, g, w = _inputs(140, 1024, 256, seed=41)
    xf = x.float()
    xf[0:8] *= 2.0 ** 100
    xf[8:16] *= 2.0 ** -60
    xf[16:24, 700:] *= 2.0 ** 20
    xf[30] = 0
    xf[139] = 0
    x2 = xf.to(torch.bfloat16)
    for eps in (0.0, 1e-4):
        O, rms = attn.rmsnorm_matmul(x2, g, w, eps=eps, with_rms=True, form="two_pass")
        torch.cuda.synchronize()
        assert attn.device_status() == 0
        assert torch.all(O[30] == 0) and torch.all(O[139] == 0)
        assert rms[30].item() == pytest.approx(math.sqrt(eps), rel=1e-6, abs=0)
        xs = x2.cpu()
        ref = rmsnorm_matmul_ref(xs, g.cpu(), w.cpu(), eps)
        for rows in (slice(8, 16), slice(16, 140)):
            _check(O[rows], ref[rows])
        # the 2^100 rows: O is that of the unscaled rows, RMS scales exactly
        ref_big = rmsnorm_matmul_ref(x.cpu()[0:8], g.cpu(), w.cpu())
        _check(O[0:8], ref_big)
        np.testing.assert_allclose(rms.cpu().numpy()[0:8].astype(np.float64) / 2.0 ** 100,
                                   rms_ref(x.cpu()[0:8]), rtol=2e-5)
        keep = [i for i in range(140) if i >= 8]
        np.testing.assert_allclose(rms.cpu().numpy()[keep], rms_ref(xs, eps)[keep], rtol=2e-5)


def test_two_pass_full_size_sampled_rows():
    """Batch 256 of the LLaMA-2-7B shape through the automatic form (which
    takes the two-pass path there), the launch the bench times."""
    cfg = W.RMS_MATMUL_CONFIGS["rmsnorm_matmul_llama7b_b256"]
    d = W.make_rmsnorm_matmul_inputs(cfg, DEV)
    O, rms = attn.rmsnorm_matmul(d["x"], d["g"], d["w"], with_rms=True, form="auto")
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    rows = sorted(set([0, 1, cfg.B - 1] + list(
        np.random.default_rng(12).choice(cfg.B, size=min(cfg.B, 13), replace=False))))
    xs = d["x"].cpu()[rows]
    _check(O, rmsnorm_matmul_ref(xs, d["g"].cpu(), d["w"].cpu()), rows=rows)
    np.testing.assert_allclose(rms.cpu().numpy()[rows], rms_ref(xs), rtol=2e-5)


def test_two_pass_rejects_small_workspace_and_unknown_form():
    x, g, w = _inputs(130, 256, 128, seed=3)
    nbytes = attn.rmsnorm_matmul_ws_bytes(130, 256)
    assert nbytes >= 130 * 256 * 2 + 2 * 130 * 4
    small = torch.empty((nbytes - 16,), dtype=torch.uint8, device=DEV)
    with pytest.raises(attn.AttnError):
        attn.rmsnorm_matmul(x, g, w, form="two_pass", workspace=small)
    with pytest.raises(ValueError):
        attn.rmsnorm_matmul(x, g, w, form="three_pass")
    # the fused form through the same entry needs no workspace
    O, _ = attn.rmsnorm_matmul(x, g, w, form="fused", workspace=small)
    torch.cuda.synchronize()
    _check(O, rmsnorm_matmul_ref(x.cpu(), g.cpu(), w.cpu()))


@pytest.mark.parametrize("B,H,D", [(16, 4096, 4096), (5, 328, 328), (256, 1024, 1024)])
def test_two_pass_chained_stack_of_layers(B, H, D):
    """Chained two-pass calls sharing one workspace: each call's X is the
    previous call's output, and its conversion pass rewrites the workspace
    the previous product kernel read. Every layer equals, bit for bit, the
    same call made plainly, and matches the oracle."""
    x, g, _ = _inputs(B, H, D, 9)
    ws = [_inputs(B, H, D, 40 + i)[2] for i in range(4)]
    work = torch.empty((attn.rmsnorm_matmul_ws_bytes(B, H),), dtype=torch.uint8, device=DEV)
    outs, rms = [], []
    cur = x
    for w in ws:
        O, R = attn.rmsnorm_matmul(cur, g, w, with_rms=True, form="two_pass", chained=True,
                                   workspace=work)
        outs.append(O)
        rms.append(R)
        cur = O
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    cur = x
    for w, O, R in zip(ws, outs, rms):
        _check(O, rmsnorm_matmul_ref(cur, g, w))
        O_plain, R_plain = attn.rmsnorm_matmul(cur, g, w, with_rms=True, form="two_pass")
        torch.cuda.synchronize()
        assert torch.equal(O, O_plain) and torch.equal(R, R_plain)
        cur = O
