"""Pins for the RMSNorm + MatMul oracle and the stable sum of squares: each
check ties the oracle to something other than itself.

Sources (page title and section):
  * 第 11 讲 · 高级 ML 编译 (CMU 15-779, Mirage) §3.1: RMS and RMSNorm, then
    O = Y W; §3.2: the fused form O = ((X ⊙ G) W) / RMS(X) equals it (the
    page's own check finds only rounding differences).
  * Neptune论文浅读 (gentlecold.top) §4: the repair h(t, r, r') must repair a
    single term and distribute over the reducer; the stable L2 norm is one of
    the reductions it covers. §6: split partials merged against the global
    producer value equal the unsplit result.
  * Library special cases: torch.nn.functional.rms_norm in float64; the
    Euclidean norm (numpy.linalg.norm, math.fsum of squares).
  * Closed forms derived here: constant rows, identity W, G = 1.
"""
import math

import numpy as np
import pytest
import torch

from oracle import (l2norm_stable, rms_ref, rmsnorm_matmul_ref, rmsnorm_ref,
                    sumsq_combine, sumsq_repair, sumsq_rolling)

RNG = np.random.default_rng(20260611)


def _case(B=5, H=24, D=7):
    X = RNG.standard_normal((B, H))
    G = 1.0 + 0.3 * RNG.standard_normal(H)
    W = RNG.standard_normal((H, D)) / math.sqrt(H)
    return X, G, W


# ------------------------------------------------------------------ RMSNorm
def test_brute_force_tiny():
    """Pure-Python loops over a 2 x 3 input and a 3 x 2 weight."""
    X = [[1.0, -2.0, 0.5], [0.0, 3.0, -1.5]]
    G = [0.5, 2.0, -1.0]
    W = [[1.0, 0.0], [0.5, -1.0], [2.0, 0.25]]
    O = rmsnorm_matmul_ref(np.array(X), np.array(G), np.array(W))
    for i in range(2):
        ms = 0.0
        for j in range(3):
            ms += X[i][j] * X[i][j]
        rms = math.sqrt(ms / 3)
        for n in range(2):
            acc = 0.0
            for j in range(3):
                acc += X[i][j] * G[j] / rms * W[j][n]
            assert O[i, n] == pytest.approx(acc, rel=1e-14, abs=1e-15)


def test_matches_torch_rms_norm():
    """Library special case: torch's rms_norm (float64) followed by @ W."""
    for H, D in ((40, 9), (16, 16)):      # square W too: catches a transposed W
        X, G, W = _case(B=6, H=H, D=D)
        for eps in (0.0, 1e-6, 0.5):
            ref = torch.nn.functional.rms_norm(torch.from_numpy(X), (H,), torch.from_numpy(G),
                                               eps=eps).numpy() @ W
            np.testing.assert_allclose(rmsnorm_matmul_ref(X, G, W, eps), ref, rtol=1e-13,
                                       atol=1e-14)


def test_fused_form_equals_definition():
    """Mirage §3.2: dividing after the product gives the same O."""
    X, G, W = _case(B=4, H=64, D=16)
    fused = ((X * G[None, :]) @ W) / np.sqrt(np.mean(X * X, axis=1))[:, None]
    np.testing.assert_allclose(rmsnorm_matmul_ref(X, G, W), fused, rtol=1e-12, atol=1e-14)


def test_constant_row_closed_form():
    """X_i = c * 1 -> RMS = |c|, Y_i = sign(c) G, O_i = sign(c) (G W)."""
    H, D = 12, 5
    G = RNG.standard_normal(H)
    W = RNG.standard_normal((H, D))
    X = np.array([[3.5] * H, [-0.25] * H])
    np.testing.assert_allclose(rms_ref(X), [3.5, 0.25], rtol=1e-15)
    O = rmsnorm_matmul_ref(X, G, W)
    np.testing.assert_allclose(O[0], G @ W, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(O[1], -(G @ W), rtol=1e-13, atol=1e-14)


def test_unit_weight_rows_have_unit_rms():
    """G = 1 -> every row of Y has RMS exactly 1; identity W -> O = Y."""
    X, _, _ = _case(B=7, H=33, D=1)
    Y = rmsnorm_ref(X, np.ones(33))
    np.testing.assert_allclose(np.sqrt(np.mean(Y * Y, axis=1)), 1.0, rtol=1e-14)
    G = RNG.standard_normal(33)
    np.testing.assert_allclose(rmsnorm_matmul_ref(X, G, np.eye(33)), rmsnorm_ref(X, G),
                               rtol=1e-14, atol=1e-15)


def test_scale_invariance_in_x():
    """With eps = 0, O(alpha X) = O(X) for any alpha > 0; -X flips the sign."""
    X, G, W = _case(B=3, H=20, D=6)
    O = rmsnorm_matmul_ref(X, G, W)
    for alpha in (2.0 ** 100, 3.7, 2.0 ** -60):
        np.testing.assert_allclose(rmsnorm_matmul_ref(alpha * X, G, W), O, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(rmsnorm_matmul_ref(-X, G, W), -O, rtol=1e-13, atol=1e-15)


def test_rms_is_mean_not_sum_and_over_hidden_axis():
    """RMS of a row with one nonzero entry a among H is |a| / sqrt(H)."""
    X = np.zeros((2, 16))
    X[0, 3] = 4.0
    X[1, 15] = -2.0
    np.testing.assert_allclose(rms_ref(X), [1.0, 0.5], rtol=1e-15)


def test_zero_row_gives_zero_output():
    X, G, W = _case(B=3, H=8, D=4)
    X[1] = 0.0
    O = rmsnorm_matmul_ref(X, G, W)
    assert np.all(O[1] == 0.0) and np.all(np.isfinite(O))
    # with eps > 0 the zero row is still zero; the others change
    O2 = rmsnorm_matmul_ref(X, G, W, eps=1e-3)
    assert np.all(O2[1] == 0.0)
    assert not np.allclose(O2[0], O[0], rtol=1e-9, atol=0)


# ------------------------------------------------- stable sum of squares
def test_repair_repairs_a_term_and_distributes():
    """Neptune §4: h(g(r, c), r, r') = g(r', c) and h(a + b) = h(a) + h(b)."""
    c = RNG.standard_normal(10)
    r, rn = 1.7, 4.2
    np.testing.assert_allclose(sumsq_repair((c / r) ** 2, r, rn), (c / rn) ** 2, rtol=1e-15)
    a, b = 0.3, 2.9
    assert sumsq_repair(a + b, r, rn) == pytest.approx(
        sumsq_repair(a, r, rn) + sumsq_repair(b, r, rn), rel=1e-15)


def test_rolling_sum_of_squares_matches_fsum():
    x = RNG.standard_normal((4, 257)) * RNG.uniform(0.01, 100.0, size=(4, 1))
    r, t = sumsq_rolling(x)
    np.testing.assert_allclose(r, np.abs(x).max(axis=1), rtol=0)
    for i in range(4):
        assert r[i] ** 2 * t[i] == pytest.approx(math.fsum(v * v for v in x[i]), rel=1e-13)
    np.testing.assert_allclose(l2norm_stable(x), np.linalg.norm(x, axis=1), rtol=1e-13)


def test_rolling_sum_of_squares_survives_overflow():
    """x * 2^600: every square overflows fp64, the norm itself does not."""
    x = RNG.standard_normal((3, 50))
    big = x * 2.0 ** 600
    with np.errstate(over="ignore"):
        assert np.all(np.isinf((big * big).sum(axis=1)))
    np.testing.assert_allclose(l2norm_stable(big) / 2.0 ** 600, np.linalg.norm(x, axis=1),
                               rtol=1e-14)


def test_split_combine_equals_unsplit():
    x = RNG.standard_normal((3, 100)) * np.array([[1.0], [1e-5], [1e8]])
    x[1, 60:] *= 1e9          # the producer value changes between splits
    r0, t0 = sumsq_rolling(x)
    for cuts in ([50], [1, 99], [10, 20, 70, 99], [33, 66]):
        edges = [0] + cuts + [100]
        parts = [sumsq_rolling(x[:, a:b]) for a, b in zip(edges[:-1], edges[1:])]
        r, t = sumsq_combine(parts)
        np.testing.assert_array_equal(r, r0)
        np.testing.assert_allclose(t, t0, rtol=1e-13)


def test_empty_and_zero_parts():
    r, t = sumsq_rolling(np.zeros((2, 5)))
    assert np.all(r == 0) and np.all(t == 0)
    x = RNG.standard_normal((2, 6))
    r1, t1 = sumsq_combine([sumsq_rolling(np.zeros((2, 3))), sumsq_rolling(x)])
    r2, t2 = sumsq_rolling(x)
    np.testing.assert_array_equal(r1, r2)
    np.testing.assert_allclose(t1, t2, rtol=1e-15)
