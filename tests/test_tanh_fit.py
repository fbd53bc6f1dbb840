"""The capped prefill's polynomial tanh (unmasked tiles whose |score / cap| is
at most 0.4 evaluate cap * tanh on the FMA pipe).

The kernel's coefficients come from a near-minimax fit of the absolute error
of y (1 + a3 y^2 + a5 y^4) to tanh y on [0, 0.4]: weighted least
squares with Lawson's reweighting (each pass multiplies a node's weight by
its current error), on Chebyshev-distributed nodes. These tests repeat that
fit, check that the constants in the kernel source are its result, and bound
the error of the polynomial as the kernel evaluates it (fp32, Horner in
y^2) against the fp64 tanh, so that cap * error stays far below the bf16
rounding of P.
"""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(__file__), "..", "online_softmax_fusion_gb300", "csrc",
                   "prefill_tc.cuh")
R = 0.4


def kernel_coefficients():
    text = open(SRC).read()
    out = []
    for name in ("kTanhA3", "kTanhA5"):
        m = re.search(r"constexpr float %s = ([-+0-9.e]+)f;" % name, text)
        assert m, name
        out.append(float(m.group(1)))
    return np.array(out)


def lawson_fit(passes=300):
    y = np.cos(np.linspace(0.0, np.pi, 4001)) * R / 2 + R / 2
    y = y[y > 0]
    A = np.stack([y ** 3, y ** 5], axis=1)
    b = np.tanh(y) - y
    w = np.ones_like(y)
    for _ in range(passes):
        sw = np.sqrt(w)
        coef, *_ = np.linalg.lstsq(A * sw[:, None], b * sw, rcond=None)
        e = np.abs(A @ coef - b)
        w = np.maximum(w * e / np.sum(w * e) * len(w), 1e-12)
    return coef


def test_kernel_constants_are_the_fit():
    np.testing.assert_allclose(kernel_coefficients(), lawson_fit(), rtol=1e-8, atol=0)
    m = re.search(r"constexpr float kTanhRange = ([0-9.]+)f;", open(SRC).read())
    assert m and float(m.group(1)) == R


def test_fit_is_near_minimax_and_beats_taylor():
    a3, a5 = kernel_coefficients()
    yy = np.linspace(0.0, R, 200001)
    fit = yy * (1 + yy ** 2 * (a3 + yy ** 2 * a5))
    err = np.abs(fit - np.tanh(yy))
    taylor5 = yy - yy ** 3 / 3 + 2 * yy ** 5 / 15
    assert err.max() < 2.5e-6
    assert err.max() < np.abs(taylor5 - np.tanh(yy)).max() / 10
    # equioscillation: the extreme error is reached, with alternating signs,
    # at several points of the interval (a least-squares fit would not)
    signed = fit - np.tanh(yy)
    big = np.abs(signed) > 0.9 * err.max()
    assert len(set(np.sign(signed[big]))) == 2


def test_fp32_evaluation_as_in_the_kernel():
    """The kernel computes x = s * Q(s^2) with the scalings folded into Q;
    in fp32 the result stays within ~2e-6 (relative to cap) of cap * tanh(s * u) over the
    whole range it is used on, for caps from 1 to 100."""
    a3, a5 = (np.float32(c) for c in kernel_coefficients())
    rng = np.random.default_rng(7)
    log2e = np.float32(1.4426950408889634)
    for cap in (1.0, 5.0, 20.0, 30.0, 100.0):
        scale = np.float32(1 / np.sqrt(128.0))
        u = np.float32(scale / np.float32(cap))            # score -> y
        k1 = np.float32(u * np.float32(cap) * log2e)       # y -> log2-domain x
        u2 = np.float32(u * u)
        k3, k5 = np.float32(k1 * a3 * u2), np.float32(k1 * a5 * u2 * u2)
        s = (rng.uniform(-1, 1, 100000) * (R / float(u))).astype(np.float32)
        w = (s * s).astype(np.float32)
        q = (k5 * w + k3) * w + k1
        x = (s * q).astype(np.float64)
        ref = float(cap) * np.tanh(s.astype(np.float64) * float(u)) * 1.4426950408889634
        assert np.max(np.abs(x - ref)) <= cap * 1.4426950408889634 * 2.5e-6 + 1e-6, cap
