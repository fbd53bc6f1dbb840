"""Plain, slow CPU fp64 reference for RMSNorm followed by a matrix product,
and for the numerically stable sum of squares with the repair.

TEST INFRASTRUCTURE ONLY: imported by tests, the smoke check and the bench's
CPU-baseline leg; never by the product path.

Definitions (第 11 讲 · 高级 ML 编译：ML 超优化 (CMU 15-779), §3.1):

  RMS(X)_i = sqrt( (1/H) * sum_j X_ij^2 )          X is B x H
  Y_ij     = X_ij * G_j / RMS(X)_i                 G has H entries
  O        = Y W                                   W is H x D, O is B x D

The same page (§3.2) fuses the two reductions by moving the division after
the product, O = ((X ⊙ G) W) / RMS(X). The oracle computes the two-step
definition above (Y materialised, then the product); the fused form is one of
the things its pins check it against.

Stable sum of squares. Neptune论文浅读 (gentlecold.top) §4 lists the
numerically stable L2 norm among the reductions its repair covers, and builds
the repair from the term function: with producer reduction r, term g(r, c)
and g invertible in c, h(t, r, r') = g(r', g^-1(r, t)). For the norm:

  r = max_j |x_j|,  g(r, x) = (x / r)^2,  g^-1(r, t) = r * sqrt(t)
  h(t, r, r') = (r * sqrt(t) / r')^2 = t * (r / r')^2

Rolling form (Neptune §5 pattern): r <- max(r, |x_j|), t <- h(t, r_old, r) +
(x_j / r)^2; then sum_j x_j^2 = r^2 * t and ||x||_2 = r * sqrt(t), and no
x_j^2 is ever formed, so nothing overflows before the final product.
Split form (Neptune §6 pattern): parts (r_s, t_s) over disjoint index sets
merge as r = max_s r_s, t = sum_s h(t_s, r_s, r).

Readings where the page is silent (listed in the design notes too):
  * eps: the page's RMS has none. An optional eps >= 0 goes under the square
    root, RMS = sqrt(mean_j X_ij^2 + eps); the default is 0.
  * a row whose RMS is 0 (all zeros with eps = 0) gives a zero output row.

Parity status: every function here is pinned by
tests/test_oracle_rmsnorm_pins.py.
"""
from __future__ import annotations

import numpy as np

from .attention import _f64


def rms_ref(X, eps: float = 0.0) -> np.ndarray:
    """RMS(X)_i = sqrt(mean_j X_ij^2 + eps) per row (Mirage §3.1)."""
    X = _f64(X)
    H = X.shape[-1]
    return np.sqrt((X * X).sum(axis=-1) / H + eps)


def rmsnorm_ref(X, G, eps: float = 0.0) -> np.ndarray:
    """Y_ij = X_ij G_j / RMS(X)_i; rows with RMS 0 give 0 (Mirage §3.1)."""
    X = _f64(X)
    G = _f64(G)
    r = rms_ref(X, eps)
    safe = np.where(r > 0, r, 1.0)
    Y = X * G[None, :] / safe[:, None]
    Y[r == 0] = 0.0
    return Y


def rmsnorm_matmul_ref(X, G, W, eps: float = 0.0) -> np.ndarray:
    """O = RMSNorm(X; G) W, the two-step (unfused) definition (Mirage §3.1)."""
    Y = rmsnorm_ref(X, G, eps)
    return Y @ _f64(W)


def sumsq_repair(t, r, r_new):
    """h(t, r, r') = t * (r / r')^2: a sum of (x / r)^2 re-expressed against r'
    (Neptune §4's construction applied to g(r, x) = (x / r)^2). An empty part
    (r = 0, t = 0) stays 0."""
    t = np.asarray(t, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    r_new = np.asarray(r_new, dtype=np.float64)
    ratio = np.where(r_new > 0, r / np.where(r_new > 0, r_new, 1.0), 0.0)
    return t * ratio * ratio


def sumsq_rolling(x):
    """Rolling stable sum of squares along the last axis, one element at a
    time: returns (r, t) with sum_j x_j^2 = r^2 t, r = max_j |x_j|."""
    x = _f64(x)
    lead = x.shape[:-1]
    r = np.zeros(lead)
    t = np.zeros(lead)
    for j in range(x.shape[-1]):
        a = np.abs(x[..., j])
        r_new = np.maximum(r, a)
        t = sumsq_repair(t, r, r_new)
        q = np.where(r_new > 0, a / np.where(r_new > 0, r_new, 1.0), 0.0)
        t = t + q * q
        r = r_new
    return r, t


def sumsq_combine(parts):
    """Merge split partials [(r_s, t_s), ...] into one (r, t) (Neptune §6
    pattern with the norm's repair)."""
    r = np.maximum.reduce([np.asarray(p[0], dtype=np.float64) for p in parts])
    t = sum(sumsq_repair(p[1], p[0], r) for p in parts)
    return r, t


def l2norm_stable(x) -> np.ndarray:
    """||x||_2 along the last axis from the rolling (r, t): r * sqrt(t)."""
    r, t = sumsq_rolling(x)
    return r * np.sqrt(t)
