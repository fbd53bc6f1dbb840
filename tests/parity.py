"""Comparison helpers shared by the GPU parity tests.

Tolerances (stated for bf16 outputs from fp32-accumulating kernels against the
fp64 oracle): O max-abs <= 2e-2 and mean-abs <= 2e-3; LSE (fp32) max-abs <=
1e-3; rows that see no key must be exactly O = 0 and LSE = -inf on both sides.
"""
import numpy as np
import torch

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3


def to64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        t = t.detach().to("cpu")
        if t.dtype in (torch.bfloat16, torch.float16):
            t = t.float()
        return t.numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


def assert_o_close(got, ref, what="O", max_abs=O_MAX_ABS, mean_abs=O_MEAN_ABS):
    g = to64(got)
    r = to64(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    err = np.abs(g - r)
    mx, mean = float(err.max(initial=0.0)), float(err.mean()) if err.size else 0.0
    assert mx <= max_abs, f"{what}: max-abs {mx:.3e} > {max_abs}"
    assert mean <= mean_abs, f"{what}: mean-abs {mean:.3e} > {mean_abs}"
    return mx, mean


def assert_lse_close(got, ref, what="LSE", tol=LSE_MAX_ABS):
    g = to64(got)
    r = to64(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    ninf_r = np.isneginf(r)
    assert np.array_equal(np.isneginf(g), ninf_r), f"{what}: -inf pattern differs"
    fin = ~ninf_r
    assert np.all(np.isfinite(g[fin])), f"{what}: non-finite values"
    err = float(np.abs(g[fin] - r[fin]).max(initial=0.0))
    assert err <= tol, f"{what}: max-abs {err:.3e} > {tol}"
    return err
