"""Comparison helpers shared by the GPU parity tests.

Tolerances (stated for bf16 outputs from fp32-accumulating kernels against the
fp64 oracle): O max-abs <= 2e-2 and mean-abs <= 2e-3; LSE (fp32) max-abs <=
1e-3; rows that see no key must be exactly O = 0 and LSE = -inf on both sides
(checked whenever the oracle's LSE is passed along with O).
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


def o_errors(got, ref):
    """(max-abs, mean-abs) error of got against ref."""
    err = np.abs(to64(got) - to64(ref))
    return float(err.max(initial=0.0)), float(err.mean()) if err.size else 0.0


def assert_o_close(got, ref, what="O", max_abs=O_MAX_ABS, mean_abs=O_MEAN_ABS, lse_ref=None):
    """O within the stated tolerance. With lse_ref (the oracle's LSE, shaped
    like O without its last axis), every row whose reference LSE is -inf (a
    row that sees no key) must be exactly zero in got."""
    g = to64(got)
    r = to64(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    if lse_ref is not None:
        empty = np.isneginf(to64(lse_ref))
        assert empty.shape == g.shape[:-1], (what, empty.shape, g.shape)
        if empty.any():
            bad = int(np.count_nonzero(g[empty]))
            assert bad == 0, f"{what}: {bad} nonzero values in rows that see no key"
            assert np.all(r[empty] == 0.0), f"{what}: oracle rows that see no key are not zero"
    mx, mean = o_errors(g, r)
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


def assert_attention_close(O, L, Or, Lr, what=""):
    """O and LSE against the oracle: the tolerances above, and rows that see
    no key exactly O = 0 with LSE = -inf."""
    o = assert_o_close(O, Or, what=f"O{what}", lse_ref=Lr)
    l = assert_lse_close(L, Lr, what=f"LSE{what}")
    return o, l
