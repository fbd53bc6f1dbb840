"""Pins for the CPU oracle: each check ties it to something other than itself.

Sources of the pins (page title and section):
  * Neptune论文浅读 (gentlecold.top) §2: stable softmax and the attention chain;
    §3: the naive fused loop is wrong, the repaired rolling loop is right;
    §4: the repair term h(t, r, r') = t * exp(r - r') distributes over +;
    §6: split-K local results merged with the global max equal the unsplit one.
  * 第 11 讲 (CMU 15-779, Mirage) §5.5: subtracting any m gives the same softmax;
    q, K scaled x40 overflow without max subtraction; §7.1: stacking a group's
    query heads equals per-head computation.
  * Library special case: torch scaled_dot_product_attention on CPU in float64
    (math path) with an explicit additive mask.
  * Closed forms derived here: uniform attention, geometric ALiBi weights,
    one-hot scores, one and two keys.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import (attend_head, attention_ref, combine_ref, decode_ref,
                    decode_split_partials_ref, naive_fused_exp_sum,
                    online_softmax_rolling, repair)

RNG = np.random.default_rng(20260520)


def _rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


def _sdpa(q, k, v, mask_add, scale):
    """fp64 CPU SDPA with an explicit additive mask (0 / bias / -inf)."""
    tq = torch.from_numpy(q)
    tk = torch.from_numpy(k)
    tv = torch.from_numpy(v)
    tm = torch.from_numpy(mask_add)
    return torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=tm, scale=scale).numpy()


def _lse_torch(q, k, mask_add, scale):
    s = torch.from_numpy(q) @ torch.from_numpy(k).transpose(-1, -2) * scale
    s = s + torch.from_numpy(mask_add)
    return torch.logsumexp(s, dim=-1).numpy()


# ---------------------------------------------------------------- library pin
@pytest.mark.parametrize("Lq,Lk,causal,G,alibi", [
    (16, 16, False, 1, False),
    (33, 33, True, 1, False),
    (7, 29, True, 2, False),      # Lq < Lk: bottom-right aligned causal mask
    (24, 24, True, 4, True),      # GQA + ALiBi + causal
    (19, 40, False, 2, True),     # non-causal ALiBi, |i' - j|
])
def test_matches_torch_sdpa_fp64(Lq, Lk, causal, G, alibi):
    B, Hkv, d = 2, 2, 16
    Hq = Hkv * G
    q = _rand(B, Hq, Lq, d)
    k = _rand(B, Hkv, Lk, d)
    v = _rand(B, Hkv, Lk, d)
    scale = 0.3
    slopes = np.array([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)])
    # Mask built entry by entry with plain loops (no shared vectorised code).
    mask = np.zeros((B, Hq, Lq, Lk))
    for h in range(Hq):
        for i in range(Lq):
            ia = i + Lk - Lq
            for j in range(Lk):
                val = 0.0
                if alibi:
                    val -= slopes[h] * abs(ia - j)
                if causal and j > ia:
                    val = -math.inf
                mask[:, h, i, j] = val
    kr = np.repeat(k, G, axis=1)
    vr = np.repeat(v, G, axis=1)
    ref = _sdpa(q, kr, vr, mask, scale)
    ref_lse = _lse_torch(q, kr, mask, scale)
    O, L = attention_ref(q, k, v, scale=scale, causal=causal,
                         alibi_slopes=slopes if alibi else None)
    assert np.max(np.abs(O - ref)) < 1e-12
    assert np.max(np.abs(L - ref_lse)) < 1e-12


# ---------------------------------------------------------- closed forms
def test_rows_sum_to_one():
    """V = 1 gives O = 1 for every visible row (softmax rows sum to 1)."""
    q = _rand(1, 2, 50, 8)
    k = _rand(1, 2, 50, 8)
    v = np.ones((1, 2, 50, 8))
    O, _ = attention_ref(q, k, v, scale=0.7, causal=True)
    assert np.max(np.abs(O - 1.0)) < 1e-14


def test_zero_query_gives_mean_of_visible_values_causal():
    """Q = 0, no bias: uniform weights over the visible keys. With v_j = j the
    output of aligned row i' is i'/2 and LSE = ln(i' + 1) exactly."""
    Lq, Lk, d = 20, 31, 4
    q = np.zeros((1, 1, Lq, d))
    k = _rand(1, 1, Lk, d)
    v = np.tile(np.arange(Lk, dtype=np.float64)[:, None], (1, d))[None, None]
    O, L = attention_ref(q, k, v, scale=1.0, causal=True)
    for i in range(Lq):
        ia = i + Lk - Lq
        assert abs(O[0, 0, i, 0] - ia / 2.0) < 1e-12
        assert abs(L[0, 0, i] - math.log(ia + 1)) < 1e-12


def test_alibi_geometric_closed_form():
    """Q = 0 with ALiBi slope a, causal: weights proportional to r^t, t = i' - j,
    r = e^{-a}. With v_j = j: O = i' - E[t], E[t] the truncated geometric mean
    r/(1-r) - (n+1) r^{n+1} / (1 - r^{n+1}), n = i'; LSE = ln((1-r^{n+1})/(1-r))."""
    Lq = Lk = 40
    a = 0.3
    q = np.zeros((1, 1, Lq, 2))
    k = _rand(1, 1, Lk, 2)
    v = np.tile(np.arange(Lk, dtype=np.float64)[:, None], (1, 2))[None, None]
    O, L = attention_ref(q, k, v, scale=1.0, causal=True, alibi_slopes=np.array([a]))
    r = math.exp(-a)
    for i in range(Lq):
        n = i
        et = r / (1 - r) - (n + 1) * r ** (n + 1) / (1 - r ** (n + 1))
        assert abs(O[0, 0, i, 0] - (i - et)) < 1e-10
        assert abs(L[0, 0, i] - math.log((1 - r ** (n + 1)) / (1 - r))) < 1e-12


def test_fully_masked_rows_are_zero_and_neg_inf():
    """Lq > Lk with bottom-right alignment: rows with i' < 0 see no key."""
    q = _rand(1, 1, 10, 4)
    k = _rand(1, 1, 6, 4)
    v = _rand(1, 1, 6, 4)
    O, L = attention_ref(q, k, v, scale=1.0, causal=True)
    for i in range(10):
        if i + 6 - 10 < 0:
            assert np.all(O[0, 0, i] == 0.0) and L[0, 0, i] == -np.inf
        else:
            assert np.isfinite(L[0, 0, i])


def test_one_hot_large_score():
    """q = alpha e_1, k_{j*} = e_1, other keys orthogonal to e_1: scores are
    alpha*s for j* and 0 elsewhere, so O = (e^{alpha s} v_{j*} + sum_{j != j*} v_j)
    / (e^{alpha s} + n - 1)."""
    n, d, s = 12, 6, 0.5
    jstar = 5
    k = _rand(n, d)
    k[:, 0] = 0.0
    k[jstar] = 0.0
    k[jstar, 0] = 1.0
    v = _rand(n, d)
    for alpha in (0.0, 3.0, 40.0, 2000.0):
        q = np.zeros((1, d))
        q[0, 0] = alpha
        o, lse = attend_head(q, [0], k, v, scale=s, Lq=1, Lk=n)
        ea = math.exp(min(alpha * s, 700.0))
        if alpha * s < 700:
            expect = (ea * v[jstar] + (v.sum(0) - v[jstar])) / (ea + n - 1)
            assert np.max(np.abs(o[0] - expect)) < 1e-12
            assert abs(lse[0] - math.log(ea + n - 1)) < 1e-12
        else:
            assert np.max(np.abs(o[0] - v[jstar])) < 1e-12
            assert abs(lse[0] - alpha * s) < 1e-12


def test_one_and_two_keys_by_hand():
    v1 = _rand(5)
    v2 = _rand(5)
    k = _rand(2, 3)
    q = _rand(1, 3)
    s = 0.8
    o, lse = attend_head(q, [0], k[:1], v1[None], scale=s)
    assert np.max(np.abs(o[0] - v1)) == 0.0
    assert abs(lse[0] - s * float(q[0] @ k[0])) < 1e-14
    o, lse = attend_head(q, [0], k, np.stack([v1, v2]), scale=s)
    x1, x2 = s * float(q[0] @ k[0]), s * float(q[0] @ k[1])
    sig = lambda z: 1.0 / (1.0 + math.exp(-z))  # noqa: E731
    expect = sig(x1 - x2) * v1 + sig(x2 - x1) * v2
    assert np.max(np.abs(o[0] - expect)) < 1e-14
    assert abs(lse[0] - (max(x1, x2) + math.log1p(math.exp(-abs(x1 - x2))))) < 1e-14


def test_permutation_invariance_and_linearity():
    q = _rand(4, 8)
    k = _rand(30, 8)
    v = _rand(30, 8)
    w = _rand(30, 8)
    o, lse = attend_head(q, np.arange(4), k, v, scale=0.4)
    perm = RNG.permutation(30)
    o2, lse2 = attend_head(q, np.arange(4), k[perm], v[perm], scale=0.4)
    assert np.max(np.abs(o - o2)) < 1e-13 and np.max(np.abs(lse - lse2)) < 1e-13
    a, b = 1.7, -0.3
    o3, _ = attend_head(q, np.arange(4), k, a * v + b * w, scale=0.4)
    ow, _ = attend_head(q, np.arange(4), k, w, scale=0.4)
    assert np.max(np.abs(o3 - (a * o + b * ow))) < 1e-12


# ------------------------------------------------------------ invariants
def test_shift_invariance():
    """Adding a constant c to every score of a row leaves O unchanged and adds
    c to LSE (an extra dimension q_{d+1} = c/s, k_{j,d+1} = 1 adds exactly c)."""
    n, d, s, c = 3, 8, 0.5, 123.25
    q = _rand(n, d)
    k = _rand(20, d)
    v = _rand(20, d)
    o, lse = attend_head(q, np.arange(n), k, v, scale=s)
    q2 = np.concatenate([q, np.full((n, 1), c / s)], axis=1)
    k2 = np.concatenate([k, np.ones((20, 1))], axis=1)
    o2, lse2 = attend_head(q2, np.arange(n), k2, v, scale=s)
    assert np.max(np.abs(o - o2)) < 1e-12
    assert np.max(np.abs(lse2 - (lse + c))) < 1e-9


def test_overflow_scaled_x40_stays_finite():
    """q and K scaled by 40 (logits ~ 2e3): the max-subtracted oracle is
    finite, rows sum to one and it matches fp64 SDPA; exp without max
    subtraction overflows on the same data."""
    q = _rand(1, 1, 32, 8) * 40
    k = _rand(1, 1, 32, 8) * 40
    v = _rand(1, 1, 32, 8)
    s = 1.0 / math.sqrt(8)
    O, L = attention_ref(q, k, v, scale=s)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
    ref = _sdpa(q, k, v, np.zeros((1, 1, 32, 32)), s)
    assert np.max(np.abs(O - ref)) < 1e-10
    logits = s * q[0, 0] @ k[0, 0].T
    assert logits.max() > 700
    with np.errstate(over="ignore", invalid="ignore"):
        e = np.exp(logits)
        naive = (e / e.sum(1, keepdims=True)) @ v[0, 0]
    assert not np.all(np.isfinite(naive))
    Ov, _ = attention_ref(q, k, np.ones_like(v), scale=s)
    assert np.max(np.abs(Ov - 1.0)) < 1e-13


# ------------------------------------------------------ the method's steps
def test_repair_distributes_over_sum():
    """h(t, r, r') = t e^{r - r'} repairs one term and distributes over +."""
    x = _rand(50)
    r, r2 = 0.7, 2.9
    terms = np.exp(x - r)
    assert np.max(np.abs(repair(terms, r, r2) - np.exp(x - r2))) < 1e-14
    assert abs(repair(terms.sum(), r, r2) - repair(terms, r, r2).sum()) < 1e-12


def test_online_rolling_equals_two_pass_naive_does_not():
    x = np.array([0.1, -2.0, 0.5, 7.0, 1.0, -0.3, 6.5])      # max arrives late
    vals = _rand(7, 5)
    m, l, o = online_softmax_rolling(x, vals)
    mt = x.max()
    e = np.exp(x - mt)
    assert m == mt
    assert abs(l - e.sum()) < 1e-14
    assert np.max(np.abs(o - (e / e.sum()) @ vals)) < 1e-14
    # agrees with the oracle's materialised path
    o2, lse2 = attend_head(x[None, :], [0], np.eye(7), vals, scale=1.0, Lq=1, Lk=7)
    assert np.max(np.abs(o - o2[0])) < 1e-14 and abs(m + math.log(l) - lse2[0]) < 1e-14
    nm, ns = naive_fused_exp_sum(x)
    assert nm == mt and abs(ns - e.sum()) > 1e-3            # stale max: wrong
    xs = np.sort(x)[::-1]                                   # max first: naive happens to be right
    assert abs(naive_fused_exp_sum(xs)[1] - np.exp(xs - xs[0]).sum()) < 1e-14


def test_rolling_with_masked_entries():
    x = np.array([-np.inf, 1.0, -np.inf, 3.0])
    m, l, o = online_softmax_rolling(x, np.eye(4))
    assert m == 3.0
    assert abs(l - (math.exp(-2.0) + 1.0)) < 1e-15
    assert o[0] == 0.0 and o[2] == 0.0


@pytest.mark.parametrize("S,split_len", [(1, 64), (2, 32), (3, 25), (64, 1), (80, 1), (5, 100)])
def test_split_then_combine_equals_unsplit(S, split_len):
    """Neptune论文浅读 §6: local (max, sum, output) per split, merged with the
    global max, equals the unsplit reduction (empty splits included)."""
    B, Hkv, G, d, Lmax = 2, 2, 3, 8, 64
    q = _rand(B, Hkv * G, d)
    k = _rand(B, Hkv, Lmax, d) * 2
    v = _rand(B, Hkv, Lmax, d)
    lens = np.array([64, 37])
    Op, Lp = decode_split_partials_ref(q, k, v, lens, scale=0.5, split_len=split_len,
                                       num_splits=S)
    O, L = combine_ref(Op, Lp)
    Ou, Lu = decode_ref(q, k, v, lens, scale=0.5)
    assert np.max(np.abs(O - Ou)) < 1e-12
    assert np.max(np.abs(L - Lu)) < 1e-12


def test_combine_empty_and_single():
    Op = _rand(2, 3, 4, 5)
    Lp = np.full((2, 3, 4), -np.inf)
    O, L = combine_ref(Op, Lp)
    assert np.all(O == 0.0) and np.all(L == -np.inf)
    Lp[:, :, 2] = 1.5
    O, L = combine_ref(Op, Lp)
    assert np.max(np.abs(O - Op[:, :, 2])) < 1e-15 and np.all(L == 1.5)


def test_decode_ignores_keys_beyond_kv_len():
    q = _rand(2, 4, 8)
    k = _rand(2, 2, 40, 8)
    v = _rand(2, 2, 40, 8)
    lens = np.array([17, 40])
    O, L = decode_ref(q, k, v, lens, scale=0.5)
    k2, v2 = k.copy(), v.copy()
    k2[0, :, 17:] = 1e6
    v2[0, :, 17:] = -1e6
    O2, L2 = decode_ref(q, k2, v2, lens, scale=0.5)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)
    # decode equals one-row prefill on the truncated keys
    Op, Lpf = attention_ref(q[:, :, None, :], k[:, :, :17], v[:, :, :17], scale=0.5,
                            batches=[0])
    assert np.max(np.abs(O[0] - Op[0, :, 0])) < 1e-14
    assert np.max(np.abs(L[0] - Lpf[0, :, 0])) < 1e-14


def test_gqa_equals_repeated_heads():
    """Stacking a group's query heads over one K/V head equals per-head
    computation with the K/V head repeated (CMU 15-779 第 11 讲 §7.1)."""
    q = _rand(1, 8, 9, 8)
    k = _rand(1, 2, 9, 8)
    v = _rand(1, 2, 9, 8)
    O, L = attention_ref(q, k, v, scale=0.6, causal=True)
    Or, Lr = attention_ref(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1),
                           scale=0.6, causal=True)
    assert np.array_equal(O, Or) and np.array_equal(L, Lr)


def test_row_subset_is_exact():
    q = _rand(1, 2, 70, 8)
    k = _rand(1, 2, 70, 8)
    v = _rand(1, 2, 70, 8)
    O, L = attention_ref(q, k, v, scale=0.5, causal=True)
    rows = np.array([0, 5, 69])
    Os, Ls = attention_ref(q, k, v, scale=0.5, causal=True, rows=rows, block_rows=2)
    assert np.max(np.abs(O[:, :, rows] - Os)) < 1e-14
    assert np.max(np.abs(L[:, :, rows] - Ls)) < 1e-14


def test_bf16_tensor_inputs_upcast_exactly():
    t = torch.randn(1, 1, 8, 4, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    O, _ = attention_ref(t, t, t, scale=0.5)
    O2, _ = attention_ref(t.float().numpy(), t.float().numpy(), t.float().numpy(), scale=0.5)
    assert np.array_equal(O, O2)


def test_oracle_is_independent_of_product():
    """The oracle imports nothing from the CUDA product package."""
    import inspect
    src = inspect.getsource(oracle.attention)
    assert "online_softmax_fusion_gb300" not in src
    assert "ctypes" not in src


# ------------------------------------------------ SoftCap and Window variants
def test_softcap_matches_sdpa_with_capped_scores():
    """SoftCap: scores become cap * tanh(score / cap). Library check: fp64 SDPA
    fed the capped logits through an additive mask on zero queries."""
    Lq, Lk, d, s, cap = 12, 20, 8, 0.9, 2.5
    q = _rand(Lq, d) * 3
    k = _rand(Lk, d) * 3
    v = _rand(Lk, d)
    o, lse = attend_head(q, np.arange(Lq), k, v, scale=s, softcap=cap, Lq=Lq, Lk=Lk)
    capped = cap * np.tanh(s * (q @ k.T) / cap)
    ref = _sdpa(np.zeros((1, 1, Lq, d)), k[None, None], v[None, None], capped[None, None], 1.0)[0, 0]
    assert np.max(np.abs(o - ref)) < 1e-12
    assert np.max(np.abs(lse - _lse_torch(np.zeros((1, 1, Lq, d)), k[None, None], capped[None, None], 1.0)[0, 0])) < 1e-12
    # bounded logits: |x| < cap, so LSE <= cap + ln(Lk)
    assert np.all(lse < cap + math.log(Lk))
    # a cap far above the logits changes nothing (tanh(z) ~ z)
    o2, l2 = attend_head(q, np.arange(Lq), k, v, scale=s, softcap=1e7, Lq=Lq, Lk=Lk)
    o3, l3 = attend_head(q, np.arange(Lq), k, v, scale=s, Lq=Lq, Lk=Lk)
    assert np.max(np.abs(o2 - o3)) < 1e-9 and np.max(np.abs(l2 - l3)) < 1e-9


def test_softcap_order_against_alibi_and_masks_by_hand():
    """SoftCap caps the scaled score first; the ALiBi bias is added to the
    capped score (unscaled); then the causal and window masks apply. Worked
    by hand on three keys with one-dimensional heads, where capping after the
    bias, scaling the bias, or dropping the cap all give different numbers."""
    s, cap, slope = 0.5, 2.0, 0.5
    q = np.array([[4.0], [3.0], [2.0]])             # rows i = 0, 1, 2 (Lq = Lk = 3)
    k = np.array([[3.0], [-1.0], [3.0]])
    v = np.array([[1.0, -2.0], [4.0, 0.5], [-3.0, 2.0]])

    def by_hand(i, keys):
        xs = []
        for j in keys:
            y = s * float(q[i, 0]) * float(k[j, 0])        # scaled score
            x = cap * math.tanh(y / cap)                     # capped
            x -= slope * abs(i - j)                          # ALiBi, not scaled
            xs.append(x)
        m = max(xs)
        w = [math.exp(x - m) for x in xs]
        tot = sum(w)
        o = sum((wj / tot) * v[j] for wj, j in zip(w, keys))
        return o, m + math.log(tot)

    o, lse = attend_head(q, np.arange(3), k, v, scale=s, causal=True, slope=slope, softcap=cap,
                         Lq=3, Lk=3)
    for i in range(3):
        oh, lh = by_hand(i, list(range(i + 1)))           # causal: keys 0..i
        assert np.max(np.abs(o[i] - oh)) < 1e-14
        assert abs(lse[i] - lh) < 1e-14
    # row 0 sees key 0 only: O = v_0, LSE = cap * tanh(s q k / cap)
    assert np.max(np.abs(o[0] - v[0])) < 1e-15
    assert abs(lse[0] - cap * math.tanh(s * 12.0 / cap)) < 1e-14
    # a left window of one key drops key 0 from row 2
    o, lse = attend_head(q, np.arange(3), k, v, scale=s, causal=True, slope=slope, softcap=cap,
                         window_left=1, Lq=3, Lk=3)
    oh, lh = by_hand(2, [1, 2])
    assert np.max(np.abs(o[2] - oh)) < 1e-14 and abs(lse[2] - lh) < 1e-14
    # the other orders are far from it on this data
    o, lse = attend_head(q, np.arange(3), k, v, scale=s, causal=True, slope=slope, softcap=cap,
                         Lq=3, Lk=3)
    y = s * q[2, 0] * k[:, 0]
    dist = np.array([2.0, 1.0, 0.0])
    for x_alt in (cap * np.tanh((y - slope * dist) / cap),    # cap after the bias
                  cap * np.tanh(y / cap) - s * slope * dist,  # bias scaled
                  y - slope * dist):                          # no cap
        assert abs(lse[2] - (x_alt.max() + math.log(np.exp(x_alt - x_alt.max()).sum()))) > 0.05


def test_window_zero_selects_the_aligned_key():
    """Window 0 on both sides: row i' sees only key i', so O_i = v_{i'} and
    LSE = its scaled score."""
    Lq, Lk, d = 9, 14, 6
    q = _rand(Lq, d)
    k = _rand(Lk, d)
    v = _rand(Lk, d)
    o, lse = attend_head(q, np.arange(Lq), k, v, scale=0.7, window_left=0, window_right=0,
                         Lq=Lq, Lk=Lk)
    for i in range(Lq):
        ia = i + Lk - Lq
        assert np.max(np.abs(o[i] - v[ia])) < 1e-15
        assert abs(lse[i] - 0.7 * float(q[i] @ k[ia])) < 1e-13


def test_window_uniform_closed_form():
    """Q = 0, causal, left window w: row i' averages keys max(0, i'-w)..i'; with
    v_j = j, O = (lo + i') / 2 and LSE = ln(i' - lo + 1)."""
    L, w = 30, 7
    q = np.zeros((L, 3))
    k = _rand(L, 3)
    v = np.tile(np.arange(L, dtype=np.float64)[:, None], (1, 3))
    o, lse = attend_head(q, np.arange(L), k, v, scale=1.0, causal=True, window_left=w)
    for i in range(L):
        lo = max(0, i - w)
        assert abs(o[i, 0] - (lo + i) / 2.0) < 1e-12
        assert abs(lse[i] - math.log(i - lo + 1)) < 1e-12


def test_window_matches_sdpa_with_band_mask():
    Lq = Lk = 25
    q = _rand(1, 2, Lq, 8)
    k = _rand(1, 2, Lk, 8)
    v = _rand(1, 2, Lk, 8)
    wl, wr = 4, 2
    mask = np.full((1, 2, Lq, Lk), -math.inf)
    for i in range(Lq):
        for j in range(Lk):
            if i - wl <= j <= i + wr:
                mask[:, :, i, j] = 0.0
    O, L = attention_ref(q, k, v, scale=0.5, window_left=wl, window_right=wr)
    assert np.max(np.abs(O - _sdpa(q, k, v, mask, 0.5))) < 1e-12
    assert np.max(np.abs(L - _lse_torch(q, k, mask, 0.5))) < 1e-12


# ------------------------------------------------------------- backward pass
@pytest.mark.parametrize("Lq,Lk,causal,G,alibi", [
    (12, 12, False, 1, False),
    (17, 17, True, 2, False),
    (9, 21, True, 1, True),      # Lq < Lk, bottom-right causal, ALiBi
    (20, 20, True, 4, True),     # GQA: dK, dV summed over the group
])
def test_backward_matches_torch_autograd_fp64(Lq, Lk, causal, G, alibi):
    from oracle import attention_backward_ref
    B, Hkv, d, s = 2, 2, 8, 0.6
    Hq = Hkv * G
    q = _rand(B, Hq, Lq, d)
    k = _rand(B, Hkv, Lk, d)
    v = _rand(B, Hkv, Lk, d)
    g = _rand(B, Hq, Lq, d)
    slopes = np.array([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)])
    mask = np.zeros((1, Hq, Lq, Lk))
    for h in range(Hq):
        for i in range(Lq):
            for j in range(Lk):
                ia = i + Lk - Lq
                val = -slopes[h] * abs(ia - j) if alibi else 0.0
                if causal and j > ia:
                    val = -math.inf
                mask[0, h, i, j] = val
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    out = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(G, dim=1), tv.repeat_interleave(G, dim=1),
        attn_mask=torch.tensor(mask), scale=s)
    out.backward(torch.tensor(g))
    dQ, dK, dV = attention_backward_ref(q, k, v, g, scale=s, causal=causal,
                                        alibi_slopes=slopes if alibi else None)
    assert np.max(np.abs(dQ - tq.grad.numpy())) < 1e-11
    assert np.max(np.abs(dK - tk.grad.numpy())) < 1e-11
    assert np.max(np.abs(dV - tv.grad.numpy())) < 1e-11


def test_backward_finite_differences_tiny():
    """Central differences of L = sum(dO * O) with the oracle's own forward
    (brute force on a 2-head, 5-row problem)."""
    from oracle import attention_backward_ref
    q = _rand(1, 2, 5, 3)
    k = _rand(1, 1, 5, 3)
    v = _rand(1, 1, 5, 3)
    g = _rand(1, 2, 5, 3)
    s = 0.8

    def loss(q_, k_, v_):
        O, _ = attention_ref(q_, k_, v_, scale=s, causal=True)
        return float((O * g).sum())

    dQ, dK, dV = attention_backward_ref(q, k, v, g, scale=s, causal=True)
    eps = 1e-6
    for arr, grad in ((q, dQ), (k, dK), (v, dV)):
        for idx in [(0, 0, 0, 0), (0, 0, 3, 2), (0, arr.shape[1] - 1, 4, 1)]:
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += eps
            minus[idx] -= eps
            args_p = [plus if a is arr else a for a in (q, k, v)]
            args_m = [minus if a is arr else a for a in (q, k, v)]
            num = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(num - grad[idx]) < 1e-7, (idx, num, grad[idx])


def test_backward_value_gradient_is_probability_weighted():
    """dV_j = sum_i P_ij dO_i: with dO = 1 every dV row is the column sum of
    P, and those sums add up to the number of rows that see a key."""
    from oracle import attention_backward_ref
    q = _rand(1, 1, 11, 4)
    k = _rand(1, 1, 11, 4)
    v = _rand(1, 1, 11, 4)
    g = np.ones((1, 1, 11, 4))
    _, _, dV = attention_backward_ref(q, k, v, g, scale=0.5, causal=True)
    assert abs(dV[0, 0, :, 0].sum() - 11.0) < 1e-12
    # the last key is seen only by the last row, with its probability
    O, L = attention_ref(q, k, v, scale=0.5, causal=True)
    p_last = math.exp(0.5 * float(q[0, 0, 10] @ k[0, 0, 10]) - L[0, 0, 10])
    assert abs(dV[0, 0, 10, 0] - p_last) < 1e-12
