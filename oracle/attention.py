"""Plain, slow CPU fp64 reference for single-head and batched attention.

TEST INFRASTRUCTURE ONLY: imported by tests, the smoke check and the bench's
CPU-baseline leg; never by the product path.

What it computes is the plain definition, materialised and two-pass (the
result the fused online method reaches up to rounding order):

  x_ij = s * (q_i . k_j) + bias_h(i, j)            scores, scale s
  x_ij = -inf  where key j is not visible to query i
  m_i  = max_j x_ij                                 pass 1
  l_i  = sum_j exp(x_ij - m_i)                      pass 2
  O_i  = sum_j exp(x_ij - m_i) / l_i * v_j
  LSE_i = m_i + ln l_i

Sources: the stable softmax softmax(x_j) = exp(x_j - m) / sum_k exp(x_k - m)
with m = max_k x_k and the attention chain QK^T -> score/mask/bias -> softmax
-> .V are Neptune论文浅读 (gentlecold.top) §2. The mask/bias variants (Causal,
ALiBi, GQA) are the ones named in its §9.

Readings where the pages are silent (each one is listed in the design notes):
  * causal alignment when Lq != Lk is bottom-right: query row i sees keys
    j <= i + (Lk - Lq);
  * ALiBi adds -slope_h * |i' - j| (i' the aligned row) after scaling; it is
    not multiplied by s;
  * GQA maps query head h to KV head floor(h / G), G = Hq / Hkv;
  * SoftCap (named in §9, not defined there) replaces the scaled score x by
    cap * tanh(x / cap) before the bias, the mask and the softmax;
  * Window (named in §9, not defined there) is local attention: aligned row
    i' sees keys j with i' - window_left <= j <= i' + window_right (a
    negative bound means unlimited on that side); with causal, keys after i'
    stay masked;
  * a row that sees no key has O = 0 and LSE = -inf;
  * a split of the Split-K form stores its normalised output O_s = O/l and
    its LSE_s = m + ln l; the merge recovers the raw sums from them.

Parity status: every function here is pinned by tests/test_oracle_pins.py.
"""
from __future__ import annotations

import math

import numpy as np

NEG_INF = -np.inf


def _f64(x) -> np.ndarray:
    """Exact upcast (bf16/fp16/fp32 values are all representable in fp64)."""
    if hasattr(x, "detach"):  # a torch tensor: go through fp32, which is exact for bf16
        import torch
        t = x.detach().to("cpu")
        if t.dtype in (torch.bfloat16, torch.float16):
            t = t.to(torch.float32)
        return t.numpy().astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def attend_head(q_rows, row_pos, k, v, *, scale, causal=False, slope=None,
                Lq=None, Lk=None, kv_len=None, softcap=0.0, window_left=-1,
                window_right=-1):
    """Attention of some query rows of one head against one K/V head.

    q_rows  [n, d]   query rows (any float dtype; upcast exactly to fp64)
    row_pos [n]      each row's index i in [0, Lq)
    k, v    [Lk_buf, d]
    Lq, Lk  nominal lengths used for causal alignment (default: n rows / len(k))
    kv_len  keys [0, kv_len) are visible (default Lk)
    softcap > 0: scores become softcap * tanh(score / softcap)
    window_left / window_right >= 0: keys outside
            [i' - window_left, i' + window_right] are not visible

    Returns (O [n, d] fp64, LSE [n] fp64).
    Follows Neptune论文浅读 §2: materialise the scores, take the row max, then
    exp and sum, then divide and multiply by V.
    """
    q = _f64(q_rows)
    kk = _f64(k)
    vv = _f64(v)
    pos = np.asarray(row_pos, dtype=np.int64)
    if Lk is None:
        Lk = kk.shape[0]
    if Lq is None:
        Lq = q.shape[0]
    if kv_len is None:
        kv_len = Lk
    n, d = q.shape
    out = np.zeros((n, vv.shape[1]), dtype=np.float64)
    lse = np.full((n,), NEG_INF, dtype=np.float64)
    if kv_len <= 0 or n == 0:
        return out, lse
    kk = kk[:kv_len]
    vv = vv[:kv_len]
    x = scale * (q @ kk.T)                                  # [n, kv_len]
    if softcap and softcap > 0.0:
        x = float(softcap) * np.tanh(x / float(softcap))
    j = np.arange(kv_len, dtype=np.int64)[None, :]
    i_al = (pos + (Lk - Lq))[:, None]                       # bottom-right aligned row
    if slope is not None:
        x = x - float(slope) * np.abs(i_al - j).astype(np.float64)
    if causal:
        x = np.where(j > i_al, NEG_INF, x)
    if window_left is not None and window_left >= 0:
        x = np.where(j < i_al - int(window_left), NEG_INF, x)
    if window_right is not None and window_right >= 0:
        x = np.where(j > i_al + int(window_right), NEG_INF, x)
    m = x.max(axis=1)                                       # pass 1: row max
    live = np.isfinite(m)
    if not live.any():
        return out, lse
    xl = x[live]
    ml = m[live]
    e = np.exp(xl - ml[:, None])                            # pass 2: exp and sum
    l = e.sum(axis=1)
    p = e / l[:, None]
    out[live] = p @ vv
    lse[live] = ml + np.log(l)
    return out, lse


def attention_ref(q, k, v, *, scale, causal=False, alibi_slopes=None,
                  rows=None, heads=None, batches=None, block_rows=512,
                  softcap=0.0, window_left=-1, window_right=-1):
    """Batched attention with GQA, causal mask and ALiBi.

    q [B, Hq, Lq, d], k/v [B, Hkv, Lk, d] (numpy arrays or torch tensors).
    rows: optional 1-D array of query-row indices evaluated for every head
    (rows are independent, so a subset is an exact check of those rows).
    heads / batches: optional subsets of query heads / batch entries.
    Returns (O [nb, nh, nr, d], LSE [nb, nh, nr]) in fp64.
    """
    B, Hq, Lq, d = tuple(q.shape)
    Hkv, Lk = int(k.shape[1]), int(k.shape[2])
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    rows = np.arange(Lq) if rows is None else np.asarray(rows, dtype=np.int64)
    heads = list(range(Hq)) if heads is None else list(heads)
    batches = list(range(B)) if batches is None else list(batches)
    slopes = None if alibi_slopes is None else _f64(alibi_slopes).reshape(-1)
    O = np.zeros((len(batches), len(heads), len(rows), d), dtype=np.float64)
    L = np.zeros((len(batches), len(heads), len(rows)), dtype=np.float64)
    for bi, b in enumerate(batches):
        for hi, h in enumerate(heads):
            kv = h // G
            kh = _f64(k[b, kv])
            vh = _f64(v[b, kv])
            for r0 in range(0, len(rows), block_rows):
                rr = rows[r0:r0 + block_rows]
                qr = _f64(q[b, h][rr])
                o, lse = attend_head(qr, rr, kh, vh, scale=scale, causal=causal,
                                     slope=None if slopes is None else slopes[h],
                                     Lq=Lq, Lk=Lk, softcap=softcap,
                                     window_left=window_left, window_right=window_right)
                O[bi, hi, r0:r0 + len(rr)] = o
                L[bi, hi, r0:r0 + len(rr)] = lse
    return O, L


def decode_ref(q, k, v, kv_lens, *, scale, batches=None, kv_heads=None):
    """Single-token decode: q [B, Hq, d] against the first kv_lens[b] keys of
    K/V [B, Hkv, Lk_max, d]. No mask beyond the sequence length.
    Returns (O [nb, nkv*G, d], LSE [nb, nkv*G]) for the chosen batch entries and
    KV heads (all query heads of each chosen KV head, in order)."""
    B, Hq, d = tuple(q.shape)
    Hkv = int(k.shape[1])
    G = Hq // Hkv
    lens = [int(x) for x in np.asarray(_f64(kv_lens)).reshape(-1)]
    batches = list(range(B)) if batches is None else list(batches)
    kv_heads = list(range(Hkv)) if kv_heads is None else list(kv_heads)
    O = np.zeros((len(batches), len(kv_heads) * G, d), dtype=np.float64)
    L = np.zeros((len(batches), len(kv_heads) * G), dtype=np.float64)
    for bi, b in enumerate(batches):
        for ki, kv in enumerate(kv_heads):
            n = lens[b]
            kh = _f64(k[b, kv, :n])
            vh = _f64(v[b, kv, :n])
            qr = _f64(q[b, kv * G:(kv + 1) * G])
            o, lse = attend_head(qr, np.zeros(G, dtype=np.int64), kh, vh,
                                 scale=scale, Lq=1, Lk=n, kv_len=n)
            O[bi, ki * G:(ki + 1) * G] = o
            L[bi, ki * G:(ki + 1) * G] = lse
    return O, L


def decode_split_partials_ref(q, k, v, kv_lens, *, scale, split_len, num_splits):
    """Local reductions of the Split-K form (Neptune论文浅读 §6): the key axis
    is cut into splits of split_len keys; split s covers keys
    [s*split_len, (s+1)*split_len) clipped to [0, kv_len_b). Each split is the
    full two-pass computation over its own keys.

    Returns (O_part [B, Hq, S, d], LSE_part [B, Hq, S]); an empty split has
    O_part = 0 and LSE_part = -inf.
    """
    B, Hq, d = tuple(q.shape)
    Hkv = int(k.shape[1])
    G = Hq // Hkv
    lens = [int(x) for x in np.asarray(_f64(kv_lens)).reshape(-1)]
    O = np.zeros((B, Hq, num_splits, d), dtype=np.float64)
    L = np.full((B, Hq, num_splits), NEG_INF, dtype=np.float64)
    for b in range(B):
        for kv in range(Hkv):
            kh = _f64(k[b, kv, :lens[b]])
            vh = _f64(v[b, kv, :lens[b]])
            qr = _f64(q[b, kv * G:(kv + 1) * G])
            for s in range(num_splits):
                lo = s * split_len
                hi = min((s + 1) * split_len, lens[b])
                if hi <= lo:
                    continue
                o, lse = attend_head(qr, np.zeros(G, dtype=np.int64), kh[lo:hi],
                                     vh[lo:hi], scale=scale, Lq=1, Lk=hi - lo)
                O[b, kv * G:(kv + 1) * G, s] = o
                L[b, kv * G:(kv + 1) * G, s] = lse
    return O, L


def combine_ref(O_part, LSE_part):
    """Global reduction of the Split-K form (Neptune论文浅读 §6): take the
    global max over the splits and repair every split's sum and output with it.

    With O_s = o_s / l_s and LSE_s = m_s + ln l_s, split s contributes raw sums
    l_s e^{m_s} = e^{LSE_s} and o_s e^{m_s} = O_s e^{LSE_s}. Relative to the
    global max M = max_s LSE_s the weights are w_s = exp(LSE_s - M), so
    O = sum_s w_s O_s / sum_s w_s and LSE = M + ln sum_s w_s.
    Splits with LSE_s = -inf get weight 0; if all are -inf, O = 0, LSE = -inf.
    """
    Op = _f64(O_part)
    Lp = _f64(LSE_part)
    M = Lp.max(axis=-1)                                     # [..]
    finite = np.isfinite(M)
    Msafe = np.where(finite, M, 0.0)
    w = np.where(np.isfinite(Lp), np.exp(Lp - Msafe[..., None]), 0.0)
    wsum = w.sum(axis=-1)
    num = (w[..., None] * Op).sum(axis=-2)
    O = np.where(finite[..., None], num / np.where(finite, wsum, 1.0)[..., None], 0.0)
    LSE = np.where(finite, Msafe + np.log(np.where(finite, wsum, 1.0)), NEG_INF)
    return O, LSE


def repair(t, r, r_new):
    """The repair term of Neptune论文浅读 §4 for the softmax sum: with
    g(r, x) = exp(x - r), h(t, r, r') = g(r', g^{-1}(r, t)) = t * exp(r - r')."""
    return np.asarray(t, dtype=np.float64) * np.exp(np.float64(r) - np.float64(r_new))


def online_softmax_rolling(x, vals=None):
    """One-pass rolling update of Neptune论文浅读 §3 (the repaired loop), with
    the output accumulator o carried the same way (the CANN FlashAttention
    blog's online-softmax section, read with its output update as
    o <- o * exp(m - m_new) + exp(x - m_new) * v and the result divided by l).

    x [n] scores, vals [n, dv] (optional). Returns (m, l, o / l) in fp64;
    o / l is None when vals is None.
    """
    xs = np.asarray(x, dtype=np.float64).reshape(-1)
    vv = None if vals is None else np.asarray(vals, dtype=np.float64).reshape(len(xs), -1)
    m_old = NEG_INF
    l = 0.0
    o = None if vv is None else np.zeros(vv.shape[1], dtype=np.float64)
    for j, xj in enumerate(xs):
        m_new = max(m_old, xj)
        if m_new == NEG_INF:          # nothing visible yet
            continue
        corr = math.exp(m_old - m_new) if m_old != NEG_INF else 0.0
        pj = math.exp(xj - m_new)
        l = corr * l + pj
        if o is not None:
            o = corr * o + pj * vv[j]
        m_old = m_new
    if o is None:
        return m_old, l, None
    return m_old, l, (o / l if l > 0 else o)


def naive_fused_exp_sum(x):
    """The naive fusion of Neptune论文浅读 §3 (the wrong one): the running max
    and the running exp-sum in one loop with no repair, so early terms keep a
    stale max. Returns (max, sum)."""
    xs = np.asarray(x, dtype=np.float64).reshape(-1)
    xmax = NEG_INF
    s = 0.0
    for xj in xs:
        xmax = max(xmax, xj)
        s += math.exp(xj - xmax)
    return xmax, s


def attention_backward_ref(q, k, v, dO, *, scale, causal=False, alibi_slopes=None):
    """Gradients of attention (the backward pass; its single-pass structure on
    tensor cores is described in the Twill review (xllm-io) §七 7.2).

    Plain definition per (b, h), kv = h // G, with P the forward probabilities
    (materialised, two-pass) and O = P V:
      dV_j  = sum_i P_ij dO_i                  (summed over the group's heads)
      dP_ij = dO_i . v_j
      D_i   = sum_j P_ij dP_ij  (= dO_i . O_i)
      dS_ij = P_ij (dP_ij - D_i)
      dQ_i  = s sum_j dS_ij k_j
      dK_j  = s sum_i dS_ij q_i                (summed over the group's heads)
    Masked pairs have P = 0; the ALiBi bias does not depend on Q or K.
    Returns (dQ [B,Hq,Lq,d], dK [B,Hkv,Lk,d], dV [B,Hkv,Lk,d]) in fp64.
    """
    qq, kk, vv, gg = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, Hq, Lq, d = qq.shape
    Hkv, Lk = kk.shape[1], kk.shape[2]
    G = Hq // Hkv
    slopes = None if alibi_slopes is None else _f64(alibi_slopes).reshape(-1)
    dQ = np.zeros_like(qq)
    dK = np.zeros_like(kk)
    dV = np.zeros_like(vv)
    i_al = (np.arange(Lq) + (Lk - Lq))[:, None]
    j = np.arange(Lk)[None, :]
    for b in range(B):
        for h in range(Hq):
            kv = h // G
            x = scale * (qq[b, h] @ kk[b, kv].T)
            if slopes is not None:
                x = x - slopes[h] * np.abs(i_al - j).astype(np.float64)
            if causal:
                x = np.where(j > i_al, NEG_INF, x)
            m = x.max(axis=1, keepdims=True)
            live = np.isfinite(m[:, 0])
            P = np.zeros_like(x)
            e = np.exp(x[live] - m[live])
            P[live] = e / e.sum(axis=1, keepdims=True)
            dV[b, kv] += P.T @ gg[b, h]
            dP = gg[b, h] @ vv[b, kv].T
            D = (P * dP).sum(axis=1, keepdims=True)
            dS = P * (dP - D)
            dQ[b, h] = scale * (dS @ kk[b, kv])
            dK[b, kv] += scale * (dS.T @ qq[b, h])
    return dQ, dK, dV
