"""Oracle: exact attention by forming the full score matrix in fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring). Plain NumPy, float64.

Definitions followed
--------------------
* Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k)) V -- "Module 09: Efficient
  Attention", section "The Math: Sharing Keys and Values".
* Query head h reads key/value head floor(h / n_rep), n_rep = Hq / Hkv -- same
  section; the grouping order is the one of ``repeat_interleave`` (section
  "Common Pitfalls", items 2 and 3: Hkv must divide Hq).
* Standard attention materialises S = Q K^T, P = softmax(S), O = P V --
  "Cache KV, atención flash y optimización de la inferencia", section
  "La atención de flash el truco de la balsa" (the three-pass listing).
* Max-subtracted ("stable") softmax -- "Генерация и KV-кэш", section
  "KV-кэш для одной головы на NumPy" (``decode_step`` and ``full_causal``).
* Causal mask aligned to the bottom-right corner when there are fewer queries
  than keys: the newest query sits at the last key position -- "Генерация и
  KV-кэш", section "Три ловушки, на которых спотыкаются все", trap 2 (the
  top-left ``is_causal`` of SDPA lets one query see only key 0; the mask must
  be built from the bottom-right corner).
* Sliding window: key j is visible from the query at position p iff
  p - W < j <= p (the diagonal counts toward W) -- "Module 09: Efficient
  Attention", section "Attention Mask Gallery", the printed
  ``sliding_window_mask(6, window=3)`` matrix.
* The online recurrence s_k = s_{k-1} e^{d_{k-1}-d_k} + sum e^{a_i-d_k} and the
  matching update of O -- "Ли Хунъи ... 2026", lecture "Ускоряем генерацию,
  часть 1: FlashAttention", the two displayed formulas.

Readings where the pages are silent:
* LSE is the natural log of the sum of exp(scaled score) over visible keys:
  lse = m + ln(l), one value per (query row, query head).
* A query with no visible key (only possible when a sequence has no keys) gets
  O = 0 and lse = -inf.
* A window with causal=False is not defined by the pages and is rejected.
"""

import numpy as np

__all__ = [
    "attention_mask",
    "sdpa",
    "sdpa_rows",
    "sdpa_varlen",
    "sdpa_backward",
    "sdpa_backward_varlen",
    "sdpa_backward_sampled",
    "online_softmax_attention",
    "merge_splits",
]


def _as_f64(x):
    """Promote to float64 (bf16/fp32 inputs are represented exactly)."""
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu")
        import torch

        x = x.to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _check_heads(hq, hkv):
    if hkv <= 0 or hq % hkv != 0:
        raise ValueError(f"num_kv_heads={hkv} must divide num_heads={hq}")
    return hq // hkv


def kv_head_of(h, num_heads, num_kv_heads):
    """Key/value head read by query head h: floor(h / n_rep), n_rep = Hq / Hkv."""
    return h // (num_heads // num_kv_heads)


def default_scale(d):
    """1 / sqrt(d_k)."""
    return 1.0 / np.sqrt(d)


def attention_mask(len_q, len_k, causal, window=0):
    """Boolean visibility matrix [len_q, len_k]; True = the query may attend.

    Query row i sits at absolute position p_i = len_k - len_q + i (bottom-right
    alignment). Causal: j <= p_i. Window W > 0: additionally j > p_i - W.
    """
    i = np.arange(len_q)[:, None]
    j = np.arange(len_k)[None, :]
    return visible(query_position(i, len_q, len_k), j, causal, window)


def query_position(i, len_q, len_k):
    """Absolute position of query row i: the last query sits at the last key
    (bottom-right alignment)."""
    return len_k - len_q + i


def visible(pos, j, causal, window):
    """May the query at absolute position ``pos`` see key ``j``? (broadcasts)"""
    if window > 0 and not causal:
        raise ValueError("a sliding window is only defined together with causal masking")
    allowed = np.ones(np.broadcast(pos, j).shape, dtype=bool)
    if causal:
        allowed &= j <= pos
    if window > 0:
        allowed &= j > pos - window
    return allowed


def _softmax_rows(scores, allowed, v):
    """Max-subtracted softmax of each row of ``scores`` over ``allowed`` keys,
    times V. Returns (o [rows, d], lse [rows])."""
    s = np.where(allowed, scores, -np.inf)
    rows = s.shape[0]
    d = v.shape[1]
    o = np.zeros((rows, d), dtype=np.float64)
    lse = np.full(rows, -np.inf, dtype=np.float64)
    has_key = allowed.any(axis=1)
    if has_key.any():
        sv = s[has_key]
        m = sv.max(axis=1, keepdims=True)
        p = np.exp(sv - m)
        l = p.sum(axis=1, keepdims=True)
        o[has_key] = (p @ v) / l
        lse[has_key] = m[:, 0] + np.log(l[:, 0])
    return o, lse


def sdpa(q, k, v, *, causal, window=0, scale=None):
    """Exact attention for ONE sequence, full score matrix in fp64.

    q: [len_q, Hq, d]; k, v: [len_k, Hkv, d] (token-major).
    Returns o [len_q, Hq, d] float64 and lse [Hq, len_q] float64.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    len_q, hq, d = q.shape
    len_k, hkv, _ = k.shape
    _check_heads(hq, hkv)
    if scale is None:
        scale = default_scale(d)
    allowed = attention_mask(len_q, len_k, causal, window)
    o = np.zeros((len_q, hq, d), dtype=np.float64)
    lse = np.full((hq, len_q), -np.inf, dtype=np.float64)
    for h in range(hq):
        kv_head = kv_head_of(h, hq, hkv)
        scores = scale * (q[:, h, :] @ k[:, kv_head, :].T)  # [len_q, len_k]
        o[:, h, :], lse[h] = _softmax_rows(scores, allowed, v[:, kv_head, :])
    return o, lse


def sdpa_rows(q, k, v, rows, *, causal, window=0, scale=None):
    """The same definition as :func:`sdpa`, evaluated only for chosen query rows.

    ``rows`` is a list of (query_row, query_head). ``q`` holds the whole
    sequence's queries (its length fixes the bottom-right alignment).
    Returns o [len(rows), d] and lse [len(rows)].
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    len_q, hq, d = q.shape
    len_k, hkv, _ = k.shape
    _check_heads(hq, hkv)
    if scale is None:
        scale = default_scale(d)
    o = np.zeros((len(rows), d), dtype=np.float64)
    lse = np.full(len(rows), -np.inf, dtype=np.float64)
    for n, (i, h) in enumerate(rows):
        kv_head = kv_head_of(h, hq, hkv)
        allowed = visible(query_position(i, len_q, len_k), np.arange(len_k), causal, window)
        scores = scale * (k[:, kv_head, :] @ q[i, h, :])  # [len_k]
        oo, ll = _softmax_rows(scores[None, :], allowed[None, :], v[:, kv_head, :])
        o[n], lse[n] = oo[0], ll[0]
    return o, lse


def sdpa_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, *, causal, window=0, scale=None):
    """Packed variable-length batch: sequence b owns rows
    [cu_q[b], cu_q[b+1]) of q and [cu_k[b], cu_k[b+1]) of k and v.

    Returns o [T_q, Hq, d] and lse [Hq, T_q] (float64).
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    cu_q = [int(x) for x in cu_seqlens_q]
    cu_k = [int(x) for x in cu_seqlens_k]
    t_q, hq, d = q.shape
    o = np.zeros((t_q, hq, d), dtype=np.float64)
    lse = np.full((hq, t_q), -np.inf, dtype=np.float64)
    for b in range(len(cu_q) - 1):
        q0, q1 = cu_q[b], cu_q[b + 1]
        k0, k1 = cu_k[b], cu_k[b + 1]
        if q1 == q0:
            continue
        ob, lb = sdpa(q[q0:q1], k[k0:k1], v[k0:k1], causal=causal, window=window, scale=scale)
        o[q0:q1] = ob
        lse[:, q0:q1] = lb
    return o, lse


def sdpa_backward(q, k, v, dout, *, causal, window=0, scale=None):
    """Gradients of :func:`sdpa`'s output for ONE sequence, in fp64.

    Given dL/dO = dout [len_q, Hq, d], returns (dq [len_q, Hq, d],
    dk [len_k, Hkv, d], dv [len_k, Hkv, d]) of L through O = softmax(S) V with
    S = scale * Q K^T (masked keys excluded). Written from the chain rule of
    those two steps ("Cache KV, atención flash ...", section "La atención de
    flash el truco de la balsa": the backward pass recomputes S and P from Q,
    K and the saved row statistics instead of storing P):
        dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij = sum_c dO_ic O_ic,
        dS = P * (dP - D),  dQ = scale * dS K,  dK = scale * dS^T Q.
    Query heads of one KV group add their dK, dV into that group's KV head.
    """
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    len_q, hq, d = q.shape
    len_k, hkv, _ = k.shape
    _check_heads(hq, hkv)
    if scale is None:
        scale = default_scale(d)
    allowed = attention_mask(len_q, len_k, causal, window)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for h in range(hq):
        g = kv_head_of(h, hq, hkv)
        dq_h, dk_h, dv_h = _head_backward(q[:, h, :], k[:, g, :], v[:, g, :], dout[:, h, :],
                                          allowed, scale)
        dq[:, h, :] = dq_h
        dk[:, g, :] += dk_h
        dv[:, g, :] += dv_h
    return dq, dk, dv


def _softmax_backward(p, dp, drow):
    """dS = P * (dP - D): the softmax's Jacobian applied row by row."""
    return p * (dp - drow)


def _head_backward(qh, kg, vg, doh, allowed, scale):
    """One query head's (dq, dk, dv) contributions; the forward recomputed."""
    s = np.where(allowed, scale * (qh @ kg.T), -np.inf)
    p = np.zeros_like(s)
    has_key = allowed.any(axis=1)
    if has_key.any():
        sv = s[has_key]
        e = np.exp(sv - sv.max(axis=1, keepdims=True))
        p[has_key] = e / e.sum(axis=1, keepdims=True)
    o = p @ vg
    dv = p.T @ doh
    dp = doh @ vg.T
    drow = (doh * o).sum(axis=1, keepdims=True)
    ds = _softmax_backward(p, dp, drow)
    return scale * (ds @ kg), scale * (ds.T @ qh), dv


def sdpa_backward_varlen(q, k, v, dout, cu_seqlens, *, causal, window=0, scale=None):
    """:func:`sdpa_backward` of packed sequences (Lq = Lk per sequence)."""
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(len(cu_seqlens) - 1):
        a, e = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        if e == a:
            continue
        dq[a:e], dk[a:e], dv[a:e] = sdpa_backward(q[a:e], k[a:e], v[a:e], dout[a:e],
                                                  causal=causal, window=window, scale=scale)
    return dq, dk, dv


def sdpa_backward_sampled(q, k, v, dout, kv_head, q_rows, k_rows, *, causal, window=0,
                          scale=None, chunk=1024):
    """Selected entries of :func:`sdpa_backward` for ONE (long) sequence.

    Returns (dq [len(q_rows), G, d] for the G query heads of ``kv_head``,
    dk [len(k_rows), d], dv [len(k_rows), d] of ``kv_head``), the same
    formulas evaluated only where asked. The score matrix is formed ``chunk``
    query rows at a time to get every row's LSE and D (dK and dV of one key
    need P and D of every query that sees it); then
        dq_i = scale * sum_j P_ij (dP_ij - D_i) k_j,
        dv_j = sum_i P_ij dO_i,  dk_j = scale * sum_i P_ij (dP_ij - D_i) q_i.
    """
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    len_q, hq, d = q.shape
    len_k, hkv, _ = k.shape
    _check_heads(hq, hkv)
    if scale is None:
        scale = default_scale(d)
    heads = [h for h in range(hq) if kv_head_of(h, hq, hkv) == kv_head]
    kg, vg = k[:, kv_head, :], v[:, kv_head, :]
    pos = query_position(np.arange(len_q), len_q, len_k)
    keys = np.arange(len_k)
    dq = np.zeros((len(q_rows), len(heads), d))
    dk = np.zeros((len(k_rows), d))
    dv = np.zeros((len(k_rows), d))
    for hi, h in enumerate(heads):
        qh, doh = q[:, h, :], dout[:, h, :]
        lse = np.full(len_q, -np.inf)
        drow = np.zeros(len_q)
        for r0 in range(0, len_q, chunk):
            r1 = min(len_q, r0 + chunk)
            allowed = visible(pos[r0:r1, None], keys[None, :], causal, window)
            s = np.where(allowed, scale * (qh[r0:r1] @ kg.T), -np.inf)
            m = s.max(axis=1, keepdims=True)
            ok = np.isfinite(m[:, 0])
            e = np.where(allowed, np.exp(s - np.where(np.isfinite(m), m, 0.0)), 0.0)
            l = e.sum(axis=1)
            lse[r0:r1] = np.where(ok, m[:, 0] + np.log(np.where(ok, l, 1.0)), -np.inf)
            o = (e / np.where(ok, l, 1.0)[:, None]) @ vg
            drow[r0:r1] = (doh[r0:r1] * o).sum(axis=1)
        for n, i in enumerate(q_rows):
            allowed = visible(pos[i], keys, causal, window)
            p = np.where(allowed, np.exp(np.where(allowed, scale * (kg @ qh[i]), 0.0) - lse[i]), 0.0)
            ds = p * (vg @ doh[i] - drow[i])
            dq[n, hi] = scale * (ds @ kg)
        for n, j in enumerate(k_rows):
            allowed = visible(pos, j, causal, window)
            p = np.where(allowed, np.exp(np.where(allowed, scale * (qh @ kg[j]), 0.0) - lse), 0.0)
            dv[n] += p @ doh
            ds = p * (doh @ vg[j] - drow)
            dk[n] += scale * (ds @ qh)
    return dq, dk, dv


def online_softmax_attention(q, k, v, block, *, scale=None):
    """FlashAttention's streaming recurrence for one head, in fp64.

    q: [len_q, d]; k, v: [len_k, d]; no mask. Keys are consumed in blocks of
    ``block``; per query row a running maximum d, running denominator s and
    running (unnormalised) output are carried, and the old totals are rescaled
    by e^{d_old - d_new} when a block raises the maximum. Returns
    (o [len_q, d], s_history) where s_history[k] holds the running denominator
    after block k (relative to the running maximum), for checking the
    lecture's worked example.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    len_q, d = q.shape
    len_k = k.shape[0]
    if scale is None:
        scale = default_scale(d)
    m = np.full(len_q, -np.inf)
    s = np.zeros(len_q)
    acc = np.zeros((len_q, d))
    history = []
    for start in range(0, len_k, block):
        a = scale * (q @ k[start:start + block].T)  # scores of this block
        m_new = np.maximum(m, a.max(axis=1))
        # e^{m_old - m_new}; the first block has nothing to rescale
        corr = np.where(np.isneginf(m), 0.0, np.exp(m - m_new))
        e = np.exp(a - m_new[:, None])
        s = s * corr + e.sum(axis=1)
        acc = acc * corr[:, None] + e @ v[start:start + block]
        m = m_new
        history.append(s.copy())
    return acc / s[:, None], history


def merge_splits(o_parts, lse_parts):
    """Combine attention computed over disjoint key subsets.

    o_parts: [S, ..., d] each normalised over its own subset; lse_parts: [S, ...].
    lse = ln sum_s e^{lse_s};  o = sum_s e^{lse_s - lse} o_s. Subsets with
    lse_s = -inf (no visible key) contribute nothing. This is the block
    recurrence above applied once more, with each split playing one block.
    """
    o_parts = _as_f64(o_parts)
    lse_parts = _as_f64(lse_parts)
    m = lse_parts.max(axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.exp(lse_parts - m_safe)  # e^{-inf} = 0 for empty splits
    total = w.sum(axis=0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, total, 1.0)), -np.inf)
    o = (w[..., None] * o_parts).sum(axis=0) / np.where(finite, total, 1.0)[..., None]
    o = np.where(finite[..., None], o, 0.0)
    return o, lse
