"""fp64 reference definitions of exact attention (test infrastructure only).

All functions take numpy arrays (any float dtype; they are upcast to float64)
in (batch, heads, seq_len, head_dim) layout.  K and V may have fewer heads
than Q (grouped-query attention): query head h reads key/value head
h // (H // Hkv), i.e. contiguous groups of G = H / Hkv query heads share one
K/V head, which equals repeating each K/V head G times along the head axis.

Sources (page title, section):
  [FA]  "Flash Attention原理：分块计算与重计算，如何降低O(n^2)的显存占用"
  [SDPA] "SDPA backend 与 FlashAttention"
  [SEL] "PyTorch scaled dot product attention怎样选择高效注意力后端"
"""
from __future__ import annotations

import math

import numpy as np


def gqa_kv_head(h: int, H: int, Hkv: int) -> int:
    """K/V head read by query head h.  [SEL] (section on why the same code can
    select different backends) only says the query and key/value head counts
    must satisfy a constraint; the reading taken is Hkv divides H and
    contiguous groups: h -> h // (H / Hkv)."""
    if H % Hkv:
        raise ValueError("Hkv must divide H")
    return h // (H // Hkv)


def _check(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("expected (B, H, N, d) tensors")
    B, H, N, d = q.shape
    if k.shape[0] != B or v.shape[0] != B or k.shape[1] != v.shape[1]:
        raise ValueError("batch / kv-head mismatch")
    if k.shape[2] != v.shape[2] or k.shape[3] != d:
        raise ValueError("key length / head_dim mismatch")
    gqa_kv_head(0, H, k.shape[1])
    return B, H, k.shape[1], N, k.shape[2], d


def _scores(qh, kh, scale, causal, rows=None, q_offset=0):
    """S = scale * Q K^T for one head, with the causal mask applied.

    [FA] §一 step 1-2 (S = Q K^T, softmax of S / sqrt(d)); the causal mask of
    [SDPA] §3 (is_causal=True) sets S_ij = -inf for key j > query position
    i.  Query row i sits at position q_offset + i (0 when queries and keys
    share positions 0..N-1).  ``rows`` selects query rows.
    """
    if rows is None:
        rows = np.arange(qh.shape[0])
    S = scale * (qh[rows] @ kh.T)
    if causal:
        cols = np.arange(kh.shape[0])
        S = np.where(cols[None, :] > q_offset + np.asarray(rows)[:, None], -np.inf, S)
    return S


def visibility(Nq, Nk, causal=False, q_offset=0, window=None, key_length=None, mask=None):
    """Boolean (Nq, Nk) matrix: may query row i attend to key j?

    Query row i sits at position q_offset + i.  The conditions combine by
    AND ([SDPA] §3: is_causal, and attn_mask with True = take part):
      causal      j <= q_offset + i
      window      (wl, wr): j >= q_offset + i - wl when wl >= 0 and
                  j <= q_offset + i + wr when wr >= 0 (a sliding window, the
                  [PROF] section on changing the architecture: cost n * w
                  instead of n^2); -1 leaves that side open
      key_length  j < key_length (a padding mask: the keys past a batch
                  element's length are padding)
      mask        an explicit boolean (Nq, Nk) matrix ([FA] FAQ Q11).
    """
    i = q_offset + np.arange(Nq)[:, None]
    j = np.arange(Nk)[None, :]
    vis = np.ones((Nq, Nk), dtype=bool)
    if causal:
        vis &= j <= i
    if window is not None:
        wl, wr = window
        if wl >= 0:
            vis &= j >= i - wl
        if wr >= 0:
            vis &= j <= i + wr
    if key_length is not None:
        vis &= j < key_length
    if mask is not None:
        vis &= np.asarray(mask, dtype=bool)
    return vis


def _mask_plane(mask, b, h):
    """The (Nq, Nk) plane of a (Bm, Hm, Nq, Nk) boolean mask that batch b,
    head h reads (Bm, Hm of 1 broadcast)."""
    if mask is None:
        return None
    m = np.asarray(mask, dtype=bool)
    return m[b if m.shape[0] > 1 else 0, h if m.shape[1] > 1 else 0]


def _masked_scores(q, k, scale, vis, bias):
    """scale * q k^T, plus the additive mask when there is one, with the
    invisible entries at -inf."""
    S = scale * (q @ k.T)
    if bias is not None:
        S = S + bias
    return np.where(vis, S, -np.inf)


def _bias_plane(bias, b, h):
    """The (Nq, Nk) float64 plane of a (Bb, Hb, Nq, Nk) additive mask that
    batch b, head h adds (Bb, Hb of 1 broadcast)."""
    if bias is None:
        return None
    a = np.asarray(bias, dtype=np.float64)
    return a[b if a.shape[0] > 1 else 0, h if a.shape[1] > 1 else 0]


def attention_masked_forward(q, k, v, scale=None, causal=False, window=None, key_lengths=None, mask=None,
                             bias=None):
    """Attention under any combination of the masks of ``visibility``, with
    query row i at position Nk - Nq + i (the alignment of
    ``attention_decode``; i itself when Nq = Nk).  key_lengths: (B,) ints or
    None; mask: boolean (Bm, Hm, Nq, Nk), Bm in {1, B}, Hm in {1, H}, or
    None; bias: an additive float mask of the same broadcasting shape, added
    to the scaled scores before the softmax (SDPA's float attn_mask; finite
    or -inf entries, -inf hiding the key), or None.  Rows that see no key:
    O = 0, lse = -inf.  Returns O (B, H, Nq, d_v) and lse (B, H, Nq)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, Hkv, Nq, Nk, d = _check(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    O = np.zeros((B, H, Nq, v.shape[3]))
    lse = np.full((B, H, Nq), -np.inf)
    for b in range(B):
        for h in range(H):
            hk = gqa_kv_head(h, H, Hkv)
            vis = visibility(Nq, Nk, causal, Nk - Nq, window,
                             None if key_lengths is None else int(key_lengths[b]), _mask_plane(mask, b, h))
            S = _masked_scores(q[b, h], k[b, hk], scale, vis, _bias_plane(bias, b, h))
            live = np.isfinite(S).any(axis=1)
            if live.any():
                P, m, l = softmax_rows(S[live])
                O[b, h][live] = P @ v[b, hk]
                lse[b, h][live] = m + np.log(l)
    return O, lse


def attention_masked_backward(q, k, v, do, scale=None, causal=False, window=None, key_lengths=None, mask=None,
                              bias=None):
    """Gradients of ``attention_masked_forward`` by the chain rule of
    ``attention_backward`` (masked entries have P = 0; rows that see no key
    contribute nothing; the additive mask enters through P only and gets no
    gradient).  Returns dQ, dK, dV in float64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, H, Hkv, Nq, Nk, d = _check(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            hk = gqa_kv_head(h, H, Hkv)
            vis = visibility(Nq, Nk, causal, Nk - Nq, window,
                             None if key_lengths is None else int(key_lengths[b]), _mask_plane(mask, b, h))
            S = _masked_scores(q[b, h], k[b, hk], scale, vis, _bias_plane(bias, b, h))
            live = np.isfinite(S).any(axis=1)
            P = np.zeros_like(S)
            if live.any():
                P[live] = softmax_rows(S[live])[0]
            dv[b, hk] += P.T @ do[b, h]
            dP = do[b, h] @ v[b, hk].T
            D = (P * dP).sum(axis=1)
            dS = P * (dP - D[:, None])
            dq[b, h] = scale * (dS @ k[b, hk])
            dk[b, hk] += scale * (dS.T @ q[b, h])
    return dq, dk, dv


def softmax_rows(S):
    """Max-subtracted softmax along the last axis ([FA] §四:
    softmax(x_i) = exp(x_i - max x) / sum_j exp(x_j - max x)).
    Returns (P, m, l) with m the row max and l the row sum of exp(S - m)."""
    S = np.asarray(S, dtype=np.float64)
    m = S.max(axis=-1, keepdims=True)
    E = np.exp(S - m)
    l = E.sum(axis=-1, keepdims=True)
    return E / l, m[..., 0], l[..., 0]


def softmax_two_block(x):
    """The two-block merge of [FA] §四 on the last axis of x.

    The last axis is split in half; each half gets its own max m1, m2 and
    exp-sum e1, e2; the global max is m = max(m1, m2) and the global sum is
    l = e1 * exp(m1 - m) + e2 * exp(m2 - m); both halves are then normalised
    with the global m and l.  Works in x's own float dtype (the page's check
    is in float32)."""
    x = np.asarray(x)
    mid = x.shape[-1] // 2
    x1, x2 = x[..., :mid], x[..., mid:]
    m1 = x1.max(axis=-1, keepdims=True)
    m2 = x2.max(axis=-1, keepdims=True)
    m = np.maximum(m1, m2)
    e1 = np.exp(x1 - m1).sum(axis=-1, keepdims=True)
    e2 = np.exp(x2 - m2).sum(axis=-1, keepdims=True)
    l = e1 * np.exp(m1 - m) + e2 * np.exp(m2 - m)
    return np.concatenate([np.exp(x1 - m) / l, np.exp(x2 - m) / l], axis=-1)


def attention_forward(q, k, v, scale=None, causal=False, q_offset=0):
    """O = softmax(scale * Q K^T [+ causal mask]) V and lse, in float64.

    [FA] §一 (standard attention: S, P and O materialised per head) with the
    stable softmax of §四.  lse_i = m_i + ln(l_i) is the natural-log
    logsumexp of row i of the scaled, masked scores: the single per-row
    statistic that replaces the m and l of §五.  Query row i sits at
    position q_offset + i for the causal mask.  A row whose keys are all
    masked has lse = -inf and O = 0.
    Returns O (B, H, N, d_v) and lse (B, H, N).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, Hkv, N, Nk, d = _check(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    O = np.empty((B, H, N, v.shape[3]))
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            hk = gqa_kv_head(h, H, Hkv)
            S = _scores(q[b, h], k[b, hk], scale, causal, q_offset=q_offset)
            live = np.isfinite(S).any(axis=1)
            P = np.zeros_like(S)
            m = np.full(S.shape[0], -np.inf)
            l = np.zeros(S.shape[0])
            if live.any():
                P[live], m[live], l[live] = softmax_rows(S[live])
            O[b, h] = P @ v[b, hk]
            with np.errstate(divide="ignore"):
                lse[b, h] = m + np.log(l)
    return O, lse


def attention_decode(q, k, v, scale=None, causal=False):
    """Attention of a block of Nq new queries against a cache of Nk >= Nq
    keys/values (decode with a KV cache).

    The pages place decode next to prefill ([FA] FAQ on inference, KV cache
    and P99 decode latency) without a formula; the computation is the same
    softmax(scale * Q K^T) V over every cached key.  Reading taken for the
    causal mask: the new queries are the last Nq positions of the sequence,
    so query t sits at position Nk - Nq + t and sees keys 0..Nk-Nq+t (with
    Nq = Nk this is the ordinary causal mask).
    Returns O (B, H, Nq, d_v) and lse (B, H, Nq)."""
    Nq, Nk = np.shape(q)[2], np.shape(k)[2]
    if Nq > Nk:
        raise ValueError("decode needs Nq <= Nk")
    return attention_forward(q, k, v, scale, causal, q_offset=Nk - Nq)


def attention_cross_backward(q, k, v, do, scale=None, causal=False):
    """Gradients of the Nq-query, Nk-key attention of ``attention_decode``
    (same causal reading: query t at position Nk - Nq + t), by the chain rule
    of ``attention_backward``.  Returns dQ (B, H, Nq, d), dK, dV (B, Hkv, Nk, d)."""
    Nq, Nk = np.shape(q)[2], np.shape(k)[2]
    if causal and Nq > Nk:
        raise ValueError("causal cross attention needs Nq <= Nk")
    return attention_backward(q, k, v, do, scale, causal, q_offset=Nk - Nq)


def attention_decode_paged(q, k_cache, v_cache, block_table, seq_lens, scale=None, causal=False):
    """Decode against a paged KV cache ([FA] FAQ Q12-Q13: the KV cache with
    PagedAttention, the cache kept in fixed-size pages found through a block
    table).  Batch element b's cached keys are the first seq_lens[b] tokens
    of its pages block_table[b, 0], block_table[b, 1], ..., in that order;
    k_cache, v_cache: (num_pages, page_size, Hkv, d).  The keys are gathered
    into one sequence per batch element and ``attention_decode`` applies.
    Returns O (B, H, Nq, d_v) and lse (B, H, Nq)."""
    q = np.asarray(q, dtype=np.float64)
    k_cache = np.asarray(k_cache, dtype=np.float64)
    v_cache = np.asarray(v_cache, dtype=np.float64)
    B, H, Nq, _ = q.shape
    ps = k_cache.shape[1]
    O = np.zeros((B, H, Nq, v_cache.shape[3]))
    lse = np.full((B, H, Nq), -np.inf)
    for b in range(B):
        L = int(seq_lens[b])
        npg = -(-L // ps)
        pages = [int(x) for x in np.asarray(block_table)[b, :npg]]
        kb = k_cache[pages].reshape(npg * ps, *k_cache.shape[2:])[:L].transpose(1, 0, 2)[None]
        vb = v_cache[pages].reshape(npg * ps, *v_cache.shape[2:])[:L].transpose(1, 0, 2)[None]
        O[b:b + 1], lse[b:b + 1] = attention_decode(q[b:b + 1], kb, vb, scale, causal)
    return O, lse


def merge_splits(O_parts, lse_parts):
    """Combine attention computed over disjoint key ranges ("splits").

    The two-block merge of [FA] §四 for any number of blocks, on normalised
    partial results: with lse_s the logsumexp of split s and O_s its
    normalised output, lse = ln sum_s exp(lse_s) and
    O = sum_s exp(lse_s - lse) O_s.  Splits with lse_s = -inf (every key
    masked) carry weight 0.
    O_parts: (S, ..., d), lse_parts: (S, ...).  Returns O (..., d), lse (...)."""
    O_parts = np.asarray(O_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = lse_parts.max(axis=0)
    safe = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(lse_parts - safe)
    tot = w.sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(tot > 0, safe + np.log(tot), -np.inf)
        O = np.where(tot[..., None] > 0, (w[..., None] * O_parts).sum(axis=0) / np.where(tot > 0, tot, 1.0)[..., None], 0.0)
    return O, lse


def attention_forward_rows(qh, kh, vh, rows, scale, causal=False, q_offset=0):
    """Forward for a subset of absolute query rows of ONE head.

    Same definition as ``attention_forward``; the causal mask uses the
    absolute row indices (query row i at position q_offset + i), so sampled
    rows of a full-size head can be checked one by one.  qh: (N, d), kh/vh:
    (Nk, d).  Returns O (len(rows), d_v), lse (len(rows),)."""
    qh = np.asarray(qh, dtype=np.float64)
    kh = np.asarray(kh, dtype=np.float64)
    vh = np.asarray(vh, dtype=np.float64)
    rows = np.asarray(rows)
    S = _scores(qh, kh, scale, causal, rows, q_offset=q_offset)
    P, m, l = softmax_rows(S)
    return P @ vh, m + np.log(l)


def attention_forward_online(q, k, v, scale=None, causal=False, block=64):
    """Forward by the blockwise online-softmax recurrence of [FA] §三-§四.

    Keys/values are visited in blocks of ``block`` columns.  For each row a
    running max m and normaliser l are kept together with the unnormalised
    output acc; when block j arrives with local max m_j:
        m_new = max(m, m_j)
        acc   = acc * exp(m - m_new) + exp(S_j - m_new) V_j
        l     = l   * exp(m - m_new) + rowsum(exp(S_j - m_new))
    and at the end O = acc / l, lse = m + ln l.  No blocking beyond the key
    blocks; used only to pin the two-pass = online equivalence.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, Hkv, N, Nk, d = _check(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    O = np.empty((B, H, N, v.shape[3]))
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            hk = gqa_kv_head(h, H, Hkv)
            S = _scores(q[b, h], k[b, hk], scale, causal)
            m = np.full(N, -np.inf)
            l = np.zeros(N)
            acc = np.zeros((N, v.shape[3]))
            for j0 in range(0, Nk, block):
                Sj = S[:, j0:j0 + block]
                m_new = np.maximum(m, Sj.max(axis=1))
                # rows whose every key so far is masked keep m = -inf
                alive = np.isfinite(m_new)
                shift = np.where(alive, m_new, 0.0)
                alpha = np.where(np.isfinite(m), np.exp(m - shift), 0.0)
                E = np.exp(Sj - shift[:, None])
                acc = acc * alpha[:, None] + E @ v[b, hk, j0:j0 + block]
                l = l * alpha + E.sum(axis=1)
                m = m_new
            O[b, h] = acc / l[:, None]
            lse[b, h] = m + np.log(l)
    return O, lse


def attention_backward(q, k, v, do, scale=None, causal=False, q_offset=0):
    """Analytic gradients of O = softmax(scale Q K^T [+mask]) V w.r.t. Q, K, V.

    The pages ([FA] §五 and FAQ Q19) say the backward recomputes P and follows
    the chain rule without printing it; the textbook derivation is written out
    per head with the oracle's own fp64 P:
        dV   = P^T dO
        dP   = dO V^T
        D_i  = sum_j P_ij dP_ij            (softmax Jacobian-vector product)
        dS   = P * (dP - D 1^T)            (masked entries have P = 0)
        dQ   = scale * dS K
        dK   = scale * dS^T Q
    With grouped-query attention the dK, dV of a K/V head are the sums over
    the G query heads that read it.  Query row i sits at position
    q_offset + i for the causal mask, as in ``attention_forward``; a row that
    sees no key has P = 0 and so contributes nothing.  Returns dQ, dK, dV in
    float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, H, Hkv, N, Nk, d = _check(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            hk = gqa_kv_head(h, H, Hkv)
            S = _scores(q[b, h], k[b, hk], scale, causal, q_offset=q_offset)
            live = np.isfinite(S).any(axis=1)
            P = np.zeros_like(S)
            if live.any():
                P[live] = softmax_rows(S[live])[0]
            dv[b, hk] += P.T @ do[b, h]
            dP = do[b, h] @ v[b, hk].T
            D = (P * dP).sum(axis=1)
            dS = P * (dP - D[:, None])
            dq[b, h] = scale * (dS @ k[b, hk])
            dk[b, hk] += scale * (dS.T @ q[b, h])
    return dq, dk, dv


def _varlen_bounds(cu, total):
    cu = [int(x) for x in np.asarray(cu).reshape(-1)]
    if len(cu) < 1 or cu[0] != 0 or cu[-1] != total or any(b < a for a, b in zip(cu, cu[1:])):
        raise ValueError("cu_seqlens must start at 0, be non-decreasing and end at the packed length")
    return cu


def attention_varlen_forward(q, k, v, cu_q, cu_k, scale=None, causal=False):
    """Attention over a packed batch of variable-length sequences.

    [FA] FAQ Q10: several sequences of different lengths are packed into one
    batch and delimited by cumulative offsets (cu_seqlens), so that no padding
    is computed.  Layout read here: q (total_q, H, d), k and v (total_k, Hkv,
    d), the sequences one after another; sequence b owns query rows
    cu_q[b] .. cu_q[b+1]-1 and key rows cu_k[b] .. cu_k[b+1]-1 and attends
    only within itself.  Causal: per sequence, query row i sits at position
    Nk_b - Nq_b + i (the alignment of ``attention_decode``).  A row that sees
    no key has O = 0 and lse = -inf.
    Returns O (total_q, H, d_v) and lse (H, total_q)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    cq = _varlen_bounds(cu_q, q.shape[0])
    ck = _varlen_bounds(cu_k, k.shape[0])
    if len(cq) != len(ck):
        raise ValueError("cu_seqlens_q and cu_seqlens_k describe different batch sizes")
    H = q.shape[1]
    O = np.zeros((q.shape[0], H, v.shape[2]))
    lse = np.full((H, q.shape[0]), -np.inf)
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        if q1 == q0:
            continue
        qb = q[q0:q1].transpose(1, 0, 2)[None]
        kb = k[k0:k1].transpose(1, 0, 2)[None]
        vb = v[k0:k1].transpose(1, 0, 2)[None]
        off = (k1 - k0) - (q1 - q0) if causal else 0
        Ob, lb = attention_forward(qb, kb, vb, scale, causal, q_offset=off)
        O[q0:q1] = Ob[0].transpose(1, 0, 2)
        lse[:, q0:q1] = lb[0]
    return O, lse


def attention_varlen_backward(q, k, v, do, cu_q, cu_k, scale=None, causal=False):
    """Gradients of ``attention_varlen_forward``: per sequence, the chain rule
    of ``attention_backward`` with that sequence's causal offset.  Returns
    dQ (total_q, H, d), dK and dV (total_k, Hkv, d); keys of a sequence with
    no query rows get zero gradients."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    cq = _varlen_bounds(cu_q, q.shape[0])
    ck = _varlen_bounds(cu_k, k.shape[0])
    if len(cq) != len(ck):
        raise ValueError("cu_seqlens_q and cu_seqlens_k describe different batch sizes")
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        if q1 == q0 or k1 == k0:
            continue
        t = lambda x, a, c: x[a:c].transpose(1, 0, 2)[None]
        off = (k1 - k0) - (q1 - q0) if causal else 0
        g = attention_backward(t(q, q0, q1), t(k, k0, k1), t(v, k0, k1), t(do, q0, q1), scale, causal,
                               q_offset=off)
        dq[q0:q1] = g[0][0].transpose(1, 0, 2)
        dk[k0:k1] = g[1][0].transpose(1, 0, 2)
        dv[k0:k1] = g[2][0].transpose(1, 0, 2)
    return dq, dk, dv


def score_matrix_bytes(n: int, bytes_per_elem: int = 4) -> int:
    """Bytes of one n x n score (or probability) matrix ([FA] §一)."""
    return n * n * bytes_per_elem


def row_stat_bytes(n: int, n_stats: int = 2, bytes_per_elem: int = 4) -> int:
    """Bytes of the per-row statistics kept instead of S and P ([FA] §五:
    m(n) and l(n))."""
    return n * n_stats * bytes_per_elem
