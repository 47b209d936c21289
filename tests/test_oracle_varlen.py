"""Pins for the oracle's packed variable-length attention (cu_seqlens).

Page "Flash Attention原理" (FAQ Q10): sequences of different lengths are
packed into one batch and delimited by cumulative offsets, which avoids the
wasted work of padding.  The packed result must therefore equal the padded
computation on the valid rows.  Pinned here against:
  * torch's CPU float64 SDPA on a zero-padded batch with an explicit
    key-validity (and causal) mask, forward and autograd backward;
  * the ordinary batched oracle when every sequence has the same length;
  * central differences of the packed forward;
  * independence of the sequences (no leakage across a boundary);
  * empty sequences and rows that see no key (O = 0, lse = -inf).
A planted mistake (top-left causal alignment per sequence) fails the pins.
"""
import numpy as np
import pytest

import oracle
from sdpa_inputs import make_random


def rnd(shape, seed):
    return make_random(shape, seed).astype(np.float64)


def packed(lq, lk, H, Hkv, d, seed):
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int64)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int64)
    q = rnd((int(cu_q[-1]), H, d), seed)
    k = rnd((int(cu_k[-1]), Hkv, d), seed + 1)
    v = rnd((int(cu_k[-1]), Hkv, d), seed + 2)
    do = rnd((int(cu_q[-1]), H, d), seed + 3)
    return q, k, v, do, cu_q, cu_k


def torch_padded(q, k, v, do, cu_q, cu_k, s, causal):
    """Padded (B, H, Lmax, d) batch through torch SDPA with a boolean mask:
    key j of sequence b is visible to its query i iff j < Nk_b and (causal)
    j <= Nk_b - Nq_b + i.  Returns O, dQ, dK, dV scattered back to packed
    rows (only rows that see at least one key are meaningful)."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    B = len(cu_q) - 1
    H, Hkv, d = q.shape[1], k.shape[1], q.shape[2]
    G = H // Hkv
    lq, lk = np.diff(cu_q), np.diff(cu_k)
    Lq, Lk = int(max(lq.max(), 1)), int(max(lk.max(), 1))
    Q = np.zeros((B, H, Lq, d)); K = np.zeros((B, Hkv, Lk, d)); V = np.zeros((B, Hkv, Lk, d))
    DO = np.zeros((B, H, Lq, d))
    mask = np.zeros((B, 1, Lq, Lk), dtype=bool)
    for b in range(B):
        Q[b, :, :lq[b]] = q[cu_q[b]:cu_q[b + 1]].transpose(1, 0, 2)
        DO[b, :, :lq[b]] = do[cu_q[b]:cu_q[b + 1]].transpose(1, 0, 2)
        K[b, :, :lk[b]] = k[cu_k[b]:cu_k[b + 1]].transpose(1, 0, 2)
        V[b, :, :lk[b]] = v[cu_k[b]:cu_k[b + 1]].transpose(1, 0, 2)
        for i in range(lq[b]):
            hi = lk[b] if not causal else min(lk[b], lk[b] - lq[b] + i + 1)
            mask[b, 0, i, :max(hi, 0)] = True
    # Rows with no visible key (and padding rows) see key 0 in torch so that
    # its softmax stays finite; they are excluded from every comparison.
    dead = ~mask.any(-1)
    mask[..., 0] |= dead
    tq = torch.tensor(Q, requires_grad=True)
    tk = torch.tensor(np.repeat(K, G, axis=1), requires_grad=True)
    tv = torch.tensor(np.repeat(V, G, axis=1), requires_grad=True)
    live = torch.tensor(~dead[:, :, :, None])
    to = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.tensor(mask), scale=s)
    (to * live * torch.tensor(DO)).sum().backward()
    O = np.zeros_like(q); dq = np.zeros_like(q); dk = np.zeros_like(k); dv = np.zeros_like(v)
    gk = tk.grad.numpy().reshape(B, Hkv, G, Lk, d).sum(2)
    gv = tv.grad.numpy().reshape(B, Hkv, G, Lk, d).sum(2)
    for b in range(B):
        O[cu_q[b]:cu_q[b + 1]] = to.detach().numpy()[b, :, :lq[b]].transpose(1, 0, 2)
        dq[cu_q[b]:cu_q[b + 1]] = tq.grad.numpy()[b, :, :lq[b]].transpose(1, 0, 2)
        dk[cu_k[b]:cu_k[b + 1]] = gk[b, :, :lk[b]].transpose(1, 0, 2)
        dv[cu_k[b]:cu_k[b + 1]] = gv[b, :, :lk[b]].transpose(1, 0, 2)
    live_rows = np.concatenate([~dead[b, 0, :lq[b]] for b in range(B)]) if B else np.zeros(0, bool)
    return O, dq, dk, dv, live_rows


CASES = [
    # lengths of the query and key sequences, causal
    ([5, 9, 1, 12], [5, 9, 1, 12], True),       # self-attention packing
    ([5, 9, 1, 12], [5, 9, 1, 12], False),
    ([3, 7, 4], [8, 7, 10], True),              # chunks against longer contexts
    ([6, 2, 9], [3, 11, 4], False),             # cross attention, mixed
    ([4, 0, 6], [4, 3, 0], False),              # an empty query sequence, an empty key sequence
]


@pytest.mark.parametrize("lq,lk,causal", CASES)
def test_varlen_matches_padded_masked_torch(lq, lk, causal):
    H, Hkv, d, s = 4, 2, 8, 0.35
    q, k, v, do, cu_q, cu_k = packed(lq, lk, H, Hkv, d, 300 + sum(lq))
    O, lse = oracle.attention_varlen_forward(q, k, v, cu_q, cu_k, s, causal)
    dq, dk, dv = oracle.attention_varlen_backward(q, k, v, do, cu_q, cu_k, s, causal)
    tO, tdq, tdk, tdv, live = torch_padded(q, k, v, do, cu_q, cu_k, s, causal)
    np.testing.assert_allclose(O[live], tO[live], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq[live], tdq[live], rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, tdk, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, tdv, rtol=0, atol=1e-11)
    # rows that see no key: O = 0, lse = -inf, dQ = 0
    assert np.all(O[~live] == 0) and np.all(np.isneginf(lse[:, ~live])) and np.all(dq[~live] == 0)
    assert np.all(np.isfinite(lse[:, live]))


@pytest.mark.parametrize("causal", [False, True])
def test_equal_lengths_equal_the_batched_oracle(causal):
    B, H, Hkv, N, d, s = 3, 4, 2, 11, 8, 0.3
    q4, k4, v4, do4 = rnd((B, H, N, d), 401), rnd((B, Hkv, N, d), 402), rnd((B, Hkv, N, d), 403), rnd((B, H, N, d), 404)
    pack = lambda x: x.transpose(0, 2, 1, 3).reshape(B * N, x.shape[1], d)
    cu = np.arange(B + 1) * N
    O, lse = oracle.attention_varlen_forward(pack(q4), pack(k4), pack(v4), cu, cu, s, causal)
    Ob, lb = oracle.attention_forward(q4, k4, v4, s, causal)
    np.testing.assert_allclose(O, pack(Ob), rtol=0, atol=0)
    np.testing.assert_allclose(lse, lb.transpose(1, 0, 2).reshape(H, B * N), rtol=0, atol=0)
    g = oracle.attention_varlen_backward(pack(q4), pack(k4), pack(v4), pack(do4), cu, cu, s, causal)
    gb = oracle.attention_backward(q4, k4, v4, do4, s, causal)
    for x, y in zip(g, gb):
        np.testing.assert_allclose(x, pack(y), rtol=0, atol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_backward_finite_differences(causal):
    lq, lk = [2, 3, 0], [3, 2, 2]
    H, Hkv, d, s, h = 2, 1, 3, 0.6, 1e-6
    q, k, v, do, cu_q, cu_k = packed(lq, lk, H, Hkv, d, 420 + causal)
    grads = oracle.attention_varlen_backward(q, k, v, do, cu_q, cu_k, s, causal)

    def loss(q_, k_, v_):
        O, _ = oracle.attention_varlen_forward(q_, k_, v_, cu_q, cu_k, s, causal)
        return float((O * do).sum())

    for idx, (x, g) in enumerate(zip((q, k, v), grads)):
        fd = np.zeros_like(x)
        for pos in np.ndindex(x.shape):
            args = [q, k, v]
            xp, xm = x.copy(), x.copy()
            xp[pos] += h
            xm[pos] -= h
            args[idx] = xp
            lp = loss(*args)
            args[idx] = xm
            lm = loss(*args)
            fd[pos] = (lp - lm) / (2 * h)
        assert np.linalg.norm(fd - g) <= 1e-6 * max(np.linalg.norm(g), 1e-30), idx


def test_sequences_do_not_leak_into_each_other():
    lq = lk = [7, 5, 9]
    q, k, v, do, cu_q, cu_k = packed(lq, lk, 2, 2, 8, 430)
    O1, l1 = oracle.attention_varlen_forward(q, k, v, cu_q, cu_k, 0.4, True)
    k2, v2 = k.copy(), v.copy()
    k2[7:12] += 3.0  # change only sequence 1's keys and values
    v2[7:12] -= 2.0
    O2, l2 = oracle.attention_varlen_forward(q, k2, v2, cu_q, cu_k, 0.4, True)
    for a, b in ((0, 7), (12, 21)):
        assert np.array_equal(O1[a:b], O2[a:b]) and np.array_equal(l1[:, a:b], l2[:, a:b])
    assert np.abs(O1[7:12] - O2[7:12]).max() > 1e-3


def test_causal_rows_before_the_keys_see_nothing():
    # 5 queries against 2 keys, causal: rows 0..2 sit at negative positions.
    q, k, v, do, cu_q, cu_k = packed([5], [2], 1, 1, 4, 440)
    O, lse = oracle.attention_varlen_forward(q, k, v, cu_q, cu_k, 0.5, True)
    assert np.all(O[:3] == 0) and np.all(np.isneginf(lse[:, :3]))
    assert np.all(np.isfinite(lse[:, 3:]))
    dq, dk, dv = oracle.attention_varlen_backward(q, k, v, do, cu_q, cu_k, 0.5, True)
    assert np.all(dq[:3] == 0)
    # row 3 (position 0) sees key 0 only: its output is v[0]
    np.testing.assert_allclose(O[3], v[0], rtol=0, atol=1e-15)


def test_bad_offsets_are_rejected():
    q, k, v, do, cu_q, cu_k = packed([3, 4], [3, 4], 1, 1, 4, 450)
    with pytest.raises(ValueError):
        oracle.attention_varlen_forward(q, k, v, [0, 4, 3], cu_k, 0.5)
    with pytest.raises(ValueError):
        oracle.attention_varlen_forward(q, k, v, [0, 3, 8], cu_k, 0.5)
    with pytest.raises(ValueError):
        oracle.attention_varlen_forward(q, k, v, [0, 7], cu_k, 0.5)


def test_planted_top_left_alignment_is_caught():
    # A per-sequence top-left causal mask (query i sees keys 0..i) disagrees
    # with the padded torch reference whenever Nq_b != Nk_b.
    lq, lk = [3, 7, 4], [8, 7, 10]
    q, k, v, do, cu_q, cu_k = packed(lq, lk, 2, 1, 8, 460)
    tO, _, _, _, live = torch_padded(q, k, v, do, cu_q, cu_k, 0.3, True)
    wrong = np.zeros_like(q)
    for b in range(3):
        sl_q, sl_k = slice(cu_q[b], cu_q[b + 1]), slice(cu_k[b], cu_k[b + 1])
        Ob, _ = oracle.attention_forward(q[sl_q].transpose(1, 0, 2)[None], k[sl_k].transpose(1, 0, 2)[None],
                                         v[sl_k].transpose(1, 0, 2)[None], 0.3, True, q_offset=0)
        wrong[sl_q] = Ob[0].transpose(1, 0, 2)
    assert np.abs(wrong[live] - tO[live]).max() > 1e-3
