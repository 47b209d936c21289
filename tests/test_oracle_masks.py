"""Pins for the oracle's masked attention (sliding window, key lengths,
boolean attn_mask, and their combination with causal).

Pinned against:
  * brute force per row: the attention of one query over the explicit list
    of keys it may see, written with plain loops (no mask matrix);
  * truncating K and V to a batch element's key length;
  * torch's CPU float64 SDPA with the boolean attn_mask, forward and
    autograd backward ([FA] FAQ Q11: SDPA takes an arbitrary boolean mask);
  * special cases: an all-True mask, a lower-triangular mask equal to
    is_causal, a window wide enough to be no window;
  * central differences of the masked forward;
  * rows that see no key (O = 0, lse = -inf, zero gradients).
A planted off-by-one in the window bound fails the brute-force pin.

The additive (float) mask, added to the scaled scores before the softmax
(SDPA's float attn_mask), is pinned against torch's CPU float64 SDPA with
that float mask (forward and autograd), a per-row brute force with the bias
added by hand, the identities bias = -inf where a boolean mask is False
(equal to that mask) and bias constant along each row (no change: softmax
is shift invariant), and central differences; a planted sign error in the
bias fails the brute-force pin.
"""
import math

import numpy as np
import pytest

import oracle
from sdpa_inputs import make_random


def rnd(shape, seed):
    return make_random(shape, seed).astype(np.float64)


def _qkv(B, H, Hkv, Nq, Nk, d, seed):
    return (rnd((B, H, Nq, d), seed), rnd((B, Hkv, Nk, d), seed + 1), rnd((B, Hkv, Nk, d), seed + 2),
            rnd((B, H, Nq, d), seed + 3))


def brute_row(qv, K, V, keys, s):
    """softmax over the listed keys only, by loops."""
    if not keys:
        return np.zeros(V.shape[1]), -math.inf
    sc = [s * float(qv @ K[j]) for j in keys]
    m = max(sc)
    w = [math.exp(x - m) for x in sc]
    l = sum(w)
    o = sum(wi * V[j] for wi, j in zip(w, keys)) / l
    return o, m + math.log(l)


def keys_of(i, Nq, Nk, causal, window, klen):
    pos = Nk - Nq + i
    out = []
    for j in range(Nk):
        if causal and j > pos:
            continue
        if window is not None:
            wl, wr = window
            if wl >= 0 and j < pos - wl:
                continue
            if wr >= 0 and j > pos + wr:
                continue
        if klen is not None and j >= klen:
            continue
        out.append(j)
    return out


@pytest.mark.parametrize("Nq,Nk,causal,window", [
    (13, 13, True, (4, -1)),      # causal sliding window
    (13, 13, False, (3, 2)),      # two-sided window
    (9, 20, True, (5, -1)),       # a chunk against a longer cache
    (20, 9, False, (2, 2)),       # more queries than keys
    (11, 11, False, (0, 0)),      # each query sees only its own position
    (11, 11, True, (-1, -1)),     # no window: plain causal
])
def test_window_matches_brute_force(Nq, Nk, causal, window):
    B, H, Hkv, d, s = 2, 2, 1, 5, 0.4
    q, k, v, _ = _qkv(B, H, Hkv, Nq, Nk, d, 500 + Nq + Nk)
    klen = np.array([Nk, max(Nk - 3, 1)])
    O, lse = oracle.attention_masked_forward(q, k, v, s, causal, window, klen)
    for b in range(B):
        for h in range(H):
            for i in range(Nq):
                o, l = brute_row(q[b, h, i], k[b, 0], v[b, 0], keys_of(i, Nq, Nk, causal, window, klen[b]), s)
                np.testing.assert_allclose(O[b, h, i], o, rtol=0, atol=1e-12)
                assert (l == lse[b, h, i]) if math.isinf(l) else abs(l - lse[b, h, i]) < 1e-12


def test_key_length_equals_truncated_keys():
    B, H, Hkv, N, d, s = 3, 2, 2, 17, 6, 0.5
    q, k, v, _ = _qkv(B, H, Hkv, N, N, d, 520)
    klen = np.array([17, 9, 1])
    O, lse = oracle.attention_masked_forward(q, k, v, s, False, None, klen)
    for b in range(B):
        L = klen[b]
        Ot, lt = oracle.attention_forward(q[b:b + 1], k[b:b + 1, :, :L], v[b:b + 1, :, :L], s)
        np.testing.assert_allclose(O[b], Ot[0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[b], lt[0], rtol=0, atol=1e-13)


def _random_mask(shape, seed, p=0.7):
    return np.random.default_rng(seed).random(shape) < p


@pytest.mark.parametrize("mshape", ["full", "batch", "head", "shared"])
@pytest.mark.parametrize("causal", [False, True])
def test_bool_mask_against_torch(mshape, causal):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    B, H, Hkv, Nq, Nk, d, s = 2, 4, 2, 10, 14, 8, 0.3
    q, k, v, do = _qkv(B, H, Hkv, Nq, Nk, d, 530)
    shape = {"full": (B, H, Nq, Nk), "batch": (B, 1, Nq, Nk), "head": (1, H, Nq, Nk), "shared": (1, 1, Nq, Nk)}
    mask = _random_mask(shape[mshape], 531)
    window = (6, 3)
    O, lse = oracle.attention_masked_forward(q, k, v, s, causal, window, None, mask)
    g = oracle.attention_masked_backward(q, k, v, do, s, causal, window, None, mask)
    # the same visibility built independently, broadcast to (B, H, Nq, Nk)
    pos = (Nk - Nq) + np.arange(Nq)[:, None]
    j = np.arange(Nk)[None, :]
    band = (j >= pos - window[0]) & (j <= pos + window[1]) & ((j <= pos) if causal else True)
    vis = np.broadcast_to(mask, (B, H, Nq, Nk)) & band
    live = vis.any(-1)
    safe = vis.copy()
    safe[..., 0] |= ~live  # keep torch's softmax finite on dead rows; they are not compared
    G = H // Hkv
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(np.repeat(k, G, axis=1), requires_grad=True)
    tv = torch.tensor(np.repeat(v, G, axis=1), requires_grad=True)
    to = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.tensor(safe), scale=s)
    (to * torch.tensor(live[..., None]) * torch.tensor(do)).sum().backward()
    np.testing.assert_allclose(O[live], to.detach().numpy()[live], rtol=0, atol=1e-12)
    assert np.all(O[~live] == 0) and np.all(np.isneginf(lse[~live]))
    np.testing.assert_allclose(g[0], tq.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(g[1], tk.grad.numpy().reshape(B, Hkv, G, Nk, d).sum(2), rtol=0, atol=1e-11)
    np.testing.assert_allclose(g[2], tv.grad.numpy().reshape(B, Hkv, G, Nk, d).sum(2), rtol=0, atol=1e-11)


def test_special_cases_reduce_to_unmasked_attention():
    B, H, Hkv, N, d, s = 1, 2, 1, 12, 4, 0.6
    q, k, v, do = _qkv(B, H, Hkv, N, N, d, 540)
    ref = oracle.attention_forward(q, k, v, s, False)
    ones = np.ones((1, 1, N, N), dtype=bool)
    for args in ((False, None, None, ones), (False, (N, N), None, None), (False, (-1, -1), np.array([N]), None)):
        O, lse = oracle.attention_masked_forward(q, k, v, s, *args)
        np.testing.assert_allclose(O, ref[0], rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse, ref[1], rtol=0, atol=1e-14)
    tril = np.tril(np.ones((N, N), dtype=bool))[None, None]
    O, lse = oracle.attention_masked_forward(q, k, v, s, False, None, None, tril)
    Oc, lc = oracle.attention_forward(q, k, v, s, True)
    np.testing.assert_allclose(O, Oc, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, lc, rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_masked_backward_finite_differences(causal):
    B, H, Hkv, Nq, Nk, d, s, h = 1, 2, 1, 5, 6, 3, 0.7, 1e-6
    q, k, v, do = _qkv(B, H, Hkv, Nq, Nk, d, 550 + causal)
    mask = _random_mask((1, H, Nq, Nk), 551, 0.6)
    window, klen = (3, 1), np.array([5])
    grads = oracle.attention_masked_backward(q, k, v, do, s, causal, window, klen, mask)

    def loss(q_, k_, v_):
        O, _ = oracle.attention_masked_forward(q_, k_, v_, s, causal, window, klen, mask)
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


def test_rows_without_keys_give_zero():
    B, H, Hkv, N, d = 1, 1, 1, 6, 4
    q, k, v, do = _qkv(B, H, Hkv, N, N, d, 560)
    mask = np.ones((1, 1, N, N), dtype=bool)
    mask[0, 0, 2] = False  # row 2 sees nothing
    O, lse = oracle.attention_masked_forward(q, k, v, 0.5, False, None, None, mask)
    dq, dk, dv = oracle.attention_masked_backward(q, k, v, do, 0.5, False, None, None, mask)
    assert np.all(O[0, 0, 2] == 0) and np.isneginf(lse[0, 0, 2]) and np.all(dq[0, 0, 2] == 0)
    assert np.all(np.isfinite(lse[0, 0, [0, 1, 3, 4, 5]]))


def test_planted_window_off_by_one_is_caught():
    # A window that keeps j > pos - wl instead of j >= pos - wl drops one key
    # per row; the brute-force pin sees it.
    Nq = Nk = 10
    wl = 3
    q, k, v, _ = _qkv(1, 1, 1, Nq, Nk, 4, 570)
    wrong_vis = oracle.visibility(Nq, Nk, True, 0, (wl - 1, -1))   # the planted bound
    S = np.where(wrong_vis, 0.5 * q[0, 0] @ k[0, 0].T, -np.inf)
    P = oracle.softmax_rows(S)[0]
    wrong = P @ v[0, 0]
    i = 7
    o, _ = brute_row(q[0, 0, i], k[0, 0], v[0, 0], keys_of(i, Nq, Nk, True, (wl, -1), None), 0.5)
    assert np.abs(wrong[i] - o).max() > 1e-3
    O, _ = oracle.attention_masked_forward(q, k, v, 0.5, True, (wl, -1))
    assert np.abs(O[0, 0, i] - o).max() < 1e-12


def _random_bias(shape, seed, dead=0.2):
    """Finite biases in [-3, 3) with a share of -inf entries."""
    rng = np.random.default_rng(seed)
    bias = rng.uniform(-3.0, 3.0, shape)
    bias[rng.random(shape) < dead] = -np.inf
    return bias


@pytest.mark.parametrize("bshape", ["full", "batch", "head", "shared"])
@pytest.mark.parametrize("causal", [False, True])
def test_additive_mask_against_torch(bshape, causal):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    B, H, Hkv, Nq, Nk, d, s = 2, 4, 2, 9, 13, 8, 0.35
    q, k, v, do = _qkv(B, H, Hkv, Nq, Nk, d, 580 + causal)
    shape = {"full": (B, H, Nq, Nk), "batch": (B, 1, Nq, Nk), "head": (1, H, Nq, Nk), "shared": (1, 1, Nq, Nk)}
    bias = _random_bias(shape[bshape], 581)
    O, lse = oracle.attention_masked_forward(q, k, v, s, causal, None, None, None, bias)
    g = oracle.attention_masked_backward(q, k, v, do, s, causal, None, None, None, bias)
    # torch: the causal band as -inf in the same float mask (bottom-right
    # aligned: row i at position Nk - Nq + i)
    pos = (Nk - Nq) + np.arange(Nq)[:, None]
    band = np.where(np.arange(Nk)[None, :] <= pos, 0.0, -np.inf) if causal else np.zeros((Nq, Nk))
    full = np.broadcast_to(bias, (B, H, Nq, Nk)) + band
    live = np.isfinite(full).any(-1)
    safe = full.copy()
    safe[..., 0] = np.where(live, safe[..., 0], 0.0)  # keep torch finite on dead rows; not compared
    G = H // Hkv
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(np.repeat(k, G, axis=1), requires_grad=True)
    tv = torch.tensor(np.repeat(v, G, axis=1), requires_grad=True)
    to = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.tensor(safe), scale=s)
    (to * torch.tensor(live[..., None]) * torch.tensor(do)).sum().backward()
    np.testing.assert_allclose(O[live], to.detach().numpy()[live], rtol=0, atol=1e-12)
    assert np.all(O[~live] == 0) and np.all(np.isneginf(lse[~live]))
    np.testing.assert_allclose(g[0], tq.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(g[1], tk.grad.numpy().reshape(B, Hkv, G, Nk, d).sum(2), rtol=0, atol=1e-11)
    np.testing.assert_allclose(g[2], tv.grad.numpy().reshape(B, Hkv, G, Nk, d).sum(2), rtol=0, atol=1e-11)


def brute_row_bias(qv, K, V, keys, s, brow):
    """softmax over the listed keys of s * q.k + bias, by loops."""
    sc = [s * float(qv @ K[j]) + float(brow[j]) for j in keys if np.isfinite(brow[j])]
    kept = [j for j in keys if np.isfinite(brow[j])]
    if not kept:
        return np.zeros(V.shape[1]), -math.inf
    m = max(sc)
    w = [math.exp(x - m) for x in sc]
    tot = sum(w)
    o = sum(wi * V[j] for wi, j in zip(w, kept)) / tot
    return o, m + math.log(tot)


def test_additive_mask_matches_brute_force():
    Nq, Nk, d, s = 7, 11, 5, 0.45
    q, k, v, _ = _qkv(1, 1, 1, Nq, Nk, d, 590)
    bias = _random_bias((1, 1, Nq, Nk), 591)
    window = (4, 2)
    O, lse = oracle.attention_masked_forward(q, k, v, s, True, window, None, None, bias)
    for i in range(Nq):
        keys = keys_of(i, Nq, Nk, True, window, None)
        o, l = brute_row_bias(q[0, 0, i], k[0, 0], v[0, 0], keys, s, bias[0, 0, i])
        np.testing.assert_allclose(O[0, 0, i], o, rtol=0, atol=1e-13)
        assert (np.isneginf(l) and np.isneginf(lse[0, 0, i])) or abs(lse[0, 0, i] - l) < 1e-13


def test_additive_mask_identities():
    B, H, Hkv, N, d, s = 2, 2, 1, 10, 6, 0.5
    q, k, v, do = _qkv(B, H, Hkv, N, N, d, 600)
    mask = _random_mask((B, 1, N, N), 601)
    as_bias = np.where(mask, 0.0, -np.inf)
    for f in (oracle.attention_masked_forward, ):
        a = f(q, k, v, s, True, None, None, mask)
        b = f(q, k, v, s, True, None, None, None, as_bias)
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])
    ga = oracle.attention_masked_backward(q, k, v, do, s, True, None, None, mask)
    gb = oracle.attention_masked_backward(q, k, v, do, s, True, None, None, None, as_bias)
    for x, y in zip(ga, gb):
        np.testing.assert_array_equal(x, y)
    # a bias constant along each row shifts every score of the row alike
    rowc = np.random.default_rng(602).uniform(-5, 5, (1, H, N, 1)) * np.ones((1, H, N, N))
    O0, l0 = oracle.attention_masked_forward(q, k, v, s, False)
    O1, l1 = oracle.attention_masked_forward(q, k, v, s, False, None, None, None, rowc)
    np.testing.assert_allclose(O1, O0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l0 + rowc[..., 0], rtol=0, atol=1e-12)


def test_additive_mask_backward_finite_differences():
    B, H, Hkv, Nq, Nk, d, s, h = 1, 2, 1, 4, 6, 3, 0.6, 1e-6
    q, k, v, do = _qkv(B, H, Hkv, Nq, Nk, d, 610)
    bias = _random_bias((1, H, Nq, Nk), 611, 0.15)
    grads = oracle.attention_masked_backward(q, k, v, do, s, False, None, None, None, bias)

    def loss(q_, k_, v_):
        O, _ = oracle.attention_masked_forward(q_, k_, v_, s, False, None, None, None, bias)
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


def test_planted_bias_sign_error_is_caught():
    # Subtracting the bias instead of adding it: the brute-force pin sees it.
    Nq = Nk = 8
    q, k, v, _ = _qkv(1, 1, 1, Nq, Nk, 4, 620)
    bias = np.random.default_rng(621).uniform(-2, 2, (1, 1, Nq, Nk))
    wrong, _ = oracle.attention_masked_forward(q, k, v, 0.5, False, None, None, None, -bias)
    i = 3
    o, _ = brute_row_bias(q[0, 0, i], k[0, 0], v[0, 0], list(range(Nk)), 0.5, bias[0, 0, i])
    assert np.abs(wrong[0, 0, i] - o).max() > 1e-3
