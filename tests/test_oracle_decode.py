"""Pins for the oracle's decode (KV-cache) definition and split merge.

The pages describe decode with a KV cache only in words (page "Flash
Attention原理", FAQ on inference: the cache spreads the work over decode
steps; prefill and decode are profiled separately).  What is pinned here:
  * the causal alignment reading (query t of an Nq-row block sits at position
    Nk - Nq + t) against the ordinary square causal problem and against
    torch's CPU float64 SDPA with an explicit mask;
  * the split merge (the two-block merge of §四 for any number of blocks)
    against full attention and against the page's two-block form.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import sdpa as osd
from sdpa_inputs import make_random


def _qkv(B, H, Hkv, Nq, Nk, d, seed):
    q = make_random((B, H, Nq, d), seed)
    k = make_random((B, Hkv, Nk, d), seed + 1)
    v = make_random((B, Hkv, Nk, d), seed + 2)
    return q, k, v


def test_single_query_causal_sees_every_cached_key():
    # One new token at the end of the sequence attends to the whole cache:
    # causal and non-causal agree.  (Top-left alignment would let it see key 0
    # only, which this pin rejects.)
    q, k, v = _qkv(2, 4, 2, 1, 37, 16, 11)
    Oc, lc = oracle.attention_decode(q, k, v, 0.3, causal=True)
    On, ln = oracle.attention_decode(q, k, v, 0.3, causal=False)
    np.testing.assert_allclose(Oc, On, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lc, ln, rtol=0, atol=1e-13)


@pytest.mark.parametrize("Nq", [1, 3, 8])
def test_decode_rows_equal_last_rows_of_square_causal_problem(Nq):
    # The new block continues a sequence whose first Nk - Nq queries are not
    # recomputed: its rows equal the last Nq rows of the ordinary causal
    # problem on Nk queries (whose mask is pinned in test_oracle.py).
    B, H, Hkv, Nk, d = 1, 4, 2, 29, 8
    q, k, v = _qkv(B, H, Hkv, Nq, Nk, d, 20 + Nq)
    prefix = make_random((B, H, Nk - Nq, d), 99)
    qfull = np.concatenate([prefix, q], axis=2)
    Of, lf = oracle.attention_forward(qfull, k, v, 0.4, causal=True)
    Od, ld = oracle.attention_decode(q, k, v, 0.4, causal=True)
    np.testing.assert_allclose(Od, Of[:, :, Nk - Nq:], rtol=0, atol=1e-13)
    np.testing.assert_allclose(ld, lf[:, :, Nk - Nq:], rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_decode_against_torch_with_explicit_mask(causal):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    B, H, Hkv, Nq, Nk, d = 2, 6, 2, 5, 41, 16
    q, k, v = _qkv(B, H, Hkv, Nq, Nk, d, 31)
    G = H // Hkv
    tq = torch.from_numpy(q.astype(np.float64))
    tk = torch.from_numpy(np.repeat(k.astype(np.float64), G, axis=1))
    tv = torch.from_numpy(np.repeat(v.astype(np.float64), G, axis=1))
    mask = None
    if causal:
        pos = torch.arange(Nq)[:, None] + (Nk - Nq)
        mask = torch.arange(Nk)[None, :] <= pos
    ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=0.25).numpy()
    O, _ = oracle.attention_decode(q, k, v, 0.25, causal)
    np.testing.assert_allclose(O, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("splits", [[5], [2, 3], [1, 1, 1, 2], [3, 7, 11, 2]])
def test_merge_of_splits_equals_full_attention(splits):
    # Attention over disjoint key ranges, merged by lse weights, is the
    # attention over all keys (closed form of the §四 merge).
    B, H, Hkv, Nq, d = 1, 2, 1, 4, 8
    Nk = sum(splits)
    q, k, v = _qkv(B, H, Hkv, Nq, Nk, d, 41)
    O_full, l_full = oracle.attention_forward(q, k, v, 0.5)
    Os, ls, lo = [], [], 0
    for n in splits:
        o_s, l_s = oracle.attention_forward(q, k[:, :, lo:lo + n], v[:, :, lo:lo + n], 0.5)
        Os.append(o_s)
        ls.append(l_s)
        lo += n
    O, l = oracle.merge_splits(Os, ls)
    np.testing.assert_allclose(O, O_full, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l, l_full, rtol=0, atol=1e-13)


def test_merge_of_two_splits_equals_page_two_block_form():
    # The page's two-block merge renormalises both halves of a score row with
    # the global max and sum; its probabilities times V equal the merge of
    # the two halves' attention outputs.
    rng = np.random.default_rng(5)
    x = rng.standard_normal(12)
    V = rng.standard_normal((12, 3))
    P = osd.softmax_two_block(x[None, :])[0]
    want = P @ V
    halves = []
    for part in (slice(0, 6), slice(6, 12)):
        p, m, l = osd.softmax_rows(x[None, part])
        halves.append(((p @ V[part])[0], (m + np.log(l))[0]))
    O, _ = oracle.merge_splits([h[0] for h in halves], [h[1] for h in halves])
    np.testing.assert_allclose(O, want, rtol=0, atol=1e-14)


def test_fully_masked_split_carries_no_weight():
    rng = np.random.default_rng(6)
    O1 = rng.standard_normal((3, 4))
    l1 = rng.standard_normal(3)
    O, l = oracle.merge_splits([O1, np.zeros((3, 4))], [l1, np.full(3, -np.inf)])
    np.testing.assert_allclose(O, O1, rtol=0, atol=0)
    np.testing.assert_allclose(l, l1, rtol=0, atol=0)
    # every split masked: lse = -inf and O = 0
    O, l = oracle.merge_splits([O1, O1], [np.full(3, -np.inf)] * 2)
    assert np.all(np.isneginf(l)) and np.all(O == 0)


def test_fully_masked_row_has_zero_output_and_minus_inf_lse():
    # A query whose position precedes every key (negative offset) sees no key.
    q, k, v = _qkv(1, 1, 1, 2, 3, 4, 51)
    O, l = oracle.attention_forward(q, k, v, 1.0, causal=True, q_offset=-1)
    assert np.isneginf(l[0, 0, 0]) and np.all(O[0, 0, 0] == 0)
    assert np.isfinite(l[0, 0, 1])


def test_planted_merge_mistake_is_caught():
    # Dropping the lse weights (plain average of the split outputs) must fail
    # the merge pin.
    B, H, Hkv, Nq, d = 1, 1, 1, 2, 4
    q, k, v = _qkv(B, H, Hkv, Nq, 9, d, 61)
    O_full, _ = oracle.attention_forward(q, k, v, 0.7)
    parts = [oracle.attention_forward(q, k[:, :, a:b], v[:, :, a:b], 0.7) for a, b in ((0, 4), (4, 9))]
    wrong = (parts[0][0] + parts[1][0]) / 2
    assert np.abs(wrong - O_full).max() > 1e-3
    right, _ = oracle.merge_splits([p[0] for p in parts], [p[1] for p in parts])
    assert np.abs(right - O_full).max() < 1e-13


# ----------------------------------------------------------------- paged cache
def _paged(k, v, page_size, order, max_pages):
    """Store contiguous (B, Hkv, N, d) K / V into a page pool: logical page i
    of batch element b goes to physical page order[b * max_pages + i]."""
    B, Hkv, N, d = k.shape
    num_pages = B * max_pages
    kc = np.zeros((num_pages, page_size, Hkv, d))
    vc = np.zeros((num_pages, page_size, Hkv, d))
    table = np.full((B, max_pages), -1, dtype=np.int64)
    for b in range(B):
        for i in range(-(-N // page_size)):
            phys = order[b * max_pages + i]
            table[b, i] = phys
            seg = slice(i * page_size, min(N, (i + 1) * page_size))
            n = seg.stop - seg.start
            kc[phys, :n] = k[b, :, seg].transpose(1, 0, 2)
            vc[phys, :n] = v[b, :, seg].transpose(1, 0, 2)
    return kc, vc, table


@pytest.mark.parametrize("page_size", [4, 16])
@pytest.mark.parametrize("causal", [False, True])
def test_paged_decode_equals_contiguous_decode(page_size, causal):
    B, H, Hkv, Nq, N, d = 3, 4, 2, 2, 37, 8
    q, k, v = _qkv(B, H, Hkv, Nq, N, d, 70)
    max_pages = -(-N // page_size) + 2
    order = np.random.default_rng(71).permutation(B * max_pages)   # pages scattered over the pool
    kc, vc, table = _paged(k, v, page_size, order, max_pages)
    lens = np.array([N, 23, 5])
    O, lse = oracle.attention_decode_paged(q, kc, vc, table, lens, 0.3, causal)
    for b in range(B):
        L = lens[b]
        Or, lr = oracle.attention_decode(q[b:b + 1], k[b:b + 1, :, :L], v[b:b + 1, :, :L], 0.3, causal)
        np.testing.assert_allclose(O[b], Or[0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[b], lr[0], rtol=0, atol=1e-13)


def test_planted_page_order_mistake_is_caught():
    # Reading logical page i from physical page i (ignoring the table) is a
    # plausible mistake; with scattered pages and a ragged, causal block (so
    # that the order decides which keys each query sees) it changes the
    # result.  (Without a mask the key order would not matter.)
    B, H, Hkv, Nq, N, d, ps = 1, 2, 1, 4, 30, 4, 8
    q, k, v = _qkv(B, H, Hkv, Nq, N, d, 80)
    order = np.array([3, 0, 2, 1])
    kc, vc, table = _paged(k, v, ps, order, 4)
    right, _ = oracle.attention_decode_paged(q, kc, vc, table, [N], 0.5, True)
    wrong, _ = oracle.attention_decode_paged(q, kc, vc, np.arange(4)[None], [N], 0.5, True)
    ref, _ = oracle.attention_decode(q, k, v, 0.5, True)
    assert np.abs(right - ref).max() < 1e-13 and np.abs(wrong - ref).max() > 1e-3
