"""Pins for the oracle's cross-attention backward (Nq queries, Nk keys).

Page "SDPA backend 与 FlashAttention" (§3) lets the query and key sequences
have their own lengths; the causal reading used everywhere in this project
puts query row i at position Nk - Nq + i.  The backward of that problem is
pinned here against:
  * brute-force central differences of the oracle's own cross forward;
  * the ordinary square causal problem on Nk queries whose first Nk - Nq
    rows carry no output gradient (its last Nq rows are the cross problem);
  * torch's CPU float64 SDPA and autograd with an explicit mask.
A planted mistake (top-left alignment) is shown to fail the pins.
"""
import numpy as np
import pytest

import oracle
from sdpa_inputs import make_random


def rnd(shape, seed):
    return make_random(shape, seed).astype(np.float64)


def _problem(B, H, Hkv, Nq, Nk, d, seed):
    return (rnd((B, H, Nq, d), seed), rnd((B, Hkv, Nk, d), seed + 1), rnd((B, Hkv, Nk, d), seed + 2),
            rnd((B, H, Nq, d), seed + 3))


def _loss(q, k, v, do, s, causal):
    Nq, Nk = q.shape[2], k.shape[2]
    O, _ = oracle.attention_forward(q, k, v, s, causal, q_offset=Nk - Nq if causal else 0)
    return float((O * do).sum())


@pytest.mark.parametrize("Nq,Nk,causal", [(3, 7, True), (3, 7, False), (7, 3, False), (4, 4, True)])
def test_cross_backward_finite_differences(Nq, Nk, causal):
    B, H, Hkv, d, s, h = 1, 2, 1, 3, 0.6, 1e-6
    q, k, v, do = _problem(B, H, Hkv, Nq, Nk, d, 70 + Nq + Nk)
    grads = oracle.attention_cross_backward(q, k, v, do, s, causal)
    for idx, (x, g) in enumerate(zip((q, k, v), grads)):
        assert g.shape == x.shape
        fd = np.zeros_like(x)
        for pos in np.ndindex(x.shape):
            args = [q, k, v]
            xp, xm = x.copy(), x.copy()
            xp[pos] += h
            xm[pos] -= h
            args[idx] = xp
            lp = _loss(*args, do, s, causal)
            args[idx] = xm
            lm = _loss(*args, do, s, causal)
            fd[pos] = (lp - lm) / (2 * h)
        err = np.linalg.norm(fd - g) / np.linalg.norm(g)
        assert err <= 1e-6, (idx, err)


@pytest.mark.parametrize("Nq", [1, 5, 11])
def test_cross_backward_equals_square_problem_with_silent_prefix(Nq):
    # Queries 0 .. Nk-Nq-1 of the square causal problem receive dO = 0, so
    # they add nothing to dK and dV; the remaining rows are the cross problem.
    B, H, Hkv, Nk, d, s = 1, 4, 2, 13, 6, 0.45
    q, k, v, do = _problem(B, H, Hkv, Nq, Nk, d, 80 + Nq)
    prefix = rnd((B, H, Nk - Nq, d), 90)
    qf = np.concatenate([prefix, q], axis=2)
    dof = np.concatenate([np.zeros_like(prefix), do], axis=2)
    dqf, dkf, dvf = oracle.attention_backward(qf, k, v, dof, s, True)
    dq, dk, dv = oracle.attention_cross_backward(q, k, v, do, s, True)
    np.testing.assert_allclose(dq, dqf[:, :, Nk - Nq:], rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk, dkf, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv, dvf, rtol=0, atol=1e-13)
    # the silent prefix rows still have a (dO-free) dQ of zero
    assert np.all(dqf[:, :, :Nk - Nq] == 0)


@pytest.mark.parametrize("Nq,Nk,causal", [(9, 40, True), (9, 40, False), (33, 12, False)])
def test_cross_backward_against_torch(Nq, Nk, causal):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    B, H, Hkv, d, s = 2, 6, 3, 16, 0.25
    q, k, v, do = _problem(B, H, Hkv, Nq, Nk, d, 100)
    G = H // Hkv
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(np.repeat(k, G, axis=1), requires_grad=True)
    tv = torch.tensor(np.repeat(v, G, axis=1), requires_grad=True)
    mask = None
    if causal:
        mask = torch.arange(Nk)[None, :] <= torch.arange(Nq)[:, None] + (Nk - Nq)
    to = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=s)
    to.backward(torch.tensor(do))
    dq, dk, dv = oracle.attention_cross_backward(q, k, v, do, s, causal)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy().reshape(B, Hkv, G, Nk, d).sum(2), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy().reshape(B, Hkv, G, Nk, d).sum(2), rtol=0, atol=1e-11)


def test_causal_cross_needs_nq_at_most_nk():
    q, k, v, do = _problem(1, 1, 1, 5, 3, 4, 110)
    with pytest.raises(ValueError):
        oracle.attention_cross_backward(q, k, v, do, 0.5, True)


def test_planted_top_left_alignment_is_caught():
    # Aligning the causal mask top-left (query i sees keys 0..i) is a
    # plausible mistake; with Nq < Nk it leaves the last keys without any
    # gradient, which the square-problem pin above rules out.
    B, H, Hkv, Nq, Nk, d, s = 1, 2, 1, 4, 10, 5, 0.5
    q, k, v, do = _problem(B, H, Hkv, Nq, Nk, d, 120)
    _, dk_tl, dv_tl = oracle.attention_backward(q, k, v, do, s, True, q_offset=0)
    _, dk, dv = oracle.attention_cross_backward(q, k, v, do, s, True)
    assert np.all(dv_tl[:, :, Nq:] == 0) and np.all(dk_tl[:, :, Nq:] == 0)
    assert np.abs(dv[:, :, Nq:]).max() > 1e-3
    assert np.abs(dv_tl - dv).max() > 1e-3
