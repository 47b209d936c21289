"""Pins for the CPU fp64 oracle (no GPU).

Each test checks the oracle against something other than itself: a closed
form, an invariant of exact softmax attention, brute-force finite
differences, the two-block merge identity of the "Flash Attention原理" page
(§四), the byte figures that page prints (§一, §三, §六), or an independent
library implementation (torch's CPU float64 scaled_dot_product_attention and
autograd).  ``test_planted_mistakes_are_caught`` plants plausible mistakes in
copies of the oracle and checks that the pins reject each of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import sdpa as osd
from sdpa_inputs import make_inputs, make_random, round_bf16, workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed, amp=1.0):
    return make_random(shape, seed, amp).astype(np.float64)


# --------------------------------------------------------------- softmax
def test_softmax_rows_sum_to_one():
    S = rnd((5, 33, 47), 11, 3.0)
    S[:, :, 40:] = -np.inf  # masked keys
    P, m, l = oracle.softmax_rows(S)
    assert np.all(P[:, :, 40:] == 0.0)
    np.testing.assert_allclose(P.sum(-1), 1.0, rtol=0, atol=1e-12)
    assert np.all(P >= 0)


def test_two_block_merge_fp64_exact():
    x = rnd((3, 17, 64), 12, 2.0)
    P, _, _ = oracle.softmax_rows(x)
    np.testing.assert_allclose(oracle.softmax_two_block(x), P, rtol=0, atol=1e-15)


def test_two_block_merge_page_check_fp32():
    # The page's own check (§四): x ~ 2*N(0,1) of shape (2, 512, 4096) in
    # float32; the two-block merge matches the direct softmax to ~1e-6.
    x = (np.random.default_rng(0).standard_normal((2, 512, 4096), dtype=np.float32) * 2).astype(np.float32)
    e = np.exp(x - x.max(-1, keepdims=True))
    direct = e / e.sum(-1, keepdims=True)
    merged = oracle.softmax_two_block(x)
    assert merged.dtype == np.float32
    assert np.abs(merged - direct).max() <= 1e-6


# --------------------------------------------------------------- forward pins
@pytest.mark.parametrize("causal", [False, True])
def test_uniform_v_gives_constant_rows(causal):
    B, H, N, d = 2, 3, 37, 16
    q, k = rnd((B, H, N, d), 1), rnd((B, H, N, d), 2)
    c = rnd((B, H, 1, d), 3)
    v = np.broadcast_to(c, (B, H, N, d)).copy()
    O, _ = oracle.attention_forward(q, k, v, 0.25, causal)
    np.testing.assert_allclose(O, np.broadcast_to(c, O.shape), rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_dominant_logit_returns_matching_v_row(causal):
    # q_i . k_j * scale = 2500 when j = perm^-1(i) and 0 otherwise: exp(-2500)
    # underflows in fp64, so P is exactly one-hot and O_i is exactly V_j.
    N = 12
    perm = np.arange(N) if causal else np.random.default_rng(5).permutation(N)
    q = np.zeros((1, 1, N, N))
    k = np.zeros((1, 1, N, N))
    q[0, 0, np.arange(N), np.arange(N)] = 50.0
    k[0, 0, np.arange(N), perm] = 50.0
    v = rnd((1, 1, N, 8), 6)
    O, lse = oracle.attention_forward(q, k, v, 1.0, causal)
    inv = np.argsort(perm)
    assert np.array_equal(O[0, 0], v[0, 0, inv])
    assert np.array_equal(lse[0, 0], np.full(N, 2500.0))


@pytest.mark.parametrize("d", [1, 7, 64])
def test_causal_row0_closed_form(d):
    q, k, v = rnd((2, 2, 9, d), 7), rnd((2, 2, 9, d), 8), rnd((2, 2, 9, d), 9)
    s = 0.3
    O, lse = oracle.attention_forward(q, k, v, s, True)
    np.testing.assert_array_equal(O[:, :, 0], v[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], s * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]), rtol=0, atol=1e-13)


def test_single_key_closed_form():
    q, k, v = rnd((3, 4, 1, 32), 10), rnd((3, 2, 1, 32), 11), rnd((3, 2, 1, 32), 12)
    O, lse = oracle.attention_forward(q, k, v, 0.5, False)
    kk = np.repeat(k, 2, axis=1)
    np.testing.assert_array_equal(O, np.repeat(v, 2, axis=1))
    np.testing.assert_allclose(lse, 0.5 * (q * kk).sum(-1), rtol=0, atol=1e-13)


def test_hand_worked_two_by_two():
    # N=2, d=1, scale=1: q=(1,0), k=(1,0), v=(2,4).
    # row 0 scores (1, 0): P = (e, 1)/(e+1); O = (2e+4)/(e+1); lse = ln(e+1)
    # row 1 scores (0, 0): P = (1/2, 1/2); O = 3; lse = ln 2
    e = math.e
    q = np.array([1.0, 0.0]).reshape(1, 1, 2, 1)
    k = np.array([1.0, 0.0]).reshape(1, 1, 2, 1)
    v = np.array([2.0, 4.0]).reshape(1, 1, 2, 1)
    O, lse = oracle.attention_forward(q, k, v, 1.0, False)
    np.testing.assert_allclose(O.ravel(), [(2 * e + 4) / (e + 1), 3.0], rtol=1e-15)
    np.testing.assert_allclose(lse.ravel(), [math.log(e + 1), math.log(2)], rtol=1e-15)
    # causal: row 0 sees key 0 only
    O, lse = oracle.attention_forward(q, k, v, 1.0, True)
    np.testing.assert_allclose(O.ravel(), [2.0, 3.0], rtol=1e-15)
    np.testing.assert_allclose(lse.ravel(), [1.0, math.log(2)], rtol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("block", [1, 7, 64, 200])
def test_online_recurrence_equals_two_pass(causal, block):
    q, k, v = rnd((1, 2, 200, 24), 13, 2.0), rnd((1, 2, 200, 24), 14, 2.0), rnd((1, 2, 200, 24), 15)
    O1, l1 = oracle.attention_forward(q, k, v, 0.4, causal)
    O2, l2 = oracle.attention_forward_online(q, k, v, 0.4, causal, block)
    np.testing.assert_allclose(O2, O1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance(causal):
    # K' = K + 1 u^T adds scale*q_i.u to every score of row i: P and O are
    # unchanged and lse shifts by scale*q_i.u.
    q, k, v = rnd((2, 2, 40, 16), 16), rnd((2, 2, 40, 16), 17), rnd((2, 2, 40, 16), 18)
    u = rnd((2, 2, 1, 16), 19)
    s = 0.25
    O1, l1 = oracle.attention_forward(q, k, v, s, causal)
    O2, l2 = oracle.attention_forward(q, k + u, v, s, causal)
    np.testing.assert_allclose(O2, O1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1 + s * (q * u).sum(-1), rtol=0, atol=1e-12)


def test_key_value_permutation_invariance():
    q, k, v = rnd((1, 3, 50, 8), 20), rnd((1, 3, 50, 8), 21), rnd((1, 3, 50, 8), 22)
    p = np.random.default_rng(23).permutation(50)
    O1, l1 = oracle.attention_forward(q, k, v, 0.3, False)
    O2, l2 = oracle.attention_forward(q, k[:, :, p], v[:, :, p], 0.3, False)
    np.testing.assert_allclose(O2, O1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_repeated_kv_heads(causal):
    B, H, Hkv, N, d = 2, 8, 2, 21, 8
    q, k, v, do = rnd((B, H, N, d), 24), rnd((B, Hkv, N, d), 25), rnd((B, Hkv, N, d), 26), rnd((B, H, N, d), 27)
    G = H // Hkv
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    O1, l1 = oracle.attention_forward(q, k, v, 0.3, causal)
    O2, l2 = oracle.attention_forward(q, kr, vr, 0.3, causal)
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-14)
    dq1, dk1, dv1 = oracle.attention_backward(q, k, v, do, 0.3, causal)
    dq2, dk2, dv2 = oracle.attention_backward(q, kr, vr, do, 0.3, causal)
    np.testing.assert_allclose(dq1, dq2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk1, dk2.reshape(B, Hkv, G, N, d).sum(2), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv1, dv2.reshape(B, Hkv, G, N, d).sum(2), rtol=0, atol=1e-13)
    assert [oracle.gqa_kv_head(h, 32, 8) for h in range(32)] == [h // 4 for h in range(32)]


def test_head_dim_padding_80_to_96():
    # Zero columns 80..95 of Q, K, V with scale 1/sqrt(80) reproduce the
    # unpadded d=80 result, and the padded output columns are exactly zero.
    q, k, v = rnd((1, 4, 33, 80), 28), rnd((1, 2, 33, 80), 29), rnd((1, 2, 33, 80), 30)
    pad = [(0, 0)] * 3 + [(0, 16)]
    s = 1 / math.sqrt(80)
    O80, l80 = oracle.attention_forward(q, k, v, s, True)
    O96, l96 = oracle.attention_forward(np.pad(q, pad), np.pad(k, pad), np.pad(v, pad), s, True)
    np.testing.assert_allclose(O96[..., :80], O80, rtol=0, atol=1e-14)
    assert np.all(O96[..., 80:] == 0.0)
    np.testing.assert_allclose(l96, l80, rtol=0, atol=1e-14)


def test_rows_variant_matches_full():
    q, k, v = rnd((1, 1, 70, 16), 31), rnd((1, 1, 70, 16), 32), rnd((1, 1, 70, 16), 33)
    for causal in (False, True):
        O, lse = oracle.attention_forward(q, k, v, 0.2, causal)
        rows = np.array([0, 5, 69, 33])
        Or, lr = oracle.attention_forward_rows(q[0, 0], k[0, 0], v[0, 0], rows, 0.2, causal)
        np.testing.assert_allclose(Or, O[0, 0, rows], rtol=0, atol=1e-14)
        np.testing.assert_allclose(lr, lse[0, 0, rows], rtol=0, atol=1e-14)
    # with the rows placed later in the key sequence (query i at position 30 + i)
    qs = q[:, :, :40]
    O, lse = oracle.attention_forward(qs, k, v, 0.2, True, q_offset=30)
    rows = np.array([0, 7, 39])
    Or, lr = oracle.attention_forward_rows(qs[0, 0], k[0, 0], v[0, 0], rows, 0.2, True, q_offset=30)
    np.testing.assert_allclose(Or, O[0, 0, rows], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lr, lse[0, 0, rows], rtol=0, atol=1e-14)


# --------------------------------------------------------------- backward pins
def _loss(q, k, v, do, s, causal):
    O, _ = oracle.attention_forward(q, k, v, s, causal)
    return float((O * do).sum())


@pytest.mark.parametrize("Hkv", [1, 2])
@pytest.mark.parametrize("N,d", [(5, 3), (9, 5)])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_finite_differences(Hkv, N, d, causal):
    B, H, s, h = 1, 2, 0.7, 1e-6
    q, k, v, do = rnd((B, H, N, d), 40), rnd((B, Hkv, N, d), 41), rnd((B, Hkv, N, d), 42), rnd((B, H, N, d), 43)
    grads = oracle.attention_backward(q, k, v, do, s, causal)
    for idx, (x, g) in enumerate(zip((q, k, v), grads)):
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


def test_backward_masked_entries_have_no_gradient():
    # With causal masking, key N-1 is seen only by query N-1: its dK and dV
    # come from that single row.
    q, k, v, do = rnd((1, 1, 6, 4), 44), rnd((1, 1, 6, 4), 45), rnd((1, 1, 6, 4), 46), rnd((1, 1, 6, 4), 47)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.5, True)
    S = 0.5 * q[0, 0] @ k[0, 0].T
    S[np.triu_indices(6, 1)] = -np.inf
    P, _, _ = oracle.softmax_rows(S)
    np.testing.assert_allclose(dv[0, 0, 5], P[5, 5] * do[0, 0, 5], rtol=1e-13)


# --------------------------------------------------------------- library cross-check
torch = pytest.importorskip("torch")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 2, 2, 64, 16), (2, 4, 1, 77, 32), (1, 3, 3, 130, 64)])
def test_against_torch_cpu_float64(causal, shape):
    import torch.nn.functional as F
    B, H, Hkv, N, d = shape
    q, k, v, do = rnd((B, H, N, d), 50), rnd((B, Hkv, N, d), 51), rnd((B, Hkv, N, d), 52), rnd((B, H, N, d), 53)
    s = 1 / math.sqrt(d)
    G = H // Hkv
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(np.repeat(k, G, axis=1), requires_grad=True)
    tv = torch.tensor(np.repeat(v, G, axis=1), requires_grad=True)
    to = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=s)
    to.backward(torch.tensor(do))
    O, _ = oracle.attention_forward(q, k, v, s, causal)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, s, causal)
    np.testing.assert_allclose(O, to.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy().reshape(B, Hkv, G, N, d).sum(2), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy().reshape(B, Hkv, G, N, d).sum(2), rtol=0, atol=1e-11)


# --------------------------------------------------------------- page figures
def test_page_byte_figures():
    with open(os.path.join(GOLDEN, "page_byte_figures.json")) as f:
        gold = {e["name"]: e for e in json.load(f)["entries"]}
    MiB, GiB, KiB = 2 ** 20, 2 ** 30, 2 ** 10
    S = oracle.score_matrix_bytes(4096)
    assert S / MiB == gold["S_fp32_one_head_n4096"]["printed"]
    assert S * 96 * 40 / GiB == gold["S_fp32_96heads_40layers_n4096"]["printed"]
    assert S * 96 / GiB >= gold["S_fp32_96heads_n4096"]["printed_at_least"]
    assert 2 * S / MiB == gold["S_plus_P_fp32_one_head_n4096"]["printed"]
    ml = oracle.row_stat_bytes(4096)
    assert ml / KiB == gold["m_plus_l_fp32_n4096"]["printed"]
    assert 2 * S / ml == gold["saving_ratio_n4096"]["printed"]
    assert oracle.score_matrix_bytes(64) / KiB == gold["local_S_fp32_block64"]["printed"]
    assert 3 * 4096 * 64 * 4 / MiB == gold["qkv_fp32_n4096_d64"]["printed"]


# --------------------------------------------------------------- inputs
def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(60).standard_normal(100000, dtype=np.float32) * 3
    x[:4] = [1.00390625, 1.01171875, -1.00390625, 0.0]  # exact ties and zero
    ours = round_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(ours, ref)


def test_workload_inputs_are_seeded_and_padded():
    w = workload("c4p", N=64, H=4, Hkv=2)
    a, b = make_inputs(w), make_inputs(w)
    assert all(np.array_equal(a[n], b[n]) for n in a)
    assert a["q"].shape == (1, 4, 64, 96)
    assert np.all(a["q"][..., 80:] == 0) and np.any(a["q"][..., :80] != 0)
    assert np.array_equal(round_bf16(a["k"]), a["k"])
    assert abs(w.softmax_scale - 1 / math.sqrt(80)) < 1e-15


# --------------------------------------------------------------- planted mistakes
def _mut_forward(kind):
    def fwd(q, k, v, scale=None, causal=False):
        q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
        B, H, N, d = q.shape
        Hkv = k.shape[1]
        scale = 1 / math.sqrt(d) if scale is None else scale
        O = np.empty((B, H, N, v.shape[3])); lse = np.empty((B, H, N))
        for b in range(B):
            for h in range(H):
                hk = (h % Hkv) if kind == "gqa_mod" else h // (H // Hkv)
                s = 1.0 if kind == "no_scale" else scale
                S = s * q[b, h] @ k[b, hk].T
                if causal:
                    tri = np.tril_indices(N, -1) if kind == "mask_flipped" else np.triu_indices(N, 1)
                    S[tri] = -np.inf
                m = S.max(1, keepdims=True)
                E = np.exp(S - m)
                l = E.sum(1, keepdims=True)
                if kind == "no_max_in_lse":
                    lse[b, h] = np.log(l[:, 0])
                else:
                    lse[b, h] = (m + np.log(l))[:, 0]
                P = E / l
                O[b, h] = (P.T @ v[b, hk]) if kind == "transposed_P" else P @ v[b, hk]
        return O, lse
    return fwd


@pytest.mark.parametrize("kind", ["no_scale", "mask_flipped", "gqa_mod", "no_max_in_lse", "transposed_P"])
def test_planted_mistakes_are_caught(kind):
    bad = _mut_forward(kind)
    B, H, Hkv, N, d = 1, 4, 2, 16, 8
    q, k, v = rnd((B, H, N, d), 70), rnd((B, Hkv, N, d), 71), rnd((B, Hkv, N, d), 72)
    good_O, good_l = oracle.attention_forward(q, k, v, 0.3, True)
    caught = []
    # causal row 0 closed form
    Ob, lb = bad(q, k, v, 0.3, True)
    kk = np.repeat(k, 2, axis=1)
    caught.append(not np.allclose(lb[:, :, 0], 0.3 * (q[:, :, 0] * kk[:, :, 0]).sum(-1)))
    caught.append(not np.allclose(Ob[:, :, 0], np.repeat(v, 2, axis=1)[:, :, 0]))
    # GQA against repeated heads
    Ob2, lb2 = bad(q, kk, np.repeat(v, 2, axis=1), 0.3, True)
    caught.append(not (np.allclose(Ob, Ob2) and np.allclose(lb, lb2)))
    # torch cross-check
    import torch.nn.functional as F
    ref = F.scaled_dot_product_attention(torch.tensor(q), torch.tensor(kk), torch.tensor(np.repeat(v, 2, axis=1)),
                                         is_causal=True, scale=0.3).numpy()
    caught.append(not np.allclose(Ob, ref))
    # key shift invariance of the lse
    u = rnd((B, Hkv, 1, d), 73)
    _, ls = bad(q, k + u, v, 0.3, True)
    uu = np.repeat(u, 2, axis=1)
    caught.append(not np.allclose(ls, lb + 0.3 * (q * uu).sum(-1)))
    assert any(caught), kind
    # and the real oracle passes the same checks
    assert np.allclose(good_O, ref)


def test_planted_backward_mistake_is_caught():
    # Dropping the rowsum term D from dS, or the scale from dK, fails the
    # finite-difference pin.
    q, k, v, do = rnd((1, 1, 5, 3), 80), rnd((1, 1, 5, 3), 81), rnd((1, 1, 5, 3), 82), rnd((1, 1, 5, 3), 83)
    s = 0.7
    S = s * q[0, 0] @ k[0, 0].T
    P, _, _ = oracle.softmax_rows(S)
    dP = do[0, 0] @ v[0, 0].T
    bad_dq = s * (P * dP) @ k[0, 0]          # D term dropped
    bad_dk = (P * (dP - (P * dP).sum(1, keepdims=True))).T @ q[0, 0]  # scale dropped
    h = 1e-6
    fd_q = np.zeros((5, 3)); fd_k = np.zeros((5, 3))
    for pos in np.ndindex(5, 3):
        for arr, fd, which in ((q, fd_q, 0), (k, fd_k, 1)):
            xp, xm = arr.copy(), arr.copy()
            xp[(0, 0) + pos] += h; xm[(0, 0) + pos] -= h
            a = [q, k, v]; a[which] = xp; lp = _loss(*a, do, s, False)
            a[which] = xm; lm = _loss(*a, do, s, False)
            fd[pos] = (lp - lm) / (2 * h)
    assert np.linalg.norm(bad_dq - fd_q) / np.linalg.norm(fd_q) > 1e-2
    assert np.linalg.norm(bad_dk - fd_k) / np.linalg.norm(fd_k) > 1e-2
    dq, dk, _ = oracle.attention_backward(q, k, v, do, s, False)
    assert np.linalg.norm(dq[0, 0] - fd_q) / np.linalg.norm(fd_q) < 1e-6
    assert np.linalg.norm(dk[0, 0] - fd_k) / np.linalg.norm(fd_k) < 1e-6
