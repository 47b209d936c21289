"""GPU parity of the packed variable-length path (attn_fwd_varlen /
attn_bwd_varlen through the C ABI) against the fp64 oracle, on seeded bf16
inputs.  The backward consumes the GPU forward's O and lse."""
import math

import numpy as np
import pytest

import oracle
from sdpa_inputs import make_random
from tests.parity import GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS, check_grads, check_same_but_rounding, dev, host, rel_fro

pytestmark = pytest.mark.gpu


def _packed(lq, lk, H, Hkv, d, seed):
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    q = make_random((int(cu_q[-1]), H, d), seed)
    k = make_random((int(cu_k[-1]), Hkv, d), seed + 1)
    v = make_random((int(cu_k[-1]), Hkv, d), seed + 2)
    do = make_random((int(cu_q[-1]), H, d), seed + 3)
    return q, k, v, do, cu_q, cu_k


def _cu(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _run(lib, lq, lk, H, Hkv, d, causal, seed, grads=True):
    q, k, v, do, cu_q, cu_k = _packed(lq, lk, H, Hkv, d, seed)
    s = 1 / math.sqrt(d)
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    cq, ck = _cu(cu_q), _cu(cu_k)
    mq, mk = max(max(lq), 1), max(max(lk), 1)
    O, lse = lib.forward_varlen(tq, tk, tv, cq, ck, mq, mk, s, causal)
    out = {"O": host(O), "lse": host(lse)}
    if grads:
        g = lib.backward_varlen(tq, tk, tv, O, lse, tdo, cq, ck, mq, mk, s, causal)
        out["grads"] = [host(x) for x in g]
    assert lib.attn_get_device_status(None) == lib.Status.OK
    return (q, k, v, do, cu_q, cu_k, s), out


def _check_forward(O, lse, Or, lr, what):
    live = np.isfinite(lr)                      # (H, total_q)
    assert np.all(np.isneginf(lse[~live])), what
    rows_dead = ~live.T                         # (total_q, H)
    assert np.all(O[rows_dead] == 0), what
    err = np.abs(O[~rows_dead] - Or[~rows_dead])
    assert err.max() <= O_MAX_ABS and err.mean() <= O_MEAN_ABS, f"{what}: O err {err.max():.3e} / {err.mean():.3e}"
    assert np.abs(lse[live] - lr[live]).max() <= LSE_MAX_ABS, what


CASES = [
    # lengths of the query and key sequences, heads, kv heads, d
    ([300, 17, 128, 1000, 1], None, 4, 2, 128),          # self-attention packing (lk = lq)
    ([129, 256, 5], None, 2, 2, 64),
    ([200, 77, 384], None, 6, 3, 96),
    ([100, 257, 0, 64], [400, 250, 33, 0], 4, 2, 128),   # cross lengths, empty sequences, Nq_b > Nk_b
    ([4097, 129], [4097, 1000], 2, 1, 128),              # a long sequence; tiles beyond a short one
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "q%s_k%s_H%d_KV%d_d%d" % (
    "-".join(map(str, c[0])), "-".join(map(str, c[1] or c[0])), c[2], c[3], c[4]))
def test_varlen_matches_oracle(cuda_lib, case, causal):
    lq, lk, H, Hkv, d = case
    lk = lk or lq
    (q, k, v, do, cu_q, cu_k, s), out = _run(cuda_lib, lq, lk, H, Hkv, d, causal, 30000 + sum(lq) + d)
    Or, lr = oracle.attention_varlen_forward(q, k, v, cu_q, cu_k, s, causal)
    _check_forward(out["O"], out["lse"], Or, lr, f"{case} causal={causal}")
    ref = oracle.attention_varlen_backward(q, k, v, do, cu_q, cu_k, s, causal)
    check_grads(out["grads"], ref, f"{case} causal={causal}")
    # keys of an empty query sequence, rows that see no key: exact zeros
    for b in range(len(lq)):
        if lq[b] == 0:
            assert np.all(out["grads"][1][cu_k[b]:cu_k[b + 1]] == 0)
            assert np.all(out["grads"][2][cu_k[b]:cu_k[b + 1]] == 0)


def test_many_short_sequences(cuda_lib):
    rng = np.random.default_rng(31)
    lq = [int(x) for x in rng.integers(1, 60, size=40)]
    (q, k, v, do, cu_q, cu_k, s), out = _run(cuda_lib, lq, lq, 4, 1, 128, True, 31001)
    Or, lr = oracle.attention_varlen_forward(q, k, v, cu_q, cu_k, s, True)
    _check_forward(out["O"], out["lse"], Or, lr, "many short")
    ref = oracle.attention_varlen_backward(q, k, v, do, cu_q, cu_k, s, True)
    check_grads(out["grads"], ref, "many short")


def test_equal_lengths_equal_the_dense_batch(cuda_lib):
    # B sequences of one length: the packed path and the dense (B, H, N, d)
    # path run the same tiles, so the results agree bit for bit.
    B, H, Hkv, N, d = 3, 4, 2, 333, 128
    q4, k4, v4, do4 = (make_random(sh, 32000 + i) for i, sh in
                       enumerate([(B, H, N, d), (B, Hkv, N, d), (B, Hkv, N, d), (B, H, N, d)]))
    pack = lambda x: np.ascontiguousarray(x.transpose(0, 2, 1, 3).reshape(B * N, x.shape[1], d))
    cu = _cu(np.arange(B + 1) * N)
    for causal in (False, True):
        Od, ld = cuda_lib.forward(dev(q4), dev(k4), dev(v4), 0.1, causal)
        gd = cuda_lib.backward(dev(q4), dev(k4), dev(v4), Od, ld, dev(do4), 0.1, causal)
        tq, tk, tv, tdo = dev(pack(q4)), dev(pack(k4)), dev(pack(v4)), dev(pack(do4))
        Op, lp = cuda_lib.forward_varlen(tq, tk, tv, cu, cu, N, N, 0.1, causal)
        gp = cuda_lib.backward_varlen(tq, tk, tv, Op, lp, tdo, cu, cu, N, N, 0.1, causal)
        assert np.array_equal(host(Op), pack(host(Od)))
        assert np.array_equal(host(lp), host(ld).transpose(1, 0, 2).reshape(H, B * N))
        for a, b in zip(gp, gd):
            assert np.array_equal(host(a), pack(host(b)))


def test_varlen_backward_is_deterministic(cuda_lib):
    lq = [500, 3, 260]
    a = _run(cuda_lib, lq, lq, 4, 2, 128, True, 33001)[1]["grads"]
    b = _run(cuda_lib, lq, lq, 4, 2, 128, True, 33001)[1]["grads"]
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_packed_neighbours_are_not_overwritten(cuda_lib):
    # Partial last tiles are stored row by row: the rows of the following
    # sequence keep the values their own CTAs wrote, whatever the order.
    lq = [130, 126, 131]
    (q, k, v, do, cu_q, cu_k, s), out = _run(cuda_lib, lq, lq, 2, 2, 64, False, 34001)
    Or, _ = oracle.attention_varlen_forward(q, k, v, cu_q, cu_k, s, False)
    for b in range(3):
        sl = slice(cu_q[b], cu_q[b + 1])
        assert np.abs(out["O"][sl] - Or[sl]).max() <= O_MAX_ABS
    ref = oracle.attention_varlen_backward(q, k, v, do, cu_q, cu_k, s, False)
    for b in range(3):
        sl = slice(cu_q[b], cu_q[b + 1])
        for g, r in zip(out["grads"], ref):
            assert rel_fro(g[sl], r[sl]) <= GRAD_REL_FRO


def test_inconsistent_offsets_are_reported(cuda_lib):
    # Offsets that decrease, or a sequence longer than the stated maximum,
    # are caught by the kernels' own checks: nothing is read or written for
    # that sequence and the device status says ATTN_ERR_INVALID_ARG.
    H, d = 2, 64
    q = dev(make_random((100, H, d), 35001))
    k = dev(make_random((100, H, d), 35002))
    v = dev(make_random((100, H, d), 35003))
    for cu, mx in (([0, 60, 40, 100], 60), ([0, 70, 100], 50)):
        c = _cu(np.array(cu))
        cuda_lib.forward_varlen(q, k, v, c, c, mx, mx, 0.125, False)
        assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.INVALID_ARG
    # the status word is cleared by the read
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK


def test_varlen_stages_equal_the_combined_call(cuda_lib):
    import torch
    lq = [300, 17, 700]
    H, Hkv, d = 4, 2, 128
    q, k, v, do, cu_q, cu_k = _packed(lq, lq, H, Hkv, d, 36001)
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    cq = _cu(cu_q)
    O, lse = cuda_lib.forward_varlen(tq, tk, tv, cq, cq, 700, 700, 0.1, True)
    want = [host(g) for g in cuda_lib.backward_varlen(tq, tk, tv, O, lse, tdo, cq, cq, 700, 700, 0.1, True)]
    ws_bytes = cuda_lib.attn_bwd_varlen_workspace_size(3, H, Hkv, int(cu_q[-1]), d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(tq), torch.empty_like(tk), torch.empty_like(tv)
    sp = torch.cuda.current_stream().cuda_stream
    P = lambda t: t.data_ptr()
    # 8 then 2 (dQ with the row vectors, then dK / dV) is the combined call
    # bit for bit; 1, 2, 4 (separate prep) differs only in D's rounding.
    for order in ((8, 2), (1, 2, 4)):
        for stages in order:
            assert cuda_lib.attn_bwd_varlen_stages(P(tq), P(tk), P(tv), P(O), P(lse), P(tdo), P(dq), P(dk), P(dv),
                                                   P(cq), P(cq), P(ws), ws_bytes, 3, H, Hkv, int(cu_q[-1]),
                                                   int(cu_q[-1]), 700, 700, d, 0.1, 1, stages, sp) == 0
        got = [host(g) for g in (dq, dk, dv)]
        if order == (8, 2):
            for g, w in zip(got, want):
                assert np.array_equal(g, w)
        else:
            check_same_but_rounding(got, want, "varlen stages 1, 2, 4")
    for bad in (0, 16, 17):
        assert cuda_lib.attn_bwd_varlen_stages(P(tq), P(tk), P(tv), P(O), P(lse), P(tdo), P(dq), P(dk), P(dv),
                                               P(cq), P(cq), P(ws), ws_bytes, 3, H, Hkv, int(cu_q[-1]),
                                               int(cu_q[-1]), 700, 700, d, 0.1, 1, bad, sp) == cuda_lib.Status.INVALID_ARG
