"""Full-size parity of the workloads bench.py times beyond the first path
(cross attention, packed varlen, masks, the additive mask, FP8, decode): each test makes the
same call on the same seeded inputs as the benchmark, then checks sampled
heads, sequences or query rows against the fp64 oracle, one by one."""
import math

import numpy as np
import pytest

import oracle
from sdpa_inputs import (e4m3_decode, make_inputs, make_varlen_inputs, prefix_lm_mask, quantize_e4m3,
                         varlen_lengths, workload)
from tests.parity import check_grads, check_o_lse, dev, host, sample_rows

pytestmark = pytest.mark.gpu


def _rows_check(O, lse, x, w, heads, q_offset, name, deq=None):
    G = w.H // w.Hkv
    got, ref = [], []
    for (b, h) in heads:
        rows = sample_rows(w.n_queries, seed=b * 1000 + h)
        qh = x["q"][b, h] if deq is None else deq[0][b, h]
        kh = x["k"][b, h // G] if deq is None else deq[1][b, h // G]
        vh = x["v"][b, h // G] if deq is None else deq[2][b, h // G]
        Or, lr = oracle.attention_forward_rows(qh, kh, vh, rows, w.softmax_scale, w.causal, q_offset=q_offset)
        got.append((O[b, h, rows], lse[b, h, rows]))
        ref.append((Or, lr))
    return (np.concatenate([g[0] for g in got]), np.concatenate([g[1] for g in got]),
            np.concatenate([r[0] for r in ref]), np.concatenate([r[1] for r in ref]))


def test_cp1_chunked_prefill(cuda_lib):
    w = workload("cp1")
    x = make_inputs(w)
    O, lse = cuda_lib.forward_cross(dev(x["q"]), dev(x["k"]), dev(x["v"]), w.softmax_scale, w.causal)
    O, lse = host(O), host(lse)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(lse))
    check_o_lse(*_rows_check(O, lse, x, w, [(0, 0), (0, 13), (0, 31)], w.N - w.n_queries, "cp1"), "cp1")


def test_cx_encoder_decoder_fwd_bwd(cuda_lib):
    w = workload("cx")
    x = make_inputs(w)
    s = w.softmax_scale
    tq, tk, tv, tdo = dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(x["do"])
    O, lse = cuda_lib.forward_cross(tq, tk, tv, s, False)
    grads = [host(g) for g in cuda_lib.backward_cross(tq, tk, tv, O, lse, tdo, s, False)]
    for (b, h) in [(0, 0), (5, 11)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        Or, lr = oracle.attention_forward(x["q"][sl], x["k"][sl], x["v"][sl], s, False)
        check_o_lse(host(O)[sl], host(lse)[sl], Or, lr, f"cx ({b},{h})")
        ref = oracle.attention_cross_backward(x["q"][sl], x["k"][sl], x["v"][sl], x["do"][sl], s, False)
        check_grads([g[sl] for g in grads], ref, f"cx ({b},{h})")


def test_vl1_packed_batch(cuda_lib):
    import torch
    w = workload("vl1")
    x = make_varlen_inputs(w)
    cu, lens = x["cu"], x["lengths"]
    tcu = torch.from_numpy(cu).cuda()
    s, mx = w.softmax_scale, int(lens.max())
    tq, tk, tv, tdo = dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(x["do"])
    O, lse = cuda_lib.forward_varlen(tq, tk, tv, tcu, tcu, mx, mx, s, True)
    grads = [host(g) for g in cuda_lib.backward_varlen(tq, tk, tv, O, lse, tdo, tcu, tcu, mx, mx, s, True)]
    O, lse = host(O), host(lse)
    # whole heads of the two shortest sequences, forward and backward
    for seq in np.argsort(lens)[:2]:
        a, e = int(cu[seq]), int(cu[seq + 1])
        for h in (0, 9):
            pk = lambda t: t[a:e, h:h + 1].transpose(1, 0, 2)[None]
            Or, lr = oracle.attention_forward(pk(x["q"]), pk(x["k"]), pk(x["v"]), s, True)
            check_o_lse(pk(O), lse[h:h + 1, a:e][None], Or, lr, f"vl1 seq {seq} head {h}")
            ref = oracle.attention_backward(pk(x["q"]), pk(x["k"]), pk(x["v"]), pk(x["do"]), s, True)
            check_grads([pk(g) for g in grads], ref, f"vl1 seq {seq} head {h}")
    # sampled rows of the longest sequence
    seq = int(np.argmax(lens))
    a, e = int(cu[seq]), int(cu[seq + 1])
    rows = sample_rows(e - a, seed=seq)
    got, ref = [], []
    for h in (3, 15):
        Or, lr = oracle.attention_forward_rows(x["q"][a:e, h], x["k"][a:e, h], x["v"][a:e, h], rows, s, True)
        got.append((O[a + rows, h], lse[h, a + rows]))
        ref.append((Or, lr))
    check_o_lse(np.concatenate([g[0] for g in got]), np.concatenate([g[1] for g in got]),
                np.concatenate([r[0] for r in ref]), np.concatenate([r[1] for r in ref]), "vl1 longest")


def test_sw1_sliding_window_rows(cuda_lib):
    w = workload("sw1")
    x = make_inputs(w)
    s, wl = w.softmax_scale, w.window[0]
    O, lse = cuda_lib.forward_masked(dev(x["q"]), dev(x["k"]), dev(x["v"]), s, True, w.window)
    O, lse = host(O), host(lse)
    G = w.H // w.Hkv
    # blocks of 128 query rows with the keys their windows reach: the masked
    # oracle on those slices aligns row r0 + i at key position r0 + i
    for (h, r0) in [(0, 0), (5, 4000), (17, 9000), (31, 16256)]:
        k0 = max(0, r0 - wl)
        sq = x["q"][:1, h:h + 1, r0:r0 + 128]
        sk = x["k"][:1, h // G:h // G + 1, k0:r0 + 128]
        sv = x["v"][:1, h // G:h // G + 1, k0:r0 + 128]
        Or, lr = oracle.attention_masked_forward(sq, sk, sv, s, True, w.window)
        check_o_lse(O[:1, h:h + 1, r0:r0 + 128], lse[:1, h:h + 1, r0:r0 + 128], Or, lr, f"sw1 ({h},{r0})")


def test_pl1_prefix_lm_fwd_bwd(cuda_lib):
    import torch
    w = workload("pl1")
    x = make_inputs(w)
    s = w.softmax_scale
    mask = prefix_lm_mask(w.N, w.prefix)
    tm = torch.from_numpy(mask.astype(np.uint8)).cuda()
    tq, tk, tv, tdo = dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(x["do"])
    O, lse = cuda_lib.forward_masked(tq, tk, tv, s, False, None, None, tm)
    grads = [host(g) for g in cuda_lib.backward_masked(tq, tk, tv, O, lse, tdo, s, False, None, None, tm)]
    for (b, h) in [(0, 0), (6, 13)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        Or, lr = oracle.attention_masked_forward(x["q"][sl], x["k"][sl], x["v"][sl], s, False, None, None, mask)
        check_o_lse(host(O)[sl], host(lse)[sl], Or, lr, f"pl1 ({b},{h})")
        ref = oracle.attention_masked_backward(x["q"][sl], x["k"][sl], x["v"][sl], x["do"][sl], s, False,
                                               None, None, mask)
        check_grads([g[sl] for g in grads], ref, f"pl1 ({b},{h})")


def test_ab1_additive_mask_fwd_bwd(cuda_lib):
    import torch
    from sdpa_inputs import distance_bias
    w = workload("ab1")
    x = make_inputs(w)
    s = w.softmax_scale
    bias = distance_bias(w.N, w.bias_slope)
    tb = torch.from_numpy(bias).cuda()
    tq, tk, tv, tdo = dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(x["do"])
    O, lse = cuda_lib.forward_masked(tq, tk, tv, s, False, None, None, None, tb)
    grads = [host(g) for g in cuda_lib.backward_masked(tq, tk, tv, O, lse, tdo, s, False, None, None, None, tb)]
    for (b, h) in [(0, 0), (7, 15)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        Or, lr = oracle.attention_masked_forward(x["q"][sl], x["k"][sl], x["v"][sl], s, False, None, None, None,
                                                 bias)
        check_o_lse(host(O)[sl], host(lse)[sl], Or, lr, f"ab1 ({b},{h})")
        ref = oracle.attention_masked_backward(x["q"][sl], x["k"][sl], x["v"][sl], x["do"][sl], s, False,
                                               None, None, None, bias)
        check_grads([g[sl] for g in grads], ref, f"ab1 ({b},{h})")


def test_c4f8_fp8_rows(cuda_lib):
    import torch
    from tests.fp8_model import FP8_MODEL_REL_FRO, O_MEAN_ABS_FP8, O_REL_FRO_FP8, p_rounding_model
    from tests.parity import LSE_MAX_ABS
    w = workload("c4f8")
    x = make_inputs(w)
    qz = [quantize_e4m3(x[n]) for n in ("q", "k", "v")]
    u8 = lambda a: torch.from_numpy(a).cuda()
    O, lse = cuda_lib.forward_fp8(u8(qz[0][0]), u8(qz[1][0]), u8(qz[2][0]), qz[0][1], qz[1][1], qz[2][1],
                                  w.softmax_scale, True)
    deq = [e4m3_decode(b) * sc for b, sc in qz]
    heads = [(0, 0), (0, 7), (0, 30)]
    O_s, l_s, O_r, l_r = _rows_check(host(O), host(lse), x, w, heads, 0, "c4f8", deq)
    O_m = np.concatenate([p_rounding_model(deq[0][b, h], deq[1][b, h // 4], deq[2][b, h // 4], w.softmax_scale, True,
                                           0, sample_rows(w.N, seed=b * 1000 + h)) for (b, h) in heads])
    assert np.linalg.norm(O_s - O_m) / np.linalg.norm(O_m) <= FP8_MODEL_REL_FRO
    assert np.linalg.norm(O_s - O_r) / np.linalg.norm(O_r) <= O_REL_FRO_FP8
    assert np.abs(O_s - O_r).mean() <= O_MEAN_ABS_FP8
    assert np.abs(l_s - l_r).max() <= LSE_MAX_ABS


@pytest.mark.parametrize("name", ["dec1", "dec4"])
def test_decode_full_size(cuda_lib, name):
    w = workload(name)
    x = make_inputs(w)
    O, lse = cuda_lib.decode(dev(x["q"]), dev(x["k"]), dev(x["v"]), w.softmax_scale, w.causal)
    for b in (0, 5):
        sl = slice(b, b + 1)
        Or, lr = oracle.attention_decode(x["q"][sl], x["k"][sl], x["v"][sl], w.softmax_scale, w.causal)
        check_o_lse(host(O)[sl], host(lse)[sl], Or, lr, f"{name} batch {b}")
