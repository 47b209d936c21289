"""GPU parity of attn_bwd_cross (Nq query rows against Nk key rows, causal
rows at positions Nk - Nq + i) against the fp64 oracle, through the C ABI.

The backward consumes the GPU's own attn_fwd_cross O and lse, as a training
step does; the reference is the oracle's analytic gradient with its own fp64
P, so forward and backward errors are both inside the comparison."""
import math

import numpy as np
import pytest

import oracle
from sdpa_inputs import make_random
from tests.parity import check_grads, check_same_but_rounding, dev, host

pytestmark = pytest.mark.gpu

SHAPES = [
    # B, H, Hkv, Nq, Nk, d
    (1, 2, 2, 128, 384, 64),     # tile-aligned chunk against a longer cache
    (1, 4, 2, 200, 1000, 128),   # ragged both ways, GQA
    (2, 2, 1, 300, 301, 96),     # offset of one key
    (1, 4, 4, 64, 2048, 128),    # short chunk, long cache (one query tile)
    (1, 2, 2, 513, 777, 128),    # odd offset 264
    (1, 2, 1, 100, 1000, 64),    # offset 900: every key tile but the last fully visible
]


def _problem(shape, seed):
    B, H, Hkv, Nq, Nk, d = shape
    return (make_random((B, H, Nq, d), seed), make_random((B, Hkv, Nk, d), seed + 1),
            make_random((B, Hkv, Nk, d), seed + 2), make_random((B, H, Nq, d), seed + 3))


def _run(lib, q, k, v, do, s, causal):
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    O, lse = lib.forward_cross(tq, tk, tv, s, causal)
    grads = lib.backward_cross(tq, tk, tv, O, lse, tdo, s, causal)
    assert lib.attn_get_device_status(None) == lib.Status.OK
    return [host(g) for g in grads]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dH%dKV%dQ%dK%dd%d" % s)
def test_bwd_cross_matches_oracle(cuda_lib, shape, causal):
    d = shape[-1]
    q, k, v, do = _problem(shape, 16000 + shape[3] + shape[4])
    s = 1 / math.sqrt(d)
    grads = _run(cuda_lib, q, k, v, do, s, causal)
    ref = oracle.attention_cross_backward(q, k, v, do, s, causal)
    check_grads(grads, ref, f"{shape} causal={causal}")


def test_bwd_cross_more_queries_than_keys(cuda_lib):
    shape = (1, 2, 1, 700, 150, 64)
    q, k, v, do = _problem(shape, 17001)
    grads = _run(cuda_lib, q, k, v, do, 0.125, False)
    ref = oracle.attention_cross_backward(q, k, v, do, 0.125, False)
    check_grads(grads, ref, "Nq > Nk")


def test_bwd_cross_with_equal_lengths_is_the_backward(cuda_lib):
    B, H, Hkv, N, d = 1, 4, 2, 333, 128
    q, k, v, do = (dev(x) for x in _problem((B, H, Hkv, N, N, d), 18001))
    for causal in (False, True):
        O, lse = cuda_lib.forward(q, k, v, 0.09, causal)
        a = cuda_lib.backward_cross(q, k, v, O, lse, do, 0.09, causal)
        b = cuda_lib.backward(q, k, v, O, lse, do, 0.09, causal)
        for x, y in zip(a, b):
            assert np.array_equal(host(x), host(y))


def test_bwd_cross_is_deterministic(cuda_lib):
    q, k, v, do = (dev(x) for x in _problem((1, 4, 2, 257, 1100, 128), 19001))
    O, lse = cuda_lib.forward_cross(q, k, v, 0.1, True)
    a = [host(g) for g in cuda_lib.backward_cross(q, k, v, O, lse, do, 0.1, True)]
    b = [host(g) for g in cuda_lib.backward_cross(q, k, v, O, lse, do, 0.1, True)]
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_bwd_cross_chunk_keys_checked_on_their_own(cuda_lib):
    # Causal chunk of 128 rows at the end of 1024 keys: keys 0..895 are seen
    # by every query row, keys 896..1023 only by part of the chunk (the
    # masked triangle).  Each key range is compared on its own, so an error
    # confined to the masked tile is not hidden in the norm of the bulk.
    shape = (1, 2, 2, 128, 1024, 128)
    q, k, v, do = _problem(shape, 20001)
    s = 1 / math.sqrt(128)
    dq, dk, dv = _run(cuda_lib, q, k, v, do, s, True)
    rq, rk, rv = oracle.attention_cross_backward(q, k, v, do, s, True)
    check_grads([dq, dk[:, :, :896], dv[:, :, :896]], [rq, rk[:, :, :896], rv[:, :, :896]], "before chunk")
    check_grads([dq, dk[:, :, 896:], dv[:, :, 896:]], [rq, rk[:, :, 896:], rv[:, :, 896:]], "inside chunk")


def test_bwd_cross_stages_equal_the_combined_call(cuda_lib):
    import torch
    B, H, Hkv, Nq, Nk, d = 1, 4, 2, 300, 700, 128
    q, k, v, do = (dev(x) for x in _problem((B, H, Hkv, Nq, Nk, d), 21001))
    s = 1 / math.sqrt(d)
    for causal in (False, True):
        O, lse = cuda_lib.forward_cross(q, k, v, s, causal)
        want = [host(g) for g in cuda_lib.backward_cross(q, k, v, O, lse, do, s, causal)]
        ws_bytes = cuda_lib.attn_bwd_workspace_size(B, H, Hkv, Nq, d)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        sp = torch.cuda.current_stream().cuda_stream
        # dQ with the row vectors, then dK / dV: the combined call, bit for bit
        assert cuda_lib.attn_bwd_dq_rows(q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(), lse.data_ptr(),
                                         do.data_ptr(), dq.data_ptr(), ws.data_ptr(), ws_bytes, B, H, Hkv, Nq, Nk,
                                         d, s, causal, sp) == 0
        assert cuda_lib.attn_bwd_grad_cross(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(), dk.data_ptr(),
                                            dv.data_ptr(), ws.data_ptr(), ws_bytes, B, H, Hkv, Nq, Nk, d, s,
                                            causal, sp) == 0
        for got, w in zip((dq, dk, dv), want):
            assert np.array_equal(host(got), w)
        # prep, grad, dq: the same up to the order of D's additions
        assert cuda_lib.attn_bwd_prep(O.data_ptr(), lse.data_ptr(), do.data_ptr(), ws.data_ptr(), ws_bytes,
                                      B, H, Hkv, Nq, d, sp) == 0
        assert cuda_lib.attn_bwd_grad_cross(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(), dk.data_ptr(),
                                            dv.data_ptr(), ws.data_ptr(), ws_bytes, B, H, Hkv, Nq, Nk, d, s,
                                            causal, sp) == 0
        assert cuda_lib.attn_bwd_dq_cross(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(), dq.data_ptr(),
                                          ws.data_ptr(), ws_bytes, B, H, Hkv, Nq, Nk, d, s, causal, sp) == 0
        check_same_but_rounding([host(g) for g in (dq, dk, dv)], want, f"cross stages causal={causal}")
