"""GPU parity of attn_fwd_cross (Nq query rows against Nk key rows, causal
rows at positions Nk - Nq + i) against the fp64 oracle, through the C ABI."""
import math

import numpy as np
import pytest

import oracle
from sdpa_inputs import make_random
from tests.parity import check_o_lse, dev, host

pytestmark = pytest.mark.gpu

SHAPES = [
    # B, H, Hkv, Nq, Nk, d
    (1, 2, 2, 128, 384, 64),     # tile-aligned chunk against a longer cache
    (1, 4, 2, 200, 1000, 128),   # ragged both ways, GQA
    (2, 2, 1, 300, 301, 96),     # offset of one key
    (1, 8, 8, 64, 4096, 128),    # short chunk, long cache
    (1, 2, 2, 513, 777, 128),    # odd offset 264
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dH%dKV%dQ%dK%dd%d" % s)
def test_cross_matches_oracle(cuda_lib, shape, causal):
    B, H, Hkv, Nq, Nk, d = shape
    q = make_random((B, H, Nq, d), 12000 + Nq)
    k = make_random((B, Hkv, Nk, d), 12001 + Nk)
    v = make_random((B, Hkv, Nk, d), 12002 + d)
    s = 1 / math.sqrt(d)
    O, lse = cuda_lib.forward_cross(dev(q), dev(k), dev(v), s, causal)
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK
    Or, lr = oracle.attention_forward(q, k, v, s, causal, q_offset=(Nk - Nq) if causal else 0)
    check_o_lse(host(O), host(lse), Or, lr, (shape, causal))


def test_cross_non_causal_with_more_queries_than_keys(cuda_lib):
    B, H, Hkv, Nq, Nk, d = 1, 2, 1, 700, 150, 64
    q = make_random((B, H, Nq, d), 13001)
    k = make_random((B, Hkv, Nk, d), 13002)
    v = make_random((B, Hkv, Nk, d), 13003)
    O, lse = cuda_lib.forward_cross(dev(q), dev(k), dev(v), 0.125, False)
    Or, lr = oracle.attention_forward(q, k, v, 0.125, False)
    check_o_lse(host(O), host(lse), Or, lr, "Nq > Nk")


def test_cross_with_equal_lengths_is_the_forward(cuda_lib):
    B, H, Hkv, N, d = 1, 4, 2, 333, 128
    q = dev(make_random((B, H, N, d), 14001))
    k = dev(make_random((B, Hkv, N, d), 14002))
    v = dev(make_random((B, Hkv, N, d), 14003))
    for causal in (False, True):
        Oc, lc = cuda_lib.forward_cross(q, k, v, 0.09, causal)
        Of, lf = cuda_lib.forward(q, k, v, 0.09, causal)
        assert np.array_equal(host(Oc), host(Of)) and np.array_equal(host(lc), host(lf))


def test_cross_chunk_agrees_with_decode_path(cuda_lib):
    # A short causal chunk against a cache: the tiled forward and the decode
    # path (split over keys, merged) compute the same rows.
    B, H, Hkv, Nq, Nk, d = 1, 8, 2, 16, 2000, 128
    q = dev(make_random((B, H, Nq, d), 15001))
    k = dev(make_random((B, Hkv, Nk, d), 15002))
    v = dev(make_random((B, Hkv, Nk, d), 15003))
    Oc, lc = cuda_lib.forward_cross(q, k, v, 0.1, True)
    Od, ld = cuda_lib.decode(q, k, v, 0.1, True)
    assert np.abs(host(Oc) - host(Od)).max() <= 2e-2
    assert np.abs(host(lc) - host(ld)).max() <= 2e-3
