"""GPU parity of attn_decode (KV-cache decode, split over the keys) against
the fp64 oracle's attention_decode, through the C ABI."""
import math

import numpy as np
import pytest

import oracle
from sdpa_inputs import make_random
from tests.parity import LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS, dev, host

pytestmark = pytest.mark.gpu


def _run(lib, B, H, Hkv, Nq, Nk, d, causal, seed, scale=None):
    q = make_random((B, H, Nq, d), seed)
    k = make_random((B, Hkv, Nk, d), seed + 1)
    v = make_random((B, Hkv, Nk, d), seed + 2)
    s = scale if scale is not None else 1 / math.sqrt(d)
    O, lse = lib.decode(dev(q), dev(k), dev(v), s, causal)
    assert lib.attn_get_device_status(None) == lib.Status.OK
    Or, lr = oracle.attention_decode(q, k, v, s, causal)
    return host(O), host(lse), Or, lr


def _check(O, lse, Or, lr, what):
    err = np.abs(O - Or)
    assert err.max() <= O_MAX_ABS and err.mean() <= O_MEAN_ABS, (what, err.max(), err.mean())
    fin = np.isfinite(lr)
    assert np.array_equal(np.isfinite(lse), fin), what
    assert np.abs(lse[fin] - lr[fin]).max() <= LSE_MAX_ABS, (what, np.abs(lse[fin] - lr[fin]).max())


SHAPES = [
    # B, H, Hkv, Nq, Nk, d
    (1, 1, 1, 1, 1, 64),        # one key
    (2, 8, 8, 1, 300, 128),     # MHA decode, ragged last tile
    (1, 32, 8, 1, 4096, 128),   # GQA 4:1
    (2, 16, 2, 4, 1000, 96),    # G*Nq = 32 rows, speculative block of 4
    (1, 64, 8, 8, 777, 64),     # G*Nq = 64 rows
    (1, 64, 4, 8, 1500, 128),   # G*Nq = 128 rows (the limit)
    (3, 4, 1, 3, 129, 128),     # MQA, one key past a tile
    (1, 8, 4, 2, 5000, 128),    # many chunks
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dH%dKV%dQ%dK%dd%d" % s)
def test_decode_matches_oracle(cuda_lib, shape, causal):
    B, H, Hkv, Nq, Nk, d = shape
    O, lse, Or, lr = _run(cuda_lib, B, H, Hkv, Nq, Nk, d, causal, 9000 + Nk + d)
    _check(O, lse, Or, lr, (shape, causal))


def test_decode_equal_lengths_causal_matches_forward(cuda_lib):
    # With Nq = Nk the decode alignment is the ordinary causal mask: decode
    # equals the forward kernel's result within the output tolerances.
    B, H, Hkv, N, d = 1, 4, 2, 60, 64     # G * Nq = 120 rows: within the 128-row limit
    q = dev(make_random((B, H, N, d), 301))
    k = dev(make_random((B, Hkv, N, d), 302))
    v = dev(make_random((B, Hkv, N, d), 303))
    Od, ld = cuda_lib.decode(q, k, v, 0.2, True)
    Of, lf = cuda_lib.forward(q, k, v, 0.2, True)
    assert np.abs(host(Od) - host(Of)).max() <= 2 * O_MAX_ABS
    assert np.abs(host(ld) - host(lf)).max() <= 2 * LSE_MAX_ABS


def test_decode_dominant_key_returns_its_value_row(cuda_lib):
    # One key aligned with the query and large scores: O is that key's V row
    # (the dominant-logit case of the pages' softmax), across chunk borders.
    import torch
    B, H, Hkv, Nq, Nk, d = 1, 2, 1, 1, 2000, 64
    rng = np.random.default_rng(7)
    k = rng.standard_normal((B, Hkv, Nk, d)).astype(np.float32) * 0.01
    hot = 1500
    k[0, 0, hot] = 1.0
    q = np.ones((B, H, Nq, d), dtype=np.float32)
    v = rng.standard_normal((B, Hkv, Nk, d)).astype(np.float32)
    O, lse = cuda_lib.decode(dev(q), dev(k), dev(v), 1.0, False)
    want = host(dev(v))[0, 0, hot]
    np.testing.assert_allclose(host(O)[0, 0, 0], want, atol=1e-2)
    np.testing.assert_allclose(host(O)[0, 1, 0], want, atol=1e-2)


def test_decode_workspace_and_outputs_stay_inside_buffers(cuda_lib):
    import torch
    B, H, Hkv, Nq, Nk, d = 1, 8, 2, 2, 700, 128
    q = dev(make_random((B, H, Nq, d), 401))
    k = dev(make_random((B, Hkv, Nk, d), 402))
    v = dev(make_random((B, Hkv, Nk, d), 403))
    pad = 4096
    ws_bytes = cuda_lib.attn_decode_workspace_size(B, H, Hkv, Nq, Nk, d)
    wsb = torch.full((ws_bytes + 2 * pad,), 0x5A, dtype=torch.uint8, device="cuda")
    ob = torch.full((q.numel() + 2 * pad,), -7.0, dtype=torch.bfloat16, device="cuda")
    lb = torch.full((B * H * Nq + 2 * pad,), -7.0, dtype=torch.float32, device="cuda")
    o = ob[pad:pad + q.numel()].view(q.shape)
    l = lb[pad:pad + B * H * Nq].view(B, H, Nq)
    st = cuda_lib.attn_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(),
                              wsb.data_ptr() + pad, ws_bytes, B, H, Hkv, Nq, Nk, d, 0.1, 1, None)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.all(wsb[:pad] == 0x5A) and torch.all(wsb[-pad:] == 0x5A)
    assert torch.all(ob[:pad] == -7.0) and torch.all(ob[-pad:] == -7.0)
    assert torch.all(lb[:pad] == -7.0) and torch.all(lb[-pad:] == -7.0)
    Or, lr = oracle.attention_decode(host(q), host(k), host(v), 0.1, True)
    _check(host(o), host(l), Or, lr, "guarded")
