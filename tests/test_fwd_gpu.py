"""GPU parity of the forward pass (attn_fwd through the C ABI) against the
CPU fp64 oracle on the same seeded bf16 inputs: small and ragged shapes,
every element, and the invariants the oracle is pinned by.  The full-size
workloads are compared element by element in test_fullsize_gpu.py."""
import math

import numpy as np
import pytest

import oracle
from sdpa_inputs import make_inputs, make_random, workload
from tests.parity import LSE_MAX_ABS, check_o_lse, dev, host

pytestmark = pytest.mark.gpu

SMALL = [
    # B, H, Hkv, N, d
    (1, 2, 2, 1, 64),
    (1, 2, 2, 17, 128),
    (1, 1, 1, 64, 96),
    (2, 2, 2, 127, 64),
    (1, 2, 1, 128, 128),
    (1, 2, 2, 129, 96),
    (1, 4, 2, 255, 64),
    (1, 2, 2, 256, 128),
    (3, 2, 2, 300, 64),
    (1, 8, 1, 300, 128),
    (1, 2, 2, 513, 96),
    (1, 1, 1, 1000, 128),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "B%dH%dKV%dN%dd%d" % s)
def test_forward_small_shapes(cuda_lib, shape, causal):
    B, H, Hkv, N, d = shape
    seed = 1000 + N + d + H
    q = make_random((B, H, N, d), seed)
    k = make_random((B, Hkv, N, d), seed + 1)
    v = make_random((B, Hkv, N, d), seed + 2)
    s = 1 / math.sqrt(d)
    O, lse = cuda_lib.forward(dev(q), dev(k), dev(v), s, causal)
    O_ref, lse_ref = oracle.attention_forward(q, k, v, s, causal)
    check_o_lse(host(O), host(lse), O_ref, lse_ref, f"{shape} causal={causal}")


def test_forward_c1_full(cuda_lib):
    w = workload("c1")
    x = make_inputs(w)
    O, lse = cuda_lib.forward(dev(x["q"]), dev(x["k"]), dev(x["v"]), w.softmax_scale, w.causal)
    O_ref, lse_ref = oracle.attention_forward(x["q"], x["k"], x["v"], w.softmax_scale, w.causal)
    check_o_lse(host(O), host(lse), O_ref, lse_ref, "c1")


# ----------------------------------------------------------------- invariants
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_dominant_logit_is_exact_on_gpu(cuda_lib, d, causal):
    # q_i . k_j = 256 for j = perm^-1(i), else 0 (scale 1): every other
    # exponent is 2^-369, which is 0 in fp32, so O_i is exactly a V row.
    N = d
    perm = np.arange(N) if causal else np.random.default_rng(d).permutation(N)
    q = np.zeros((1, 1, N, d), np.float32)
    k = np.zeros((1, 1, N, d), np.float32)
    q[0, 0, np.arange(N), np.arange(N)] = 16.0
    k[0, 0, np.arange(N), perm] = 16.0
    v = make_random((1, 1, N, d), 7)
    O, lse = cuda_lib.forward(dev(q), dev(k), dev(v), 1.0, causal)
    inv = np.argsort(perm)
    assert np.array_equal(host(O)[0, 0], v[0, 0, inv].astype(np.float64))
    assert np.abs(host(lse) - 256.0).max() <= LSE_MAX_ABS


@pytest.mark.parametrize("d", [64, 96, 128])
def test_uniform_v_and_causal_row0(cuda_lib, d):
    B, H, N = 1, 2, 300
    q = make_random((B, H, N, d), 11)
    k = make_random((B, H, N, d), 12)
    c = make_random((B, H, 1, d), 13)
    v = np.broadcast_to(c, (B, H, N, d)).copy()
    s = 1 / math.sqrt(d)
    for causal in (False, True):
        O, lse = cuda_lib.forward(dev(q), dev(k), dev(v), s, causal)
        assert np.abs(host(O) - c).max() <= 1e-2
    v = make_random((B, H, N, d), 14)
    O, lse = cuda_lib.forward(dev(q), dev(k), dev(v), s, True)
    assert np.array_equal(host(O)[:, :, 0], v[:, :, 0].astype(np.float64))
    l0 = s * (q[:, :, 0].astype(np.float64) * k[:, :, 0]).sum(-1)
    assert np.abs(host(lse)[:, :, 0] - l0).max() <= LSE_MAX_ABS


def test_outputs_stay_inside_their_buffers(cuda_lib):
    """Guard bands: sentinel-filled margins around O and lse are untouched."""
    import torch
    B, H, N, d = 1, 3, 200, 96
    q = dev(make_random((B, H, N, d), 21))
    k = dev(make_random((B, H, N, d), 22))
    v = dev(make_random((B, H, N, d), 23))
    pad = 4096
    obuf = torch.full((2 * pad + B * H * N * d,), -7.0, dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((2 * pad + B * H * N,), -7.0, dtype=torch.float32, device="cuda")
    o = obuf[pad:pad + B * H * N * d].view(B, H, N, d)
    l = lbuf[pad:pad + B * H * N].view(B, H, N)
    for causal in (False, True):
        cuda_lib.forward(q, k, v, 0.1, causal, out=o, lse=l)
        torch.cuda.synchronize()
        assert torch.all(obuf[:pad] == -7.0) and torch.all(obuf[-pad:] == -7.0)
        assert torch.all(lbuf[:pad] == -7.0) and torch.all(lbuf[-pad:] == -7.0)
        assert torch.all(torch.isfinite(o)) and torch.all(torch.isfinite(l))


# ----------------------------------------------------------------- boundary
def test_device_argument_errors(cuda_lib):
    import torch
    q = torch.zeros((1, 2, 64, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 2, 64), dtype=torch.float32, device="cuda")
    host_buf = torch.zeros((1, 2, 64, 64), dtype=torch.bfloat16).pin_memory()
    S = cuda_lib.Status
    st = cuda_lib.attn_fwd(q.data_ptr(), q.data_ptr(), host_buf.data_ptr(), o.data_ptr(), lse.data_ptr(),
                           1, 2, 2, 64, 64, 0.125, 0, None)
    assert st == S.INVALID_ARG  # host memory is refused, never silently used
    st = cuda_lib.attn_fwd(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr() + 4,
                           1, 2, 2, 64, 64, 0.125, 0, None)
    assert st == S.MISALIGNED
    assert cuda_lib.attn_get_device_status(None) == S.OK


def test_bounded_wait_times_out_and_context_survives(cuda_lib):
    import torch
    S = cuda_lib.Status
    assert cuda_lib.attn_get_device_status(None) == S.OK
    assert cuda_lib.attn_selftest_wait_timeout(20000, None) == S.OK   # 20 ms limit
    st, info = cuda_lib.attn_get_timeout_info(None)
    assert st == S.OK and info[0] >> 16 == 0x01 and info[1] == 0 and info[3] >= 19000
    assert cuda_lib.attn_get_device_status(None) == S.TIMEOUT
    assert cuda_lib.attn_get_device_status(None) == S.OK              # cleared by the read
    # the context is still usable: a normal forward runs and is correct
    q = make_random((1, 2, 130, 64), 31)
    k = make_random((1, 2, 130, 64), 32)
    v = make_random((1, 2, 130, 64), 33)
    O, lse = cuda_lib.forward(dev(q), dev(k), dev(v), 0.125, True)
    torch.cuda.synchronize()
    O_ref, lse_ref = oracle.attention_forward(q, k, v, 0.125, True)
    check_o_lse(host(O), host(lse), O_ref, lse_ref, "after timeout")
    assert cuda_lib.attn_get_device_status(None) == S.OK
