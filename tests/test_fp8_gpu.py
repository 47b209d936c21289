"""GPU parity of the FP8 (e4m3) forward (attn_fwd_fp8 through the C ABI)
against the fp64 oracle on the dequantised e4m3 inputs.

Tolerance (the pages give none for FP8): the kernel rounds P to e4m3 before
the P V product, which moves each probability by up to 2^-4 of itself
(3-bit mantissa, round to nearest).  A CPU simulation of that rounding alone
on these shapes gives a relative Frobenius error of O of 1.0-2.4% per head;
the bound used is twice the largest, 5e-2 per (batch, head), with a mean
absolute error of O <= 8e-3.  lse comes from float32 scores of exact e4m3
products, so it keeps the bf16 path's bound, 1e-3."""
import math

import numpy as np
import pytest

import oracle
from sdpa_inputs import e4m3_decode, make_random, quantize_e4m3
from tests.parity import LSE_MAX_ABS, host

pytestmark = pytest.mark.gpu

O_REL_FRO_FP8 = 5e-2
O_MEAN_ABS_FP8 = 8e-3


def _u8(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def _run(lib, shape, causal, seed, amp=1.0):
    B, H, Hkv, Nq, Nk, d = shape
    q = make_random((B, H, Nq, d), seed, amp)
    k = make_random((B, Hkv, Nk, d), seed + 1, amp)
    v = make_random((B, Hkv, Nk, d), seed + 2)
    (qb, qs), (kb, ks), (vb, vs) = quantize_e4m3(q), quantize_e4m3(k), quantize_e4m3(v)
    s = 1 / math.sqrt(d)
    O, lse = lib.forward_fp8(_u8(qb), _u8(kb), _u8(vb), qs, ks, vs, s, causal)
    assert lib.attn_get_device_status(None) == lib.Status.OK
    qd, kd, vd = e4m3_decode(qb) * qs, e4m3_decode(kb) * ks, e4m3_decode(vb) * vs
    off = (Nk - Nq) if causal else 0
    Or, lr = oracle.attention_forward(qd, kd, vd, s, causal, q_offset=off)
    return host(O), host(lse), Or, lr


def _check(O, lse, Or, lr, what):
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(lse)), what
    B, H = O.shape[:2]
    for b in range(B):
        for h in range(H):
            e = np.linalg.norm(O[b, h] - Or[b, h]) / np.linalg.norm(Or[b, h])
            assert e <= O_REL_FRO_FP8, f"{what} (b={b}, h={h}): O rel Frobenius {e:.3e}"
    assert np.abs(O - Or).mean() <= O_MEAN_ABS_FP8, what
    assert np.abs(lse - lr).max() <= LSE_MAX_ABS, f"{what}: lse err {np.abs(lse - lr).max():.3e}"


SHAPES = [
    # B, H, Hkv, Nq, Nk, d
    (1, 2, 2, 512, 512, 128),
    (2, 4, 2, 700, 700, 128),    # ragged, GQA
    (1, 2, 1, 129, 129, 128),
    (1, 4, 4, 256, 1024, 128),   # cross: Nq < Nk
    (1, 2, 2, 1, 300, 128),      # one query row
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dH%dKV%dQ%dK%dd%d" % s)
def test_fp8_forward_matches_oracle(cuda_lib, shape, causal):
    O, lse, Or, lr = _run(cuda_lib, shape, causal, 50000 + shape[3] + shape[4])
    _check(O, lse, Or, lr, f"{shape} causal={causal}")


@pytest.mark.parametrize("amp", [0.25, 3.0])
def test_fp8_forward_score_ranges(cuda_lib, amp):
    # Flat (small scores) and peaked (large scores) softmax rows.
    shape = (1, 2, 2, 384, 384, 128)
    O, lse, Or, lr = _run(cuda_lib, shape, True, 51000, amp)
    _check(O, lse, Or, lr, f"amp={amp}")


def test_fp8_rejects_other_head_dims(cuda_lib):
    import torch
    z = torch.zeros((1, 1, 16, 64), dtype=torch.uint8, device="cuda")
    with pytest.raises(cuda_lib.AttnError):
        cuda_lib.forward_fp8(z, z, z, 1.0, 1.0, 1.0)
