"""GPU parity of the backward pass (attn_bwd through the C ABI) against the
CPU fp64 oracle's analytic gradients on the same seeded bf16 inputs.

The GPU backward consumes the GPU forward's O and lse (as a training step
does); the reference is the pure oracle (its own fp64 P), so forward and
backward errors are both inside the comparison.  The full-size training
workload is compared element by element in test_fullsize_gpu.py."""
import math

import numpy as np
import pytest

import oracle
from sdpa_inputs import make_inputs, make_random, workload
from tests.parity import check_same_but_rounding, check_grads, dev, host, rel_fro

pytestmark = pytest.mark.gpu

SMALL = [
    # B, H, Hkv, N, d
    (1, 1, 1, 1, 64),
    (1, 2, 2, 17, 128),
    (1, 2, 2, 128, 64),
    (1, 2, 1, 129, 96),
    (2, 2, 2, 200, 128),
    (1, 4, 2, 256, 64),
    (1, 4, 1, 300, 128),
    (1, 2, 2, 513, 96),
    (1, 8, 2, 384, 64),
    (1, 1, 1, 1000, 128),
]


def _run(lib, q, k, v, do, s, causal):
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    O, lse = lib.forward(tq, tk, tv, s, causal)
    return [host(g) for g in lib.backward(tq, tk, tv, O, lse, tdo, s, causal)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "B%dH%dKV%dN%dd%d" % s)
def test_backward_small_shapes(cuda_lib, shape, causal):
    B, H, Hkv, N, d = shape
    seed = 5000 + N + d + H
    q = make_random((B, H, N, d), seed)
    k = make_random((B, Hkv, N, d), seed + 1)
    v = make_random((B, Hkv, N, d), seed + 2)
    do = make_random((B, H, N, d), seed + 3)
    s = 1 / math.sqrt(d)
    grads = _run(cuda_lib, q, k, v, do, s, causal)
    ref = oracle.attention_backward(q, k, v, do, s, causal)
    check_grads(grads, ref, f"{shape} causal={causal}")


def test_backward_gqa_group_sum_long(cuda_lib):
    # GQA with a long sequence: dK/dV sum over the 4 query heads of a group.
    B, H, Hkv, N, d = 1, 8, 2, 1536, 128
    q = make_random((B, H, N, d), 71, 0.5)
    k = make_random((B, Hkv, N, d), 72, 0.5)
    v = make_random((B, Hkv, N, d), 73, 0.5)
    do = make_random((B, H, N, d), 74)
    s = 1 / math.sqrt(d)
    grads = _run(cuda_lib, q, k, v, do, s, True)
    ref = oracle.attention_backward(q, k, v, do, s, True)
    check_grads(grads, ref, "gqa long")


def test_backward_padded_head_dim(cuda_lib):
    # head_dim 80 zero-padded to 96: gradients equal the unpadded d=80 oracle
    # and the pad columns of dQ, dK, dV are exactly zero.
    B, H, Hkv, N = 1, 4, 2, 333
    q = make_random((B, H, N, 80), 81)
    k = make_random((B, Hkv, N, 80), 82)
    v = make_random((B, Hkv, N, 80), 83)
    do = make_random((B, H, N, 80), 84)
    pad = [(0, 0)] * 3 + [(0, 16)]
    s = 1 / math.sqrt(80)
    grads = _run(cuda_lib, np.pad(q, pad), np.pad(k, pad), np.pad(v, pad), np.pad(do, pad), s, True)
    for g in grads:
        assert np.all(g[..., 80:] == 0.0)
    ref = oracle.attention_backward(q, k, v, do, s, True)
    check_grads([g[..., :80] for g in grads], ref, "padded d=96")


def test_backward_outputs_stay_inside_buffers_and_workspace_checks(cuda_lib):
    import torch
    B, H, Hkv, N, d = 1, 2, 1, 150, 64
    q = dev(make_random((B, H, N, d), 91))
    k = dev(make_random((B, Hkv, N, d), 92))
    v = dev(make_random((B, Hkv, N, d), 93))
    do = dev(make_random((B, H, N, d), 94))
    O, lse = cuda_lib.forward(q, k, v, 0.125, True)
    pad = 2048
    bufs = [torch.full((2 * pad + t.numel(),), -3.0, dtype=torch.bfloat16, device="cuda") for t in (q, k, v)]
    views = [bb[pad:pad + t.numel()].view(t.shape) for bb, t in zip(bufs, (q, k, v))]
    ws_bytes = cuda_lib.attn_bwd_workspace_size(B, H, Hkv, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    S = cuda_lib.Status
    args = [q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(), lse.data_ptr(), do.data_ptr(),
            views[0].data_ptr(), views[1].data_ptr(), views[2].data_ptr()]
    assert cuda_lib.attn_bwd(*args, ws.data_ptr(), ws_bytes - 16, B, H, Hkv, N, d, 0.125, 1, None) == S.WORKSPACE
    assert cuda_lib.attn_bwd(*args, 0, ws_bytes, B, H, Hkv, N, d, 0.125, 1, None) == S.WORKSPACE
    assert cuda_lib.attn_bwd(*args, ws.data_ptr(), ws_bytes, B, H, Hkv, N, d, 0.125, 1, None) == S.OK
    torch.cuda.synchronize()
    for bb in bufs:
        assert torch.all(bb[:pad] == -3.0) and torch.all(bb[-pad:] == -3.0)
    ref = oracle.attention_backward(host(q), host(k), host(v), host(do), 0.125, True)
    check_grads([host(t) for t in views], ref, "views")
    assert cuda_lib.attn_get_device_status(None) == S.OK


def test_backward_stages_equal_the_combined_call(cuda_lib):
    # attn_bwd_dq_rows + attn_bwd_grad on one stream are attn_bwd, bit for
    # bit; attn_bwd_prep + attn_bwd_grad + attn_bwd_dq differ only by the
    # order of D's float32 additions, and both write the same row vectors.
    import torch
    B, H, Hkv, N, d = 1, 4, 2, 260, 96
    q = dev(make_random((B, H, N, d), 111))
    k = dev(make_random((B, Hkv, N, d), 112))
    v = dev(make_random((B, Hkv, N, d), 113))
    do = dev(make_random((B, H, N, d), 114))
    O, lse = cuda_lib.forward(q, k, v, 0.1, False)
    ref = [host(g) for g in cuda_lib.backward(q, k, v, O, lse, do, 0.1, False)]
    ws_bytes = cuda_lib.attn_bwd_workspace_size(B, H, Hkv, N, d)
    sp = torch.cuda.current_stream().cuda_stream
    P = lambda t: t.data_ptr()
    vecs = []
    for order in ("rows", "prep"):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.full((ws_bytes // 4,), float("nan"), dtype=torch.float32, device="cuda")
        if order == "rows":
            assert cuda_lib.attn_bwd_dq_rows(P(q), P(k), P(v), P(O), P(lse), P(do), P(dq), P(ws), ws_bytes,
                                             B, H, Hkv, N, N, d, 0.1, 0, sp) == 0
            assert cuda_lib.attn_bwd_grad(P(q), P(k), P(v), P(do), P(dk), P(dv), P(ws), ws_bytes,
                                          B, H, Hkv, N, d, 0.1, 0, sp) == 0
        else:
            assert cuda_lib.attn_bwd_prep(P(O), P(lse), P(do), P(ws), ws_bytes, B, H, Hkv, N, d, sp) == 0
            assert cuda_lib.attn_bwd_grad(P(q), P(k), P(v), P(do), P(dk), P(dv), P(ws), ws_bytes,
                                          B, H, Hkv, N, d, 0.1, 0, sp) == 0
            assert cuda_lib.attn_bwd_dq(P(q), P(k), P(v), P(do), P(dq), P(ws), ws_bytes,
                                        B, H, Hkv, N, d, 0.1, 0, sp) == 0
        got = [host(g) for g in (dq, dk, dv)]
        if order == "rows":
            for g, r in zip(got, ref):
                assert np.array_equal(g, r)
        else:
            check_same_but_rounding(got, ref, "prep + grad + dq")
        vecs.append(ws.cpu().numpy().reshape(2, B * H, -1))
    # -D close, -lse2 identical; the padding rows (260..383) -D = 0, -lse2 = -inf
    assert np.allclose(vecs[0][0], vecs[1][0], rtol=1e-5, atol=1e-6)
    assert np.array_equal(vecs[0][1], vecs[1][1])
    for vv in vecs:
        assert np.all(vv[0][:, N:] == 0) and np.all(np.isneginf(vv[1][:, N:]))


def test_backward_is_deterministic(cuda_lib):
    # dK, dV (per key tile) and dQ (per query tile) each accumulate in tensor
    # memory in a fixed order and have one writer: bit-identical across runs.
    B, H, Hkv, N, d = 1, 4, 2, 700, 128
    q = make_random((B, H, N, d), 101)
    k = make_random((B, Hkv, N, d), 102)
    v = make_random((B, Hkv, N, d), 103)
    do = make_random((B, H, N, d), 104)
    g1 = _run(cuda_lib, q, k, v, do, 0.1, True)
    g2 = _run(cuda_lib, q, k, v, do, 0.1, True)
    for a, b in zip(g1, g2):
        assert np.array_equal(a, b)
