"""The production kernels' failure path, without a GPU fault.

attn_debug_drop_load arms one launch: the first CTA's TMA producer skips one
ring load and every on-chip wait is limited to 20 ms.  The consumers of that
load must give up, record ATTN_ERR_TIMEOUT with the CTA and the wait site,
and every role of the CTA must stop and exit (each named barrier is reached
whatever a wait returned), so that the launch ends and the context stays
usable.  The CTAs that lost nothing complete normally, and the next normal
call is correct.  One case per kernel: forward, dQ, dK/dV, the
persistent forward, dK/dV and dQ kernels, and the FP8 forward (both
schedules).
"""
import math

import numpy as np
import pytest

import oracle
from sdpa_inputs import make_random
from tests.parity import check_grads, check_o_lse, dev, host

pytestmark = pytest.mark.gpu

LIMIT_US = 20000
FWD_SITES = {0x51, 0x52, 0x53, 0x54, 0x61, 0x71, 0x72, 0x73, 0x74, 0x75, 0x76, 0x77, 0x78, 0x79, 0x7a}
DQ_SITES = {0x81, 0x82, 0x83, 0x84, 0x85, 0x91, 0x92, 0x93} | set(range(0xa1, 0xa9))
GRAD_SITES = {0x11, 0x12, 0x13, 0x14, 0x31, 0x32} | set(range(0x41, 0x48))


def _inputs(B, H, N, d, seed):
    return [make_random((B, H, N, d), seed + i) for i in range(4)]


def _expect_timeout_in_cta0(lib, sites):
    import torch
    torch.cuda.synchronize()
    st, info = lib.attn_get_timeout_info(None)
    assert st == lib.Status.OK
    assert lib.attn_get_device_status(None) == lib.Status.TIMEOUT
    assert lib.attn_get_device_status(None) == lib.Status.OK  # cleared by the read
    site = info[0] >> 16
    assert site in sites, hex(site)
    assert info[1] == 0  # the CTA whose load was dropped
    assert info[3] >= LIMIT_US * 0.9


def test_forward_dropped_load_times_out_and_recovers(cuda_lib):
    B, H, N, d = 1, 2, 512, 128
    q, k, v, _ = _inputs(B, H, N, d, 61000)
    s = 1 / math.sqrt(d)
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK
    # CTA 0 = head 0, query tiles 2 and 3 (four key tiles, eight ring loads): drop K_1
    assert cuda_lib.attn_debug_drop_load(0, 2, LIMIT_US) == cuda_lib.Status.OK
    O, lse = cuda_lib.forward(dev(q), dev(k), dev(v), s, True)
    _expect_timeout_in_cta0(cuda_lib, FWD_SITES)
    O_ref, lse_ref = oracle.attention_forward(q, k, v, s, True)
    O, lse = host(O), host(lse)
    # the other CTAs (head 0 rows 0..255, all of head 1) completed normally
    check_o_lse(O[:, 1], lse[:, 1], O_ref[:, 1], lse_ref[:, 1], "head 1 beside the dropped load")
    check_o_lse(O[:, 0, :256], lse[:, 0, :256], O_ref[:, 0, :256], lse_ref[:, 0, :256], "head 0, first CTA")
    # the next call is whole and correct
    O, lse = cuda_lib.forward(dev(q), dev(k), dev(v), s, True)
    check_o_lse(host(O), host(lse), O_ref, lse_ref, "after the timeout")
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK


@pytest.mark.parametrize("kernel,load,sites", [(1, 3, DQ_SITES), (2, 1, GRAD_SITES)], ids=["dq_V1", "dkdv_Q1"])
def test_backward_dropped_load_times_out_and_recovers(cuda_lib, kernel, load, sites):
    B, H, N, d = 1, 2, 512, 128
    q, k, v, do = _inputs(B, H, N, d, 62000 + kernel)
    s = 1 / math.sqrt(d)
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    O, lse = cuda_lib.forward(tq, tk, tv, s, True)
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK
    # dQ: CTA 0 = head 0, query tile 3, drop V_1; dK/dV: CTA 0 = head 0, key tile 0, drop Q_1
    assert cuda_lib.attn_debug_drop_load(kernel, load, LIMIT_US) == cuda_lib.Status.OK
    cuda_lib.backward(tq, tk, tv, O, lse, tdo, s, True)
    _expect_timeout_in_cta0(cuda_lib, sites)
    grads = [host(g) for g in cuda_lib.backward(tq, tk, tv, O, lse, tdo, s, True)]
    check_grads(grads, oracle.attention_backward(q, k, v, do, s, True), "after the timeout")
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK


PERSIST_SITES = {0x51, 0x52, 0x53, 0x54, 0x5a, 0x61, 0x64, 0x65, 0x66} | set(range(0x71, 0x7b))


def test_persistent_forward_dropped_load_times_out_and_recovers(cuda_lib):
    # The persistent forward (attn_fwd's dense calls): the CTA that takes the
    # first work unit (head 0, query tiles 2 and 3) skips that unit's K_1.
    # Which CTA that is depends on the queue, so only the status, the site
    # and the next call are checked.
    import torch
    B, H, N, d = 1, 2, 512, 128
    q, k, v, _ = _inputs(B, H, N, d, 63000)
    s = 1 / math.sqrt(d)
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK
    assert cuda_lib.attn_debug_drop_load(3, 2, LIMIT_US) == cuda_lib.Status.OK
    cuda_lib.forward(dev(q), dev(k), dev(v), s, True)
    torch.cuda.synchronize()
    st, info = cuda_lib.attn_get_timeout_info(None)
    assert st == cuda_lib.Status.OK
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.TIMEOUT
    assert info[0] >> 16 in PERSIST_SITES, hex(info[0] >> 16)
    assert info[3] >= LIMIT_US * 0.9
    O_ref, lse_ref = oracle.attention_forward(q, k, v, s, True)
    O, lse = cuda_lib.forward(dev(q), dev(k), dev(v), s, True)
    check_o_lse(host(O), host(lse), O_ref, lse_ref, "after the timeout")
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK


PERSIST_GRAD_SITES = {0x11, 0x12, 0x13, 0x14, 0x1a, 0x31, 0x32, 0x34, 0x35} | set(range(0x41, 0x49))


def test_persistent_dkdv_dropped_load_times_out_and_recovers(cuda_lib):
    # The persistent dK/dV kernel (attn_bwd's dense second stage): the CTA
    # that takes the first work unit skips that unit's Q_1 load.
    import torch
    B, H, N, d = 1, 2, 512, 128
    q, k, v, do = _inputs(B, H, N, d, 64000)
    s = 1 / math.sqrt(d)
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    O, lse = cuda_lib.forward(tq, tk, tv, s, True)
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK
    assert cuda_lib.attn_debug_drop_load(4, 1, LIMIT_US) == cuda_lib.Status.OK
    cuda_lib.backward(tq, tk, tv, O, lse, tdo, s, True)
    torch.cuda.synchronize()
    st, info = cuda_lib.attn_get_timeout_info(None)
    assert st == cuda_lib.Status.OK
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.TIMEOUT
    assert info[0] >> 16 in PERSIST_GRAD_SITES, hex(info[0] >> 16)
    assert info[3] >= LIMIT_US * 0.9
    grads = [host(g) for g in cuda_lib.backward(tq, tk, tv, O, lse, tdo, s, True)]
    check_grads(grads, oracle.attention_backward(q, k, v, do, s, True), "after the timeout")
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK


PERSIST_DQ_SITES = set(range(0xb0, 0xc0)) | {0xf1, 0xf2}


def test_persistent_dq_dropped_load_times_out_and_recovers(cuda_lib):
    # The persistent dQ kernel (attn_bwd's dense first stage): the CTA that
    # takes the first work unit (head 0, query tile 3: four key tiles) skips
    # that unit's K_1 load.
    import torch
    B, H, N, d = 1, 2, 512, 128
    q, k, v, do = _inputs(B, H, N, d, 65000)
    s = 1 / math.sqrt(d)
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    O, lse = cuda_lib.forward(tq, tk, tv, s, True)
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK
    assert cuda_lib.attn_debug_drop_load(5, 1, LIMIT_US) == cuda_lib.Status.OK
    cuda_lib.backward(tq, tk, tv, O, lse, tdo, s, True)
    torch.cuda.synchronize()
    st, info = cuda_lib.attn_get_timeout_info(None)
    assert st == cuda_lib.Status.OK
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.TIMEOUT
    assert info[0] >> 16 in PERSIST_DQ_SITES, hex(info[0] >> 16)
    assert info[3] >= LIMIT_US * 0.9
    grads = [host(g) for g in cuda_lib.backward(tq, tk, tv, O, lse, tdo, s, True)]
    check_grads(grads, oracle.attention_backward(q, k, v, do, s, True), "after the timeout")
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK


FP8_SITES = set(range(0xc1, 0xc6)) | set(range(0xd1, 0xd5)) | set(range(0xe1, 0xeb))


@pytest.mark.parametrize("d", [128, 64], ids=["d128_per_unit", "d64_persistent"])
def test_fp8_forward_dropped_load_times_out_and_recovers(cuda_lib, d):
    # The FP8 forward (one CTA per unit at d = 128, persistent at d = 64):
    # the first CTA's producer skips K_1.  The next call equals a call made
    # before the hook was armed, bit for bit.
    import torch
    from sdpa_inputs import quantize_e4m3
    B, H, N = 1, 2, 512
    q, k, v, _ = _inputs(B, H, N, d, 66000 + d)
    (q8, qs), (k8, ks), (v8, vs) = (quantize_e4m3(x) for x in (q, k, v))
    t8 = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (q8, k8, v8)]
    s = 1 / math.sqrt(d)
    O_ref, lse_ref = cuda_lib.forward_fp8(*t8, qs, ks, vs, s, True)
    torch.cuda.synchronize()
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK
    assert cuda_lib.attn_debug_drop_load(6, 2, LIMIT_US) == cuda_lib.Status.OK
    cuda_lib.forward_fp8(*t8, qs, ks, vs, s, True)
    torch.cuda.synchronize()
    st, info = cuda_lib.attn_get_timeout_info(None)
    assert st == cuda_lib.Status.OK
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.TIMEOUT
    assert info[0] >> 16 in FP8_SITES, hex(info[0] >> 16)
    assert info[3] >= LIMIT_US * 0.9
    O, lse = cuda_lib.forward_fp8(*t8, qs, ks, vs, s, True)
    torch.cuda.synchronize()
    assert torch.equal(O, O_ref) and torch.equal(lse, lse_ref)
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK
