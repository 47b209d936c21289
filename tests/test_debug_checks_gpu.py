"""The debug build's in-kernel index checks (-DATTN_DEBUG), standing in for
compute-sanitizer's bounds checking, which this pool does not offer.

* test_debug_build_runs_the_suite builds _lib/libsdpa08_debug.so, checks
  that it gives the release build's outputs bit for bit, then runs the
  small-shape GPU tests (dense, cross, packed batches, masks, the additive
  mask, decode, paged decode, FP8) against it in a subprocess: each test
  must pass and end without a failed check (tests/conftest.py).
* The planted-index tests run only against the debug build (inside that
  subprocess): one armed launch computes an element index past the end of
  an output array in a production kernel, and the check must catch it,
  skip the store and leave the context usable.
"""
import ctypes
import math
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from sdpa_inputs import make_random
from tests.parity import check_grads, check_o_lse, dev, host

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITE = ["tests/test_fwd_gpu.py", "tests/test_bwd_gpu.py", "tests/test_fwd_cross_gpu.py",
         "tests/test_bwd_cross_gpu.py", "tests/test_varlen_gpu.py", "tests/test_masked_gpu.py",
         "tests/test_decode_gpu.py", "tests/test_decode_paged_gpu.py", "tests/test_fp8_gpu.py",
         "tests/test_debug_checks_gpu.py"]
SENTINEL = 12345.0


def _raw(path):
    """The fwd/bwd entry points of one library file, as a separate handle."""
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib = ctypes.CDLL(path)
    lib.attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, P]
    lib.attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, I, I, I, I, I, F, I, P]
    lib.attn_bwd_workspace_size.argtypes = [I, I, I, I, I]
    lib.attn_bwd_workspace_size.restype = ctypes.c_size_t
    lib.attn_get_device_status.argtypes = [P]
    lib.attn_debug_build.restype = I
    return lib


def _fwd_bwd(lib, q, k, v, do, s, causal):
    import torch
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsb = lib.attn_bwd_workspace_size(B, H, Hkv, N, d)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    P = lambda t: t.data_ptr()
    assert lib.attn_fwd(P(q), P(k), P(v), P(o), P(lse), B, H, Hkv, N, d, s, int(causal), None) == 0
    assert lib.attn_bwd(P(q), P(k), P(v), P(o), P(lse), P(do), P(dq), P(dk), P(dv), P(ws), wsb, B, H, Hkv, N, d, s,
                        int(causal), None) == 0
    torch.cuda.synchronize()
    assert lib.attn_get_device_status(None) == 0
    return [t.cpu() for t in (o, lse, dq, dk, dv)]


def test_debug_build_runs_the_suite(cuda_lib):
    import torch
    from scaled_dot_product_08_gb300.build import build
    if os.environ.get("SDPA08_LIBRARY"):
        pytest.skip("already running against a library named by SDPA08_LIBRARY")
    path = build(debug=True)
    dbg, rel = _raw(path), _raw(cuda_lib.library_path())
    assert dbg.attn_debug_build() == 1 and rel.attn_debug_build() == 0
    assert cuda_lib.attn_debug_plant_index(0) == cuda_lib.Status.INVALID_ARG  # nothing to arm in the release build
    # The checks change no arithmetic: the same outputs, bit for bit.
    for (B, H, Hkv, N, d, causal) in [(2, 4, 2, 1000, 64, True), (1, 2, 2, 384, 128, False), (1, 3, 1, 257, 96, True)]:
        q = dev(make_random((B, H, N, d), 71000 + N))
        k, v = dev(make_random((B, Hkv, N, d), 71001 + N)), dev(make_random((B, Hkv, N, d), 71002 + N))
        do = dev(make_random((B, H, N, d), 71003 + N))
        a = _fwd_bwd(dbg, q, k, v, do, 1 / math.sqrt(d), causal)
        b = _fwd_bwd(rel, q, k, v, do, 1 / math.sqrt(d), causal)
        for x, y, name in zip(a, b, ("O", "lse", "dQ", "dK", "dV")):
            assert torch.equal(x, y), f"debug and release builds differ in {name} at {(B, H, Hkv, N, d, causal)}"
    env = dict(os.environ, SDPA08_LIBRARY=path)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu and not slow", "-p", "no:cacheprovider",
                        *SUITE], cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-25:])
    assert r.returncode == 0, f"GPU tests under the debug build failed:\n{tail}"
    print("\n" + tail.splitlines()[-1], end="")


def _need_debug_build(lib):
    if lib.attn_debug_build() != 1:
        pytest.skip("runs against the debug build (test_debug_build_runs_the_suite runs it)")


def _expect_check(lib, site):
    import torch
    torch.cuda.synchronize()
    st, info = lib.attn_get_timeout_info(None)
    assert st == lib.Status.OK
    assert lib.attn_get_device_status(None) == lib.Status.CHECK
    assert lib.attn_get_device_status(None) == lib.Status.OK  # cleared by the read
    assert info[0] >> 16 == site, hex(info[0] >> 16)
    assert info[1] == 0  # the CTA that planted the index
    return info


def test_planted_forward_lse_index_is_caught(cuda_lib):
    import torch
    _need_debug_build(cuda_lib)
    B, H, N, d = 1, 2, 512, 128
    q, k, v = (make_random((B, H, N, d), 72000 + i) for i in range(3))
    s = 1 / math.sqrt(d)
    tq, tk, tv = dev(q), dev(k), dev(v)
    lse = torch.full((B, H, N), SENTINEL, dtype=torch.float32, device="cuda")
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK
    assert cuda_lib.attn_debug_plant_index(0) == cuda_lib.Status.OK
    O, lse = cuda_lib.forward(tq, tk, tv, s, True, lse=lse)
    info = _expect_check(cuda_lib, 0x103)
    assert info[3] >= B * H * N  # the planted index lies past the lse array
    O_ref, lse_ref = oracle.attention_forward(q, k, v, s, True)
    O, lse = host(O), host(lse)
    # CTA 0 (head 0, query rows 256..511) skipped its lse store; O (a TMA
    # store) and every other row are whole
    assert np.all(lse[0, 0, 256:] == SENTINEL)
    check_o_lse(O, np.where(lse == SENTINEL, lse_ref, lse), O_ref, lse_ref, "beside the planted index")
    O, lse = cuda_lib.forward(tq, tk, tv, s, True)
    check_o_lse(host(O), host(lse), O_ref, lse_ref, "the next call")
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK


def test_planted_dq_workspace_index_is_caught(cuda_lib):
    _need_debug_build(cuda_lib)
    B, H, N, d = 1, 2, 512, 64
    q, k, v, do = (make_random((B, H, N, d), 73000 + i) for i in range(4))
    s = 1 / math.sqrt(d)
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    O, lse = cuda_lib.forward(tq, tk, tv, s, True)
    ref = oracle.attention_backward(q, k, v, do, s, True)
    assert cuda_lib.attn_debug_plant_index(1) == cuda_lib.Status.OK
    dq, _, _ = cuda_lib.backward(tq, tk, tv, O, lse, tdo, s, True)
    _expect_check(cuda_lib, 0x204)
    # the dQ kernel keeps its own row vectors in registers: dQ is whole
    check_grads([host(dq), ref[1], ref[2]], ref, "dQ beside the planted index")
    grads = [host(g) for g in cuda_lib.backward(tq, tk, tv, O, lse, tdo, s, True)]
    check_grads(grads, ref, "the next call")
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK
