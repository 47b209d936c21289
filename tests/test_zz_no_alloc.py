"""attn_bwd_noalloc against attn_bwd, called through the C ABI.

attn_bwd_noalloc is for callers that cannot allocate device memory: code
running inside a custom allocator (which must not call cudaMalloc on
itself), a runtime that has already given the whole device memory to its
own pool, or a plug-in interface that hands over only tensor pointers.  It
takes no workspace and uses a fixed 64 MiB scratch array inside the library
instead.  These tests check, on two calls in a row (with different shapes,
so the second call starts from the first call's leftover scratch), that its
gradients equal those of attn_bwd with a caller-provided workspace bit for
bit (the same deterministic kernels on the same inputs: a row vector read
from stale scratch would change them), and that a shape needing more scratch
than the fixed array is refused.

The file name sorts last, so a run that stops at the first failure has run
every other test before this one.
"""
import math

import numpy as np
import pytest

from sdpa_inputs import make_random
from tests.parity import dev, host, rel_fro

pytestmark = pytest.mark.gpu


def _grads_both_ways(lib, B, H, Hkv, N, d, causal, seed):
    import torch
    q = dev(make_random((B, H, N, d), seed))
    k = dev(make_random((B, Hkv, N, d), seed + 1))
    v = dev(make_random((B, Hkv, N, d), seed + 2))
    do = dev(make_random((B, H, N, d), seed + 3))
    s = 1 / math.sqrt(d)
    O, lse = lib.forward(q, k, v, s, causal)
    ref = [host(g) for g in lib.backward(q, k, v, O, lse, do, s, causal)]
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    st = lib.attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(), lse.data_ptr(),
                              do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                              B, H, Hkv, N, d, s, causal, torch.cuda.current_stream().cuda_stream)
    assert st == lib.Status.OK, lib.attn_status_string(st)
    torch.cuda.synchronize()
    assert lib.attn_get_device_status(None) == lib.Status.OK
    return [host(g) for g in (dq, dk, dv)], ref


def test_noalloc_backward_matches_attn_bwd_on_two_calls_in_a_row(cuda_lib):
    for shape, causal, seed in (((1, 4, 2, 300, 128), True, 7001), ((2, 2, 2, 129, 64), False, 7101)):
        got, ref = _grads_both_ways(cuda_lib, *shape, causal, seed)
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert np.all(np.isfinite(g)), name
            assert np.array_equal(g, r), (shape, name, rel_fro(g, r))


def test_noalloc_refuses_shapes_beyond_its_fixed_scratch(cuda_lib):
    # B=16, H=32, N=32768, d=128 needs 128 MiB of workspace, more than the
    # 64 MiB scratch: refused before anything is read or launched.
    assert cuda_lib.attn_bwd_workspace_size(16, 32, 32, 32768, 128) > 64 << 20
    fake = 0x10000
    st = cuda_lib.attn_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                   16, 32, 32, 32768, 128, 0.1, 1, None)
    assert st == cuda_lib.Status.WORKSPACE
