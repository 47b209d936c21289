"""GPU parity of decode against a paged KV cache (attn_decode_paged through
the C ABI) against the fp64 oracle.  The pages of each sequence are
scattered over the pool; the slots past each sequence (the tail of its last
page, pages no table points at) hold NaN, so a kernel that let them into a
product would fail."""
import math

import numpy as np
import pytest

import oracle
from sdpa_inputs import make_random
from tests.parity import check_o_lse, dev, host

pytestmark = pytest.mark.gpu


def _pool(k, v, lens, page_size, seed, spare=3):
    """Scatter contiguous (B, Hkv, N, d) K / V into a NaN-filled page pool."""
    B, Hkv, N, d = k.shape
    max_pages = -(-N // page_size) + 1
    num_pages = B * max_pages + spare
    order = np.random.default_rng(seed).permutation(num_pages)
    kc = np.full((num_pages, page_size, Hkv, d), np.nan, dtype=np.float32)
    vc = np.full((num_pages, page_size, Hkv, d), np.nan, dtype=np.float32)
    table = np.full((B, max_pages), -1, dtype=np.int32)
    for b in range(B):
        L = int(lens[b])
        for i in range(-(-L // page_size)):
            phys = int(order[b * max_pages + i])
            table[b, i] = phys
            a, e = i * page_size, min(L, (i + 1) * page_size)
            kc[phys, :e - a] = k[b, :, a:e].transpose(1, 0, 2)
            vc[phys, :e - a] = v[b, :, a:e].transpose(1, 0, 2)
    return kc, vc, table


def _int32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _run(lib, B, H, Hkv, Nq, N, d, lens, page_size, causal, seed):
    q = make_random((B, H, Nq, d), seed)
    k = make_random((B, Hkv, N, d), seed + 1)
    v = make_random((B, Hkv, N, d), seed + 2)
    kc, vc, table = _pool(k, v, lens, page_size, seed + 3)
    s = 1 / math.sqrt(d)
    O, lse = lib.decode_paged(dev(q), dev(kc), dev(vc), _int32(table), _int32(lens), s, causal)
    status = lib.attn_get_device_status(None)
    Or, lr = oracle.attention_decode_paged(q, np.nan_to_num(kc), np.nan_to_num(vc), table, lens, s, causal)
    return host(O), host(lse), Or, lr, status


@pytest.mark.parametrize("page_size", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_paged_decode_matches_oracle(cuda_lib, page_size, causal):
    lens = np.array([1000, 37, 513])
    O, lse, Or, lr, status = _run(cuda_lib, 3, 8, 2, 4, 1000, 128, lens, page_size, causal, 60000 + page_size)
    assert status == cuda_lib.Status.OK
    check_o_lse(O, lse, Or, lr, f"page {page_size} causal={causal}")


@pytest.mark.parametrize("d", [64, 96])
def test_paged_decode_head_dims(cuda_lib, d):
    lens = np.array([300, 129])
    O, lse, Or, lr, status = _run(cuda_lib, 2, 4, 4, 1, 300, d, lens, 32, True, 61000 + d)
    assert status == cuda_lib.Status.OK
    check_o_lse(O, lse, Or, lr, f"d={d}")


def test_paged_decode_long_cache(cuda_lib):
    # A long sequence split over many key chunks, next to a short one.
    lens = np.array([20000, 200])
    O, lse, Or, lr, status = _run(cuda_lib, 2, 16, 2, 1, 20000, 128, lens, 64, False, 62000)
    assert status == cuda_lib.Status.OK
    check_o_lse(O, lse, Or, lr, "long")


def test_paged_decode_bad_table_entry_is_reported(cuda_lib):
    # A page the sequence needs points outside the pool: the kernel reads
    # zeros for it (no access outside the cache) and reports the argument.
    B, H, Hkv, Nq, N, d, ps = 1, 2, 2, 1, 100, 64, 32
    q = dev(make_random((B, H, Nq, d), 63000))
    kc = dev(make_random((4, ps, Hkv, d), 63001))
    vc = dev(make_random((4, ps, Hkv, d), 63002))
    for table, lens in (([[0, 1, 99, 2]], [N]), ([[0, 1, 2, 3]], [200])):
        cuda_lib.decode_paged(q, kc, vc, _int32(table), _int32(lens), 0.1, False)
        assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.INVALID_ARG
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK
