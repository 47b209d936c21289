"""GPU parity of the masked path (attn_fwd_masked / attn_bwd_masked through
the C ABI: sliding windows, per-batch key lengths, boolean masks and their
combinations) against the fp64 oracle on seeded bf16 inputs.  The backward
consumes the GPU forward's O and lse."""
import math

import numpy as np
import pytest

import oracle
from sdpa_inputs import make_random, round_bf16
from tests.parity import LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS, check_grads, dev, host

pytestmark = pytest.mark.gpu


def _problem(B, H, Hkv, Nq, Nk, d, seed):
    return (make_random((B, H, Nq, d), seed), make_random((B, Hkv, Nk, d), seed + 1),
            make_random((B, Hkv, Nk, d), seed + 2), make_random((B, H, Nq, d), seed + 3))


def _t(a, dtype):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype).cuda()


def _check_forward(O, lse, Or, lr, what):
    live = np.isfinite(lr)
    assert np.all(np.isneginf(lse[~live])), what
    assert np.all(O[~live] == 0), what
    err = np.abs(O[live] - Or[live])
    assert err.max() <= O_MAX_ABS and err.mean() <= O_MEAN_ABS, f"{what}: O err {err.max():.3e} / {err.mean():.3e}"
    assert np.abs(lse[live] - lr[live]).max() <= LSE_MAX_ABS, what


def _run(lib, shape, causal, window=None, key_lengths=None, mask=None, seed=40000):
    import torch
    B, H, Hkv, Nq, Nk, d = shape
    q, k, v, do = _problem(B, H, Hkv, Nq, Nk, d, seed)
    s = 1 / math.sqrt(d)
    kl = _t(np.asarray(key_lengths, dtype=np.int32), torch.int32) if key_lengths is not None else None
    mk = _t(mask.astype(np.uint8), torch.uint8) if mask is not None else None
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    O, lse = lib.forward_masked(tq, tk, tv, s, causal, window, kl, mk)
    g = lib.backward_masked(tq, tk, tv, O, lse, tdo, s, causal, window, kl, mk)
    assert lib.attn_get_device_status(None) == lib.Status.OK
    Or, lr = oracle.attention_masked_forward(q, k, v, s, causal, window, key_lengths, mask)
    ref = oracle.attention_masked_backward(q, k, v, do, s, causal, window, key_lengths, mask)
    return host(O), host(lse), [host(x) for x in g], Or, lr, ref


CASES = [
    # (B, H, Hkv, Nq, Nk, d), causal, window, key_lengths, mask kind
    ((1, 4, 2, 700, 700, 128), True, (100, -1), None, None),       # causal sliding window
    ((1, 2, 2, 513, 513, 64), False, (64, 200), None, None),       # two-sided window
    ((2, 2, 1, 640, 640, 128), True, (300, -1), None, None),       # window spanning tiles
    ((3, 2, 2, 700, 700, 128), False, None, [700, 129, 1], None),  # padding by key length
    ((3, 2, 2, 700, 700, 96), True, None, [650, 300, 1], None),
    ((2, 4, 2, 300, 300, 96), False, None, None, "batch"),          # random boolean mask per batch element
    ((2, 4, 4, 260, 260, 128), True, None, None, "full"),           # per (batch, head), with causal
    ((1, 2, 1, 384, 384, 64), False, None, None, "shared"),
    ((2, 2, 2, 512, 512, 128), False, None, None, "documents"),     # block-diagonal document mask
    ((2, 4, 2, 200, 600, 128), True, (250, -1), [600, 450], "batch"),  # all of it, Nq < Nk
    ((1, 2, 2, 300, 150, 64), True, None, None, None),              # causal with Nq > Nk: rows without keys
    ((1, 4, 2, 1536, 1536, 128), False, None, None, "doc3"),        # 3 documents: most tiles skipped
    ((2, 2, 2, 1024, 1024, 128), False, None, None, "prefix"),      # prefix-LM
    ((1, 2, 1, 1000, 1000, 96), True, (200, -1), None, "doc3"),     # documents, causal, window
]


def _mask(kind, B, H, Nq, Nk, seed):
    rng = np.random.default_rng(seed)
    if kind is None:
        return None
    if kind == "documents":
        m = np.zeros((B, 1, Nq, Nk), dtype=bool)
        for b in range(B):
            cuts = np.sort(rng.choice(np.arange(1, Nq), size=4, replace=False))
            edges = [0, *cuts.tolist(), Nq]
            for a, e in zip(edges, edges[1:]):
                m[b, 0, a:e, a:e] = True
        return m
    if kind == "doc3":  # three documents of uneven lengths, one plane for all (b, h)
        m = np.zeros((1, 1, Nq, Nk), dtype=bool)
        edges = [0, Nq // 5, (3 * Nq) // 5, Nq]
        for a, e in zip(edges, edges[1:]):
            m[0, 0, a:e, a:e] = True
        return m
    if kind == "prefix":  # prefix-LM over the first quarter
        i = np.arange(Nq)[:, None]
        j = np.arange(Nk)[None, :]
        return ((j < Nk // 4) | (j <= i))[None, None]
    shape = {"batch": (B, 1, Nq, Nk), "full": (B, H, Nq, Nk), "shared": (1, 1, Nq, Nk)}[kind]
    return rng.random(shape) < 0.7


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dH%dKV%dQ%dK%dd%d" % c[0] + f"_c{int(c[1])}_w{c[2]}_kl{c[3] is not None}_{c[4]}")
def test_masked_matches_oracle(cuda_lib, case):
    shape, causal, window, kl, kind = case
    B, H, Hkv, Nq, Nk, d = shape
    mask = _mask(kind, B, H, Nq, Nk, 41000 + Nq)
    O, lse, g, Or, lr, ref = _run(cuda_lib, shape, causal, window, kl, mask, seed=42000 + Nq + Nk)
    _check_forward(O, lse, Or, lr, str(case))
    check_grads(g, ref, str(case))


def test_rows_without_keys_are_zero(cuda_lib):
    B, H, Hkv, N, d = 1, 2, 2, 256, 128
    mask = np.ones((1, 1, N, N), dtype=bool)
    mask[0, 0, [0, 5, 130, 255]] = False
    O, lse, g, Or, lr, ref = _run(cuda_lib, (B, H, Hkv, N, N, d), False, None, None, mask, seed=43000)
    for r in (0, 5, 130, 255):
        assert np.all(O[:, :, r] == 0) and np.all(np.isneginf(lse[:, :, r])) and np.all(g[0][:, :, r] == 0)
    _check_forward(O, lse, Or, lr, "dead rows")
    check_grads(g, ref, "dead rows")


def test_keys_nobody_sees_get_zero_gradients(cuda_lib):
    # Key length 100 of 600: keys 100.. are padding for every query.
    shape = (1, 2, 2, 300, 600, 128)
    O, lse, g, Or, lr, ref = _run(cuda_lib, shape, False, None, [100], None, seed=44000)
    assert np.all(g[1][:, :, 100:] == 0) and np.all(g[2][:, :, 100:] == 0)
    check_grads(g, ref, "padding keys")


@pytest.mark.parametrize("d,N", [(128, 777), (96, 333), (64, 461)])
def test_plain_causal_through_the_masked_path_is_the_dense_result(cuda_lib, d, N):
    # No window, no lengths, no mask: the masked instance visits the same
    # tiles and masks the same entries as the dense causal kernels (which
    # are the persistent ones, so this also checks them against the
    # launch-per-unit kernels bit for bit, epilogues of every head dim
    # included).
    B, H, Hkv = 2, 4, 2
    q, k, v, do = (dev(x) for x in _problem(B, H, Hkv, N, N, d, 45000 + d))
    for causal in (False, True):
        Od, ld = cuda_lib.forward(q, k, v, 0.1, causal)
        gd = cuda_lib.backward(q, k, v, Od, ld, do, 0.1, causal)
        Om, lm = cuda_lib.forward_masked(q, k, v, 0.1, causal)
        gm = cuda_lib.backward_masked(q, k, v, Om, lm, do, 0.1, causal)
        assert np.array_equal(host(Om), host(Od)) and np.array_equal(host(lm), host(ld))
        for a, b in zip(gm, gd):
            assert np.array_equal(host(a), host(b))


def test_masked_backward_is_deterministic(cuda_lib):
    shape = (2, 4, 2, 300, 300, 96)
    mask = _mask("batch", 2, 4, 300, 300, 46000)
    a = _run(cuda_lib, shape, True, (120, -1), [300, 200], mask, seed=46001)[2]
    b = _run(cuda_lib, shape, True, (120, -1), [300, 200], mask, seed=46001)[2]
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_mask_bytes_nonzero_values_and_unaligned_base(cuda_lib):
    # Any nonzero byte marks a visible key, whether the packer reads the rows
    # 16 bytes at a time (Nk a multiple of 16, base 16-byte aligned) or byte
    # by byte (base one byte past the allocation's start): both give the
    # result of the same mask as 0 / 1 bytes.
    import torch
    B, H, Hkv, N, d = 1, 2, 2, 512, 64
    q, k, v, do = (dev(x) for x in _problem(B, H, Hkv, N, N, d, 47000))
    mask = _mask("batch", B, H, N, N, 47001)
    codes = np.where(mask, np.random.default_rng(47002).integers(1, 256, mask.shape), 0).astype(np.uint8)
    ref = _t(mask.astype(np.uint8), torch.uint8)
    aligned = _t(codes, torch.uint8)
    buf = torch.zeros(codes.size + 1, dtype=torch.uint8, device="cuda")
    shifted = buf[1:].view(codes.shape)
    shifted.copy_(aligned)
    assert shifted.data_ptr() % 16 == 1
    O0, l0 = cuda_lib.forward_masked(q, k, v, 0.125, False, None, None, ref)
    g0 = cuda_lib.backward_masked(q, k, v, O0, l0, do, 0.125, False, None, None, ref)
    for m in (aligned, shifted):
        O1, l1 = cuda_lib.forward_masked(q, k, v, 0.125, False, None, None, m)
        g1 = cuda_lib.backward_masked(q, k, v, O1, l1, do, 0.125, False, None, None, m)
        assert np.array_equal(host(O1), host(O0)) and np.array_equal(host(l1), host(l0))
        for a, b in zip(g1, g0):
            assert np.array_equal(host(a), host(b))
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK


def test_masked_stage_orders(cuda_lib):
    # Stages 8 then 2 (dQ forming the row vectors and packing the mask, then
    # dK / dV) are attn_bwd_masked bit for bit; 1, 2, 4 (prep and packing,
    # dK / dV, dQ) differ only in D's rounding.  Other stage words are
    # refused.
    import torch
    from tests.parity import check_same_but_rounding
    B, H, Hkv, N, d = 2, 4, 2, 384, 128
    q, k, v, do = (dev(x) for x in _problem(B, H, Hkv, N, N, d, 48000))
    mask = _mask("documents", B, H, N, N, 48001)
    tm = _t(mask.astype(np.uint8), torch.uint8)
    O, lse = cuda_lib.forward_masked(q, k, v, 0.1, True, (200, -1), None, tm)
    want = [host(g) for g in cuda_lib.backward_masked(q, k, v, O, lse, do, 0.1, True, (200, -1), None, tm)]
    m = cuda_lib.make_mask((200, -1), None, tm, B, H)
    wsb = cuda_lib.attn_masked_workspace_size(B, H, Hkv, N, N, d, m, 1)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    sp = torch.cuda.current_stream().cuda_stream
    P = lambda t: t.data_ptr()
    for order in ((8, 2), (1, 2, 4)):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        for st in order:
            assert cuda_lib.attn_bwd_masked_stages(P(q), P(k), P(v), P(O), P(lse), P(do), P(dq), P(dk), P(dv),
                                                   B, H, Hkv, N, N, d, 0.1, 1, m, P(ws), wsb, st, sp) == 0
        got = [host(g) for g in (dq, dk, dv)]
        if order == (8, 2):
            for g, w in zip(got, want):
                assert np.array_equal(g, w)
        else:
            check_same_but_rounding(got, want, "masked stages 1, 2, 4")
    for bad in (0, 16):
        assert cuda_lib.attn_bwd_masked_stages(P(q), P(k), P(v), P(O), P(lse), P(do), P(dq), P(dk), P(dv),
                                               B, H, Hkv, N, N, d, 0.1, 1, m, P(ws), wsb, bad,
                                               sp) == cuda_lib.Status.INVALID_ARG
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK


def _bias(shape, seed, dead=0.1):
    """Finite biases in [-4, 4) with a share of -inf entries."""
    rng = np.random.default_rng(seed)
    b = rng.uniform(-4.0, 4.0, shape).astype(np.float32)
    b[rng.random(shape) < dead] = -np.inf
    return b


BIAS_CASES = [
    # (B, H, Hkv, Nq, Nk, d), causal, window, key_lengths, bool mask kind, bias shape kind
    ((2, 4, 2, 300, 300, 128), True, None, None, None, "full"),     # per (batch, head), causal
    ((1, 4, 4, 513, 513, 64), False, None, None, None, "shared"),   # one plane for all
    ((2, 2, 1, 260, 700, 96), True, None, None, None, "batch"),     # Nq < Nk, GQA
    ((2, 4, 2, 384, 384, 128), True, (150, -1), [384, 200], "batch", "head"),  # with every other mask
    # Nk a multiple of 8: a bf16 bias is staged by TMA (the others load it per thread)
    ((1, 4, 4, 520, 520, 64), False, None, None, None, "shared"),   # ragged last key tile
    ((2, 2, 1, 264, 712, 96), True, None, None, None, "batch"),     # Nq < Nk, GQA
]


@pytest.mark.parametrize("bias_dtype", ["float32", "bfloat16"])
@pytest.mark.parametrize("case", BIAS_CASES, ids=lambda c: "B%dH%dKV%dQ%dK%dd%d" % c[0] + f"_c{int(c[1])}_{c[4]}_{c[5]}")
def test_additive_mask_matches_oracle(cuda_lib, case, bias_dtype):
    import torch
    shape, causal, window, kl, kind, bkind = case
    B, H, Hkv, Nq, Nk, d = shape
    q, k, v, do = _problem(B, H, Hkv, Nq, Nk, d, 49000 + Nq)
    mask = _mask(kind, B, H, Nq, Nk, 49100 + Nq)
    bshape = {"full": (B, H, Nq, Nk), "batch": (B, 1, Nq, Nk), "head": (1, H, Nq, Nk), "shared": (1, 1, Nq, Nk)}
    bias = _bias(bshape[bkind], 49200 + Nq)
    if bias_dtype == "bfloat16":  # the values a bf16 bias holds (round to nearest even); -inf stays -inf
        bias = round_bf16(bias)
    s = 1 / math.sqrt(d)
    kt = _t(np.asarray(kl, dtype=np.int32), torch.int32) if kl is not None else None
    mt = _t(mask.astype(np.uint8), torch.uint8) if mask is not None else None
    bt = _t(bias, getattr(torch, bias_dtype))
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    O, lse = cuda_lib.forward_masked(tq, tk, tv, s, causal, window, kt, mt, bt)
    g = cuda_lib.backward_masked(tq, tk, tv, O, lse, tdo, s, causal, window, kt, mt, bt)
    assert cuda_lib.attn_get_device_status(None) == cuda_lib.Status.OK
    Or, lr = oracle.attention_masked_forward(q, k, v, s, causal, window, kl, mask, bias)
    ref = oracle.attention_masked_backward(q, k, v, do, s, causal, window, kl, mask, bias)
    _check_forward(host(O), host(lse), Or, lr, str(case))
    check_grads([host(x) for x in g], ref, str(case))


def test_additive_mask_of_zeros_and_neg_inf_is_the_boolean_mask(cuda_lib):
    # bias = 0 where the boolean mask is True and -inf where it is False
    # gives the boolean mask's result (up to the extra add of zero).
    import torch
    B, H, Hkv, N, d = 2, 2, 2, 320, 128
    q, k, v, do = (dev(x) for x in _problem(B, H, Hkv, N, N, d, 49500))
    mask = _mask("batch", B, H, N, N, 49501)
    bias = np.where(mask, 0.0, -np.inf).astype(np.float32)
    Om, lm = cuda_lib.forward_masked(q, k, v, 0.1, False, None, None, _t(mask.astype(np.uint8), torch.uint8))
    Ob, lb = cuda_lib.forward_masked(q, k, v, 0.1, False, None, None, None, _t(bias, torch.float32))
    # (the boolean mask also skips the tiles it hides; the bias path visits
    # them and adds exact zeros)
    assert np.abs(host(Om) - host(Ob)).max() <= 2 ** -8
    assert np.abs(host(lm) - host(lb)).max() <= 1e-5


def test_rows_whose_bias_hides_every_key(cuda_lib):
    import torch
    B, H, Hkv, N, d = 1, 2, 2, 200, 64
    q, k, v, do = _problem(B, H, Hkv, N, N, d, 49600)
    bias = _bias((1, 1, N, N), 49601, 0.0)
    bias[0, 0, [3, 150]] = -np.inf
    bt = _t(bias, torch.float32)
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    O, lse = cuda_lib.forward_masked(tq, tk, tv, 0.125, False, None, None, None, bt)
    g = cuda_lib.backward_masked(tq, tk, tv, O, lse, tdo, 0.125, False, None, None, None, bt)
    O, lse = host(O), host(lse)
    for r in (3, 150):
        assert np.all(O[:, :, r] == 0) and np.all(np.isneginf(lse[:, :, r])) and np.all(host(g[0])[:, :, r] == 0)
    Or, lr = oracle.attention_masked_forward(q, k, v, 0.125, False, None, None, None, bias)
    _check_forward(O, lse, Or, lr, "bias dead rows")
    check_grads([host(x) for x in g], oracle.attention_masked_backward(q, k, v, do, 0.125, False, None, None, None,
                                                                      bias), "bias dead rows")


@pytest.mark.parametrize("shape,causal", [((2, 4, 2, 300, 384, 128), True), ((1, 2, 2, 520, 520, 64), False)])
def test_bf16_bias_staged_equals_loaded(cuda_lib, shape, causal):
    """A bf16 additive mask with Nk a multiple of 8 on a 16-byte boundary is
    staged by TMA; the same values one element into a buffer (2-byte aligned)
    go through per-thread loads.  Both add the same values in the same order:
    O and lse agree bit for bit."""
    import torch
    B, H, Hkv, Nq, Nk, d = shape
    q, k, v, _ = _problem(B, H, Hkv, Nq, Nk, d, 49500 + Nq)
    bias = round_bf16(_bias((1, H, Nq, Nk), 49600 + Nq))
    s = 1 / math.sqrt(d)
    staged = _t(bias, torch.bfloat16)
    buf = torch.zeros(bias.size + 8, dtype=torch.bfloat16, device="cuda")
    buf[1:1 + bias.size] = staged.reshape(-1)
    loaded = buf[1:1 + bias.size].view(1, H, Nq, Nk)
    assert staged.data_ptr() % 16 == 0 and loaded.data_ptr() % 16 != 0
    tq, tk, tv = dev(q), dev(k), dev(v)
    O1, l1 = cuda_lib.forward_masked(tq, tk, tv, s, causal, None, None, None, staged)
    O2, l2 = cuda_lib.forward_masked(tq, tk, tv, s, causal, None, None, None, loaded)
    assert torch.equal(O1, O2) and torch.equal(l1, l2)


def test_bf16_bias_staged_equals_loaded_backward(cuda_lib):
    """The dK/dV kernel stages a bf16 additive mask by TMA unless a boolean
    mask comes with it; an all-visible boolean mask changes no value but
    selects per-thread loads.  dQ, dK and dV agree bit for bit."""
    import torch
    B, H, Hkv, Nq, Nk, d = 1, 2, 2, 384, 384, 128
    q, k, v, do = _problem(B, H, Hkv, Nq, Nk, d, 49700)
    bias = _t(round_bf16(_bias((1, H, Nq, Nk), 49800)), torch.bfloat16)
    ones = _t(np.ones((1, 1, Nq, Nk), dtype=np.uint8), torch.uint8)
    s = 1 / math.sqrt(d)
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    O, lse = cuda_lib.forward_masked(tq, tk, tv, s, True, None, None, None, bias)
    staged = cuda_lib.backward_masked(tq, tk, tv, O, lse, tdo, s, True, None, None, None, bias)
    loaded = cuda_lib.backward_masked(tq, tk, tv, O, lse, tdo, s, True, None, None, ones, bias)
    for a, b, name in zip(staged, loaded, ("dQ", "dK", "dV")):
        assert torch.equal(a, b), name
