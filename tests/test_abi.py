"""C-ABI checks that need no GPU: the library builds, loads, exports every
function include/attn.h declares, and rejects bad arguments before touching
the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import scaled_dot_product_08_gb300 as sdpa
    sdpa.build()
    return sdpa.load()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("attn_fwd", "attn_bwd", "attn_bwd_workspace_size", "attn_get_device_status",
              "attn_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    import scaled_dot_product_08_gb300 as sdpa
    for s in sdpa.Status:
        assert sdpa.attn_status_string(int(s)) == "ATTN_" + ("OK" if s == 0 else "ERR_" + s.name)
    assert sdpa.attn_status_string(99) == "ATTN_ERR_UNKNOWN"
    assert lib.attn_abi_version() == 3


def test_workspace_size_formula(lib):
    import scaled_dot_product_08_gb300 as sdpa
    # two float32 row vectors (-D and -lse*log2 e) of B*H*Npad rows each
    assert sdpa.attn_bwd_workspace_size(8, 16, 16, 4096, 128) == 8 * 16 * 4096 * 2 * 4
    assert sdpa.attn_bwd_workspace_size(1, 2, 1, 129, 64) == 2 * 256 * 2 * 4
    assert sdpa.attn_bwd_workspace_size(1, 3, 2, 128, 64) == 0      # H % Hkv != 0
    assert sdpa.attn_bwd_workspace_size(1, 2, 2, 128, 80) == 0      # unsupported d
    assert sdpa.attn_bwd_workspace_size(1, 2, 2, 0, 64) == 0


# Argument errors are detected on the host before any CUDA call, so they can
# be checked here without a GPU.  Fake, 16-byte aligned addresses are never
# dereferenced because a shape error is reported first.
FAKE = 0x10000


@pytest.mark.parametrize("B,H,Hkv,N,d,expect", [
    (1, 2, 2, 128, 80, 2),    # d not supported
    (1, 2, 2, 128, 32, 2),
    (1, 3, 2, 128, 64, 2),    # H % Hkv
    (1, 2, 2, 0, 64, 2),      # N < 1
    (0, 2, 2, 16, 64, 2),     # B < 1
    (1, 2, 0, 16, 64, 2),     # Hkv < 1
])
def test_fwd_rejects_bad_shapes(lib, B, H, Hkv, N, d, expect):
    import scaled_dot_product_08_gb300 as sdpa
    st = sdpa.attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, B, H, Hkv, N, d, 0.125, 0, None)
    assert st == expect


@pytest.mark.parametrize("scale,causal", [(float("nan"), 0), (float("inf"), 0), (0.0, 0), (-0.1, 1), (0.1, 2)])
def test_fwd_rejects_bad_scale_or_flag(lib, scale, causal):
    import scaled_dot_product_08_gb300 as sdpa
    assert sdpa.attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 2, 64, 64, scale, causal, None) == sdpa.Status.INVALID_ARG


def test_fwd_rejects_null_and_misaligned(lib):
    import scaled_dot_product_08_gb300 as sdpa
    assert sdpa.attn_fwd(0, FAKE, FAKE, FAKE, FAKE, 1, 2, 2, 64, 64, 0.1, 0, None) == sdpa.Status.INVALID_ARG
    assert sdpa.attn_fwd(FAKE + 8, FAKE, FAKE, FAKE, FAKE, 1, 2, 2, 64, 64, 0.1, 0, None) == sdpa.Status.MISALIGNED


def test_bwd_rejects_bad_arguments(lib):
    import scaled_dot_product_08_gb300 as sdpa
    args = [FAKE] * 9
    assert sdpa.attn_bwd(*args, FAKE, 1 << 20, 1, 2, 2, 64, 96 - 16, 0.1, 0, None) == sdpa.Status.UNSUPPORTED_SHAPE
    assert sdpa.attn_bwd(*args, FAKE, 1 << 20, 1, 2, 2, 64, 64, float("nan"), 0, None) == sdpa.Status.INVALID_ARG
    bad = list(args)
    bad[6] = FAKE + 4
    assert sdpa.attn_bwd(*bad, FAKE, 1 << 20, 1, 2, 2, 64, 64, 0.1, 0, None) == sdpa.Status.MISALIGNED


def test_bwd_noalloc_checks_arguments_before_its_scratch(lib):
    # attn_bwd_noalloc reports attn_bwd's own status for a bad argument
    # before it looks up its scratch array (which needs a device).
    import scaled_dot_product_08_gb300 as sdpa
    args = [FAKE] * 9
    assert sdpa.attn_bwd_noalloc(*args, 1, 2, 2, 64, 80, 0.1, 0, None) == sdpa.Status.UNSUPPORTED_SHAPE
    assert sdpa.attn_bwd_noalloc(*args, 1, 2, 2, 64, 64, float("nan"), 0, None) == sdpa.Status.INVALID_ARG
    assert sdpa.attn_bwd_noalloc(*args, 1, 2, 2, 64, 64, 0.1, 2, None) == sdpa.Status.INVALID_ARG
    bad = list(args)
    bad[7] = FAKE + 4
    assert sdpa.attn_bwd_noalloc(*bad, 1, 2, 2, 64, 64, 0.1, 0, None) == sdpa.Status.MISALIGNED
    bad[7] = 0
    assert sdpa.attn_bwd_noalloc(*bad, 1, 2, 2, 64, 64, 0.1, 0, None) == sdpa.Status.INVALID_ARG


def test_debug_drop_load_checks_its_arguments(lib):
    # The failure-path test hook arms nothing on bad arguments (host only).
    import scaled_dot_product_08_gb300 as sdpa
    assert sdpa.attn_debug_drop_load(7, 0, 20000) == sdpa.Status.INVALID_ARG
    assert sdpa.attn_debug_drop_load(-1, 0, 20000) == sdpa.Status.INVALID_ARG
    assert sdpa.attn_debug_drop_load(0, -1, 20000) == sdpa.Status.INVALID_ARG
    assert sdpa.attn_debug_drop_load(0, 0, 999) == sdpa.Status.INVALID_ARG
    assert sdpa.attn_debug_drop_load(0, 0, 60000001) == sdpa.Status.INVALID_ARG


def _decode_chunks(B, Hkv, Nk):
    # The documented chunk plan: whole 128-key tiles, about 1216 CTAs in all
    # (ceil(1216 / (B * Hkv)) chunks while tiles last).
    tiles = -(-Nk // 128)
    want = -(-1216 // (B * Hkv))
    ns0 = min(tiles, want)
    per = -(-tiles // ns0)
    return -(-tiles // per)


@pytest.mark.parametrize("B,H,Hkv,Nq,Nk,d", [(8, 32, 8, 1, 32768, 128), (1, 8, 8, 4, 4096, 64),
                                             (2, 16, 2, 2, 1000, 96), (1, 1, 1, 1, 1, 128)])
def test_decode_workspace_size_formula(lib, B, H, Hkv, Nq, Nk, d):
    import scaled_dot_product_08_gb300 as sdpa
    ns = _decode_chunks(B, Hkv, Nk)
    assert sdpa.attn_decode_workspace_size(B, H, Hkv, Nq, Nk, d) == B * H * Nq * ns * (d + 1) * 4


def test_decode_rejects_bad_arguments(lib):
    import scaled_dot_product_08_gb300 as sdpa
    S = sdpa.Status
    f = lambda *a: sdpa.attn_decode(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, *a)
    assert f(1, 8, 8, 5, 4, 128, 0.1, 0, None) == S.UNSUPPORTED_SHAPE      # Nq > Nk
    assert f(1, 8, 8, 0, 4, 128, 0.1, 0, None) == S.UNSUPPORTED_SHAPE      # Nq < 1
    assert f(1, 64, 1, 3, 64, 128, 0.1, 0, None) == S.UNSUPPORTED_SHAPE    # G * Nq = 192 > 128
    assert f(1, 8, 3, 1, 64, 128, 0.1, 0, None) == S.UNSUPPORTED_SHAPE     # Hkv does not divide H
    assert f(1, 8, 8, 1, 64, 80, 0.1, 0, None) == S.UNSUPPORTED_SHAPE      # d
    assert f(1, 8, 8, 1, 64, 128, float("inf"), 0, None) == S.INVALID_ARG
    assert f(1, 8, 8, 1, 64, 128, 0.1, 2, None) == S.INVALID_ARG
    assert sdpa.attn_decode(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 1, 8, 8, 1, 64, 128, 0.1, 0, None) == S.WORKSPACE
    assert sdpa.attn_decode(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 1 << 30, 1, 8, 8, 1, 64, 128, 0.1, 0, None) == S.WORKSPACE
    assert sdpa.attn_decode(FAKE + 4, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, 1, 8, 8, 1, 64, 128, 0.1, 0,
                            None) == S.MISALIGNED
    assert sdpa.attn_decode_workspace_size(1, 8, 8, 5, 4, 128) == 0


def test_fwd_cross_rejects_bad_arguments(lib):
    import scaled_dot_product_08_gb300 as sdpa
    S = sdpa.Status
    f = lambda *a: sdpa.attn_fwd_cross(FAKE, FAKE, FAKE, FAKE, FAKE, *a)
    assert f(1, 2, 2, 300, 200, 128, 0.1, 1, None) == S.UNSUPPORTED_SHAPE   # causal with Nq > Nk
    assert f(1, 2, 2, 0, 200, 128, 0.1, 0, None) == S.UNSUPPORTED_SHAPE     # Nq < 1
    assert f(1, 2, 2, 10, 0, 128, 0.1, 0, None) == S.UNSUPPORTED_SHAPE      # Nk < 1
    assert f(1, 2, 2, 10, 20, 80, 0.1, 0, None) == S.UNSUPPORTED_SHAPE      # d
    assert f(1, 2, 2, 10, 20, 128, -1.0, 0, None) == S.INVALID_ARG


def test_bwd_cross_rejects_bad_arguments(lib):
    import scaled_dot_product_08_gb300 as sdpa
    S = sdpa.Status
    ws = sdpa.attn_bwd_workspace_size(1, 2, 2, 300, 128)

    def f(Nq, Nk, d, scale, causal, wsb=ws, w=FAKE, q=FAKE):
        return sdpa.attn_bwd_cross(q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, w, wsb,
                                   1, 2, 2, Nq, Nk, d, scale, causal, None)
    assert f(300, 200, 128, 0.1, 1) == S.UNSUPPORTED_SHAPE   # causal with Nq > Nk
    assert f(0, 200, 128, 0.1, 0) == S.UNSUPPORTED_SHAPE     # Nq < 1
    assert f(10, 0, 128, 0.1, 0) == S.UNSUPPORTED_SHAPE      # Nk < 1
    assert f(10, 20, 80, 0.1, 0) == S.UNSUPPORTED_SHAPE      # d
    assert f(10, 20, 128, -1.0, 0) == S.INVALID_ARG
    assert f(10, 20, 128, 0.1, 2) == S.INVALID_ARG
    # the workspace is sized by the query rows
    assert f(300, 400, 128, 0.1, 1, wsb=ws - 1) == S.WORKSPACE
    assert f(300, 400, 128, 0.1, 1, w=0) == S.WORKSPACE
    assert f(300, 400, 128, 0.1, 1, q=FAKE + 2) == S.MISALIGNED


def test_bwd_cross_stages_reject_bad_arguments(lib):
    import scaled_dot_product_08_gb300 as sdpa
    S = sdpa.Status
    ws = sdpa.attn_bwd_workspace_size(1, 2, 2, 300, 128)
    g = lambda Nq, Nk, causal: sdpa.attn_bwd_grad_cross(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws,
                                                        1, 2, 2, Nq, Nk, 128, 0.1, causal, None)
    q = lambda Nq, Nk, causal: sdpa.attn_bwd_dq_cross(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws,
                                                      1, 2, 2, Nq, Nk, 128, 0.1, causal, None)
    for f in (g, q):
        assert f(300, 200, 1) == S.UNSUPPORTED_SHAPE
        assert f(300, 0, 0) == S.UNSUPPORTED_SHAPE
        assert f(385, 400, 0) == S.WORKSPACE      # workspace sized for 300 (padded: 384) query rows


def test_bwd_dq_rows_rejects_bad_arguments(lib):
    # attn_bwd_dq_rows also reads o and lse: both are checked like the rest.
    import scaled_dot_product_08_gb300 as sdpa
    S = sdpa.Status
    ws = sdpa.attn_bwd_workspace_size(1, 2, 2, 300, 128)

    def f(Nq=300, Nk=400, causal=0, wsb=ws, o=FAKE, lse=FAKE, scale=0.1, d=128):
        return sdpa.attn_bwd_dq_rows(FAKE, FAKE, FAKE, o, lse, FAKE, FAKE, FAKE, wsb, 1, 2, 2, Nq, Nk, d, scale,
                                     causal, None)
    assert f(Nq=300, Nk=200, causal=1) == S.UNSUPPORTED_SHAPE   # a causal row would see no key
    assert f(d=80) == S.UNSUPPORTED_SHAPE
    assert f(scale=float("inf")) == S.INVALID_ARG
    assert f(causal=2) == S.INVALID_ARG
    assert f(wsb=ws - 1) == S.WORKSPACE
    assert f(o=0) == S.INVALID_ARG
    assert f(lse=0) == S.INVALID_ARG
    assert f(o=FAKE + 2) == S.MISALIGNED


def test_varlen_rejects_bad_arguments(lib):
    import scaled_dot_product_08_gb300 as sdpa
    S = sdpa.Status
    f = lambda B, tq, tk, mq, mk, d=128, scale=0.1, causal=0: sdpa.attn_fwd_varlen(
        FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, 4, 2, tq, tk, mq, mk, d, scale, causal, None)
    assert f(2, 0, 10, 8, 8) == S.UNSUPPORTED_SHAPE        # no query rows
    assert f(2, 10, 0, 8, 8) == S.UNSUPPORTED_SHAPE        # no key rows
    assert f(2, 17, 10, 8, 8) == S.UNSUPPORTED_SHAPE       # total_q > B * max_seqlen_q
    assert f(2, 10, 10, 0, 8) == S.UNSUPPORTED_SHAPE       # max_seqlen_q < 1
    assert f(2, 10, 10, 8, 8, d=80) == S.UNSUPPORTED_SHAPE
    assert f(2, 10, 10, 8, 8, scale=float("nan")) == S.INVALID_ARG
    assert f(2, 10, 10, 8, 8, causal=3) == S.INVALID_ARG
    ws = sdpa.attn_bwd_varlen_workspace_size(2, 4, 2, 10, 128)
    assert ws == 4 * 8 * (((10 + 264 + 3) // 4) * 4 + 128)
    assert sdpa.attn_bwd_varlen_workspace_size(2, 4, 2, 0, 128) == 0
    g = lambda wsb, w=FAKE: sdpa.attn_bwd_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                                 w, wsb, 2, 4, 2, 10, 10, 8, 8, 128, 0.1, 1, None)
    assert g(ws - 1) == S.WORKSPACE
    assert g(ws, w=0) == S.WORKSPACE


def test_masked_rejects_bad_arguments(lib):
    import scaled_dot_product_08_gb300 as sdpa
    S = sdpa.Status
    M = lambda wl=-1, wr=-1, kl=0, m=0, mb=1, mh=1, bias=0, bb=1, bh=1, bf=0: sdpa.AttnMask(
        wl, wr, kl, m, mb, mh, bias, bb, bh, bf)
    f = lambda mask, ws=FAKE, wsb=1 << 20, causal=0: sdpa.attn_fwd_masked(
        FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 2, 100, 300, 128, 0.1, causal, mask, ws, wsb, None)
    assert f(M(wl=-2)) == S.INVALID_ARG
    assert f(M(wr=-3)) == S.INVALID_ARG
    assert f(M(kl=FAKE + 2)) == S.MISALIGNED                 # key lengths are int32
    assert f(M(m=FAKE, mb=3)) == S.INVALID_ARG               # mask batch must be 1 or B
    assert f(M(m=FAKE, mh=2)) == S.INVALID_ARG               # mask heads must be 1 or H
    need = sdpa.attn_masked_workspace_size(2, 4, 2, 100, 300, 128, M(m=FAKE, mb=2), 0)
    assert need == 2 * 100 * 12 * 4 + 16                     # one bit per (query, key) + tile flags
    assert f(M(m=FAKE, mb=2), wsb=need - 1) == S.WORKSPACE
    assert f(M(m=FAKE, mb=2), ws=0) == S.WORKSPACE
    assert sdpa.attn_masked_workspace_size(2, 4, 2, 100, 300, 128, M(), 0) == 0
    assert sdpa.attn_masked_workspace_size(2, 4, 2, 100, 300, 128, M(), 1) == sdpa.attn_bwd_workspace_size(
        2, 4, 2, 100, 128)
    g = lambda stages, wsb=1 << 20: sdpa.attn_bwd_masked_stages(
        FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 2, 100, 300, 128, 0.1, 0, M(), FAKE, wsb,
        stages, None)
    assert g(0) == S.INVALID_ARG and g(16) == S.INVALID_ARG and g(17) == S.INVALID_ARG
    assert g(7, wsb=16) == S.WORKSPACE
    # the additive mask: float32 (4-byte aligned) or bf16 (2-byte aligned), (1 or B, 1 or H, Nq, Nk)
    assert f(M(bias=FAKE + 2)) == S.MISALIGNED
    assert f(M(bias=FAKE + 1, bf=1)) == S.MISALIGNED
    assert f(M(bias=FAKE, bf=2)) == S.INVALID_ARG
    for bf, size in ((0, 4), (1, 2)):  # the backward's transpose of the bias, in its own type
        assert sdpa.attn_masked_workspace_size(2, 4, 2, 100, 300, 128, M(bias=FAKE, bb=2, bf=bf), 1) == (
            sdpa.attn_bwd_workspace_size(2, 4, 2, 100, 128) + -(-2 * 100 * 300 * size // 16) * 16)
    assert f(M(bias=FAKE, bb=3)) == S.INVALID_ARG
    assert f(M(bias=FAKE, bh=2)) == S.INVALID_ARG
    # its transpose (float32, Nk x Nq per plane) joins the backward's workspace only
    assert sdpa.attn_masked_workspace_size(2, 4, 2, 100, 300, 128, M(bias=FAKE, bh=4), 0) == 0
    assert sdpa.attn_masked_workspace_size(2, 4, 2, 100, 300, 128, M(bias=FAKE, bh=4), 1) == \
        sdpa.attn_bwd_workspace_size(2, 4, 2, 100, 128) + 4 * 100 * 300 * 4


def test_fp8_rejects_bad_arguments(lib):
    import scaled_dot_product_08_gb300 as sdpa
    S = sdpa.Status
    f = lambda d=128, scale=0.1, qs=1.0, ks=1.0, vs=1.0, causal=0, Nq=100, Nk=200: sdpa.attn_fwd_fp8(
        FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 2, Nq, Nk, d, scale, qs, ks, vs, causal, None)
    assert f(d=80) == S.UNSUPPORTED_SHAPE  # head_dim 64, 96 and 128 are served
    assert f(d=256) == S.UNSUPPORTED_SHAPE
    assert f(qs=0.0) == S.INVALID_ARG
    assert f(vs=float("inf")) == S.INVALID_ARG
    assert f(ks=-1.0) == S.INVALID_ARG
    assert f(scale=float("nan")) == S.INVALID_ARG
    assert f(causal=1, Nq=300, Nk=200) == S.UNSUPPORTED_SHAPE


def test_decode_paged_rejects_bad_arguments(lib):
    import scaled_dot_product_08_gb300 as sdpa
    S = sdpa.Status
    ws = sdpa.attn_decode_paged_workspace_size(2, 8, 2, 1, 16, 64, 128)
    assert ws == sdpa.attn_decode_workspace_size(2, 8, 2, 1, 16 * 64, 128)
    f = lambda ps=16, npg=10, mp=64, d=128, wsb=ws, causal=0: sdpa.attn_decode_paged(
        FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, wsb, 2, 8, 2, 1, ps, npg, mp, d, 0.1, causal, None)
    assert f(ps=48) == S.UNSUPPORTED_SHAPE     # neither divides 128 nor a multiple of it
    assert f(ps=100) == S.UNSUPPORTED_SHAPE
    assert f(ps=8) == S.UNSUPPORTED_SHAPE
    assert f(npg=0) == S.UNSUPPORTED_SHAPE
    assert f(mp=0) == S.UNSUPPORTED_SHAPE
    assert f(d=80) == S.UNSUPPORTED_SHAPE
    assert f(wsb=ws - 1) == S.WORKSPACE
    assert sdpa.attn_decode_paged_workspace_size(2, 8, 2, 1, 48, 64, 128) == 0
