"""Full-size parity of the workloads bench.py times beyond the first path
(cross attention, chunked prefill, packed varlen, masks, the additive mask,
FP8, decode): each test makes the benchmark's call on the benchmark's seeded
inputs, then compares every output element with the fp64 oracle, one whole
head (or sequence and head) per worker process (tests/oracle_pool.py).
Tolerances are those of the five reference workloads (O max |err| <= 1e-2,
mean <= 1e-3, lse <= 1e-3, gradients 2e-2 relative Frobenius over each
tensor); FP8 uses its own (tests/fp8_model.py)."""
import numpy as np
import pytest

import oracle
from sdpa_inputs import (e4m3_decode, make_inputs, make_varlen_inputs, prefix_lm_mask, quantize_e4m3,
                         workload)
from tests.oracle_pool import cross_head, fp8_head, make_pool, masked_head, window_head
from tests.parity import GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS, check_o_lse, dev, host

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _f32(t):
    import torch
    return t.detach().to(torch.float32).cpu().numpy()


def _run_pool(fn, tasks, bytes_per_worker):
    pool, _ = make_pool(bytes_per_worker)
    with pool:
        return list(pool.imap_unordered(fn, tasks))


def _check_parts(name, parts, grads=False):
    o_max = max(p["o_max"] for p in parts)
    o_mean = sum(p["o_sum"] for p in parts) / sum(p["o_n"] for p in parts)
    lse_max = max(p["lse_max"] for p in parts)
    worst = max(parts, key=lambda p: p["o_max"])
    print(f"\n{name}: {len(parts)} units, every element: O max {o_max:.3e} mean {o_mean:.3e}, lse max {lse_max:.3e}"
          f" (largest O error at {worst['head']}, row {worst['o_max_at'][0]})", end="")
    assert all(p["finite"] for p in parts), f"{name}: non-finite output"
    assert all(p["dead_ok"] for p in parts), f"{name}: a row that sees no key is not O = 0, lse = -inf"
    assert o_max <= O_MAX_ABS, f"{name}: O max abs err {o_max:.3e}"
    assert o_mean <= O_MEAN_ABS, f"{name}: O mean abs err {o_mean:.3e}"
    assert lse_max <= LSE_MAX_ABS, f"{name}: lse max abs err {lse_max:.3e}"
    if grads:
        for g in ("dq", "dk", "dv"):
            assert all(p[g + "_finite"] for p in parts), f"{name}: {g} not finite"
            e = float(np.sqrt(sum(p[g + "_e2"] for p in parts) / sum(p[g + "_r2"] for p in parts)))
            print(f"\n{name} {g}: rel Frobenius {e:.3e} over the tensor", end="")
            assert e <= GRAD_REL_FRO, f"{name}: {g} rel Frobenius err {e:.3e}"


def test_cp1_chunked_prefill(cuda_lib):
    w = workload("cp1")
    x = make_inputs(w)
    O, lse = cuda_lib.forward_cross(dev(x["q"]), dev(x["k"]), dev(x["v"]), w.softmax_scale, w.causal)
    O, lse = _f32(O), _f32(lse)
    G = w.H // w.Hkv
    tasks = ((x["q"][b, h], x["k"][b, h // G], x["v"][b, h // G], None, O[b, h], lse[b, h], None, None, None,
              w.softmax_scale, w.causal, (b, h)) for b in range(w.B) for h in range(w.H))
    _check_parts("cp1", _run_pool(cross_head, tasks, 7 * w.n_queries * w.N * 8))


def test_cx_encoder_decoder_fwd_bwd(cuda_lib):
    w = workload("cx")
    x = make_inputs(w)
    s = w.softmax_scale
    tq, tk, tv, tdo = dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(x["do"])
    O, lse = cuda_lib.forward_cross(tq, tk, tv, s, False)
    dq, dk, dv = (_f32(g) for g in cuda_lib.backward_cross(tq, tk, tv, O, lse, tdo, s, False))
    O, lse = _f32(O), _f32(lse)
    tasks = ((x["q"][b, h], x["k"][b, h], x["v"][b, h], x["do"][b, h], O[b, h], lse[b, h], dq[b, h], dk[b, h],
              dv[b, h], s, False, (b, h)) for b in range(w.B) for h in range(w.H))
    _check_parts("cx", _run_pool(cross_head, tasks, 10 * w.n_queries * w.N * 8), grads=True)


def test_vl1_packed_batch(cuda_lib):
    import torch
    w = workload("vl1")
    x = make_varlen_inputs(w)
    cu, lens = x["cu"], x["lengths"]
    tcu = torch.from_numpy(cu).cuda()
    s, mx = w.softmax_scale, int(lens.max())
    tq, tk, tv, tdo = dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(x["do"])
    O, lse = cuda_lib.forward_varlen(tq, tk, tv, tcu, tcu, mx, mx, s, True)
    dq, dk, dv = (_f32(g) for g in cuda_lib.backward_varlen(tq, tk, tv, O, lse, tdo, tcu, tcu, mx, mx, s, True))
    O, lse = _f32(O), _f32(lse)
    # every sequence and head: packed (total, heads, d) rows a..e of head h
    tasks = ((x["q"][a:e, h], x["k"][a:e, h], x["v"][a:e, h], x["do"][a:e, h], O[a:e, h], lse[h, a:e],
              dq[a:e, h], dk[a:e, h], dv[a:e, h], s, True, (seq, h))
             for seq, (a, e) in enumerate(zip(cu[:-1].tolist(), cu[1:].tolist())) for h in range(w.H))
    _check_parts("vl1", _run_pool(cross_head, tasks, 10 * mx * mx * 8), grads=True)


def test_sw1_sliding_window(cuda_lib):
    w = workload("sw1")
    x = make_inputs(w)
    s, wl = w.softmax_scale, w.window[0]
    O, lse = cuda_lib.forward_masked(dev(x["q"]), dev(x["k"]), dev(x["v"]), s, True, w.window)
    O, lse = _f32(O), _f32(lse)
    G = w.H // w.Hkv
    tasks = ((x["q"][0, h], x["k"][0, h // G], x["v"][0, h // G], O[0, h], lse[0, h], s, wl, (0, h))
             for h in range(w.H))
    _check_parts("sw1", _run_pool(window_head, tasks, 7 * 128 * (wl + 128) * 8 + (1 << 28)))


@pytest.mark.parametrize("name", ["pl1", "ab1", "ab1h"])
def test_masked_fwd_bwd(cuda_lib, name):
    import torch
    from sdpa_inputs import workload_bias
    w = workload(name)
    x = make_inputs(w)
    s = w.softmax_scale
    tq, tk, tv, tdo = dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(x["do"])
    if w.prefix is not None:
        recipe = ("prefix", w.prefix)
        args = (None, None, torch.from_numpy(prefix_lm_mask(w.N, w.prefix).astype(np.uint8)).cuda())
    else:
        recipe = ("distance", w.bias_slope, w.bias_bf16)
        tb = torch.from_numpy(workload_bias(w)).cuda()
        args = (None, None, None, tb.to(torch.bfloat16) if w.bias_bf16 else tb)
    O, lse = cuda_lib.forward_masked(tq, tk, tv, s, w.causal, *args)
    dq, dk, dv = (_f32(g) for g in cuda_lib.backward_masked(tq, tk, tv, O, lse, tdo, s, w.causal, *args))
    O, lse = _f32(O), _f32(lse)
    tasks = ((x["q"][b, h], x["k"][b, h], x["v"][b, h], x["do"][b, h], O[b, h], lse[b, h], dq[b, h], dk[b, h],
              dv[b, h], s, w.causal, recipe, (b, h)) for b in range(w.B) for h in range(w.H))
    _check_parts(name, _run_pool(masked_head, tasks, 12 * w.N * w.N * 8), grads=True)


@pytest.mark.parametrize("name", ["c4f8", "c3cf8"])
def test_fp8_full_size(cuda_lib, name):
    import torch
    from tests.fp8_model import FP8_MODEL_REL_FRO, O_MEAN_ABS_FP8, O_REL_FRO_FP8
    w = workload(name)
    x = make_inputs(w)
    qz = [quantize_e4m3(x[n]) for n in ("q", "k", "v")]
    u8 = lambda a: torch.from_numpy(a).cuda()
    O, lse = cuda_lib.forward_fp8(u8(qz[0][0]), u8(qz[1][0]), u8(qz[2][0]), qz[0][1], qz[1][1], qz[2][1],
                                  w.softmax_scale, True)
    O, lse = _f32(O), _f32(lse)
    deq = [(e4m3_decode(b) * sc).astype(np.float32) for b, sc in qz]
    G = w.H // w.Hkv
    tasks = ((deq[0][0, h], deq[1][0, h // G], deq[2][0, h // G], O[0, h], lse[0, h], w.softmax_scale, True, 0,
              (0, h)) for h in range(w.H))
    parts = _run_pool(fp8_head, tasks, 8 * w.N * w.N * 8)
    worst, worst_m = max(p["rel_fro"] for p in parts), max(p["rel_fro_model"] for p in parts)
    mean = sum(p["o_sum"] for p in parts) / sum(p["o_n"] for p in parts)
    lmax = max(p["lse_max"] for p in parts)
    print(f"\n{name}: {len(parts)} heads: worst rel Frobenius {worst:.3e} (against the rounding model {worst_m:.3e}),"
          f" mean |err| {mean:.3e}, lse max {lmax:.3e}", end="")
    assert all(p["finite"] for p in parts)
    assert worst <= O_REL_FRO_FP8 and worst_m <= FP8_MODEL_REL_FRO
    assert mean <= O_MEAN_ABS_FP8 and lmax <= LSE_MAX_ABS


@pytest.mark.parametrize("name", ["dec1", "dec4"])
def test_decode_full_size(cuda_lib, name):
    w = workload(name)
    x = make_inputs(w)
    O, lse = cuda_lib.decode(dev(x["q"]), dev(x["k"]), dev(x["v"]), w.softmax_scale, w.causal)
    O, lse = host(O), host(lse)
    for b in range(w.B):
        sl = slice(b, b + 1)
        Or, lr = oracle.attention_decode(x["q"][sl], x["k"][sl], x["v"][sl], w.softmax_scale, w.causal)
        check_o_lse(O[sl], lse[sl], Or, lr, f"{name} batch {b}")
