"""Full-size parity of the five reference workloads, every element.

Each test makes the benchmark's call (the launch configuration bench.py
times) on the seeded inputs of one workload, copies every output back, and
compares all of it with the fp64 oracle, one whole head per worker process
(tests/oracle_pool.py):

  c2   B=4  H=16 N=2048 d=128 causal              forward: O, lse
  c3   B=1  H=96 N=4096 d=64  non-causal          forward
  c3c  the same, causal                           forward
  c4   B=1  H=32 Hkv=8 N=8192 d=128 causal, x0.5  forward (GQA)
  c4p  c4 with head_dim 80 zero-padded to 96      forward; the pad columns of
       O must be exactly 0 and the rest equal the unpadded d=80 oracle
  c5   B=8  H=16 N=4096 d=128 causal              forward and backward:
       O, lse, dQ, dK, dV

Tolerances (bf16 inputs, fp32 accumulation): O max |err| <= 1e-2 and mean
|err| <= 1e-3 over every element, lse max |err| <= 1e-3, and dQ, dK, dV a
relative Frobenius error <= 2e-2 over each whole tensor.  The backward runs
on the GPU forward's O and lse, as a training step does; the reference is
the pure oracle, so forward and backward errors are both inside it.
"""
import numpy as np
import pytest

from sdpa_inputs import make_inputs, workload
from tests.oracle_pool import backward_head, forward_head, make_pool
from tests.parity import GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS, dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _f32(t):
    """A device tensor as float32 numpy (exact for bf16 and fp32)."""
    import torch
    return t.detach().to(torch.float32).cpu().numpy()


def _summary(name, parts):
    o_max = max(p["o_max"] for p in parts)
    o_mean = sum(p["o_sum"] for p in parts) / sum(p["o_n"] for p in parts)
    lse_max = max(p["lse_max"] for p in parts)
    worst = max(parts, key=lambda p: p["o_max"])
    print(f"\n{name}: {len(parts)} heads, every element: O max {o_max:.3e} mean {o_mean:.3e}, lse max {lse_max:.3e}"
          f" (largest O error at head {worst['head']}, row {worst['o_max_at'][0]}, column {worst['o_max_at'][1]}:"
          f" {worst['o_max_at'][2]:.6g} against {worst['o_max_at'][3]:.6g})", end="")
    assert all(p["finite"] for p in parts), f"{name}: non-finite output"
    assert o_max <= O_MAX_ABS, f"{name}: O max abs err {o_max:.3e}"
    assert o_mean <= O_MEAN_ABS, f"{name}: O mean abs err {o_mean:.3e}"
    assert lse_max <= LSE_MAX_ABS, f"{name}: lse max abs err {lse_max:.3e}"


@pytest.mark.parametrize("name", ["c2", "c3", "c3c", "c4", "c4p"])
def test_forward_every_element(cuda_lib, name):
    w = workload(name)
    x = make_inputs(w)
    O, lse = cuda_lib.forward(dev(x["q"]), dev(x["k"]), dev(x["v"]), w.softmax_scale, w.causal)
    O, lse = _f32(O), _f32(lse)
    G, d_use = w.H // w.Hkv, (w.d_draw or w.d)
    tasks = ((x["q"][b, h], x["k"][b, h // G], x["v"][b, h // G], O[b, h], lse[b, h], w.softmax_scale, w.causal, 0,
              d_use, (b, h)) for b in range(w.B) for h in range(w.H))
    pool, _ = make_pool(7 * w.N * w.N * 8)
    with pool:
        parts = list(pool.imap_unordered(forward_head, tasks))
    assert len(parts) == w.B * w.H
    if d_use != w.d:
        assert all(p["pad_zero"] for p in parts), f"{name}: padding columns of O not zero"
    _summary(name, parts)


def test_c5_forward_backward_every_element(cuda_lib):
    w = workload("c5")
    x = make_inputs(w)
    s = w.softmax_scale
    tq, tk, tv, tdo = dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(x["do"])
    O, lse = cuda_lib.forward(tq, tk, tv, s, w.causal)
    dq, dk, dv = (_f32(g) for g in cuda_lib.backward(tq, tk, tv, O, lse, tdo, s, w.causal))
    O, lse = _f32(O), _f32(lse)
    del tq, tk, tv, tdo
    tasks = ((x["q"][b, h], x["k"][b, h], x["v"][b, h], x["do"][b, h], O[b, h], lse[b, h], dq[b, h], dk[b, h],
              dv[b, h], s, w.causal, (b, h)) for b in range(w.B) for h in range(w.H))
    pool, _ = make_pool(10 * w.N * w.N * 8)
    with pool:
        parts = list(pool.imap_unordered(backward_head, tasks))
    assert len(parts) == w.B * w.H
    grad_err = {}
    for g in ("dq", "dk", "dv"):
        grad_err[g] = float(np.sqrt(sum(p[g + "_e2"] for p in parts) / sum(p[g + "_r2"] for p in parts)))
        print(f"\nc5 {g}: rel Frobenius {grad_err[g]:.3e} over the tensor "
              f"(worst head {max(p[g + '_head'] for p in parts):.3e})", end="")
    _summary("c5", parts)
    for g in ("dq", "dk", "dv"):
        assert all(p[g + "_finite"] for p in parts), f"c5: {g} not finite"
        assert grad_err[g] <= GRAD_REL_FRO, f"c5: {g} rel Frobenius err {grad_err[g]:.3e}"
