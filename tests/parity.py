"""Shared helpers for the GPU parity tests: device upload of the seeded bf16
inputs and the tolerances the comparison uses.

Tolerances (bf16 inputs, float32 accumulation, compared with the fp64
oracle on the same inputs, element by element):
  O    max |err| <= 1e-2 and mean |err| <= 1e-3 over all compared elements
  lse  max |err| <= 1e-3
  dQ, dK, dV  ||g - g*||_F / ||g*||_F <= 2e-2 per tensor
"""
import numpy as np

O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-3
GRAD_REL_FRO = 2e-2


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).cuda()


def host(t):
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def check_o_lse(O, lse, O_ref, lse_ref, what=""):
    err = np.abs(O - O_ref)
    lerr = np.abs(lse - lse_ref)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(lse)), what
    assert err.max() <= O_MAX_ABS, f"{what}: O max abs err {err.max():.3e}"
    assert err.mean() <= O_MEAN_ABS, f"{what}: O mean abs err {err.mean():.3e}"
    assert lerr.max() <= LSE_MAX_ABS, f"{what}: lse max abs err {lerr.max():.3e}"
    return {"o_max": float(err.max()), "o_mean": float(err.mean()), "lse_max": float(lerr.max())}


def rel_fro(g, g_ref):
    den = np.linalg.norm(g_ref)
    return float(np.linalg.norm(g - g_ref) / den) if den > 0 else float(np.linalg.norm(g))


def check_grads(grads, grads_ref, what=""):
    out = {}
    for name, g, r in zip(("dq", "dk", "dv"), grads, grads_ref):
        assert np.all(np.isfinite(g)), f"{what}: {name} not finite"
        e = rel_fro(g, r)
        assert e <= GRAD_REL_FRO, f"{what}: {name} rel Frobenius err {e:.3e}"
        out[name] = e
    return out


def sample_rows(N, k=24, seed=0):
    """Rows spanning tile boundaries, both ends and a seeded random spread."""
    fixed = {0, 1, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1}
    rng = np.random.default_rng(seed)
    rnd = set(rng.integers(0, N, size=k).tolist())
    return np.array(sorted(r for r in fixed | rnd if 0 <= r < N))


# The backward's two schedules (row vectors from the prep kernel, or formed
# inside the dQ kernel) sum D = rowsum(dO * O) in different float32 orders,
# so their gradients may differ in the last bits of a few elements.
STAGE_ORDER_REL_FRO = 1e-3


def check_same_but_rounding(got, want, what=""):
    for g, w in zip(got, want):
        err = rel_fro(g, w)
        assert err <= STAGE_ORDER_REL_FRO, f"{what}: rel err {err:.2e} between the two stage orders"
