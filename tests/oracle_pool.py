"""Runs the fp64 oracle over whole heads in a pool of worker processes, for
the full-size parity tests.

Every full-size comparison is element by element: each worker takes one
(batch, head) of the inputs and of the GPU's outputs (float32 copies of the
bf16 / fp32 results), computes that head with the oracle, and returns the
error sums of that head; the test adds them up over every head and checks
the tolerances on the whole tensors.  No output is sampled.

The pool uses the ``spawn`` start method, so it may be created after the
CUDA context exists (a forked child of a CUDA process can hang).  Each
worker runs single-threaded BLAS; the pool is as wide as the host's cores
and its free memory allow.
"""
from __future__ import annotations

import math
import multiprocessing as mp
import os

import numpy as np

import oracle

_BLAS_ENV = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def _free_bytes() -> int:
    try:
        return int(os.sysconf("SC_AVPHYS_PAGES")) * int(os.sysconf("SC_PAGE_SIZE"))
    except (ValueError, OSError):
        return 16 << 30


def make_pool(bytes_per_worker: int):
    """A spawn pool of single-threaded workers: one per host core, fewer if
    the free memory cannot hold ``bytes_per_worker`` for each."""
    cores = os.cpu_count() or 1
    n = max(1, min(cores, int(0.6 * _free_bytes()) // max(1, bytes_per_worker)))
    saved = {k: os.environ.get(k) for k in _BLAS_ENV}
    for k in _BLAS_ENV:
        os.environ[k] = "1"
    try:
        pool = mp.get_context("spawn").Pool(n)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return pool, n


def forward_head(task):
    """Oracle forward of one head against the GPU's O and lse of that head.

    task: (q (Nq, d), k (Nk, d), v (Nk, d), O (Nq, d_out), lse (Nq,), scale,
    causal, q_offset, d_use, head).  Columns d_use.. of O are zero-padding
    columns: they must be exactly 0, and the oracle runs on the first d_use
    columns.  ``head`` is a label returned with the result."""
    q, k, v, O, lse, scale, causal, q_offset, d_use, head = task
    one = lambda a: np.asarray(a[None, None, :, :d_use], dtype=np.float64)
    O_ref, lse_ref = oracle.attention_forward(one(q), one(k), one(v), scale, causal, q_offset=q_offset)
    err = np.abs(np.asarray(O[:, :d_use], np.float64) - O_ref[0, 0])
    lerr = np.abs(np.asarray(lse, np.float64) - lse_ref[0, 0])
    at = np.unravel_index(int(np.argmax(err)), err.shape)
    return {
        "finite": bool(np.all(np.isfinite(O)) and np.all(np.isfinite(lse))),
        "pad_zero": bool(np.all(O[:, d_use:] == 0.0)),
        "o_max": float(err.max()),
        "o_sum": float(err.sum()),
        "o_n": int(err.size),
        "lse_max": float(lerr.max()),
        "head": head,
        # where the largest O error is: (row, column, GPU value, oracle value)
        "o_max_at": (int(at[0]), int(at[1]), float(O[at]), float(O_ref[0, 0][at])),
    }


def backward_head(task):
    """Oracle forward and backward of one head (H = Hkv) against the GPU's O,
    lse, dQ, dK and dV of that head.

    task: (q, k, v, do, O, lse, dq, dk, dv, scale, causal, head).  Returns the
    forward errors of ``forward_head`` and, per gradient, the sums of squared
    errors and of squared reference values (for the relative Frobenius error
    of the whole tensor), plus the head's own relative error."""
    q, k, v, do, O, lse, dq, dk, dv, scale, causal, head = task
    out = forward_head((q, k, v, O, lse, scale, causal, 0, q.shape[1], head))
    one = lambda a: np.asarray(a[None, None], dtype=np.float64)
    ref = oracle.attention_backward(one(q), one(k), one(v), one(do), scale, causal)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        g = np.asarray(g, np.float64)
        r = r[0, 0]
        e2 = float(((g - r) ** 2).sum())
        r2 = float((r ** 2).sum())
        out[name + "_finite"] = bool(np.all(np.isfinite(g)))
        out[name + "_e2"] = e2
        out[name + "_r2"] = r2
        out[name + "_head"] = math.sqrt(e2 / r2) if r2 > 0 else math.sqrt(e2)
    return out


def _grad_errors(out, grads, ref):
    """Adds, per gradient, the sums of squared errors and squared reference
    values and the unit's own relative Frobenius error to ``out``."""
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        g = np.asarray(g, np.float64)
        r = np.asarray(r, np.float64)
        e2 = float(((g - r) ** 2).sum())
        r2 = float((r ** 2).sum())
        out[name + "_finite"] = bool(np.all(np.isfinite(g)))
        out[name + "_e2"] = e2
        out[name + "_r2"] = r2
        out[name + "_head"] = math.sqrt(e2 / r2) if r2 > 0 else math.sqrt(e2)
    return out


def _o_lse_errors(O, lse, O_ref, lse_ref, head):
    """Forward error sums of one unit; rows that see no key must be exactly
    O = 0, lse = -inf."""
    O = np.asarray(O, np.float64)
    lse = np.asarray(lse, np.float64)
    live = np.isfinite(lse_ref)
    err = np.abs(O - O_ref)
    lerr = np.abs(lse[live] - lse_ref[live]) if live.any() else np.zeros(1)
    at = np.unravel_index(int(np.argmax(err)), err.shape)
    return {
        "finite": bool(np.all(np.isfinite(O)) and np.all(np.isfinite(lse[live]))),
        "dead_ok": bool(np.all(O[~live] == 0) and np.all(np.isneginf(lse[~live]))),
        "pad_zero": True,
        "o_max": float(err.max()),
        "o_sum": float(err.sum()),
        "o_n": int(err.size),
        "lse_max": float(lerr.max()),
        "head": head,
        "o_max_at": (int(at[0]), int(at[1]), float(O[at]), float(O_ref[at])),
    }


def cross_head(task):
    """Nq queries against Nk keys of one head (causal: query row i at
    position Nk - Nq + i), forward and, when dO is given, backward.
    task: (q, k, v, do or None, O, lse, dq, dk, dv (or None), scale, causal, head)."""
    q, k, v, do, O, lse, dq, dk, dv, scale, causal, head = task
    one = lambda a: np.asarray(a[None, None], dtype=np.float64)
    off = k.shape[0] - q.shape[0] if causal else 0
    O_ref, lse_ref = oracle.attention_forward(one(q), one(k), one(v), scale, causal, q_offset=off)
    out = _o_lse_errors(O, lse, O_ref[0, 0], lse_ref[0, 0], head)
    if do is not None:
        ref = oracle.attention_backward(one(q), one(k), one(v), one(do), scale, causal, q_offset=off)
        _grad_errors(out, (dq, dk, dv), [r[0, 0] for r in ref])
    return out


def masked_head(task):
    """One head under a mask built here from its recipe: ("prefix", p) a
    prefix-LM boolean mask, ("distance", slope, bf16) the additive bias
    -slope * |i - j| (rounded to bf16 when bf16); forward and, when dO is
    given, backward.
    task: (q, k, v, do or None, O, lse, dq, dk, dv (or None), scale, causal, recipe, head)."""
    from sdpa_inputs import distance_bias, prefix_lm_mask, round_bf16
    q, k, v, do, O, lse, dq, dk, dv, scale, causal, recipe, head = task
    one = lambda a: np.asarray(a[None, None], dtype=np.float64)
    N = q.shape[0]
    mask = prefix_lm_mask(N, recipe[1]) if recipe[0] == "prefix" else None
    bias = distance_bias(N, recipe[1]) if recipe[0] == "distance" else None
    if bias is not None and len(recipe) > 2 and recipe[2]:
        bias = round_bf16(bias)
    O_ref, lse_ref = oracle.attention_masked_forward(one(q), one(k), one(v), scale, causal, None, None, mask, bias)
    out = _o_lse_errors(O, lse, O_ref[0, 0], lse_ref[0, 0], head)
    if do is not None:
        ref = oracle.attention_masked_backward(one(q), one(k), one(v), one(do), scale, causal, None, None, mask,
                                               bias)
        _grad_errors(out, (dq, dk, dv), [r[0, 0] for r in ref])
    return out


def window_head(task):
    """One head of a causal sliding window of wl keys to the left, every
    query row, in blocks of 128 rows against the keys their windows reach
    (the masked oracle aligns block row r0 + i at key position r0 + i).
    task: (q (N, d), k, v, O, lse, scale, wl, head)."""
    q, k, v, O, lse, scale, wl, head = task
    N = q.shape[0]
    O_ref = np.zeros((N, v.shape[1]))
    lse_ref = np.zeros(N)
    for r0 in range(0, N, 128):
        r1 = min(N, r0 + 128)
        k0 = max(0, r0 - wl)
        blk = lambda a, a0, a1: np.asarray(a[None, None, a0:a1], dtype=np.float64)
        Ob, lb = oracle.attention_masked_forward(blk(q, r0, r1), blk(k, k0, r1), blk(v, k0, r1), scale, True,
                                                 (wl, -1))
        O_ref[r0:r1] = Ob[0, 0]
        lse_ref[r0:r1] = lb[0, 0]
    return _o_lse_errors(O, lse, O_ref, lse_ref, head)


def fp8_head(task):
    """One head of the FP8 forward on its dequantised e4m3 inputs: errors
    against the exact oracle and against the model of the kernel's one
    added rounding (tests/fp8_model.py).
    task: (q, k, v (dequantised, (N, d)), O, lse, scale, causal, q_offset, head)."""
    from tests.fp8_model import p_rounding_model
    q, k, v, O, lse, scale, causal, off, head = task
    one = lambda a: np.asarray(a[None, None], dtype=np.float64)
    O_ref, lse_ref = oracle.attention_forward(one(q), one(k), one(v), scale, causal, q_offset=off)
    O_ref, lse_ref = O_ref[0, 0], lse_ref[0, 0]
    O_m = p_rounding_model(q, k, v, scale, causal, off)
    O = np.asarray(O, np.float64)
    return {
        "head": head,
        "finite": bool(np.all(np.isfinite(O)) and np.all(np.isfinite(lse))),
        "rel_fro": float(np.linalg.norm(O - O_ref) / np.linalg.norm(O_ref)),
        "rel_fro_model": float(np.linalg.norm(O - O_m) / np.linalg.norm(O_m)),
        "o_sum": float(np.abs(O - O_ref).sum()),
        "o_n": int(O.size),
        "lse_max": float(np.abs(np.asarray(lse, np.float64) - lse_ref).max()),
    }
