"""Seeded synthetic inputs for exact scaled-dot-product attention.

This module is shared by the CPU oracle tests, the GPU parity tests and the
benchmark.  It holds no attention arithmetic: only the workload shapes, the
seeded random draws and the round-to-nearest-even conversion to bf16 that
turns each draw into exactly representable bf16 values.

Workloads (all tensors in (batch, heads, seq_len, head_dim) layout, the layout
used by the "Flash Attention原理：分块计算与重计算" page, §一, and by the
SDPA call on "SDPA backend 与 FlashAttention", §3):

  c1   B=1  H=2   Hkv=2  N=256  d=64   non-causal   seed 1
  c2   B=4  H=16  Hkv=16 N=2048 d=128  causal       seed 2   (LLM prefill)
  c3   B=1  H=96  Hkv=96 N=4096 d=64   non-causal   seed 3   (GPT-3 layer of §一)
  c3c  same shape, causal                            seed 3
  c4   B=1  H=32  Hkv=8  N=8192 d=128  causal, x0.5 seed 4   (long-context GQA)
  c4p  same, head_dim 80 zero-padded to 96, scale 1/sqrt(80)  seed 4
  c5   B=8  H=16  Hkv=16 N=4096 d=128  causal, fwd+bwd (dO drawn)  seed 5

Decode workloads (Nq new queries per head against a cache of N keys/values;
the pages' FAQ on inference with a KV cache, decode profiled apart from
prefill; the cache length and group size are those of a long-context GQA
model):

  dec1 B=8  H=64  Hkv=8  Nq=1 N=32768 d=128  non-causal  seed 6
  dec4 same shape, Nq=4 new tokens (a speculative block), causal  seed 7
  dec1p dec1's draw with the cache in a pool of 16-token pages (the page
       size vLLM uses by default), each sequence's pages scattered over the
       pool by paged_layout (default_rng(seed + 2000).permutation)

Chunked prefill (Nq new queries per head against N keys, the tiled forward):

  cp1  B=1  H=32  Hkv=8  Nq=2048 N=16384 d=128  causal   seed 8

Encoder-decoder cross attention (Nq decoder queries against N encoder keys,
no mask), forward + backward:

  cx   B=8  H=16  Hkv=16 Nq=2048 N=4096  d=128  non-causal  seed 9

Packed variable-length batch (the pages' FAQ on variable lengths: sequences
of different lengths packed into one batch by cumulative offsets), forward +
backward, self-attention (the same lengths for queries and keys):

  vl1  32768 tokens, H=16 Hkv=16 d=128, causal, seed 10; sequence lengths
       drawn uniformly from [128, 8192] (numpy default_rng(10).integers,
       inclusive) until they reach 32768 tokens, the last one cut to fit.
       Tensors are packed token-major: (total, heads, d).  The draws of Q,
       K, V, dO use default_rng(seed + 1000) in that order.

FP8 forward (attn_fwd_fp8): c4f8 is c4's draw (seed 4, x0.5) quantised per
tensor to e4m3 (quantize_e4m3: scale = amax / 448); c3cf8 is c3c's draw
(seed 3, head_dim 64, causal) quantised the same way.

Masked workloads (attn_fwd_masked / attn_bwd_masked), forward + backward:

  sw1  B=1  H=32  Hkv=8  N=16384 d=128  causal sliding window of 4096 keys
       (window_left 4095): the [PROF] page's window attention, n * w work
  pl1  B=8  H=16  Hkv=16 N=4096  d=128  prefix-LM boolean mask, one plane for
       all (b, h): key j visible to query i when j < 1024 or j <= i
  ab1  B=8  H=16  Hkv=16 N=4096  d=128  additive float32 mask -|i - j| / 64,
       one plane for all (b, h)   seed 13
  ab1h ab1 with its mask stored in bf16 (values rounded to bf16)

Every draw is numpy's PCG64 ``default_rng(seed).standard_normal(dtype=float32)``
taken in the fixed order Q, K, V, dO, multiplied by the config's amplitude and
then rounded to bf16 (round to nearest, ties to even).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Hkv: int
    N: int
    d: int
    causal: bool
    seed: int
    amp: float = 1.0
    d_draw: int | None = None      # head_dim actually drawn (zero-padded up to d)
    with_grad: bool = False        # also draw dO
    scale: float | None = None     # default 1/sqrt(d_draw or d)
    Nq: int | None = None          # decode / cross: query rows per head (None: Nq = N)
    kind: str = "full"             # "full" (Nq = N), "decode" (attn_decode), "cross" (attn_fwd_cross),
                                   # "varlen" (attn_fwd_varlen: N = total tokens, B = 1), "masked",
                                   # "fp8" (attn_fwd_fp8 on e4m3 inputs)
    len_range: tuple[int, int] | None = None  # varlen: sequence lengths drawn from [lo, hi]
    window: tuple[int, int] | None = None     # masked: (left, right), -1 = open
    prefix: int | None = None                 # masked: prefix-LM boolean mask with this prefix
    page_size: int | None = None              # decode: the cache kept in pages of this many tokens
    bias_slope: float | None = None           # masked: additive (1, 1, N, N) bias -slope * |i - j|
    bias_bf16: bool = False                   # masked: that bias stored in bf16 (its values rounded to bf16)

    @property
    def softmax_scale(self) -> float:
        if self.scale is not None:
            return self.scale
        return 1.0 / math.sqrt(self.d_draw or self.d)

    @property
    def G(self) -> int:
        return self.H // self.Hkv

    @property
    def n_queries(self) -> int:
        return self.Nq if self.Nq is not None else self.N


WORKLOADS: dict[str, Workload] = {
    "c1": Workload("c1", 1, 2, 2, 256, 64, False, 1),
    "c2": Workload("c2", 4, 16, 16, 2048, 128, True, 2),
    "c3": Workload("c3", 1, 96, 96, 4096, 64, False, 3),
    "c3c": Workload("c3c", 1, 96, 96, 4096, 64, True, 3),
    "c4": Workload("c4", 1, 32, 8, 8192, 128, True, 4, amp=0.5),
    "c4p": Workload("c4p", 1, 32, 8, 8192, 96, True, 4, amp=0.5, d_draw=80),
    "c5": Workload("c5", 8, 16, 16, 4096, 128, True, 5, with_grad=True),
    "dec1": Workload("dec1", 8, 64, 8, 32768, 128, False, 6, Nq=1, kind="decode"),
    "dec4": Workload("dec4", 8, 64, 8, 32768, 128, True, 7, Nq=4, kind="decode"),
    "dec1p": Workload("dec1p", 8, 64, 8, 32768, 128, False, 6, Nq=1, kind="decode", page_size=16),
    "cp1": Workload("cp1", 1, 32, 8, 16384, 128, True, 8, Nq=2048, kind="cross"),
    "cx": Workload("cx", 8, 16, 16, 4096, 128, False, 9, with_grad=True, Nq=2048, kind="cross"),
    "vl1": Workload("vl1", 1, 16, 16, 32768, 128, True, 10, with_grad=True, kind="varlen", len_range=(128, 8192)),
    "c4f8": Workload("c4f8", 1, 32, 8, 8192, 128, True, 4, amp=0.5, kind="fp8"),
    "c3cf8": Workload("c3cf8", 1, 96, 96, 4096, 64, True, 3, kind="fp8"),
    "sw1": Workload("sw1", 1, 32, 8, 16384, 128, True, 11, with_grad=True, kind="masked", window=(4095, -1)),
    "pl1": Workload("pl1", 8, 16, 16, 4096, 128, False, 12, with_grad=True, kind="masked", prefix=1024),
    "ab1": Workload("ab1", 8, 16, 16, 4096, 128, False, 13, with_grad=True, kind="masked", bias_slope=1 / 64),
    "ab1h": Workload("ab1h", 8, 16, 16, 4096, 128, False, 13, with_grad=True, kind="masked", bias_slope=1 / 64,
                     bias_bf16=True),
}


def prefix_lm_mask(N: int, prefix: int) -> np.ndarray:
    """Boolean (1, 1, N, N) prefix-LM mask: key j is visible to query i when
    j < prefix (the bidirectional prefix) or j <= i (causal after it)."""
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    return ((j < prefix) | (j <= i))[None, None]


def distance_bias(N: int, slope: float) -> np.ndarray:
    """Float32 (1, 1, N, N) additive mask -slope * |i - j|: a linear
    distance penalty shared by every head (an input of the additive-mask
    workload; all entries finite)."""
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    return (-slope * np.abs(i - j)).astype(np.float32)[None, None]


def workload_bias(w: Workload) -> np.ndarray | None:
    """The additive mask of a masked workload as float32 values: the
    distance bias, rounded to bf16 (nearest even) when the workload stores it
    in bf16; None without one."""
    if w.bias_slope is None:
        return None
    b = distance_bias(w.N, w.bias_slope)
    return round_bf16(b) if w.bias_bf16 else b


def visible_pairs(w: Workload) -> int:
    """(query, key) pairs a masked self-attention workload computes, per
    (batch, head): the exact count, by closed form."""
    N = w.N
    if w.bias_slope is not None and w.prefix is None and w.window is None:
        return N * (N + 1) // 2 if w.causal else N * N  # a finite bias hides no key
    if w.prefix is not None:
        P = w.prefix
        return P * P + sum(i + 1 for i in range(P, N))
    wl = w.window[0] if w.window is not None else -1
    if w.causal:
        return sum(min(i + 1, wl + 1) if wl >= 0 else i + 1 for i in range(N))
    raise ValueError("no closed form for this mask")


def flops_masked(w: Workload) -> float:
    """Forward work of a masked workload: 4 * d per visible (query, key)
    pair and head (the convention of flops_forward with the exact count)."""
    return 4.0 * w.B * w.H * w.d * visible_pairs(w)


def varlen_lengths(w: Workload) -> list[int]:
    """Sequence lengths of a packed workload: uniform integers in
    w.len_range (inclusive) from default_rng(w.seed) until they cover w.N
    tokens; the last one is cut so that they sum to exactly w.N."""
    lo, hi = w.len_range
    rng = np.random.default_rng(w.seed)
    out, tot = [], 0
    while tot < w.N:
        n = int(rng.integers(lo, hi, endpoint=True))
        n = min(n, w.N - tot)
        out.append(n)
        tot += n
    return out


def make_varlen_inputs(w: Workload) -> dict[str, np.ndarray]:
    """Packed (total, heads, d) Q, K, V, dO of a varlen workload and its
    int32 cumulative offsets cu (B + 1 entries)."""
    lens = varlen_lengths(w)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    rng = np.random.default_rng(w.seed + 1000)
    out = {"q": draw(rng, (w.N, w.H, w.d), w.amp), "k": draw(rng, (w.N, w.Hkv, w.d), w.amp),
           "v": draw(rng, (w.N, w.Hkv, w.d), w.amp), "cu": cu, "lengths": np.array(lens)}
    if w.with_grad:
        out["do"] = draw(rng, (w.N, w.H, w.d), 1.0)
    return out


def workload(name: str, **overrides) -> Workload:
    """A named workload, optionally with fields replaced (e.g. a smaller N)."""
    w = WORKLOADS[name]
    return replace(w, **overrides) if overrides else w


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32.

    bf16 keeps the upper 16 bits of an IEEE float32.  Adding 0x7FFF plus the
    lowest kept bit before truncating implements round-to-nearest-even for
    finite inputs (the draws here are always finite).
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    r = (u + bias) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def draw(rng: np.random.Generator, shape, amp: float) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if amp != 1.0:
        x *= np.float32(amp)
    return round_bf16(x)


def make_inputs(w: Workload) -> dict[str, np.ndarray]:
    """Q, K, V (and dO when the workload has a backward pass) as float32
    arrays whose values are exactly representable in bf16."""
    rng = np.random.default_rng(w.seed)
    dd = w.d_draw or w.d
    q = draw(rng, (w.B, w.H, w.n_queries, dd), w.amp)
    k = draw(rng, (w.B, w.Hkv, w.N, dd), w.amp)
    v = draw(rng, (w.B, w.Hkv, w.N, dd), w.amp)
    out = {"q": q, "k": k, "v": v}
    if w.with_grad:
        out["do"] = draw(rng, (w.B, w.H, w.n_queries, dd), 1.0)
    if dd != w.d:
        pad = [(0, 0)] * 3 + [(0, w.d - dd)]
        out = {n: np.pad(a, pad) for n, a in out.items()}
    return out


def make_random(shape, seed: int, amp: float = 1.0) -> np.ndarray:
    """One seeded bf16-exact float32 tensor (small parity sweeps)."""
    return draw(np.random.default_rng(seed), shape, amp)


def flops_cross(B: int, H: int, Nq: int, Nk: int, d: int, causal: bool) -> float:
    """Forward work of Nq queries against Nk keys: 4*B*H*d per visible
    (query, key) pair; causal rows sit at positions Nk - Nq + i, and the
    square Nq x Nq corner is counted halved as in the Nq = Nk convention."""
    pairs = Nq * (Nk - Nq) + Nq * Nq / 2 if causal else Nq * Nk
    return 4.0 * B * H * d * pairs


def flops_varlen(lengths, H: int, d: int, causal: bool) -> float:
    """Forward work of a packed self-attention batch: the forward convention
    summed over its sequences."""
    return sum(flops_forward(1, H, int(n), d, causal) for n in lengths)


def flops_forward(B: int, H: int, N: int, d: int, causal: bool) -> float:
    """Forward work convention: 4*B*H*N^2*d, halved when causal."""
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


def flops_backward(B: int, H: int, N: int, d: int, causal: bool) -> float:
    """Backward work convention: 2.5x the forward."""
    return 2.5 * flops_forward(B, H, N, d, causal)


# ---------------------------------------------------------------- e4m3 inputs
# FP8 e4m3 (the "fn" variant: 1 sign bit, 4 exponent bits with bias 7, 3
# mantissa bits, no infinities, S.1111.111 is NaN, largest value 448,
# subnormals m / 8 * 2^-6).  Input preparation only: the FP8 forward takes
# e4m3 tensors with one dequantisation factor each.
E4M3_MAX = 448.0


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """float -> e4m3 bytes: round to nearest, ties to even, saturating at
    +-448 (finite inputs)."""
    x = np.asarray(x, dtype=np.float64)
    sign = (np.signbit(x)).astype(np.uint8) << 7
    a = np.minimum(np.abs(x), E4M3_MAX)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.clip(e, -6, 8)                       # -6: the subnormal binade shares the smallest exponent
    q = a / np.exp2(e - 3)                      # significand in units of the last place: [8, 16) or [0, 8)
    qr = np.round(q)                            # numpy rounds half to even
    carry = qr >= 16
    e = np.where(carry, e + 1, e)
    qr = np.where(carry, 8, qr)
    over = (e > 8) | ((e == 8) & (qr > 14))     # beyond 448 = 1.75 * 2^8: saturate
    e = np.where(over, 8, e)
    qr = np.where(over, 14, qr)
    normal = qr >= 8
    code = np.where(normal, ((e + 7).astype(np.int64) << 3) | (qr.astype(np.int64) - 8), qr.astype(np.int64))
    return (code.astype(np.uint8) | sign).astype(np.uint8)


def e4m3_decode(b: np.ndarray) -> np.ndarray:
    """e4m3 bytes -> float64 (NaN for S.1111.111)."""
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    s = np.where(b & 0x80, -1.0, 1.0)
    E = (b >> 3) & 0xF
    M = b & 0x7
    val = np.where(E == 0, M * 2.0 ** -9, (8 + M) * np.exp2(E - 10.0))
    val = np.where((E == 15) & (M == 7), np.nan, val)
    return s * val


def quantize_e4m3(x: np.ndarray):
    """Per-tensor e4m3 quantisation: scale = amax / 448, bytes = e4m3(x /
    scale).  Returns (bytes, scale); the tensor the FP8 path computes with is
    e4m3_decode(bytes) * scale."""
    amax = float(np.max(np.abs(x)))
    scale = np.float32(amax / E4M3_MAX if amax > 0 else 1.0)
    return e4m3_encode(np.asarray(x, dtype=np.float64) / float(scale)), float(scale)


def paged_layout(w: Workload, k: np.ndarray, v: np.ndarray):
    """A decode workload's contiguous (B, Hkv, N, d) cache stored in a page
    pool of w.page_size-token pages: (num_pages, page_size, Hkv, d) K and V
    and the (B, max_pages) int32 block table, each sequence's logical pages
    at physical pages default_rng(w.seed + 2000).permutation(num_pages)."""
    B, Hkv, N, d = k.shape
    ps = w.page_size
    max_pages = -(-N // ps)
    num_pages = B * max_pages
    order = np.random.default_rng(w.seed + 2000).permutation(num_pages)
    table = order.reshape(B, max_pages).astype(np.int32)
    kc = np.zeros((num_pages, ps, Hkv, d), dtype=k.dtype)
    vc = np.zeros((num_pages, ps, Hkv, d), dtype=v.dtype)
    for b in range(B):
        kp = np.zeros((max_pages * ps, Hkv, d), dtype=k.dtype)
        vp = np.zeros((max_pages * ps, Hkv, d), dtype=v.dtype)
        kp[:N] = k[b].transpose(1, 0, 2)
        vp[:N] = v[b].transpose(1, 0, 2)
        kc[table[b]] = kp.reshape(max_pages, ps, Hkv, d)
        vc[table[b]] = vp.reshape(max_pages, ps, Hkv, d)
    return kc, vc, table
