// attn_bwd_prep.cu — the first kernel of the backward pass: the per-row
// vectors both gradient kernels read.
//
// Method (page "Flash Attention原理：分块计算与重计算，如何降低O(n^2)的显存占用",
// §五 and FAQ Q19): with P recomputed from the forward's logsumexp, the
// softmax gradient dS = P * (dP - D) needs D_i = rowsum(dO_i * O_i), one
// scalar per query row.  This kernel writes -D and -lse * log2(e) (the
// exponent offset of the base-2 recomputation) into the workspace, padded
// to 128 rows per head.
#include <algorithm>
#include <cmath>

#include <cuda_bf16.h>

#include "kernels.h"

namespace sdpa {

// ------------------------------------------------------------------ preprocess
// Row i < N of each (head, padded row) gets -D = -(dO_i . O_i) (fp32) and
// -lse_i * log2(e); rows i >= N get -D = 0 and -lse2 = -inf (so P = 0
// there).  The negated values let the other kernels form P and dP - D with
// one packed FMA / add per pair.  A row that saw no key (lse = -inf, masked
// calls only) also gets -lse2 = -inf, so P = 0 on it.
// HBM-bound (reads O and dO once): LPR lanes take one row, 16 bytes of O and
// dO each, so a warp covers 32 / LPR rows per pass, and every thread issues
// the loads of all its PRE_IT passes (and the rows' lse) before it uses any
// of them: one round trip to memory per block.
constexpr int PRE_IT = 4;

template <int LPR>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdParams p) {
  constexpr int RPW = 32 / LPR;  // rows per warp and pass
  const long long rows = (long long)p.B * p.H * p.Npad;
  const int lane = threadIdx.x & 31, sub = lane / LPR, c = lane % LPR;
  const long long row0 = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * (RPW * PRE_IT);
  if (row0 >= rows) return;
  // A warp's RPW * PRE_IT (8 or 16) rows lie in one head: Npad is a multiple
  // of 128.  One division per thread.
  const long long bh = row0 / p.Npad;
  const int i0 = (int)(row0 - bh * p.Npad) + sub;
  const size_t base = ((size_t)bh * p.N) * p.d + c * 8;
  uint4 o[PRE_IT], g[PRE_IT];
  float lv[PRE_IT];
#pragma unroll
  for (int it = 0; it < PRE_IT; ++it) {
    const int i = i0 + it * RPW;
    o[it] = make_uint4(0, 0, 0, 0);
    g[it] = make_uint4(0, 0, 0, 0);
    lv[it] = -INFINITY;
    if (i < p.N && c * 8 < p.d && ATTN_IN_RANGE(base + (size_t)i * p.d + 7, (size_t)p.B * p.H * p.N * p.d, p, 0x401)) {
      const size_t off = base + (size_t)i * p.d;
      o[it] = *reinterpret_cast<const uint4*>(p.o + off);
      g[it] = *reinterpret_cast<const uint4*>(p.dout + off);
    }
    if (i < p.N && c == 0 && ATTN_IN_RANGE((size_t)bh * p.N + i, (size_t)p.B * p.H * p.N, p, 0x402))
      lv[it] = p.lse[(size_t)bh * p.N + i];
  }
#pragma unroll
  for (int it = 0; it < PRE_IT; ++it) {
    const uint32_t ow[4] = {o[it].x, o[it].y, o[it].z, o[it].w}, gw[4] = {g[it].x, g[it].y, g[it].z, g[it].w};
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[e]));
      const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[e]));
      dot = fmaf(of.x, gf.x, dot);
      dot = fmaf(of.y, gf.y, dot);
    }
#pragma unroll
    for (int s = LPR / 2; s > 0; s >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, s);
    const long long row = row0 + it * RPW + sub;
    const int i = i0 + it * RPW;
    if (c == 0 && row < rows && ATTN_IN_RANGE(row, vec_floats(p), p, 0x403)) {
      const float l = lv[it];
      p.dvec[row] = (i < p.N) ? -dot : 0.f;
      p.lse2[row] = (l == -INFINITY) ? -INFINITY : -l * 1.4426950408889634f;
    }
  }
}

// Packed batch: one CTA of 8 warps per (128-row tile of a sequence, head);
// warp w takes rows 16 w .. 16 w + 15 of the tile and writes them into the
// sequence's aligned region of the workspace (rows past Nq: -D = 0 and
// -lse2 = -inf).  A row that saw no key (lse = -inf) also gets -lse2 = -inf,
// so P = 0 on it.
__global__ void __launch_bounds__(256) bwd_pre_varlen_kernel(const BwdParams p) {
  const int t = (int)(blockIdx.x % p.nq);
  const int bh = (int)(blockIdx.x / p.nq);
  const int b = bh / p.H, h = bh % p.H;
  const SeqView sq = seq_view(p.vl, b, p.N, p.Nk);
  if (!sq.ok) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0, kDevBadSeqlens);
    return;
  }
  if (128 * t >= sq.nq) return;
  // 16 lanes per row (two rows per warp and pass); each warp takes 16 rows
  // of the tile in two groups and issues a group's loads (O, dO, lse) before
  // it reduces any of them.
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, sub = lane >> 4, c = lane & 15;
  const size_t vbase = (size_t)h * p.vec_stride + (size_t)varlen_vec_offset(sq.q0, b) + 128 * (size_t)t;
  for (int k0 = 16 * warp; k0 < 16 * warp + 16; k0 += 2 * PRE_IT) {
    uint4 o[PRE_IT], g[PRE_IT];
    float lv[PRE_IT];
#pragma unroll
    for (int it = 0; it < PRE_IT; ++it) {
      const int i = 128 * t + k0 + 2 * it + sub;
      o[it] = make_uint4(0, 0, 0, 0);
      g[it] = make_uint4(0, 0, 0, 0);
      lv[it] = -INFINITY;
      if (i < sq.nq) {
        const size_t off = ((size_t)(sq.q0 + i) * p.H + h) * p.d + c * 8;
        if (c * 8 < p.d && ATTN_IN_RANGE(off + 7, (size_t)p.vl.total_q * p.H * p.d, p, 0x401)) {
          o[it] = *reinterpret_cast<const uint4*>(p.o + off);
          g[it] = *reinterpret_cast<const uint4*>(p.dout + off);
        }
        if (c == 0 && ATTN_IN_RANGE((size_t)h * p.vl.total_q + sq.q0 + i, (size_t)p.H * p.vl.total_q, p, 0x402))
          lv[it] = p.lse[(size_t)h * p.vl.total_q + sq.q0 + i];
      }
    }
#pragma unroll
    for (int it = 0; it < PRE_IT; ++it) {
      const uint32_t ow[4] = {o[it].x, o[it].y, o[it].z, o[it].w}, gw[4] = {g[it].x, g[it].y, g[it].z, g[it].w};
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[e]));
        const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[e]));
        dot = fmaf(of.x, gf.x, dot);
        dot = fmaf(of.y, gf.y, dot);
      }
#pragma unroll
      for (int s = 8; s > 0; s >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, s);
      if (c == 0 && ATTN_IN_RANGE(vbase + k0 + 2 * it + sub, vec_floats(p), p, 0x403)) {
        const int k = k0 + 2 * it + sub;
        const float l = lv[it];
        p.dvec[vbase + k] = -dot;
        p.lse2[vbase + k] = (l == -INFINITY) ? -INFINITY : -l * 1.4426950408889634f;
      }
    }
  }
}

cudaError_t launch_bwd_prep(const BwdParams& p, cudaStream_t stream) {
  if (p.vl.cu_q != nullptr) {
    bwd_pre_varlen_kernel<<<(unsigned)p.nq * (unsigned)(p.B * p.H), 256, 0, stream>>>(p);
  } else {
    // 16 lanes per row for d = 96, 128 (12 of them busy at 96), 8 for d = 64.
    const long long rows = (long long)p.B * p.H * p.Npad;
    if (p.d == 64) {
      const long long per_block = 8LL * (32 / 8) * PRE_IT;
      bwd_pre_kernel<8><<<(unsigned)((rows + per_block - 1) / per_block), 256, 0, stream>>>(p);
    } else {
      const long long per_block = 8LL * (32 / 16) * PRE_IT;
      bwd_pre_kernel<16><<<(unsigned)((rows + per_block - 1) / per_block), 256, 0, stream>>>(p);
    }
  }
  return cudaGetLastError();
}

}  // namespace sdpa
