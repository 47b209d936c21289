// attn_bwd_dq.cu — dQ of exact attention on sm_103a (query-stationary).
//
// Method (page "Flash Attention原理：分块计算与重计算，如何降低O(n^2)的显存占用",
// §五): for one 128-row query tile i of one head, walk the key tiles j (up to
// the last one a row of the tile sees, when causal) and accumulate
//     S  = Q_i K_j^T,   P = exp2(S * scale * log2 e - lse_i * log2 e),
//     dP = dO_i V_j^T,  dS = P * (dP - D_i),   dQ_i += dS K_j,
// with dQ_i in tensor memory for the whole walk and the softmax scale applied
// once at the end.  Each dQ tile has exactly one writer: no atomics, no
// accumulator in global memory, and the result does not depend on timing.
//
// Warp roles (384 threads):
//   warps 0-7   compute, two warpgroups: warpgroup X takes key columns
//               [64X, 64X+64) of each 128 x 128 (queries x keys) tile, one
//               thread per query row: S -> P (registers), dP -> dS (bf16
//               pairs back into its S columns, the A operand of the dQ MMA);
//               then half of the dQ epilogue
//   warp  8     TMA producer: Q_i, dO_i once; K_j (3-slot ring), V_j (2-slot);
//               with p.rows_in_dq, O_i once into K slot 2 before K_2
//               (the compute threads then form D_i = rowsum(dO_i * O_i) and
//               lse_i in base 2, use them, and write them for the dK/dV
//               kernel; otherwise they read them from the workspace)
//   warp  9     MMA issuer (one elected lane issues)
//   warps 10-11 idle
// Tensor memory: S[0] [0,128), S[1] [128,256) (double-buffered, so S_{j+2}
// is computed while step j+1 is in the softmax), dP [256,384), dQ [384,384+d).
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {

template <int D>
struct DqTraits {
  static constexpr int NB = (D + 63) / 64;
  static constexpr int BLOCK_BYTES = 128 * 128;
  static constexpr int TILE_BYTES = NB * BLOCK_BYTES;  // one [128 rows x d] bf16 tile
  static constexpr int KSTEPS = D / 16;
  static constexpr int KS = 3, VS = 2;                 // K and V ring slots
  static constexpr int NBAR = 20;
  static constexpr int MISC = 64;                      // tmem slot, abort flag, per-CTA values
  static constexpr int SMEM = 1024 + (2 + KS + VS) * TILE_BYTES + NBAR * 8 + MISC + 2 * kMaxTileList;
  static constexpr int THREADS = 384;
};

// A query tile none of whose rows sees a key: its rows' vectors for the
// dK/dV kernel, -lse2 = -inf (P = 0) and -D = 0, one thread per row.
__device__ __noinline__ void no_key_vectors(const BwdParams& p, bool varlen, int q0, int b, int bh, int h, int i) {
  if (threadIdx.x >= 128) return;
  const size_t vrow = (varlen ? (size_t)h * p.vec_stride + (size_t)varlen_vec_offset(q0, b) : (size_t)bh * p.Npad) +
                      (size_t)i * 128 + threadIdx.x;
  if (!ATTN_IN_RANGE(vrow, vec_floats(p), p, 0x201)) return;
  p.dvec[vrow] = 0.f;
  p.lse2[vrow] = -INFINITY;
}

// MASKED: the instance that applies p.mk (causal enters as wr = 0).
template <int D, bool CAUSAL, int MASKED>
__global__ void __launch_bounds__(384, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const __grid_constant__ CUtensorMap tmdQ, const __grid_constant__ CUtensorMap tmO,
                  const BwdParams p) {
  using T = DqTraits<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1024-byte alignment
  uint8_t* const gbase = smem_raw + (base - raw);

  const uint32_t sQ = base;                          // Q_i; dQ_i staging at the end
  const uint32_t sdO = sQ + T::TILE_BYTES;           // dO_i
  const uint32_t sK = sdO + T::TILE_BYTES;           // [KS] K_j
  const uint32_t sV = sK + T::KS * T::TILE_BYTES;    // [VS] V_j
  const uint32_t sBar = sV + T::VS * T::TILE_BYTES;
  const uint32_t bQ = sBar;                  // Q_i and dO_i loaded
  const uint32_t bKf = bQ + 8;               // [KS] K slot full
  const uint32_t bKe = bKf + 8 * T::KS;      // [KS] K slot free (after dQ += dS K_j)
  const uint32_t bVf = bKe + 8 * T::KS;      // [VS] V slot full
  const uint32_t bVe = bVf + 8 * T::VS;      // [VS] V slot free (after dP_j)
  const uint32_t bS = bVe + 8 * T::VS;       // [2] S_j ready in buffer j & 1
  const uint32_t bDp = bS + 16;              // dP_j ready
  const uint32_t bDpc = bDp + 8;             // dP_j copied out of TMEM (256 arrivals)
  const uint32_t bDs = bDpc + 8;             // dS_j in TMEM (256 arrivals)
  const uint32_t bFin = bDs + 8;             // dQ_i final
  const uint32_t bDrain = bFin + 8;
  const uint32_t bO = bDrain + 8;            // O_i loaded into K slot 2 (row vectors formed here)
  const uint32_t bOc = bO + 8;               // O_i read (256 arrivals): K slot 2 free for K_2
  static_assert(1 + 2 * 3 + 2 * 2 + 2 + 5 + 2 == 20, "barrier count");
  uint8_t* const misc = gbase + (sBar - base) + 8 * T::NBAR;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  // This CTA's sequence {q0, nq, k0, nk}, first key tile, visible key count
  // and mask plane, read back where needed rather than held in registers
  // across the main loops.
  volatile int* const seq_s = reinterpret_cast<volatile int*>(misc + 8);
  // Masked instance with a tile mask: the key tiles this CTA visits, in
  // order, relative to its first key tile jlo.
  volatile uint16_t* const tile_list = reinterpret_cast<volatile uint16_t*>(misc + T::MISC);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Work unit (work_unit): head-major (the CTAs in flight share K/V heads in
  // L2), the longest causal walks of a head first; the last heads
  // level-major, for a short tail.
  int bh, lv;
  work_unit((int)blockIdx.x, p.nq, p.B * p.H, p.tail, bh, lv);
  const int i = p.nq - 1 - lv;  // query tile
  const int b = bh / p.H, h = bh % p.H;
  const int bhk = b * p.Hkv + h / p.G;
  const bool varlen = p.vl.cu_q != nullptr;
  // Tensor-map planes: b * heads + head for the dense batch, the head for a
  // packed one (maps over (total, heads)).
  const int qplane = varlen ? h : bh, kplane = varlen ? h / p.G : bhk;
  int n;  // key tiles visited
  {
    const SeqView sq = seq_view(p.vl, b, p.N, p.Nk);
    if (!sq.ok) {
      if (threadIdx.x == 0) atomicCAS(p.status, 0, kDevBadSeqlens);
      return;
    }
    if (128 * i >= sq.nq) return;  // past the end of a shorter packed sequence
    // Causal: up to the tile holding the last row's last visible key,
    // koff + 128 i + 127 (query row r at position koff + r, koff = Nk - Nq).
    const int nkv = (sq.nk + 127) / 128, koff = sq.nk - sq.nq;
    int jlo = 0, nke = sq.nk;
    if (MASKED) {
      // Key tiles from the first row's window start to the last row's
      // last visible key.
      if (p.mk.key_len != nullptr) nke = max(0, min(nke, p.mk.key_len[b]));
      int hi = nke;
      if (p.mk.wr >= 0) hi = min(hi, koff + 128 * i + 127 + p.mk.wr + 1);
      if (p.mk.wl >= 0) jlo = max(0, floor_div128(koff + 128 * i - p.mk.wl));
      n = min(nkv, (max(hi, 0) + 127) / 128) - jlo;
    } else {
      n = CAUSAL ? min(nkv, (koff + i * 128 + 127) / 128 + 1) : nkv;
    }
    if (n <= 0) {
      // No row of the tile sees a key (packed batches, masks): dQ = 0.
      // Packed: (total, H, d) rows; dense: the (b, h) plane of (B, H, Nq, d).
      if (p.rows_in_dq) no_key_vectors(p, varlen, sq.q0, b, bh, h, i);
      const uint32_t rs = varlen ? (uint32_t)(p.H * D) : (uint32_t)D;
      uint16_t* dst = varlen ? p.dq + ((long long)sq.q0 + 128 * i) * rs + (long long)h * D
                             : p.dq + ((long long)bh * p.N + 128 * i) * D;
      if (ATTN_IN_RANGE(varlen ? (long long)sq.q0 + 128 * i + min(128, sq.nq - 128 * i) - 1
                               : (long long)bh * p.N + 128 * i + min(128, sq.nq - 128 * i) - 1,
                        varlen ? (long long)p.vl.total_q : (long long)p.B * p.H * p.N, p, 0x202))
        zero_rows_bf16<D>(dst, rs, min(128, sq.nq - 128 * i));
      return;
    }
    if (threadIdx.x == 0) {
      seq_s[0] = sq.q0;
      seq_s[1] = sq.nq;
      seq_s[2] = sq.k0;
      seq_s[3] = sq.nk;
      seq_s[4] = jlo;
      seq_s[5] = nke;
      if (MASKED) seq_s[6] = mask_plane(p.mk, b, h);
    }
  }
  // Tile skipping (masked instance with tile flags): warp 0 lists the key
  // tiles of [jlo, jlo + n) whose tile with this query tile has a visible
  // entry; seq_s[7] = 1 when the list is in use, seq_s[8] its length.  No
  // tile at all: dQ = 0.
  if (MASKED) {
    if (warp == 0) {
      __syncwarp();
      int use = 0, cnt = 0;
      if (p.mk.flags != nullptr && n <= kMaxTileList) {
        use = 1;
        const uint8_t* f = p.mk.flags + ((size_t)seq_s[6] * p.mk.ftq + i) * p.mk.ftk + seq_s[4];
        for (int base = 0; base < n; base += 32) {
          const int jj = base + lane;
          const bool act = jj < n && f[jj] != 0;
          const unsigned bal = __ballot_sync(0xffffffffu, act);
          if (act) tile_list[cnt + __popc(bal & ((1u << lane) - 1u))] = (uint16_t)jj;
          cnt += __popc(bal);
        }
      }
      if (lane == 0) {
        seq_s[7] = use;
        seq_s[8] = cnt;
      }
    }
    __syncthreads();
    if (seq_s[7]) {
      n = seq_s[8];
      if (n == 0) {
        if (p.rows_in_dq) no_key_vectors(p, varlen, seq_s[0], b, bh, h, i);
        const uint32_t rs = varlen ? (uint32_t)(p.H * D) : (uint32_t)D;
        uint16_t* dst = varlen ? p.dq + ((long long)seq_s[0] + 128 * i) * rs + (long long)h * D
                               : p.dq + ((long long)bh * p.N + 128 * i) * D;
        if (ATTN_IN_RANGE(varlen ? (long long)seq_s[0] + 128 * i + min(128, seq_s[1] - 128 * i) - 1
                                 : (long long)bh * p.N + 128 * i + min(128, seq_s[1] - 128 * i) - 1,
                          varlen ? (long long)p.vl.total_q : (long long)p.B * p.H * p.N, p, 0x202))
          zero_rows_bf16<D>(dst, rs, min(128, seq_s[1] - 128 * i));
        return;
      }
    }
  }
  // The j-th visited key tile, relative to jlo.
  auto tile_at = [&](int jj) -> int { return (MASKED && seq_s[7]) ? (int)tile_list[jj] : jj; };

  if (threadIdx.x == 0) {
    mbar_init(bQ, 1);
    for (int s = 0; s < T::KS; ++s) {
      mbar_init(bKf + 8u * s, 1);
      mbar_init(bKe + 8u * s, 1);
    }
    for (int s = 0; s < T::VS; ++s) {
      mbar_init(bVf + 8u * s, 1);
      mbar_init(bVe + 8u * s, 1);
    }
    mbar_init(bS, 1);
    mbar_init(bS + 8u, 1);
    mbar_init(bDp, 1);
    mbar_init(bDpc, 256);
    mbar_init(bDs, 256);
    mbar_init(bFin, 1);
    mbar_init(bDrain, 1);
    mbar_init(bO, 1);
    mbar_init(bOc, 256);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  const WaitCtx wc{abort_flag, p.status, p.limit_ns, p.info};

  if (warp < 8) {
    setmaxnreg_inc<200>();
    reg_split_sync(384);
    // ------------------------------------------------------------ compute
    const int X = warp >> 2;
    const int r = threadIdx.x & 127;  // query row within the tile == TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tdP = tmem + 256 + 64 * X + lane_off;
    const size_t vrow = (varlen ? (size_t)h * p.vec_stride + (size_t)varlen_vec_offset(seq_s[0], b)
                                : (size_t)bh * p.Npad) + (size_t)i * 128 + r;
    float l2 = -INFINITY, nD = 0.f;  // -lse * log2(e) (-inf on padding rows: P = 0 there) and -D
    bool rows_ok = true;
    if (p.rows_in_dq) {
      // This kernel forms its rows' vectors itself and writes them for the
      // dK/dV kernel: O_i arrives by TMA in K slot 2 (free until K_2), dO_i
      // is already in shared memory.  Warpgroup X sums its half of the
      // columns, [X d / 2, (X + 1) d / 2), of dO_r * O_r; the halves meet
      // through tensor-memory columns 384 + X of lane r (dQ columns, which no
      // MMA writes before every thread has passed dS_0).  Every compute
      // thread reaches the barriers below, whatever the waits return.
      const int row = 128 * i + r;
      // the row's lse first: its load overlaps the waits below
      const size_t lidx = varlen ? (size_t)h * p.vl.total_q + seq_s[0] + row : (size_t)bh * p.N + row;
      const float l = (row < seq_s[1] && ATTN_IN_RANGE(lidx, varlen ? (size_t)p.H * p.vl.total_q
                                                                      : (size_t)p.B * p.H * p.N, p, 0x203))
                          ? p.lse[lidx]
                          : -INFINITY;
      rows_ok = __all_sync(0xffffffffu, wait_bounded(wc, bQ, 0, wait_site(0x84, 0)) &&
                                            wait_bounded(wc, bO, 0, wait_site(0x85, 0)));
      float part = 0.f;
      if (rows_ok && row < seq_s[1]) {
        const uint32_t sO = sK + 2 * T::TILE_BYTES;
#pragma unroll
        for (int cc = X * (D / 16); cc < (X + 1) * (D / 16); ++cc) {
          const uint32_t off = (uint32_t)(cc >> 3) * T::BLOCK_BYTES + sw128_offset(r, cc & 7);
          const uint4 a = ld_shared_v4u(sO + off), g = ld_shared_v4u(sdO + off);
          const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 af = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[e]));
            const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[e]));
            part = fmaf(af.x, gf.x, part);
            part = fmaf(af.y, gf.y, part);
          }
        }
      }
      mbar_arrive(bOc);  // O_i read: the producer may load K_2 over it
      tmem_st1(tmem + 384 + X + lane_off, __float_as_uint(part));
      tmem_wait_st();
      tc_fence_before();
      named_bar_sync_c<2, 256>();
      tc_fence_after();
      uint32_t other = tmem_ld1(tmem + 384 + (1 - X) + lane_off);
      tmem_wait_ld();
      asm volatile("" : "+r"(other));
      nD = row < seq_s[1] ? -(part + __uint_as_float(other)) : 0.f;
      l2 = (l == -INFINITY) ? -INFINITY : -l * 1.4426950408889634f;
      size_t vst = vrow;
      if (kDebugChecks && p.debug_plant == 2 && blockIdx.x == 0) vst += vec_floats(p);  // planted mistake (test of the checks)
      if (X == 0 && rows_ok && ATTN_IN_RANGE(vst, vec_floats(p), p, 0x204)) {
        p.dvec[vst] = nD;
        p.lse2[vst] = l2;
      }
    } else if (ATTN_IN_RANGE(vrow, vec_floats(p), p, 0x205)) {
      l2 = p.lse2[vrow];
      nD = p.dvec[vrow];
    }
    const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
    const float2 l22 = make_float2(l2, l2), nD2 = make_float2(nD, nD);
    // Key columns at or past lim0 - 128 j of the j-th visited key tile are
    // invisible to row r: keys past Nk, and for causal rows keys past
    // position koff + 128 i + r.  Masked instance: the key length and the
    // window's right edge bound lim0; columns below lom0 - 128 j (the
    // window's left edge) and those whose bit is clear are hidden too.
    int lim0, lom0 = 0;
    uint32_t rowbits = 0xffffffffu;  // word index of this row's bits (all ones: none)
    if (MASKED) {
      const int pos = seq_s[3] - seq_s[1] + 128 * i + r, jlo = seq_s[4];
      int hi = seq_s[5];
      if (p.mk.wr >= 0) hi = min(hi, pos + p.mk.wr + 1);
      lim0 = hi - 128 * jlo - 64 * X;
      lom0 = (p.mk.wl >= 0 ? pos - p.mk.wl : -(1 << 30)) - 128 * jlo - 64 * X;
      if (p.mk.bits != nullptr && 128 * i + r < p.N)
        rowbits = ((uint32_t)seq_s[6] * (uint32_t)p.N + (uint32_t)(128 * i + r)) * (uint32_t)p.mk.words +
                  4u * jlo + 2u * X;
    } else {
      lim0 = (CAUSAL ? min(seq_s[3], seq_s[3] - seq_s[1] + 128 * i + r + 1) : seq_s[3]) - 64 * X;
    }
    bool ok = rows_ok;
    for (int j = 0; j < n && ok; ++j) {
      const uint32_t tS = tmem + (j & 1) * 128 + 64 * X + lane_off;
      uint2 bt = make_uint2(~0u, ~0u);
      const int jt = MASKED ? tile_at(j) : j;  // key tile relative to jlo
      if (MASKED && rowbits != 0xffffffffu &&
          ATTN_IN_RANGE((size_t)rowbits + 4u * jt + 1u, (size_t)p.mk.mask_b * p.mk.mask_h * p.N * p.mk.words, p, 0x206))
        bt = *reinterpret_cast<const uint2*>(p.mk.bits + rowbits + 4u * jt);
      // The additive mask of this row over the warpgroup's 64 keys, loaded
      // before the wait for S; added as b / scale to the unscaled scores.
      // Columns past Nk are not read.
      float bb[MASKED >= 2 ? 64 : 1];
      if constexpr (MASKED >= 2) {
        const int row = 128 * i + r, k0 = (seq_s[4] + jt) * 128 + 64 * X;
        const size_t boff = ((size_t)bias_plane(p.mk, b, h) * p.N + (size_t)row) * p.Nk + (size_t)k0;
        int bn = row < seq_s[1] ? min(64, p.Nk - k0) : 0;
        if (bn > 0 && !ATTN_IN_RANGE(boff + bn - 1, (size_t)p.mk.bias_b * p.mk.bias_h * p.N * p.Nk, p, 0x207)) bn = 0;
        load_bias_row<64, MASKED == 3>(p.mk.bias, boff, bn, bias_rows_vec(p.mk.bias, p.Nk, MASKED == 3), bb);
      }
      ok = __all_sync(0xffffffffu, wait_bounded(wc, bS + 8u * (j & 1), (j >> 1) & 1, wait_site(0x81, j)));
      if (!ok) break;
      tc_fence_after();
      float x[64];
      {
        uint32_t ra[32], rb[32];
        tmem_ld32(tS + 0, ra);
        tmem_ld32(tS + 32, rb);
        tmem_wait_ld();
        reg_fence(ra);
        reg_fence(rb);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          x[e] = __uint_as_float(ra[e]);
          x[32 + e] = __uint_as_float(rb[e]);
        }
      }
      if constexpr (MASKED >= 2) {
#pragma unroll
        for (int k = 0; k < 64; ++k) x[k] = fmaf(bb[k], p.mk.inv_scale, x[k]);
      }
      // P[r][k] = exp2(S * scale * log2e - lse2[r]); invisible keys (past
      // the row's causal position, or past Nk) are exactly 0.
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float2 t = ffma2(make_float2(x[2 * e], x[2 * e + 1]), c2, l22);
        x[2 * e] = ex2(t.x);
        x[2 * e + 1] = ex2(t.y);
      }
      if (MASKED) {
        const int lim = lim0 - 128 * jt, lom = lom0 - 128 * jt;
        if (__any_sync(0xffffffffu, lim < 64 || lom > 0 || (bt.x & bt.y) != ~0u)) {
#pragma unroll
          for (int k = 0; k < 64; ++k)
            if (k >= lim || k < lom || !((((k < 32) ? bt.x : bt.y) >> (k & 31)) & 1u)) x[k] = 0.f;
        }
      } else {
        const int lim = lim0 - 128 * j;
        if (__any_sync(0xffffffffu, lim < 64)) {
#pragma unroll
          for (int k = 0; k < 64; ++k)
            if (k >= lim) x[k] = 0.f;
        }
      }
      ok = __all_sync(0xffffffffu, wait_bounded(wc, bDp, j & 1, wait_site(0x82, j)));
      if (!ok) break;
      tc_fence_after();
      // dS[r][k] = P * (dP - D) -> bf16 pairs over this warpgroup's S columns
      uint32_t w[32];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t g[32];
        tmem_ld32(tdP + 32 * hh, g);
        tmem_wait_ld();
        reg_fence(g);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int k = 32 * hh + 2 * e;
          const float2 ds = fmul2(make_float2(x[k], x[k + 1]),
                                  fadd2(make_float2(__uint_as_float(g[2 * e]), __uint_as_float(g[2 * e + 1])), nD2));
          w[16 * hh + e] = pack_bf16(ds.x, ds.y);
        }
      }
      tc_fence_before();
      mbar_arrive(bDpc);  // the dP columns may be overwritten
      tmem_st32(tS, w);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bDs);
    }
    // ------------------------------------------------------------ dQ out
    // dQ_i = scale * (sum_j dS K_j) -> bf16 -> the Q tile (dead once every
    // MMA has completed) -> TMA store.  Warpgroup X takes the 32-column
    // groups cc with cc % 2 == X.
    if (ok) ok = __all_sync(0xffffffffu, wait_bounded(wc, bFin, 0, wait_site(0x83, n)));
    if (ok) {
      tc_fence_after();
      const uint32_t tQd = tmem + 384 + lane_off;
      const float2 s2 = make_float2(p.scale, p.scale);
#pragma unroll
      for (int cc = X; cc < D / 32; cc += 2) {
        uint32_t o[32];
        tmem_ld32(tQd + cc * 32, o);
        tmem_wait_ld();
        reg_fence(o);
        const int blk = (cc * 32) / 64, ch0 = ((cc * 32) % 64) / 8;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t ww[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 t = fmul2(make_float2(__uint_as_float(o[q4 * 8 + 2 * e]), __uint_as_float(o[q4 * 8 + 2 * e + 1])), s2);
            ww[e] = pack_bf16(t.x, t.y);
          }
          st_shared_v4(sQ + blk * T::BLOCK_BYTES + sw128_offset(r, ch0 + q4), ww[0], ww[1], ww[2], ww[3]);
        }
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 256);
    if (ok) {
      // The dense batch clips the box at Nq; in a packed batch the rows past
      // the sequence belong to the next one, so a partial tile is stored row
      // by row instead.
      const int q0 = seq_s[0], valid = seq_s[1] - 128 * i;
      if (valid >= 128 || !varlen) {
        if (threadIdx.x == 0) {
          for (int cb = 0; cb < T::NB; ++cb)
            tma_store_3d(&tmdQ, sQ + cb * T::BLOCK_BYTES, cb * 64, q0 + i * 128, qplane);
          bulk_commit();
          bulk_wait_read_all();  // the tile has been read out of shared memory
        }
      } else {
        const uint32_t rs = (uint32_t)(p.H * D);
        if (ATTN_IN_RANGE((long long)q0 + 128 * i + valid - 1, p.vl.total_q, p, 0x208))
          store_rows_sw128<D>(sQ, p.dq + ((long long)q0 + 128 * i) * rs + (long long)h * D, rs, valid, threadIdx.x, 256);
      }
    }
    setmaxnreg_dec<168>();
  } else {
    setmaxnreg_dec<104>();
    reg_split_sync(384);
    if (warp == 8) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        const int q0 = seq_s[0], k0 = seq_s[2] + 128 * seq_s[4];  // from the first visited key tile
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        mbar_expect_tx(bQ, 2 * T::TILE_BYTES);
        for (int cb = 0; cb < T::NB; ++cb) {
          tma_load_3d(sQ + cb * T::BLOCK_BYTES, &tmQ, bQ, cb * 64, q0 + i * 128, qplane);
          tma_load_3d(sdO + cb * T::BLOCK_BYTES, &tmdO, bQ, cb * 64, q0 + i * 128, qplane);
        }
        // O_i for the row vectors, right after Q_i and dO_i: the compute
        // threads form them while K_0 and V_0 arrive and S_0 is computed.
        const bool o_issued = p.rows_in_dq != 0;
        if (o_issued) {
          mbar_expect_tx(bO, T::TILE_BYTES);
          for (int cb = 0; cb < T::NB; ++cb)
            tma_load_3d(sK + 2 * T::TILE_BYTES + cb * T::BLOCK_BYTES, &tmO, bO, cb * 64, q0 + i * 128, qplane);
        }
        int issued = 0;
        for (int j = 0; j < n; ++j) {
          const int ks = j % T::KS, kr = j / T::KS, vs = j % T::VS, vr = j / T::VS;
          if (kr > 0 && !wait_bounded(wc, bKe + 8u * ks, (kr - 1) & 1, wait_site(0x91, j))) break;
          if (o_issued && j == 2 && !wait_bounded(wc, bOc, 0, wait_site(0x93, j))) break;
          // (p.debug_drop1: a test of the bounded waits skips one load in CTA 0)
          if (!(p.debug_drop1 == 2 * j + 1 && blockIdx.x == 0)) {
            mbar_expect_tx(bKf + 8u * ks, T::TILE_BYTES);
            for (int cb = 0; cb < T::NB; ++cb)
              tma_load_3d(sK + ks * T::TILE_BYTES + cb * T::BLOCK_BYTES, &tmK, bKf + 8u * ks, cb * 64,
                          k0 + tile_at(j) * 128, kplane);
          }
          issued = 2 * j + 1;
          if (vr > 0 && !wait_bounded(wc, bVe + 8u * vs, (vr - 1) & 1, wait_site(0x92, j))) break;
          if (!(p.debug_drop1 == 2 * j + 2 && blockIdx.x == 0)) {
            mbar_expect_tx(bVf + 8u * vs, T::TILE_BYTES);
            for (int cb = 0; cb < T::NB; ++cb)
              tma_load_3d(sV + vs * T::TILE_BYTES + cb * T::BLOCK_BYTES, &tmV, bVf + 8u * vs, cb * 64,
                          k0 + tile_at(j) * 128, kplane);
          }
          issued = 2 * j + 2;
        }
        // Every copy issued above has landed before the CTA may exit.
        wait_drain(bQ, 0, p.limit_ns);
        if (o_issued) wait_drain(bO, 0, p.limit_ns);
        const int nk = (issued + 1) / 2, nv = issued / 2;  // K_0..K_{nk-1}, V_0..V_{nv-1} issued
        for (int s = 0; s < T::KS && s < nk; ++s) {
          const int last = ((nk - 1 - s) / T::KS) * T::KS + s;
          wait_drain(bKf + 8u * s, (last / T::KS) & 1, p.limit_ns);
        }
        for (int s = 0; s < T::VS && s < nv; ++s) {
          const int last = ((nv - 1 - s) / T::VS) * T::VS + s;
          wait_drain(bVf + 8u * s, (last / T::VS) & 1, p.limit_ns);
        }
      }
      __syncwarp();
    } else if (warp == 9) {
      // ------------------------------------------------------------ MMA issuer
      // Per step j: dP_{j+1} (once dP_j has been read), dQ += dS_j K_j,
      // S_{j+2} into the S buffer dS_j occupied.
      {
        const uint32_t leader = elect_one();
        constexpr uint32_t I_SS = idesc_bf16_f32(128, 128, false, false);  // S, dP (K-major x K-major)
        constexpr uint32_t I_DQ = idesc_bf16_f32(128, D, false, true);     // dQ (A in TMEM, B MN-major)
        const uint32_t tdP = tmem + 256, tdQ = tmem + 384;
        const uint64_t dQk = sdesc_sw128(sQ, 16, 1024);                 // Q, K-major A
        const uint64_t dOk = sdesc_sw128(sdO, 16, 1024);                // dO, K-major A
        const uint64_t dKk0 = sdesc_sw128(sK, 16, 1024);                // K slot 0, K-major B (S)
        const uint64_t dKmn0 = sdesc_sw128(sK, T::BLOCK_BYTES, 1024);   // K slot 0, MN-major B (dQ)
        const uint64_t dVk0 = sdesc_sw128(sV, 16, 1024);                // V slot 0, K-major B (dP)
        auto mma_kk = [&](uint32_t dst, uint64_t ad, uint64_t bd, uint32_t idesc) {
#pragma unroll
          for (int kk = 0; kk < T::KSTEPS; ++kk) {
            const uint32_t off = (kk >> 2) * T::BLOCK_BYTES + (kk & 3) * 32;
            mma_ss_p(leader, dst, sdesc_add(ad, off), sdesc_add(bd, off), idesc, kk > 0);
          }
        };
        auto wait_all = [&](uint32_t bar, uint32_t parity, int site) {
          return __all_sync(0xffffffffu, wait_bounded(wc, bar, parity, site));
        };
        // Each group's barrier checks run right after the previous group's
        // MMAs are issued and before that group's commit: the commit returns
        // only once its MMAs have nearly drained, so a check placed after it
        // would leave the tensor pipe idle for its length.  No check waits on
        // a signal that the commit it precedes would give.
        bool ok = wait_all(bQ, 0, wait_site(0xa1, 0)) && wait_all(bKf, 0, wait_site(0xa2, 0)) &&
                  wait_all(bVf, 0, wait_site(0xa3, 0));
        if (ok) {
          tc_fence_after();
          mma_kk(tmem, dQk, dKk0, I_SS);  // S_0
          mma_commit_p(leader, bS);
          mma_kk(tdP, dOk, dVk0, I_SS);  // dP_0
          if (n > 1) ok = wait_all(bKf + 8u, 0, wait_site(0xa4, 1));  // for S_1
          mma_commit_p(leader, bDp);
          mma_commit_p(leader, bVe);  // V_0 consumed
          if (ok && n > 1) {
            tc_fence_after();
            mma_kk(tmem + 128, dQk, sdesc_add(dKk0, T::TILE_BYTES), I_SS);  // S_1
            // for dP_1: V_1 loaded, dP_0 read
            ok = wait_all(bVf + 8u * (1 % T::VS), (1 / T::VS) & 1, wait_site(0xa5, 0)) &&
                 wait_all(bDpc, 0, wait_site(0xa6, 0));
            mma_commit_p(leader, bS + 8u);
          }
        }
        for (int j = 0; j < n && ok; ++j) {
          // dP_{j+1} (its conditions were checked during the previous group),
          // then dQ += dS_j K_j, then S_{j+2} into the S buffer dS_j occupied
          // (MMAs from one thread run in order, so dQ has read dS_j first).
          if (j + 1 < n) {
            const int vs = (j + 1) % T::VS;
            tc_fence_after();
            mma_kk(tdP, dOk, sdesc_add(dVk0, vs * T::TILE_BYTES), I_SS);  // dP_{j+1}
            ok = wait_all(bDs, j & 1, wait_site(0xa7, j));               // for dQ_j
            mma_commit_p(leader, bDp);
            mma_commit_p(leader, bVe + 8u * vs);
          } else {
            ok = wait_all(bDs, j & 1, wait_site(0xa7, j));
          }
          if (!ok) break;
          tc_fence_after();
          // dQ += dS_j K_j: A = dS in TMEM (keys 64X.. of warpgroup X at
          // columns 64X.., bf16 pairs), B = K_j (MN-major, N = d)
          const int ks = j % T::KS;
          const uint32_t tS = tmem + (j & 1) * 128;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts_p(leader, tdQ, tS + 64 * (kk >> 2) + (kk & 3) * 8,
                     sdesc_add(dKmn0, ks * T::TILE_BYTES + kk * 2048), I_DQ, (j > 0 || kk > 0) ? 1u : 0u);
          const int k2 = (j + 2) % T::KS;
          if (j + 2 < n) ok = wait_all(bKf + 8u * k2, ((j + 2) / T::KS) & 1, wait_site(0xa8, j));  // for S_{j+2}
          mma_commit_p(leader, bKe + 8u * ks);  // K_j consumed
          if (!ok) break;
          if (j + 2 < n) {
            tc_fence_after();
            mma_kk(tS, dQk, sdesc_add(dKk0, k2 * T::TILE_BYTES), I_SS);  // S_{j+2}
            // for dP_{j+2}: V_{j+2} loaded, dP_{j+1} read
            ok = wait_all(bVf + 8u * ((j + 2) % T::VS), ((j + 2) / T::VS) & 1, wait_site(0xa5, j + 1)) &&
                 wait_all(bDpc, (j + 1) & 1, wait_site(0xa6, j + 1));
            mma_commit_p(leader, bS + 8u * (j & 1));
          }
        }
        if (ok) mma_commit_p(leader, bFin);
        mma_commit_p(leader, bDrain);  // fires once every MMA issued above has finished
        wait_drain(bDrain, 0, p.limit_ns);
      }
      __syncwarp();
    }
    setmaxnreg_inc<168>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

size_t bwd_dq_smem_bytes(int d) {
  switch (d) {
    case 64: return DqTraits<64>::SMEM;
    case 96: return DqTraits<96>::SMEM;
    case 128: return DqTraits<128>::SMEM;
    default: return 0;
  }
}

template <int D, bool C, int M = 0>
static cudaError_t launch_dq_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& to,
                               const BwdParams& p, cudaStream_t stream) {
  auto kern = bwd_dq_kernel<D, C, M>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DqTraits<D>::SMEM);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)p.nq * (unsigned)(p.B * p.H);
  BwdParams pc = p;
  pc.tail = uniform_levels(C, p.vl, p.mk, M != 0) ? 1 : order_tail(p.nq, p.B * p.H, p.G);
  kern<<<grid, DqTraits<D>::THREADS, DqTraits<D>::SMEM, stream>>>(tq, tk, tv, tdo, tdq, to, pc);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& to, const BwdParams& p,
                          cudaStream_t stream, bool masked) {
  if (masked) {
    const bool bias = p.mk.bias != nullptr;  // the instances with the additive mask (float32, bf16)
    switch (d) {
      case 64: return bias ? (p.mk.bias_bf16 ? launch_dq_t<64, false, 3>(tq, tk, tv, tdo, tdq, to, p, stream) : launch_dq_t<64, false, 2>(tq, tk, tv, tdo, tdq, to, p, stream))
                      : launch_dq_t<64, false, 1>(tq, tk, tv, tdo, tdq, to, p, stream);
      case 96: return bias ? (p.mk.bias_bf16 ? launch_dq_t<96, false, 3>(tq, tk, tv, tdo, tdq, to, p, stream) : launch_dq_t<96, false, 2>(tq, tk, tv, tdo, tdq, to, p, stream))
                      : launch_dq_t<96, false, 1>(tq, tk, tv, tdo, tdq, to, p, stream);
      case 128: return bias ? (p.mk.bias_bf16 ? launch_dq_t<128, false, 3>(tq, tk, tv, tdo, tdq, to, p, stream) : launch_dq_t<128, false, 2>(tq, tk, tv, tdo, tdq, to, p, stream))
                      : launch_dq_t<128, false, 1>(tq, tk, tv, tdo, tdq, to, p, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  // The dense batch runs the persistent kernel; launches armed by the test
  // hooks of this kernel keep it (their tests expect its CTA mapping).
  if (p.vl.cu_q == nullptr && p.debug_drop1 == 0 && p.debug_plant == 0 && p.dq != nullptr &&
      (!p.rows_in_dq || (p.o != nullptr && p.dout != nullptr && p.lse != nullptr)))
    return launch_bwd_dq_persist(d, causal, tq, tk, tv, tdo, p, stream);
  switch (d) {
    case 64: return causal ? launch_dq_t<64, true>(tq, tk, tv, tdo, tdq, to, p, stream)
                           : launch_dq_t<64, false>(tq, tk, tv, tdo, tdq, to, p, stream);
    case 96: return causal ? launch_dq_t<96, true>(tq, tk, tv, tdo, tdq, to, p, stream)
                           : launch_dq_t<96, false>(tq, tk, tv, tdo, tdq, to, p, stream);
    case 128: return causal ? launch_dq_t<128, true>(tq, tk, tv, tdo, tdq, to, p, stream)
                            : launch_dq_t<128, false>(tq, tk, tv, tdo, tdq, to, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sdpa
