// attn_bwd_dq_persist.cu — the dQ kernel of the dense backward (no mask, no
// packed batch) as a persistent kernel on sm_103a.
//
// Method and arithmetic: those of attn_bwd_dq.cu's bwd_dq_kernel (page
// "Flash Attention原理", §五: P recomputed from lse, dP = dO V^T,
// dS = P (dP - D), dQ = scale dS K, and the row vectors D = rowsum(dO * O)
// and lse in base 2), unchanged, so the two kernels give the same bits.
// What differs is the schedule: one CTA per SM takes the (head, query tile)
// units of bwd_dq_kernel, in the same order (work_unit), from a queue until
// none is left, instead of one CTA per unit paying its launch, barrier and
// tensor-memory setup, the wait for its first tiles and its epilogue while
// the tensor core idles (about 6 us of a 22 us unit at C5).
//
// GB300 mapping: bwd_dq_kernel's roles (warps 0-7 compute, warp 8 the TMA
// producer, warp 9 the MMA issuer), with these differences:
//   * Q_i and dO_i go from shared memory into tensor memory once per unit
//     (the compute threads copy their rows), and S = Q K_j^T and
//     dP = dO V_j^T take them from there: a 128 x 128 x 16 product with both
//     operands in shared memory reads 8 KB per 64 cycles, as much as shared
//     memory delivers, so with the K/V tiles streaming in the products were
//     bound by shared-memory bandwidth; with A in tensor memory they read
//     half of that.  The tensor memory that costs is won by keeping one S
//     buffer (released as soon as the compute threads have loaded S_j, so
//     S_{j+1} runs during the exponentials) and writing dS_j over dP_j;
//     per step the products run S_{j+1}, dQ_j, dP_{j+1};
//   * warps 10-11 take the units from the queue and pass each one on through
//     a two-entry ring in shared memory, with the unit's row vectors (-lse2,
//     -D for its 128 query rows), which they form from lse, O and dO in
//     global memory (or copy from the workspace, when an earlier stage formed
//     them) while the unit before it runs; they also write the vectors to
//     the workspace for the dK/dV kernel, and ask L2 for the unit's Q and dO
//     tiles ahead of the producer's loads;
//   * the K and V rings and every per-step barrier run on across units, and
//     the shared-memory Q and dO tiles are free once copied, so the next
//     unit's tiles load while the current unit runs;
//   * dQ leaves from registers straight to global memory (each warp's rows
//     transposed across its lanes so that a store covers whole lines).
// Tensor memory: S [0,128), dP and then dS [128,256), dQ [256,256+d),
// Q [384,384+d/2), dO [448,448+d/2) (bf16 pairs).
#include <atomic>
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {

namespace {

template <int D>
struct PQTraits {
  static constexpr int NB = (D + 63) / 64;
  static constexpr int BLOCK_BYTES = 128 * 128;
  static constexpr int TILE_BYTES = NB * BLOCK_BYTES;  // one [128 rows x d] bf16 tile
  static constexpr int KSTEPS = D / 16;
  static constexpr int KS = 3, VS = 2;                 // K and V ring slots
  static constexpr int VEC_BYTES = 1024;               // -lse2[128], -D[128]
  // q_full do_full staged k_full[3] k_empty[3] v_full[2] v_empty[2]
  // s s_read dp ds fin unit_full[2] unit_vec[2] unit_empty[2] drain
  static constexpr int NBAR = 3 + 6 + 4 + 5 + 6 + 1;
  static constexpr int TILES_BYTES = (2 + KS + VS) * TILE_BYTES;  // Q, dO, K[3], V[2]
  static constexpr int MISC = 32;                                 // tmem slot, abort flag, unit ring, stop flag
  static constexpr int SMEM = TILES_BYTES + 2 * VEC_BYTES + NBAR * 8 + MISC;
  static constexpr int THREADS = 384;
};
static_assert(PQTraits<128>::SMEM <= 227 * 1024, "shared memory");

// Arrivals on unit_empty: every thread that reads a ring entry (the compute
// warpgroups, the MMA warp and the producer warp).
constexpr int kDqUnitReaders = 256 + 32 + 32;
// Named barrier of the two vector warps (ids 0, 15 and the compute
// warpgroups' are taken elsewhere).
constexpr uint32_t kVecBarrier = 5;

}  // namespace

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    bwd_dq_persist_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                          const BwdParams p) {
  using T = PQTraits<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = smem_u32(smem_raw);
  if (base & 1023u) {  // the layout needs a 1024-byte aligned start (128-byte swizzle atoms)
    if (threadIdx.x == 0) atomicCAS(p.status, 0, kDevMisaligned);
    return;
  }
  const uint32_t sQ = base;                          // Q_i
  const uint32_t sdO = sQ + T::TILE_BYTES;           // dO_i
  const uint32_t sK = sdO + T::TILE_BYTES;           // [KS] K_j
  const uint32_t sV = sK + T::KS * T::TILE_BYTES;    // [VS] V_j
  const uint32_t sVec = sV + T::VS * T::TILE_BYTES;  // [2] x {-lse2[128], -D[128]}
  const uint32_t sBar = sVec + 2 * T::VEC_BYTES;
  const uint32_t bQf = sBar;            // Q_i loaded
  const uint32_t bOf = bQf + 8;         // dO_i loaded
  const uint32_t bQs = bOf + 8;         // Q_i, dO_i copied to tensor memory (256 arrivals): shared tiles free
  const uint32_t bKf = bQs + 8;         // [KS] K slot full
  const uint32_t bKe = bKf + 8 * T::KS; // [KS] K slot free (after dQ += dS K_j)
  const uint32_t bVf = bKe + 8 * T::KS; // [VS] V slot full
  const uint32_t bVe = bVf + 8 * T::VS; // [VS] V slot free (after dP_j)
  const uint32_t bS = bVe + 8 * T::VS;  // S_j ready
  const uint32_t bSr = bS + 8;          // S_j loaded by the compute threads (256 arrivals): S buffer free
  const uint32_t bDp = bSr + 8;         // dP_j ready
  const uint32_t bDs = bDp + 8;         // dS_j in TMEM over dP_j (256 arrivals)
  const uint32_t bFin = bDs + 8;        // every MMA of the unit done
  const uint32_t bUf = bFin + 8;        // [2] unit ring entry written
  const uint32_t bUv = bUf + 16;        // [2] its row vectors written (64 arrivals)
  const uint32_t bUe = bUv + 16;        // [2] unit ring entry read
  const uint32_t bDrain = bUe + 16;
  static_assert(3 + 2 * T::KS + 2 * T::VS + 5 + 6 + 1 == T::NBAR, "barrier count");
  uint8_t* const misc = smem_raw + (sBar - base) + 8 * T::NBAR;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  volatile int* const unit_ring = reinterpret_cast<volatile int*>(misc + 8);  // [2]
  volatile int* const vec_stop = reinterpret_cast<volatile int*>(misc + 16);  // the vector warps stop
  float* const vec_s = reinterpret_cast<float*>(smem_raw + (sVec - base));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // A unit's head, query tile and key tiles visited (causal: up to the tile
  // holding the last row's last visible key, query row r at position
  // koff + r).
  auto unit_of = [&](int u, int& bh, int& i, int& n) {
    int lv;
    work_unit(u, p.nq, p.B * p.H, p.tail, bh, lv);
    i = p.nq - 1 - lv;
    n = CAUSAL ? min(p.nkv, (p.koff + i * 128 + 127) / 128 + 1) : p.nkv;
  };

  if (threadIdx.x == 0) {
    mbar_init(bQf, 1);
    mbar_init(bOf, 1);
    mbar_init(bQs, 256);
    for (int s = 0; s < T::KS; ++s) {
      mbar_init(bKf + 8u * s, 1);
      mbar_init(bKe + 8u * s, 1);
    }
    for (int s = 0; s < T::VS; ++s) {
      mbar_init(bVf + 8u * s, 1);
      mbar_init(bVe + 8u * s, 1);
    }
    mbar_init(bS, 1);
    mbar_init(bSr, 256);
    mbar_init(bDp, 1);
    mbar_init(bDs, 256);
    mbar_init(bFin, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bUf + 8u * s, 1);
      mbar_init(bUv + 8u * s, 64);
      mbar_init(bUe + 8u * s, kDqUnitReaders);
    }
    mbar_init(bDrain, 1);
    *abort_flag = 0;
    *vec_stop = 0;
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
  // The k-th unit this CTA takes, as read from the ring by the producer or
  // the MMA warp (-1: none left, or the vector warps stopped).
  auto next_unit = [&](int k, bool& ok) -> int {
    const int e = k & 1;
    ok = __all_sync(0xffffffffu, wait_bounded(wc, bUf + 8u * e, (k >> 1) & 1, wait_site(0xb0, k)));
    const int u = ok ? unit_ring[e] : -1;
    mbar_arrive(bUe + 8u * e);
    return u;
  };

  if (warp < 8) {
    setmaxnreg_inc<200>();
    reg_split_sync(384);
    // ------------------------------------------------------------ compute
    // Warpgroup X takes key columns [64X, 64X + 64) of each 128 x 128
    // (queries x keys) tile, one thread per query row; the body is
    // bwd_dq_kernel's for the dense batch.
    const int X = warp >> 2;
    const int r = threadIdx.x & 127;  // query row within the tile == TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + 64 * X + lane_off;          // S columns of this half
    const uint32_t tdP = tmem + 128 + 64 * X + lane_off;   // dP columns of this half; dS pairs after
    const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
    // Row r of a [128 x D] bf16 tile in shared memory (128-byte swizzle,
    // 64-column blocks), columns [X D/2, (X + 1) D/2), as bf16 pairs into
    // tensor-memory columns [X D/4, (X + 1) D/4) from tcol: the A operand
    // layout (column c holds elements 2c, 2c + 1 of the row).
    auto stage_half = [&](uint32_t stile, uint32_t tcol) {
      constexpr int CH = D / 16;  // 16-byte chunks in the half
      uint32_t w[4 * CH];
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int cg = X * CH + c;
        const uint4 v = ld_shared_v4u(stile + (uint32_t)(cg >> 3) * T::BLOCK_BYTES + sw128_offset(r, cg & 7));
        w[4 * c] = v.x;
        w[4 * c + 1] = v.y;
        w[4 * c + 2] = v.z;
        w[4 * c + 3] = v.w;
      }
      const uint32_t t0 = tcol + X * (D / 4) + lane_off;
#pragma unroll
      for (int o = 0; o + 16 <= 4 * CH; o += 16) {
        uint32_t q[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) q[e] = w[o + e];
        tmem_st16(t0 + o, q);
      }
      if constexpr ((4 * CH) % 16 != 0) {
        uint32_t q[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) q[e] = w[4 * CH - 8 + e];
        tmem_st8(t0 + 4 * CH - 8, q);
      }
    };
    uint32_t gs = 0;  // steps over all units so far
    int kf = 0;       // units with steps whose products are done
    int ks = 0;       // units with steps whose Q and dO were copied
    // A unit as read from ring entry k & 1, with this row's vectors.  The
    // entry is released when the unit is done (release()), so that the
    // vector warps run one unit ahead, not two: their reads of O and dO
    // then come close enough to the producer's dO load for it to find dO in
    // L2.
    struct CUnit {
      int u, bh, i, n;
      float l2, nD;  // -lse * log2(e) (-inf on padding rows: P = 0 there) and -D
    };
    auto take = [&](int k, CUnit& c) -> bool {
      const int e = k & 1;
      bool got = __all_sync(0xffffffffu, wait_bounded(wc, bUf + 8u * e, (k >> 1) & 1, wait_site(0xb1, k)));
      c.u = got ? unit_ring[e] : -1;
      c.l2 = -INFINITY;
      c.nD = 0.f;
      if (c.u >= 0) {
        got = __all_sync(0xffffffffu, wait_bounded(wc, bUv + 8u * e, (k >> 1) & 1, wait_site(0xb2, k)));
        if (got) {
          c.l2 = vec_s[e * 256 + r];
          c.nD = vec_s[e * 256 + 128 + r];
        }
      }
      if (c.u < 0) mbar_arrive(bUe + 8u * e);
      c.bh = c.i = c.n = 0;
      if (c.u >= 0) unit_of(c.u, c.bh, c.i, c.n);
      return got;
    };
    // Q_i and dO_i of a unit with steps into tensor memory; the unit before
    // has finished every product (the caller waited for that), so their
    // columns are free.  Then the next unit's tiles may load.
    auto stage = [&](int k) -> bool {
      if (!__all_sync(0xffffffffu, wait_bounded(wc, bQf, ks & 1, wait_site(0xf1, k)) &&
                                       wait_bounded(wc, bOf, ks & 1, wait_site(0xf2, k))))
        return false;
      stage_half(sQ, tmem + 384);
      stage_half(sdO, tmem + 448);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bQs);  // (also: the shared Q and dO tiles may be overwritten)
      ++ks;
      return true;
    };
    auto release = [&](int k) { mbar_arrive(bUe + 8u * (k & 1)); };
    CUnit cur;
    bool ok = take(0, cur);
    if (ok && cur.u >= 0 && cur.n > 0) ok = stage(0);
    for (int k = 0; ok && cur.u >= 0; ++k) {
      const int i = cur.i, n = cur.n, bh = cur.bh;
      if (n <= 0) {
        // No row of the tile sees a key: dQ = 0 (the vector warps wrote the
        // rows' vectors).
        const int row = 128 * i + r;
        uint16_t* const dqrow = p.dq + ((size_t)bh * p.N + row) * D;
        if (row < p.N && ATTN_IN_RANGE(((size_t)bh * p.N + row) * D + D - 1, (size_t)p.B * p.H * p.N * D, p, 0x209))
          for (int c8 = X * (D / 16); c8 < (X + 1) * (D / 16); ++c8)
            *reinterpret_cast<uint4*>(dqrow + 8 * c8) = make_uint4(0, 0, 0, 0);
        release(k);
        CUnit nx;
        ok = take(k + 1, nx);
        if (ok && nx.u >= 0 && nx.n > 0) ok = stage(k + 1);
        cur = nx;
        continue;
      }
      const float2 l22 = make_float2(cur.l2, cur.l2), nD2 = make_float2(cur.nD, cur.nD);
      // Key columns at or past lim0 - 128 j of key tile j are invisible to
      // row r: keys past Nk, and for causal rows keys past position
      // koff + 128 i + r.
      const int lim0 = (CAUSAL ? min(p.Nk, p.koff + 128 * i + r + 1) : p.Nk) - 64 * X;
      for (int j = 0; j < n; ++j, ++gs) {
        ok = __all_sync(0xffffffffu, wait_bounded(wc, bS, gs & 1, wait_site(0xb3, j)));
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
          for (int q = 0; q < 32; ++q) {
            x[q] = __uint_as_float(ra[q]);
            x[32 + q] = __uint_as_float(rb[q]);
          }
        }
        tc_fence_before();
        mbar_arrive(bSr);  // the S buffer may take S_{j+1}
        // P[r][k] = exp2(S * scale * log2e - lse2[r]); invisible keys (past
        // the row's causal position, or past Nk) are exactly 0.
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const float2 t = ffma2(make_float2(x[2 * q], x[2 * q + 1]), c2, l22);
          x[2 * q] = ex2(t.x);
          x[2 * q + 1] = ex2(t.y);
        }
        {
          const int lim = lim0 - 128 * j;
          if (__any_sync(0xffffffffu, lim < 64)) {
#pragma unroll
            for (int q = 0; q < 64; ++q)
              if (q >= lim) x[q] = 0.f;
          }
        }
        ok = __all_sync(0xffffffffu, wait_bounded(wc, bDp, gs & 1, wait_site(0xb4, j)));
        if (!ok) break;
        tc_fence_after();
        // dS[r][k] = P * (dP - D) -> bf16 pairs over this warpgroup's first
        // 32 dP columns (read before they are written)
        uint32_t w[32];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t g[32];
          tmem_ld32(tdP + 32 * hh, g);
          tmem_wait_ld();
          reg_fence(g);
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int c = 32 * hh + 2 * q;
            const float2 ds = fmul2(make_float2(x[c], x[c + 1]),
                                    fadd2(make_float2(__uint_as_float(g[2 * q]), __uint_as_float(g[2 * q + 1])), nD2));
            w[16 * hh + q] = pack_bf16(ds.x, ds.y);
          }
        }
        tmem_st32(tdP, w);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bDs);
      }
      if (!ok) break;
      // ---------------------------------------------------------- dQ out
      // Once every product of the unit is done: the next unit from the
      // ring, its Q and dO into tensor memory (so that its first products
      // run during what follows), then dQ_i = scale * (sum_j dS K_j) -> bf16
      // -> dQ, from registers: warpgroup X takes the 32-column groups
      // [X GH, min(G, (X + 1) GH)), and each warp writes its 32 rows a row
      // slice per group of lanes (store_rows_transposed), whole lines per
      // store.  The next unit's first dQ product, which overwrites the
      // accumulator, waits for this warpgroup's next dS, published after
      // these loads.
      ok = __all_sync(0xffffffffu, wait_bounded(wc, bFin, kf & 1, wait_site(0xb5, k)));
      if (!ok) break;
      ++kf;
      tc_fence_after();
      CUnit nx;
      ok = take(k + 1, nx);
      if (ok && nx.u >= 0 && nx.n > 0) ok = stage(k + 1);
      if (!ok) break;
      {
        constexpr int G = D / 32, GH = (G + 1) / 2;
        const uint32_t tQd = tmem + 256 + lane_off;
        const float2 s2 = make_float2(p.scale, p.scale);
        const int wr0 = 128 * i + 32 * (warp & 3);  // the warp's first row
        uint16_t* const wdst = p.dq + ((size_t)bh * p.N + wr0) * D;
        int nvalid = min(32, p.N - wr0);
        if (nvalid > 0 && !ATTN_IN_RANGE(((size_t)bh * p.N + wr0 + nvalid) * D - 1, (size_t)p.B * p.H * p.N * D, p, 0x209))
          nvalid = 0;
        // Columns 32 cc .. 32 cc + 31 of this thread's row as four bf16 chunks.
        auto chunks = [&](int cc, uint4* ch) {
          uint32_t o[32];
          tmem_ld32(tQd + cc * 32, o);
          tmem_wait_ld();
          reg_fence(o);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t ww[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float2 t =
                  fmul2(make_float2(__uint_as_float(o[q4 * 8 + 2 * q]), __uint_as_float(o[q4 * 8 + 2 * q + 1])), s2);
              ww[q] = pack_bf16(t.x, t.y);
            }
            ch[q4] = make_uint4(ww[0], ww[1], ww[2], ww[3]);
          }
        };
        // Columns 32 cc .. 32 cc + 63 (two groups): both loads in flight before one wait.
        auto chunks2 = [&](int cc, uint4 (&ch)[8]) {
          uint32_t o0[32], o1[32];
          tmem_ld32(tQd + cc * 32, o0);
          tmem_ld32(tQd + cc * 32 + 32, o1);
          tmem_wait_ld();
          reg_fence(o0);
          reg_fence(o1);
          auto cvt = [&](const uint32_t (&o)[32], uint4* c) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint32_t wq[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 t = fmul2(make_float2(__uint_as_float(o[q4 * 8 + 2 * e]), __uint_as_float(o[q4 * 8 + 2 * e + 1])), s2);
                wq[e] = pack_bf16(t.x, t.y);
              }
              c[q4] = make_uint4(wq[0], wq[1], wq[2], wq[3]);
            }
          };
          cvt(o0, ch);
          cvt(o1, ch + 4);
        };
        if (X == 0 && GH == 2) {
          uint4 ch[8];
          chunks2(0, ch);
          store_rows_transposed<8>(ch, wdst, D, nvalid);
        } else if (X == 0) {
          uint4 ch[4];
          chunks(0, ch);
          store_rows_transposed<4>(ch, wdst, D, nvalid);
        } else if (G - GH == 2) {
          uint4 ch[8];
          chunks2(GH, ch);
          store_rows_transposed<8>(ch, wdst + GH * 32, D, nvalid);
        } else {
          uint4 ch[4];
          chunks(GH, ch);
          store_rows_transposed<4>(ch, wdst + GH * 32, D, nvalid);
        }
      }
      release(k);
      cur = nx;
    }
    setmaxnreg_dec<168>();
  } else {
    setmaxnreg_dec<104>();
    reg_split_sync(384);
    if (warp == 8) {
      // ------------------------------------------------------------ producer: Q, dO, K, V
      // Per unit: Q_i and dO_i (once the compute threads have copied the
      // previous unit's tiles to tensor memory), then K_j, V_j in the order
      // the MMA warp consumes them.  The K and V slots and phases follow the
      // step count over all units.
      bool ok = true;
      int kq = 0;       // units with steps whose Q and dO were issued
      uint32_t gk = 0;  // K tiles issued over all units (== steps)
      uint32_t gv = 0;  // V tiles issued
      if (lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmdO);
      }
      for (int k = 0; ok; ++k) {
        const int u = next_unit(k, ok);
        if (u < 0) break;
        int bh, i, n;
        unit_of(u, bh, i, n);
        if (n <= 0) continue;
        if (lane == 0) {
          const int b = bh / p.H, h = bh % p.H;
          const int bhk = b * p.Hkv + h / p.G;
          auto load_k = [&](int j) -> bool {
            const uint32_t s = gk % T::KS, rd = gk / T::KS;
            if (rd > 0 && !wait_bounded(wc, bKe + 8u * s, (rd - 1) & 1, wait_site(0xb9, j))) return false;
            // (p.debug_drop_p: a test of the bounded waits skips one K load of unit 0)
            if (!(u == 0 && p.debug_drop_p == j + 1)) {
              mbar_expect_tx(bKf + 8u * s, T::TILE_BYTES);
              for (int cb = 0; cb < T::NB; ++cb)
                tma_load_3d(sK + s * T::TILE_BYTES + cb * T::BLOCK_BYTES, &tmK, bKf + 8u * s, cb * 64, j * 128, bhk);
            }
            ++gk;
            return true;
          };
          auto load_v = [&](int j) -> bool {
            const uint32_t s = gv % T::VS, rd = gv / T::VS;
            if (rd > 0 && !wait_bounded(wc, bVe + 8u * s, (rd - 1) & 1, wait_site(0xba, j))) return false;
            mbar_expect_tx(bVf + 8u * s, T::TILE_BYTES);
            for (int cb = 0; cb < T::NB; ++cb)
              tma_load_3d(sV + s * T::TILE_BYTES + cb * T::BLOCK_BYTES, &tmV, bVf + 8u * s, cb * 64, j * 128, bhk);
            ++gv;
            return true;
          };
          ok = kq == 0 || wait_bounded(wc, bQs, (kq - 1) & 1, wait_site(0xb8, k));
          if (ok) {
            mbar_expect_tx(bQf, T::TILE_BYTES);
            for (int cb = 0; cb < T::NB; ++cb) tma_load_3d(sQ + cb * T::BLOCK_BYTES, &tmQ, bQf, cb * 64, i * 128, bh);
            mbar_expect_tx(bOf, T::TILE_BYTES);
            for (int cb = 0; cb < T::NB; ++cb) tma_load_3d(sdO + cb * T::BLOCK_BYTES, &tmdO, bOf, cb * 64, i * 128, bh);
            ++kq;
          }
          for (int j = 0; j < n && ok; ++j) ok = load_k(j) && load_v(j);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      // Every copy issued above has landed before the CTA may exit (bounded:
      // after an abort, or a load the test hook skipped, some never do).
      if (lane == 0) {
        if (kq > 0) {
          wait_drain(bQf, (kq - 1) & 1, p.limit_ns);
          wait_drain(bOf, (kq - 1) & 1, p.limit_ns);
        }
        for (uint32_t s = 0; s < T::KS && s < gk; ++s) {
          const uint32_t last = ((gk - 1 - s) / T::KS) * T::KS + s;
          wait_drain(bKf + 8u * s, (last / T::KS) & 1, p.limit_ns);
        }
        for (uint32_t s = 0; s < T::VS && s < gv; ++s) {
          const uint32_t last = ((gv - 1 - s) / T::VS) * T::VS + s;
          wait_drain(bVf + 8u * s, (last / T::VS) & 1, p.limit_ns);
        }
      }
      __syncwarp();
    } else if (warp == 9) {
      // ------------------------------------------------------------ MMA issuer
      // Per unit: S_0 and dP_0 once Q_i and dO_i are in tensor memory; then
      // per step j: S_{j+1} once the compute threads have loaded S_j,
      // dQ += dS_j K_j once dS_j is written, dP_{j+1} over dS_j (MMAs from
      // one thread run in order, so dQ_j has read dS_j first).  Slots and
      // per-step barrier phases follow the step count over all units.
      {
        const uint32_t leader = elect_one();
        constexpr uint32_t I_S = idesc_bf16_f32(128, 128, false, false);  // S, dP (A in TMEM, B K-major)
        constexpr uint32_t I_DQ = idesc_bf16_f32(128, D, false, true);    // dQ (A in TMEM, B MN-major)
        const uint32_t tS = tmem, tdP = tmem + 128, tdQ = tmem + 256, tQ = tmem + 384, tO = tmem + 448;
        const uint64_t dKk0 = sdesc_sw128(sK, 16, 1024);                // K slot 0, K-major B (S)
        const uint64_t dKmn0 = sdesc_sw128(sK, T::BLOCK_BYTES, 1024);   // K slot 0, MN-major B (dQ)
        const uint64_t dVk0 = sdesc_sw128(sV, 16, 1024);                // V slot 0, K-major B (dP)
        // D (+)= A[tmem] B[smem] over d: A = Q or dO (bf16 pairs, 8 columns
        // per 16 elements), B = a K-major K or V tile.
        auto mma_td = [&](uint32_t dst, uint32_t a, uint64_t bd) {
#pragma unroll
          for (int kk = 0; kk < T::KSTEPS; ++kk)
            mma_ts_p(leader, dst, a + 8 * kk, sdesc_add(bd, (kk >> 2) * T::BLOCK_BYTES + (kk & 3) * 32), I_S,
                     kk > 0 ? 1u : 0u);
        };
        auto wait_all = [&](uint32_t bar, uint32_t parity, int site) {
          return __all_sync(0xffffffffu, wait_bounded(wc, bar, parity, site));
        };
        // K_g and V_g (step g over all units) loaded.
        auto k_full = [&](uint32_t g, int site) { return wait_all(bKf + 8u * (g % T::KS), (g / T::KS) & 1, site); };
        auto v_full = [&](uint32_t g, int site) { return wait_all(bVf + 8u * (g % T::VS), (g / T::VS) & 1, site); };
        auto k_tile = [&](uint32_t g) { return (g % T::KS) * T::TILE_BYTES; };
        auto v_tile = [&](uint32_t g) { return (g % T::VS) * T::TILE_BYTES; };
        bool ok = true;
        uint32_t gs = 0;  // steps over all units
        int kq = 0;       // units with steps so far
        for (int k = 0; ok; ++k) {
          const int u = next_unit(k, ok);
          if (u < 0) break;
          int bh, i, n;
          unit_of(u, bh, i, n);
          if (n <= 0) continue;
          const uint32_t g0 = gs;
          // S_0 and dP_0.  (As in the loop, the checks for a product run
          // before the commit of the one issued before it.)
          ok = wait_all(bQs, kq & 1, wait_site(0xbb, k)) && k_full(g0, wait_site(0xbc, 0));
          if (!ok) break;
          tc_fence_after();
          mma_td(tS, tQ, sdesc_add(dKk0, k_tile(g0)));  // S_0
          ok = v_full(g0, wait_site(0xbd, 0));
          mma_commit_p(leader, bS);
          if (!ok) break;
          tc_fence_after();
          mma_td(tdP, tO, sdesc_add(dVk0, v_tile(g0)));  // dP_0
          if (n > 1) ok = wait_all(bSr, g0 & 1, wait_site(0xbe, 0)) && k_full(g0 + 1, wait_site(0xbc, 1));  // for S_1
          mma_commit_p(leader, bDp);
          mma_commit_p(leader, bVe + 8u * (g0 % T::VS));  // V_0 consumed
          for (int j = 0; j < n && ok; ++j) {
            const uint32_t g = g0 + j;
            if (j + 1 < n) {
              tc_fence_after();
              mma_td(tS, tQ, sdesc_add(dKk0, k_tile(g + 1)));  // S_{j+1}, over S_j (loaded)
            }
            ok = wait_all(bDs, g & 1, wait_site(0xbf, j));  // for dQ_j
            if (j + 1 < n) mma_commit_p(leader, bS);
            if (!ok) break;
            tc_fence_after();
            // dQ += dS_j K_j: A = dS in TMEM (keys 64X.. of warpgroup X at
            // dP columns 64X.., bf16 pairs), B = K_j (MN-major, N = d)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts_p(leader, tdQ, tdP + 64 * (kk >> 2) + (kk & 3) * 8,
                       sdesc_add(dKmn0, k_tile(g) + kk * 2048), I_DQ, (j > 0 || kk > 0) ? 1u : 0u);
            if (j + 1 < n) ok = v_full(g + 1, wait_site(0xbd, j + 1));  // for dP_{j+1}
            mma_commit_p(leader, bKe + 8u * (g % T::KS));               // K_j consumed
            if (!ok) break;
            if (j + 1 < n) {
              tc_fence_after();
              mma_td(tdP, tO, sdesc_add(dVk0, v_tile(g + 1)));  // dP_{j+1}, over dS_j (read by dQ_j)
              // for S_{j+2}: S_{j+1} loaded, K_{j+2} loaded
              if (j + 2 < n)
                ok = wait_all(bSr, (g + 1) & 1, wait_site(0xbe, j + 1)) && k_full(g + 2, wait_site(0xbc, j + 2));
              mma_commit_p(leader, bDp);
              mma_commit_p(leader, bVe + 8u * ((g + 1) % T::VS));
            }
          }
          if (!ok) break;
          mma_commit_p(leader, bFin);
          gs += n;
          ++kq;
        }
        mma_commit_p(leader, bDrain);  // fires once every MMA issued above has finished
        wait_drain(bDrain, 0, p.limit_ns);
      }
      __syncwarp();
    } else {
      // ------------------------------------------------------------ warps 10-11: queue, row vectors
      // Warp 10 takes the next unit once ring entry k & 1 is free; then both
      // warps write that unit's row vectors into the entry.  Their barrier
      // is reached by both warps in every round, so that a stop is seen by
      // both.
      const int t = (int)threadIdx.x - 320;  // 0..63
      for (int k = 0;; ++k) {
        const int e = k & 1;
        if (warp == 10) {
          const bool ok =
              k < 2 || __all_sync(0xffffffffu, wait_bounded(wc, bUe + 8u * e, ((k - 2) >> 1) & 1, wait_site(0xb6, k)));
          if (lane == 0) {
            if (ok) {
              // CTA b's first unit is unit b (no queue round trip before the first
              // loads); the counter hands out the rest, from gridDim.x on.
              int u = k == 0 ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(p.sched, 1);
              if (u >= p.n_units) u = -1;
              unit_ring[e] = u;
              mbar_arrive(bUf + 8u * e);  // (release: the entry is visible to the roles that wait for it)
            } else {
              *vec_stop = 1;
            }
          }
        }
        named_bar_sync(kVecBarrier, 64);
        const int u = unit_ring[e];
        if (*vec_stop || u < 0) break;
        int bh, i, n;
        unit_of(u, bh, i, n);
        if (t == 0 && n > 0) {
          // Q_i and dO_i into L2 ahead of the producer's loads.
          for (int cb = 0; cb < T::NB; ++cb) {
            tma_prefetch_l2_3d(&tmQ, cb * 64, i * 128, bh);
            tma_prefetch_l2_3d(&tmdO, cb * 64, i * 128, bh);
          }
        }
        float* const ve = vec_s + e * 256;
        for (int rr = t; rr < 128; rr += 64) {
          const int row = 128 * i + rr;
          const size_t vrow = (size_t)bh * p.Npad + row;
          float l2 = -INFINITY, nD = 0.f;  // rows that see no key: P = 0
          if (n > 0 && p.rows_in_dq) {
            // -lse * log2(e) and -D = -rowsum(dO * O), D as the sum of the
            // two column halves' sums, each summed in column order (the
            // order of bwd_dq_kernel, so that the bits agree).
            float l = -INFINITY, part[2] = {0.f, 0.f};
            const size_t orow = (size_t)bh * p.N + row;
            if (row < p.N && ATTN_IN_RANGE(orow * D + D - 1, (size_t)p.B * p.H * p.N * D, p, 0x20a)) {
              l = p.lse[orow];
              const uint4* po = reinterpret_cast<const uint4*>(p.o + orow * D);
              const uint4* pg = reinterpret_cast<const uint4*>(p.dout + orow * D);
#pragma unroll
              for (int X = 0; X < 2; ++X) {
                uint4 a[D / 16], g[D / 16];
#pragma unroll
                for (int c = 0; c < D / 16; ++c) {
                  a[c] = __ldg(po + X * (D / 16) + c);
                  g[c] = __ldg(pg + X * (D / 16) + c);
                }
                float s = 0.f;
#pragma unroll
                for (int c = 0; c < D / 16; ++c) {
                  const uint32_t aw[4] = {a[c].x, a[c].y, a[c].z, a[c].w}, gw[4] = {g[c].x, g[c].y, g[c].z, g[c].w};
#pragma unroll
                  for (int q = 0; q < 4; ++q) {
                    const float2 af = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[q]));
                    const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[q]));
                    s = fmaf(af.x, gf.x, s);
                    s = fmaf(af.y, gf.y, s);
                  }
                }
                part[X] = s;
              }
            }
            nD = row < p.N ? -(part[0] + part[1]) : 0.f;
            l2 = (l == -INFINITY) ? -INFINITY : -l * 1.4426950408889634f;
          } else if (n > 0 && ATTN_IN_RANGE(vrow, vec_floats(p), p, 0x20b)) {
            // formed by an earlier stage
            l2 = p.lse2[vrow];
            nD = p.dvec[vrow];
          }
          ve[rr] = l2;
          ve[128 + rr] = nD;
          if (p.rows_in_dq && ATTN_IN_RANGE(vrow, vec_floats(p), p, 0x20c)) {
            p.dvec[vrow] = nD;
            p.lse2[vrow] = l2;
          }
        }
        mbar_arrive(bUv + 8u * e);  // (release: the vectors are visible to the compute threads)
      }
    }
    setmaxnreg_inc<168>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // The last CTA to finish resets the queue for the next launch that uses
  // this slot (every CTA's vector warps have stopped taking units by now).
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.sched + 1, 1) == (int)gridDim.x - 1) {
      atomicExch(p.sched, 0);
      atomicExch(p.sched + 1, 0);
    }
  }
}

namespace {

// Queue slots (next unit, CTAs done), one per launch in flight (see
// attn_fwd_persist.cu).
constexpr int kDqQueueSlots = 256;
__device__ int g_dq_queue[kDqQueueSlots][2];

int* dq_queue_slot() {
  static std::atomic<unsigned> next{0};
  static int* base[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (base[dev] == nullptr) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_dq_queue) != cudaSuccess) return nullptr;
    base[dev] = static_cast<int*>(a);
  }
  return base[dev] + 2 * (next.fetch_add(1) % kDqQueueSlots);
}

template <int D, bool C>
cudaError_t launch_dq_persist_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& tdo, const BwdParams& p, cudaStream_t stream) {
  using T = PQTraits<D>;
  auto kern = bwd_dq_persist_kernel<D, C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidValue;
  BwdParams pc = p;
  pc.n_units = p.nq * p.B * p.H;
  pc.tail = uniform_levels(C, p.vl, p.mk, false) ? 1 : order_tail(p.nq, p.B * p.H, p.G);
  pc.sched = dq_queue_slot();
  if (pc.sched == nullptr) return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)min(pc.n_units, sms);  // one CTA per SM
  kern<<<grid, T::THREADS, T::SMEM, stream>>>(tq, tk, tv, tdo, pc);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq_persist(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                  const CUtensorMap& tv, const CUtensorMap& tdo, const BwdParams& p,
                                  cudaStream_t stream) {
  switch (d) {
    case 64: return causal ? launch_dq_persist_t<64, true>(tq, tk, tv, tdo, p, stream) : launch_dq_persist_t<64, false>(tq, tk, tv, tdo, p, stream);
    case 96: return causal ? launch_dq_persist_t<96, true>(tq, tk, tv, tdo, p, stream) : launch_dq_persist_t<96, false>(tq, tk, tv, tdo, p, stream);
    case 128:
      return causal ? launch_dq_persist_t<128, true>(tq, tk, tv, tdo, p, stream) : launch_dq_persist_t<128, false>(tq, tk, tv, tdo, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sdpa
