// attn_bwd_persist.cu — the dK/dV kernel of the dense backward (no mask, no
// packed batch) as a persistent kernel on sm_103a.
//
// Method and arithmetic: those of attn_bwd.cu's bwd_main_kernel (page
// "Flash Attention原理", §五 and FAQ Q19: P^T recomputed from lse, dV = P^T dO,
// dP^T = V dO^T, dS^T = P^T (dP^T - D), dK = scale dS^T Q), unchanged, so the
// two kernels give the same bits.  What differs is the schedule: one CTA per
// SM takes the (K/V head, key tile) units of bwd_main_kernel, in the same
// order (work_unit), from a queue until none is left, instead of one CTA per
// unit paying its launch, barrier and tensor-memory setup, the wait for its
// first tiles and an epilogue while the tensor core idles (about 5 us of a
// 25 us unit at C5).
//
// GB300 mapping: bwd_main_kernel's roles (warps 0-7 compute, warp 8 the K, V
// and Q producer, which also takes the units from the queue, warp 9 the MMA
// issuer, warp 10 the dO producer), with these differences:
//   * a unit ring of two entries in shared memory carries the unit index to
//     the other roles;
//   * the Q and dO rings, and every per-step barrier, run on across units;
//   * K and V have an empty barrier, committed once the unit's last S^T and
//     dP^T products are issued (its last step needs only dV and dK, which
//     read neither), so the next unit's K and V load during that step;
//   * dK and dV leave from registers to global memory, each warp's rows
//     transposed through a 4 KB shared-memory scratch of its own so that a
//     store covers whole lines;
//   * a unit whose keys no query sees (causal cross attention) writes zeros
//     and takes no loads or products.
#include <atomic>
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {

namespace {

template <int D>
struct PBTraits {
  static constexpr int NB = (D + 63) / 64;
  static constexpr int BLOCK_BYTES = 128 * 128;
  static constexpr int TILE_BYTES = NB * BLOCK_BYTES;  // one [128 rows x d] bf16 tile
  static constexpr int KSTEPS = D / 16;
  static constexpr int VEC_BYTES = 1024;               // -lse2[128] + -D[128]
  // kv_full kv_empty q_full[2] q_empty[2] do_full[2] do_empty[2] s p dp ds fin
  // unit_full[2] unit_empty[2] drain
  static constexpr int NBAR = 2 + 8 + 5 + 4 + 1;
  static constexpr int TILES_BYTES = 6 * TILE_BYTES;  // K, V, Q[2], dO[2]
  static constexpr int MISC = 32;                      // tmem slot, abort flag, unit ring
  static constexpr int SCRATCH_BYTES = 8 * 4096;      // a 4 KB epilogue scratch per compute warp
  static constexpr int SMEM = TILES_BYTES + SCRATCH_BYTES + 2 * VEC_BYTES + NBAR * 8 + MISC;
  static constexpr int THREADS = 384;
};

static_assert(PBTraits<128>::SMEM <= 227 * 1024, "shared memory");

// Arrivals on unit_empty: every thread that reads a ring entry (the compute
// warpgroups, the MMA warp and the dO producer warp).
constexpr int kBwdUnitReaders = 256 + 32 + 32;

}  // namespace

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    bwd_persist_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const BwdParams p) {
  using T = PBTraits<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = smem_u32(smem_raw);
  if (base & 1023u) {  // the layout needs a 1024-byte aligned start (128-byte swizzle atoms)
    if (threadIdx.x == 0) atomicCAS(p.status, 0, kDevMisaligned);
    return;
  }
  const uint32_t sK = base;
  const uint32_t sV = sK + T::TILE_BYTES;
  const uint32_t sQ = sV + T::TILE_BYTES;            // [2]
  const uint32_t sdO = sQ + 2 * T::TILE_BYTES;       // [2]
  const uint32_t sScr = sdO + 2 * T::TILE_BYTES;     // [8] epilogue scratch, one per compute warp
  const uint32_t sVec = sScr + T::SCRATCH_BYTES;     // [2] x {-lse2[128], -D[128]}
  const uint32_t sBar = sVec + 2 * T::VEC_BYTES;
  const uint32_t bKV = sBar;          // K, V of the unit loaded
  const uint32_t bKVe = bKV + 8;      // K, V no longer read
  const uint32_t bQf = bKVe + 8;      // [2] Q_i + vectors loaded
  const uint32_t bQe = bQf + 16;      // [2] Q stage free (after dK_i)
  const uint32_t bDf = bQe + 16;      // [2] dO_i loaded
  const uint32_t bDe = bDf + 16;      // [2] dO stage free (after dV_i)
  const uint32_t bS = bDe + 16;       // S^T ready
  const uint32_t bP = bS + 8;         // P^T in TMEM (256 arrivals)
  const uint32_t bDp = bP + 8;        // dP^T ready
  const uint32_t bDs = bDp + 8;       // dS^T in TMEM (256 arrivals)
  const uint32_t bFin = bDs + 8;      // every MMA of the unit done
  const uint32_t bUf = bFin + 8;      // [2] unit ring entry written
  const uint32_t bUe = bUf + 16;      // [2] unit ring entry read
  const uint32_t bDrain = bUe + 16;
  uint8_t* const misc = smem_raw + (sBar - base) + 8 * T::NBAR;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  volatile int* const unit_ring = reinterpret_cast<volatile int*>(misc + 8);  // [2]
  const float* const vec_g = reinterpret_cast<const float*>(smem_raw + (sVec - base));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = (p.N + 127) / 128;  // query tiles per head
  // A unit's K/V head and key tile, its first query tile and its steps
  // (head in group x query tile; 0 when no query sees its keys).
  struct Unit {
    int bhk, j, i0, ni, total;
  };
  auto unit_of = [&](int u) {
    Unit x;
    work_unit(u, p.nkv, p.B * p.Hkv, p.tail, x.bhk, x.j);
    // Causal: the first query tile with a row at position >= 128 j (query
    // row i at position koff + i).
    x.i0 = CAUSAL ? max(0, (x.j * 128 - p.koff) / 128) : 0;
    x.ni = nq - x.i0;
    x.total = x.ni > 0 ? p.G * x.ni : 0;
    return x;
  };

  if (threadIdx.x == 0) {
    mbar_init(bKV, 1);
    mbar_init(bKVe, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bQf + 8u * s, 1);
      mbar_init(bQe + 8u * s, 1);
      mbar_init(bDf + 8u * s, 1);
      mbar_init(bDe + 8u * s, 1);
      mbar_init(bUf + 8u * s, 1);
      mbar_init(bUe + 8u * s, kBwdUnitReaders);
    }
    mbar_init(bS, 1);
    mbar_init(bP, 256);
    mbar_init(bDp, 1);
    mbar_init(bDs, 256);
    mbar_init(bFin, 1);
    mbar_init(bDrain, 1);
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
  // The k-th unit this CTA takes, as read from the ring by a consumer role
  // (-1: none left, or the producer stopped); every reader arrives on the
  // entry's empty barrier after reading.
  auto next_unit = [&](int k, bool& ok) -> int {
    const int e = k & 1;
    ok = __all_sync(0xffffffffu, wait_bounded(wc, bUf + 8u * e, (k >> 1) & 1, wait_site(0x1a, k)));
    const int u = ok ? unit_ring[e] : -1;
    mbar_arrive(bUe + 8u * e);
    return u;
  };

  if (warp < 8) {
    setmaxnreg_inc<200>();
    reg_split_sync(384);
    // ------------------------------------------------------------ compute
    // Warpgroup X takes query columns [64X, 64X + 64) of every score tile for
    // all 128 key rows (thread = key row = TMEM lane); the body is
    // bwd_main_kernel's for the dense batch.
    const int X = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + 64 * X + lane_off;           // S^T columns of this half
    const uint32_t tP = tmem + 64 * X + lane_off;           // P^T (bf16 pairs), first 32 of them
    const uint32_t tdP = tmem + 128 + 64 * X + lane_off;    // dP^T columns of this half; dS^T pairs after
    const float c = p.scale_log2;
    const float2 c2 = make_float2(c, c);
    uint32_t gs = 0;  // steps over all units so far
    int kf = 0;       // units with steps so far
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int u = next_unit(k, ok);
      if (u < 0) break;
      const Unit x = unit_of(u);
      const int kr = 128 * x.j + r;  // this thread's key row
      // dV (warpgroup 0) or dK (warpgroup 1) row kr of K/V head bhk.
      uint16_t* const drow = (X ? p.dk : p.dv) + ((size_t)x.bhk * p.Nk + kr) * D;
      const bool row_ok = kr < p.Nk && ATTN_IN_RANGE(((size_t)x.bhk * p.Nk + kr) * D + D - 1,
                                                     (size_t)p.B * p.Hkv * p.Nk * D, p, 0x306);
      if (x.total == 0) {
        // No query sees these keys: dK = dV = 0.
        if (row_ok)
          for (int c8 = 0; c8 < D / 8; ++c8) *reinterpret_cast<uint4*>(drow + 8 * c8) = make_uint4(0, 0, 0, 0);
        continue;
      }
      // Query column q of tile i cannot see key row kr when q < qmin0 - 128 i:
      // every column for key rows past Nk, and for causal rows the queries at
      // positions koff + 128 i + 64 X + q below the key.
      const int qmin0 = (kr >= p.Nk) ? (1 << 30) : CAUSAL ? kr - p.koff - 64 * X : -(1 << 30);
      for (int it = 0; it < x.total; ++it, ++gs) {
        const int i = x.i0 + it % x.ni;
        const float* vl = vec_g + (gs & 1) * (T::VEC_BYTES / 4) + 64 * X;  // -lse2 of this half; -D at +128
        // The vectors come from the bulk copy of this step: observe its
        // barrier before reading them, and read this half's -lse2 while S^T
        // is still being computed.
        ok = __all_sync(0xffffffffu, wait_bounded(wc, bQf + 8u * (gs & 1), (gs >> 1) & 1, wait_site(0x11, it)));
        if (!ok) break;
        float4 lv[16];
#pragma unroll
        for (int q4 = 0; q4 < 16; ++q4) lv[q4] = *reinterpret_cast<const float4*>(vl + 4 * q4);
        ok = __all_sync(0xffffffffu, wait_bounded(wc, bS, gs & 1, wait_site(0x12, it)));
        if (!ok) break;
        tc_fence_after();
        float xs[64];
        {
          uint32_t ra[32], rb[32];
          tmem_ld32(tS + 0, ra);
          tmem_ld32(tS + 32, rb);
          tmem_wait_ld();
          reg_fence(ra);
          reg_fence(rb);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            xs[e] = __uint_as_float(ra[e]);
            xs[32 + e] = __uint_as_float(rb[e]);
          }
        }
        // P^T[r][q] = exp2(S^T * scale * log2e - lse2[q]); masked entries and
        // padding key rows are exactly 0.
#pragma unroll
        for (int q4 = 0; q4 < 16; ++q4) {
          const float4 l4 = lv[q4];
          const float2 t0 = ffma2(make_float2(xs[4 * q4 + 0], xs[4 * q4 + 1]), c2, make_float2(l4.x, l4.y));
          const float2 t1 = ffma2(make_float2(xs[4 * q4 + 2], xs[4 * q4 + 3]), c2, make_float2(l4.z, l4.w));
          xs[4 * q4 + 0] = ex2(t0.x);
          xs[4 * q4 + 1] = ex2(t0.y);
          xs[4 * q4 + 2] = ex2(t1.x);
          xs[4 * q4 + 3] = ex2(t1.y);
        }
        {
          const int qmin = qmin0 - 128 * i;
          if (__any_sync(0xffffffffu, qmin > 0)) {
#pragma unroll
            for (int q = 0; q < 64; ++q)
              if (q < qmin) xs[q] = 0.f;
          }
        }
        uint32_t pk[32];  // P^T as bf16 pairs: to TMEM for the dV MMA, kept for dS
#pragma unroll
        for (int e = 0; e < 32; ++e) pk[e] = pack_bf16(xs[2 * e], xs[2 * e + 1]);
        tmem_st32(tP, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bP);
        // dS^T[r][q] = P^T[r][q] * (dP^T[r][q] - D[q]) -> bf16 pairs over the
        // first 32 of this half's dP^T columns.
        ok = __all_sync(0xffffffffu, wait_bounded(wc, bDp, gs & 1, wait_site(0x14, it)));
        if (!ok) break;
        tc_fence_after();
        uint32_t g0[32], g1[32];
        tmem_ld32(tdP + 0, g0);
        tmem_ld32(tdP + 32, g1);
        tmem_wait_ld();
        reg_fence(g0);
        reg_fence(g1);
        const float4* Dv = reinterpret_cast<const float4*>(vl + 128);
        uint32_t w[32];
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
          const float4 da = Dv[2 * q8], db = Dv[2 * q8 + 1];
          const float2 dd[4] = {make_float2(da.x, da.y), make_float2(da.z, da.w), make_float2(db.x, db.y),
                                make_float2(db.z, db.w)};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int q = q8 * 8 + 2 * e;  // column within the half
            const uint32_t gx = (q < 32) ? g0[q] : g1[q - 32];
            const uint32_t gy = (q < 32) ? g0[q + 1] : g1[q - 31];
            const uint32_t pp = pk[q >> 1];
            const float2 pf = make_float2(__uint_as_float(pp << 16), __uint_as_float(pp & 0xffff0000u));
            const float2 ds = fmul2(pf, fadd2(make_float2(__uint_as_float(gx), __uint_as_float(gy)), dd[e]));
            w[q >> 1] = pack_bf16(ds.x, ds.y);
          }
        }
        tmem_st32(tdP, w);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bDs);
      }
      if (!ok) break;
      // ---------------------------------------------------------- dK / dV out
      // Warpgroup 0 writes dV, warpgroup 1 dK = scale * (dS^T Q), each row
      // from registers.  The next unit's first dV / dK product, which
      // overwrites these accumulators, waits for this warpgroup's next P^T /
      // dS^T, published after these loads.
      ok = __all_sync(0xffffffffu, wait_bounded(wc, bFin, kf & 1, wait_site(0x13, k)));
      if (!ok) break;
      ++kf;
      tc_fence_after();
      const uint32_t src = tmem + (X ? 256u : 384u) + lane_off;
      const float2 f2 = X ? make_float2(p.scale, p.scale) : make_float2(1.f, 1.f);
      // The warp's 32 key rows 128 j + 32 (warp % 4) + lane, written a row
      // slice per group of lanes through the warp's shared-memory scratch
      // (store_rows_staged): whole 128-byte lines per store rather than 32
      // separate 16-byte pieces.
      const int wr0 = 128 * x.j + 32 * (warp & 3);
      uint16_t* const wdst = (X ? p.dk : p.dv) + ((size_t)x.bhk * p.Nk + wr0) * D;
      const uint32_t scr = sScr + (uint32_t)warp * 4096u;  // this warp's scratch
      int nvalid = min(32, p.Nk - wr0);
      if (nvalid > 0 && !ATTN_IN_RANGE(((size_t)x.bhk * p.Nk + wr0 + nvalid) * D - 1, (size_t)p.B * p.Hkv * p.Nk * D, p, 0x306))
        nvalid = 0;
      // Columns 32 cc .. 32 cc + 31 of this thread's row as four bf16 chunks.
      auto chunks = [&](int cc, uint4* ch) {
        uint32_t o[32];
        tmem_ld32(src + cc * 32, o);
        tmem_wait_ld();
        reg_fence(o);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t wq[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 t = fmul2(make_float2(__uint_as_float(o[q4 * 8 + 2 * e]),
                                               __uint_as_float(o[q4 * 8 + 2 * e + 1])), f2);
            wq[e] = pack_bf16(t.x, t.y);
          }
          ch[q4] = make_uint4(wq[0], wq[1], wq[2], wq[3]);
        }
      };
      // Columns 32 cc .. 32 cc + 63 (two groups): both loads in flight before one wait.
      auto chunks2 = [&](int cc, uint4 (&ch)[8]) {
        uint32_t o0[32], o1[32];
        tmem_ld32(src + cc * 32, o0);
        tmem_ld32(src + cc * 32 + 32, o1);
        tmem_wait_ld();
        reg_fence(o0);
        reg_fence(o1);
        auto cvt = [&](const uint32_t (&o)[32], uint4* c) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t wq[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 t = fmul2(make_float2(__uint_as_float(o[q4 * 8 + 2 * e]), __uint_as_float(o[q4 * 8 + 2 * e + 1])), f2);
              wq[e] = pack_bf16(t.x, t.y);
            }
            c[q4] = make_uint4(wq[0], wq[1], wq[2], wq[3]);
          }
        };
        cvt(o0, ch);
        cvt(o1, ch + 4);
      };
#pragma unroll
      for (int cc = 0; cc + 1 < D / 32; cc += 2) {
        uint4 ch[8];
        chunks2(cc, ch);
        store_rows_staged<8>(ch, scr, wdst + cc * 32, D, nvalid);
      }
      if constexpr ((D / 32) % 2 != 0) {
        uint4 ch[4];
        chunks(D / 32 - 1, ch);
        store_rows_staged<4>(ch, scr, wdst + (D / 32 - 1) * 32, D, nvalid);
      }
    }
    setmaxnreg_dec<168>();
  } else {
    setmaxnreg_dec<104>();
    reg_split_sync(384);
    if (warp == 8) {
      // ------------------------------------------------------------ unit queue; producer: K, V, Q
      if (lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        bool ok = true;
        uint32_t gq = 0;  // steps over all units whose Q was issued: stage gq & 1
        int kkv = 0;      // units with steps whose K, V were issued
        for (int k = 0; ok; ++k) {
          const int e = k & 1;
          // CTA b's first unit is unit b (no queue round trip before the first
          // loads); the counter hands out the rest, from gridDim.x on.
          int u = k == 0 ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(p.sched, 1);
          if (u >= p.n_units) u = -1;
          if (k >= 2 && !(ok = wait_bounded(wc, bUe + 8u * e, ((k - 2) >> 1) & 1, wait_site(0x34, k)))) break;
          unit_ring[e] = u;
          mbar_arrive(bUf + 8u * e);  // (release: the entry is visible to the roles that wait for it)
          if (u < 0) break;
          const Unit x = unit_of(u);
          if (x.total == 0) continue;
          const int b = x.bhk / p.Hkv, hk = x.bhk % p.Hkv;
          // K, V once the previous unit's last S^T and dP^T have read them.
          if (kkv > 0 && !(ok = wait_bounded(wc, bKVe, (kkv - 1) & 1, wait_site(0x35, k)))) break;
          mbar_expect_tx(bKV, 2 * T::TILE_BYTES);
          for (int cb = 0; cb < T::NB; ++cb) {
            tma_load_3d(sK + cb * T::BLOCK_BYTES, &tmK, bKV, cb * 64, x.j * 128, x.bhk);
            tma_load_3d(sV + cb * T::BLOCK_BYTES, &tmV, bKV, cb * 64, x.j * 128, x.bhk);
          }
          ++kkv;
          for (int it = 0; it < x.total; ++it) {
            const int st = gq & 1, rd = gq >> 1;
            const int g = it / x.ni, i = x.i0 + it % x.ni;
            const int bh = b * p.H + hk * p.G + g;
            if (rd > 0 && !(ok = wait_bounded(wc, bQe + 8u * st, (rd - 1) & 1, wait_site(0x31, it)))) break;
            if (u == 0 && p.debug_drop_p == it + 1) {  // test of the bounded waits only
              ++gq;
              continue;
            }
            const uint32_t barq = bQf + 8u * st;
            mbar_expect_tx(barq, T::TILE_BYTES + T::VEC_BYTES);
            for (int cb = 0; cb < T::NB; ++cb)
              tma_load_3d(sQ + st * T::TILE_BYTES + cb * T::BLOCK_BYTES, &tmQ, barq, cb * 64, i * 128, bh);
            size_t voff = (size_t)bh * p.Npad + (size_t)i * 128;
            // (a failed check reads in-range vectors instead, so that the step's barrier still completes)
            if (!ATTN_IN_RANGE(voff + 127, vec_floats(p), p, 0x307)) voff = 0;
            bulk_load(sVec + st * T::VEC_BYTES, p.lse2 + voff, 512, barq);
            bulk_load(sVec + st * T::VEC_BYTES + 512, p.dvec + voff, 512, barq);
            ++gq;
          }
        }
        // Every copy issued above has landed before the CTA may exit.
        if (kkv > 0) wait_drain(bKV, (kkv - 1) & 1, p.limit_ns);
        for (uint32_t st = 0; st < 2 && st < gq; ++st)
          wait_drain(bQf + 8u * st, ((((gq - 1 - st) / 2) * 2 + st) >> 1) & 1, p.limit_ns);
      }
      __syncwarp();
    } else if (warp == 10) {
      // ------------------------------------------------------------ producer: dO
      bool ok = true;
      uint32_t gd = 0;  // steps over all units whose dO was issued
      for (int k = 0; ok; ++k) {
        const int u = next_unit(k, ok);
        if (u < 0) break;
        const Unit x = unit_of(u);
        if (lane == 0) {
          const int b = x.bhk / p.Hkv, hk = x.bhk % p.Hkv;
          for (int it = 0; it < x.total; ++it) {
            const int st = gd & 1, rd = gd >> 1;
            const int g = it / x.ni, i = x.i0 + it % x.ni;
            const int bh = b * p.H + hk * p.G + g;
            if (rd > 0 && !(ok = wait_bounded(wc, bDe + 8u * st, (rd - 1) & 1, wait_site(0x32, it)))) break;
            const uint32_t bard = bDf + 8u * st;
            mbar_expect_tx(bard, T::TILE_BYTES);
            for (int cb = 0; cb < T::NB; ++cb)
              tma_load_3d(sdO + st * T::TILE_BYTES + cb * T::BLOCK_BYTES, &tmdO, bard, cb * 64, i * 128, bh);
            ++gd;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (lane == 0)
        for (uint32_t st = 0; st < 2 && st < gd; ++st)
          wait_drain(bDf + 8u * st, ((((gd - 1 - st) / 2) * 2 + st) >> 1) & 1, p.limit_ns);
      __syncwarp();
    } else if (warp == 9) {
      // ------------------------------------------------------------ MMA issuer
      // bwd_main_kernel's schedule for each unit in turn; per step i: dV(i),
      // S^T(i+1), dK(i), dP^T(i+1) (MMAs from one thread run in order, so
      // S^T(i+1) overwrites P^T(i) only after dV(i), and dP^T(i+1) dS^T(i)
      // only after dK(i)).  Stages and per-step barrier phases follow the
      // step count over all units.
      {
        const uint32_t leader = elect_one();
        constexpr uint32_t I_SS = idesc_bf16_f32(128, 128, false, false);   // S^T, dP^T (K-major x K-major)
        constexpr uint32_t I_TB = idesc_bf16_f32(128, D, false, true);      // dV, dK (A in TMEM, B MN-major)
        const uint32_t tS = tmem, tdP = tmem + 128, tdK = tmem + 256, tdV = tmem + 384;
        const uint64_t dKk = sdesc_sw128(sK, 16, 1024);                  // K as K-major A (S^T)
        const uint64_t dVk = sdesc_sw128(sV, 16, 1024);                  // V as K-major A (dP^T)
        const uint64_t dQk0 = sdesc_sw128(sQ, 16, 1024);                 // Q stage 0, K-major B (S^T)
        const uint64_t dQmn0 = sdesc_sw128(sQ, T::BLOCK_BYTES, 1024);    // Q stage 0, MN-major B (dK)
        const uint64_t dOk0 = sdesc_sw128(sdO, 16, 1024);                // dO stage 0, K-major B (dP^T)
        const uint64_t dOmn0 = sdesc_sw128(sdO, T::BLOCK_BYTES, 1024);   // dO stage 0, MN-major B (dV)
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
        bool ok = true;
        uint32_t gs = 0;  // steps over all units
        int kf = 0;       // units with steps so far
        for (int k = 0; ok; ++k) {
          const int u = next_unit(k, ok);
          if (u < 0) break;
          const Unit x = unit_of(u);
          if (x.total == 0) continue;
          const uint32_t st0 = gs & 1;
          if (!(ok = wait_all(bKV, kf & 1, wait_site(0x41, k)) && wait_all(bQf + 8u * st0, (gs >> 1) & 1, wait_site(0x42, k)) &&
                     wait_all(bDf + 8u * st0, (gs >> 1) & 1, wait_site(0x48, k))))
            break;
          tc_fence_after();
          mma_kk(tS, dKk, sdesc_add(dQk0, st0 * T::TILE_BYTES), I_SS);  // S^T of the unit's first step
          mma_commit_p(leader, bS);
          mma_kk(tdP, dVk, sdesc_add(dOk0, st0 * T::TILE_BYTES), I_SS);  // dP^T of its first step
          mma_commit_p(leader, bDp);
          if (x.total == 1) mma_commit_p(leader, bKVe);  // K, V read for the last time
          for (int it = 0; it < x.total && ok; ++it, ++gs) {
            const int st = gs & 1, sn = st ^ 1;
            const bool nx = it + 1 < x.total;
            const uint32_t so = st * T::TILE_BYTES, sno = sn * T::TILE_BYTES;
            if (!(ok = wait_all(bP, gs & 1, wait_site(0x44, it)))) break;
            tc_fence_after();
            // dV += P^T dO_i: A = P^T in TMEM, B = dO_i (MN-major)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts_p(leader, tdV, tS + 64 * (kk >> 2) + 8 * (kk & 3), sdesc_add(dOmn0, so + kk * 2048), I_TB,
                       (it > 0 || kk > 0) ? 1u : 0u);
            mma_commit_p(leader, bDe + 8u * st);  // dO_i no longer needed
            if (nx) {
              if (!(ok = wait_all(bQf + 8u * sn, ((gs + 1) >> 1) & 1, wait_site(0x46, it)))) break;
              tc_fence_after();
              mma_kk(tS, dKk, sdesc_add(dQk0, sno), I_SS);  // S^T_{i+1}
              mma_commit_p(leader, bS);
            }
            if (!(ok = wait_all(bDs, gs & 1, wait_site(0x45, it)))) break;
            tc_fence_after();
            // dK += dS^T Q_i: A = dS^T in TMEM, B = Q_i (MN-major)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts_p(leader, tdK, tdP + 64 * (kk >> 2) + 8 * (kk & 3), sdesc_add(dQmn0, so + kk * 2048), I_TB,
                       (it > 0 || kk > 0) ? 1u : 0u);
            mma_commit_p(leader, bQe + 8u * st);  // Q_i (and its vectors) no longer needed
            if (nx) {
              if (!(ok = wait_all(bDf + 8u * sn, ((gs + 1) >> 1) & 1, wait_site(0x47, it)))) break;
              tc_fence_after();
              mma_kk(tdP, dVk, sdesc_add(dOk0, sno), I_SS);  // dP^T_{i+1}
              mma_commit_p(leader, bDp);
              if (it + 2 == x.total) mma_commit_p(leader, bKVe);  // K, V read for the last time
            }
          }
          if (!ok) break;
          mma_commit_p(leader, bFin);
          ++kf;
        }
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
  // The last CTA to finish resets the queue for the next launch that uses
  // this slot (every CTA's producer has stopped taking units by now).
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
constexpr int kBwdQueueSlots = 256;
__device__ int g_bwd_queue[kBwdQueueSlots][2];

int* bwd_queue_slot() {
  static std::atomic<unsigned> next{0};
  static int* base[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (base[dev] == nullptr) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_bwd_queue) != cudaSuccess) return nullptr;
    base[dev] = static_cast<int*>(a);
  }
  return base[dev] + 2 * (next.fetch_add(1) % kBwdQueueSlots);
}

template <int D, bool C>
cudaError_t launch_bwd_persist_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const CUtensorMap& tdo, const BwdParams& p, cudaStream_t stream) {
  using T = PBTraits<D>;
  auto kern = bwd_persist_kernel<D, C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidValue;
  BwdParams pc = p;
  pc.n_units = p.nkv * p.B * p.Hkv;
  pc.tail = uniform_levels(C, p.vl, p.mk, false) ? 1 : order_tail(p.nkv, p.B * p.Hkv, 1);
  pc.sched = bwd_queue_slot();
  if (pc.sched == nullptr) return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)min(pc.n_units, sms);  // one CTA per SM
  kern<<<grid, T::THREADS, T::SMEM, stream>>>(tq, tk, tv, tdo, pc);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_grad_persist(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                    const CUtensorMap& tv, const CUtensorMap& tdo, const BwdParams& p,
                                    cudaStream_t stream) {
  switch (d) {
    case 64: return causal ? launch_bwd_persist_t<64, true>(tq, tk, tv, tdo, p, stream) : launch_bwd_persist_t<64, false>(tq, tk, tv, tdo, p, stream);
    case 96: return causal ? launch_bwd_persist_t<96, true>(tq, tk, tv, tdo, p, stream) : launch_bwd_persist_t<96, false>(tq, tk, tv, tdo, p, stream);
    case 128:
      return causal ? launch_bwd_persist_t<128, true>(tq, tk, tv, tdo, p, stream) : launch_bwd_persist_t<128, false>(tq, tk, tv, tdo, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sdpa
