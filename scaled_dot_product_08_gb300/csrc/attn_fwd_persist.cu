// attn_fwd_persist.cu — the dense forward of exact attention (no mask, no
// packed batch) as a persistent kernel on sm_103a.
//
// Method and arithmetic: those of attn_fwd.cu (page "Flash Attention原理", §三
// tiling, §四 online softmax with a lazily raised max, §五 only O and the
// row logsumexp leave the chip), unchanged, so the two kernels give the same
// bits.  What differs is the schedule: one CTA per SM takes work units —
// the (head, pair of 128-row query tiles) units of attn_fwd.cu, in the same
// order (work_unit) — from a queue until none is left.  A launch-per-unit
// kernel pays, per unit, the CTA launch, barrier and tensor-memory setup,
// the wait for its first Q and K tiles, and an epilogue during which the
// tensor core idles: about 5 us, a fifth to a third of a unit at N = 2048 to
// 4096.  Here the producer runs ahead into the next unit (its Q tiles load
// once the last Q K^T of the current unit is issued, its K/V through the
// same ring), so the next unit's first Q K^T overlaps the current epilogue.
//
// GB300 mapping: the roles of attn_fwd.cu (warps 0-7 softmax, one
// warpgroup per query tile; warp 8 TMA producer, which also takes the units
// from the queue; warp 9 MMA issuer), with these differences:
//   * a unit ring of two entries in shared memory (unit_full / unit_empty
//     barriers) carries the unit index from warp 8 to the other roles;
//   * every barrier's phase runs on across units, and the Q tiles have an
//     empty barrier, committed after each tile's last Q K^T;
//   * O leaves from registers to global memory (rows past Nq are not
//     written), so the Q tiles are never used as a staging buffer; each
//     warp's rows go through a 4 KB shared-memory scratch of its own, whole
//     128-byte lines per store (not at d = 64 with a causal mask, where the
//     rows go straight out), and the scratch takes one stage of the K/V ring
//     at d = 128 and 96;
//   * the queue is a per-launch counter pair in global memory (next unit,
//     CTAs done); the last CTA to finish resets it for the next launch.
#include <atomic>
#include <cmath>
#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {

namespace {

template <int D>
struct PTraits {
  static constexpr int NB = (D + 63) / 64;           // 64-column (128-byte) blocks per row
  static constexpr int BLOCK_BYTES = 128 * 128;      // [128 rows x 128 B]
  static constexpr int TILE_BYTES = NB * BLOCK_BYTES;
  static constexpr int NSTAGE = (D == 64) ? 8 : 4;   // K/V ring depth
  static constexpr int KSTEPS = D / 16;              // K=16 steps of Q K^T
  // q_full[2] q_empty[2] kv_full[NSTAGE] kv_empty[NSTAGE] s_full[2] p_full[2][2]
  // o_full[2] unit_full[2] unit_empty[2] drain
  static constexpr int NBAR = 2 + 2 + 2 * NSTAGE + 2 + 4 + 2 + 2 + 2 + 1;
  static constexpr int MISC = 32;                    // tmem slot, abort flag, unit ring
  static constexpr int SCRATCH_BYTES = 8 * 4096;  // a 4 KB O-epilogue scratch per softmax warp
  static constexpr int SMEM = 1024 + (2 + NSTAGE) * TILE_BYTES + SCRATCH_BYTES + NBAR * 8 + MISC;
  static constexpr int THREADS = 384;
};

static_assert(PTraits<128>::SMEM <= 227 * 1024 && PTraits<96>::SMEM <= 227 * 1024, "shared memory");

// Arrivals on unit_empty: every thread that reads a ring entry (the MMA
// warp and both softmax warpgroups).
constexpr int kUnitReaders = 32 + 256;

}  // namespace

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    fwd_persist_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using T = PTraits<D>;
  constexpr bool STAGED_O = !(D == 64 && CAUSAL);  // O rows through the per-warp scratch
  static_assert(!STAGED_O || T::SCRATCH_BYTES == 8 * 4096, "O-epilogue scratch");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);

  const uint32_t sQ = base;                          // 2 query tiles
  const uint32_t sKV = base + 2 * T::TILE_BYTES;     // K/V ring
  const uint32_t sScr = sKV + T::NSTAGE * T::TILE_BYTES;  // [8] O-epilogue scratch, one per softmax warp
  const uint32_t sBar = sScr + T::SCRATCH_BYTES;
  const uint32_t bQ = sBar;                          // q_full[2]
  const uint32_t bQe = bQ + 16u;                     // q_empty[2]
  const uint32_t bKVf = bQe + 16u;                   // kv_full[NSTAGE]
  const uint32_t bKVe = bKVf + 8u * T::NSTAGE;       // kv_empty[NSTAGE]
  const uint32_t bS = bKVe + 8u * T::NSTAGE;         // s_full[2]
  const uint32_t bP = bS + 16u;                      // p_full[2][2] (tile, half of the keys)
  const uint32_t bO = bP + 32u;                      // o_full[2]
  const uint32_t bUf = bO + 16u;                     // unit_full[2]
  const uint32_t bUe = bUf + 16u;                    // unit_empty[2]
  const uint32_t bDrain = bUe + 16u;
  uint8_t* const misc = gbase + (sBar - base) + 8 * T::NBAR;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  volatile int* const unit_ring = reinterpret_cast<volatile int*>(misc + 8);  // [2]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // A unit's head and query-tile pair, and the key tiles query tile s of it
  // visits (causal: up to the tile holding its last row's last visible key,
  // query row i at position koff + i).
  auto unit_of = [&](int u, int& bh, int& mt) {
    int lv;
    work_unit(u, p.n_mtiles, p.B * p.H, p.tail, bh, lv);
    mt = p.n_mtiles - 1 - lv;
  };
  auto ntiles = [&](int mt, int s) -> int {
    return CAUSAL ? max(1, min((p.koff + 256 * mt + 128 * s + 127) / 128 + 1, p.nkv)) : p.nkv;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bQ + 8u * s, 1);
      mbar_init(bQe + 8u * s, 1);
      mbar_init(bS + 8u * s, 1);
      mbar_init(bP + 16u * s, 128);
      mbar_init(bP + 16u * s + 8u, 128);
      mbar_init(bO + 8u * s, 1);
      mbar_init(bUf + 8u * s, 1);
      mbar_init(bUe + 8u * s, kUnitReaders);
    }
    for (int i = 0; i < T::NSTAGE; ++i) {
      mbar_init(bKVf + 8u * i, 1);
      mbar_init(bKVe + 8u * i, 1);
    }
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
    ok = __all_sync(0xffffffffu, wait_bounded(wc, bUf + 8u * e, (k >> 1) & 1, wait_site(0x5a, k)));
    const int u = ok ? unit_ring[e] : -1;
    mbar_arrive(bUe + 8u * e);
    return u;
  };

  if (warp < 8) {
    setmaxnreg_inc<208>();
    reg_split_sync(384);
    // ------------------------------------------------------------ softmax
    // Warpgroup s takes query tile s of every unit (one thread per row);
    // the body is attn_fwd.cu's for a dense row.
    const int s = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + s * 128 + lane_off;
    const uint32_t tO = tmem + 256 + s * 128 + lane_off;
    const uint32_t barS = bS + 8u * s, barP = bP + 16u * s, barO = bO + 8u * s;
    const float c = p.scale_log2;
    uint32_t ns = 0;  // S tiles of this query tile consumed so far, over all units
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int u = next_unit(k, ok);
      if (u < 0) break;
      int bh, mt;
      unit_of(u, bh, mt);
      const int qi = 2 * mt + s;
      const int n = ntiles(mt, s);
      // Columns at or past lim0 - 128 j of key tile j are invisible to row
      // r: keys past Nk, and for causal rows keys past position koff + 128 qi + r.
      const int lim0 = CAUSAL ? min(p.Nk, p.koff + qi * 128 + r + 1) : p.Nk;
      // Running max from -1e30 (see attn_fwd.cu); l sums the fp32 p, lo the
      // normaliser of O (bf16-rounded p on a row's first tile with hidden columns).
      float m = -1e30f, l = 0.f, lo = 0.f;
      for (int j = 0; j < n; ++j, ++ns) {
        ok = __all_sync(0xffffffffu, wait_bounded(wc, barS, ns & 1, wait_site(0x51 + s, j)));
        if (!ok) break;
        tc_fence_after();
        float x[128];
        {
          uint32_t ra[32], rb[32], rc[32], rd[32];
          tmem_ld32(tS + 0, ra);
          tmem_ld32(tS + 32, rb);
          tmem_ld32(tS + 64, rc);
          tmem_ld32(tS + 96, rd);
          tmem_wait_ld();
          reg_fence(ra);
          reg_fence(rb);
          reg_fence(rc);
          reg_fence(rd);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            x[i] = __uint_as_float(ra[i]);
            x[32 + i] = __uint_as_float(rb[i]);
            x[64 + i] = __uint_as_float(rc[i]);
            x[96 + i] = __uint_as_float(rd[i]);
          }
        }
        // Only the diagonal and the ragged last tile have masked columns.
        const int lim = lim0 - j * 128;
        const bool edge = __any_sync(0xffffffffu, lim < 128);
        if (edge) {
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i >= lim) x[i] = -INFINITY;
        }
        float mx[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) mx[q] = x[q];
#pragma unroll
        for (int i = 8; i < 128; i += 2) mx[(i >> 1) & 7] = fmax3(mx[(i >> 1) & 7], x[i], x[i + 1]);
        const float tile_max = fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], fmax3(mx[4], mx[5], mx[6]), mx[7]));
        const float mc = tile_max * c;
        const bool raise = mc > m + 8.0f;  // always true on the first tile
        float alpha = 1.f;
        if (raise) {
          alpha = ex2(m - mc);
          m = mc;
        }
        if (j > 0 && __any_sync(0xffffffffu, raise)) {
          // O_acc <- alpha * O_acc (P V of tile j-1 has completed: its
          // commit precedes S_j's).
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + cc * 32, o);
            tmem_wait_ld();
            reg_fence(o);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 t = fmul2(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])),
                                     make_float2(alpha, alpha));
              o[i] = __float_as_uint(t.x);
              o[i + 1] = __float_as_uint(t.y);
            }
            tmem_st32(tO + cc * 32, o);
          }
        }
        const float2 c2 = make_float2(c, c), nm2 = make_float2(-m, -m);
        float2 sum[4], sumr = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 4; ++q) sum[q] = make_float2(0.f, 0.f);
        auto publish = [&](auto rounded) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int i = 64 * h + 2 * e;
              const float2 t = ffma2(make_float2(x[i], x[i + 1]), c2, nm2);
              const float2 pp = make_float2(ex2(t.x), ex2(t.y));
              if constexpr (decltype(rounded)::value)
                sum[e & 1] = fadd2(sum[e & 1], pp);
              else
                sum[e & 3] = fadd2(sum[e & 3], pp);
              pk[e] = pack_bf16(pp.x, pp.y);
            }
            tmem_st32(tS + 32 * h, pk);
            if constexpr (decltype(rounded)::value) {
#pragma unroll
              for (int e = 0; e < 32; ++e)
                sumr = fadd2(sumr, make_float2(__uint_as_float(pk[e] << 16), __uint_as_float(pk[e] & 0xffff0000u)));
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(barP + 8u * h);
          }
        };
        if (edge && j == 0) {
          publish(std::true_type{});
          const float2 s01 = fadd2(sum[0], sum[1]);
          l = l * alpha + (s01.x + s01.y);
          lo = lo * alpha + (sumr.x + sumr.y);
        } else {
          publish(std::false_type{});
          const float2 s01 = fadd2(sum[0], sum[1]), s23 = fadd2(sum[2], sum[3]);
          const float st = (s01.x + s23.x) + (s01.y + s23.y);
          l = l * alpha + st;
          lo = lo * alpha + st;
        }
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      // O / lo in bf16 from registers to this row of O, and lse.  The next
      // unit's first P V, which overwrites O in tensor memory, waits for
      // this warpgroup's next P, published after these loads.
      // Each warp's 32 rows go through its shared-memory scratch
      // (store_rows_staged), so that a store covers whole 128-byte row
      // slices rather than 32 separate 16-byte pieces; at d = 64 with a
      // causal mask they go straight out (A/B, staged against direct: c3c
      // 217.1 -> 218.9 us, c3 401.4 -> 393.2, c4p 296.5 -> 288.8, c5
      // 366.6 -> 356.4, cx 341 -> 328, cp1 329 -> 332).
      ok = __all_sync(0xffffffffu, wait_bounded(wc, barO, k & 1, wait_site(0x53 + s, k)));
      if (!ok) break;
      tc_fence_after();
      const int row = qi * 128 + r;
      const float inv = lo > 0.f ? 1.f / lo : 0.f;
      if constexpr (STAGED_O) {
        const int wr0 = qi * 128 + 32 * (warp & 3);  // the warp's first row
        uint16_t* const wdst = p.o + ((size_t)bh * p.Nq + wr0) * D;
        int nvalid = min(32, p.Nq - wr0);
        if (nvalid > 0 && !ATTN_IN_RANGE(((size_t)bh * p.Nq + wr0 + nvalid) * D - 1, (size_t)p.B * p.H * p.Nq * D, p, 0x105))
          nvalid = 0;
        const uint32_t scr = sScr + (uint32_t)warp * 4096u;
        // 32 columns of this thread's row (from o) as four bf16 chunks.
        auto pack4 = [&](const uint32_t (&o)[32], uint4* ch) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16(__uint_as_float(o[q4 * 8 + 2 * e]) * inv, __uint_as_float(o[q4 * 8 + 2 * e + 1]) * inv);
            ch[q4] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        };
#pragma unroll
        for (int cc = 0; cc + 1 < D / 32; cc += 2) {  // 64 columns: two loads per wait
          uint32_t oa[32], ob[32];
          tmem_ld32(tO + cc * 32, oa);
          tmem_ld32(tO + cc * 32 + 32, ob);
          tmem_wait_ld();
          reg_fence(oa);
          reg_fence(ob);
          uint4 ch[8];
          pack4(oa, ch);
          pack4(ob, ch + 4);
          store_rows_staged<8>(ch, scr, wdst + cc * 32, D, nvalid);
        }
        if constexpr (D % 64 != 0) {  // d = 96: the last 32 columns
          uint32_t oa[32];
          tmem_ld32(tO + (D / 32 - 1) * 32, oa);
          tmem_wait_ld();
          reg_fence(oa);
          uint4 ch[4];
          pack4(oa, ch);
          store_rows_staged<4>(ch, scr, wdst + (D - 32), D, nvalid);
        }
      } else {
        uint16_t* const orow = p.o + ((size_t)bh * p.Nq + row) * D;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + cc * 32, o);
          tmem_wait_ld();
          reg_fence(o);
          if (row < p.Nq && ATTN_IN_RANGE(((size_t)bh * p.Nq + row) * D + cc * 32 + 31, (size_t)p.B * p.H * p.Nq * D, p, 0x105)) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w[e] = pack_bf16(__uint_as_float(o[q4 * 8 + 2 * e]) * inv, __uint_as_float(o[q4 * 8 + 2 * e + 1]) * inv);
              *reinterpret_cast<uint4*>(orow + cc * 32 + q4 * 8) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
      if (row < p.Nq && ATTN_IN_RANGE((size_t)bh * p.Nq + row, (size_t)p.B * p.H * p.Nq, p, 0x106))
        p.lse[(size_t)bh * p.Nq + row] = (m + log2f(l)) * 0.69314718055994531f;
    }
    setmaxnreg_dec<168>();  // one register budget again for the common teardown
  } else {
    setmaxnreg_dec<88>();
    reg_split_sync(384);
    if (warp == 8) {
      // ------------------------------------------------------------ unit queue and TMA producer
      // Takes the next unit of the launch's order (work_unit) from the
      // queue, hands it to the other roles through the unit ring, then loads
      // its Q tiles (once the previous unit's last Q K^T of that tile has
      // read the buffer) and its K_j / V_j into the ring, which runs on
      // across units.
      if (lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        bool ok = true;
        int t = 0;  // ring slot counter over all units: K_j is slot t, V_j slot t + 1
        int nq = 0; // units whose Q tiles were issued
        for (int k = 0; ok; ++k) {
          const int e = k & 1;
          // CTA b's first unit is unit b (no queue round trip before the first
          // loads); the counter hands out the rest, from gridDim.x on.
          int u = k == 0 ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(p.sched, 1);
          if (u >= p.n_units) u = -1;
          if (k >= 2 && !(ok = wait_bounded(wc, bUe + 8u * e, ((k - 2) >> 1) & 1, wait_site(0x64, k)))) break;
          unit_ring[e] = u;
          mbar_arrive(bUf + 8u * e);  // (release: the entry is visible to the roles that wait for it)
          if (u < 0) break;
          int bh, mt;
          unit_of(u, bh, mt);
          const int bhk = (bh / p.H) * p.Hkv + (bh % p.H) / p.G;
          const int n1 = ntiles(mt, 1);
          for (int s = 0; s < 2 && ok; ++s) {
            if (k >= 1 && !(ok = wait_bounded(wc, bQe + 8u * s, (k - 1) & 1, wait_site(0x65 + s, k)))) break;
            mbar_expect_tx(bQ + 8u * s, T::TILE_BYTES);
            for (int cb = 0; cb < T::NB; ++cb)
              tma_load_3d(sQ + s * T::TILE_BYTES + cb * T::BLOCK_BYTES, &tmQ, bQ + 8u * s, cb * 64,
                          (2 * mt + s) * 128, bh);
          }
          if (!ok) break;
          nq = k + 1;
          for (int j = 0; j < n1 && ok; ++j) {
            for (int w = 0; w < 2; ++w) {
              const int st = t % T::NSTAGE, rd = t / T::NSTAGE;
              if (rd > 0 && !(ok = wait_bounded(wc, bKVe + 8u * st, (rd - 1) & 1, wait_site(0x61, t)))) break;
              if (u == 0 && p.debug_drop_p == 2 * j + w + 1) {  // test of the bounded waits only
                ++t;
                continue;
              }
              mbar_expect_tx(bKVf + 8u * st, T::TILE_BYTES);
              const CUtensorMap* m = (w == 0) ? &tmK : &tmV;
              for (int cb = 0; cb < T::NB; ++cb)
                tma_load_3d(sKV + st * T::TILE_BYTES + cb * T::BLOCK_BYTES, m, bKVf + 8u * st, cb * 64, j * 128,
                            bhk);
              ++t;
            }
          }
        }
        // Every copy this thread issued has landed before the CTA may exit
        // (immediate on the normal path; matters after an abort).
        if (nq > 0)
          for (int s = 0; s < 2; ++s) wait_drain(bQ + 8u * s, (nq - 1) & 1, p.limit_ns);
        for (int i = 0; i < T::NSTAGE && i < t; ++i) {
          const int last = ((t - 1 - i) / T::NSTAGE) * T::NSTAGE + i;
          wait_drain(bKVf + 8u * i, (last / T::NSTAGE) & 1, p.limit_ns);
        }
      }
      __syncwarp();
    } else if (warp == 9) {
      // ------------------------------------------------------------ MMA issuer
      // attn_fwd.cu's schedule for each unit in turn; the ring slot counter
      // and the P barriers' phases run on across units.
      {
        const uint32_t leader = elect_one();
        constexpr uint32_t IQK = idesc_bf16_f32(128, 128, false, false);
        constexpr uint32_t IPV = idesc_bf16_f32(128, D, false, true);
        const uint32_t tS0 = tmem, tS1 = tmem + 128, tO0 = tmem + 256, tO1 = tmem + 384;
        const uint64_t dQ0 = sdesc_sw128(sQ, 16, 1024), dQ1 = sdesc_sw128(sQ + T::TILE_BYTES, 16, 1024);
        const uint64_t dK0 = sdesc_sw128(sKV, 16, 1024);             // K slots (K-major)
        const uint64_t dV0 = sdesc_sw128(sKV, T::BLOCK_BYTES, 1024);  // V slots (MN-major)
        auto qk = [&](uint32_t dS, uint64_t qd, uint64_t kd) {
#pragma unroll
          for (int kk = 0; kk < T::KSTEPS; ++kk) {
            const uint32_t off = (kk >> 2) * T::BLOCK_BYTES + (kk & 3) * 32;
            mma_ss_p(leader, dS, sdesc_add(qd, off), sdesc_add(kd, off), IQK, kk > 0);
          }
        };
        // O += P V over keys [64h, 64h + 64) once half h of P is in TMEM.
        auto pv_half = [&](uint32_t dO, uint32_t p_tmem, uint64_t vd, bool acc, int h) {
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int kk = 4 * h + k4;
            mma_ts_p(leader, dO, p_tmem + kk * 8, sdesc_add(vd, kk * 2048), IPV, (acc || kk > 0) ? 1u : 0u);
          }
        };
        auto wait_all = [&](uint32_t bar, uint32_t parity, int site) {
          return __all_sync(0xffffffffu, wait_bounded(wc, bar, parity, site));
        };
        bool ok = true;
        int tb = 0;               // ring index of this unit's K_0
        uint32_t np0 = 0, np1 = 0;  // P tiles each softmax warpgroup has published so far
        for (int k = 0; ok; ++k) {
          const int u = next_unit(k, ok);
          if (u < 0) break;
          int bh, mt;
          unit_of(u, bh, mt);
          const int n0 = ntiles(mt, 0), n1 = ntiles(mt, 1);  // key tiles of query tiles 0 / 1 (n0 <= n1)
          const uint32_t qp = k & 1;
          const uint64_t dKf = sdesc_add(dK0, (tb % T::NSTAGE) * T::TILE_BYTES);
          if (!(ok = wait_all(bKVf + 8u * (tb % T::NSTAGE), (tb / T::NSTAGE) & 1, wait_site(0x71, k)) &&
                     wait_all(bQ, qp, wait_site(0x72, k))))
            break;
          tc_fence_after();
          qk(tS0, dQ0, dKf);
          mma_commit_p(leader, bS);
          if (n0 == 1) mma_commit_p(leader, bQe);  // Q tile 0 read for the last time
          if (!(ok = wait_all(bQ + 8u, qp, wait_site(0x73, k)))) break;
          tc_fence_after();
          qk(tS1, dQ1, dKf);
          mma_commit_p(leader, bS + 8u);
          if (n1 == 1) mma_commit_p(leader, bQe + 8u);
          mma_commit_p(leader, bKVe + 8u * (tb % T::NSTAGE));  // K_0 consumed
          for (int j = 0; j < n1 && ok; ++j) {
            const int t = tb + 2 * j + 1;  // V_j; K_{j+1} is t + 1
            const int sv = t % T::NSTAGE, sk = (t + 1) % T::NSTAGE;
            const bool next = j + 1 < n1;
            const uint64_t vd = sdesc_add(dV0, sv * T::TILE_BYTES), kd = sdesc_add(dK0, sk * T::TILE_BYTES);
            // V_j is needed now; K_{j+1} only for the next Q K^T.
            if (!(ok = wait_all(bKVf + 8u * sv, (t / T::NSTAGE) & 1, wait_site(0x74, j)))) break;
            if (j < n0) {
              if (!(ok = wait_all(bP, np0 & 1, wait_site(0x76, j)))) break;  // keys 0-63
              tc_fence_after();
              pv_half(tO0, tS0, vd, j > 0, 0);
              if (!(ok = wait_all(bP + 8u, np0 & 1, wait_site(0x78, j)))) break;  // keys 64-127
              tc_fence_after();
              pv_half(tO0, tS0, vd, j > 0, 1);
              ++np0;
              if (j + 1 < n0) {
                if (!(ok = wait_all(bKVf + 8u * sk, ((t + 1) / T::NSTAGE) & 1, wait_site(0x75, j)))) break;
                tc_fence_after();
                qk(tS0, dQ0, kd);
                mma_commit_p(leader, bS);
                if (j + 2 == n0) mma_commit_p(leader, bQe);
              } else {
                mma_commit_p(leader, bO);
              }
            }
            if (!(ok = wait_all(bP + 16u, np1 & 1, wait_site(0x77, j)))) break;
            tc_fence_after();
            pv_half(tO1, tS1, vd, j > 0, 0);
            if (!(ok = wait_all(bP + 24u, np1 & 1, wait_site(0x79, j)))) break;
            tc_fence_after();
            pv_half(tO1, tS1, vd, j > 0, 1);
            ++np1;
            if (next) {
              if (!(ok = wait_all(bKVf + 8u * sk, ((t + 1) / T::NSTAGE) & 1, wait_site(0x7a, j)))) break;
              tc_fence_after();
              qk(tS1, dQ1, kd);
              mma_commit_p(leader, bS + 8u);
              if (j + 2 == n1) mma_commit_p(leader, bQe + 8u);
            } else {
              mma_commit_p(leader, bO + 8u);
            }
            mma_commit_p(leader, bKVe + 8u * sv);
            if (next) mma_commit_p(leader, bKVe + 8u * sk);
          }
          tb += 2 * n1;
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

// Queue slots (next unit, CTAs done), one per launch in flight: launches
// take slots in turn, and a slot is back at zero when its launch ends, so
// up to kQueueSlots launches may run at once on different streams.
constexpr int kQueueSlots = 256;
__device__ int g_fwd_queue[kQueueSlots][2];

int* queue_slot() {
  static std::atomic<unsigned> next{0};
  static int* base[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (base[dev] == nullptr) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_fwd_queue) != cudaSuccess) return nullptr;
    base[dev] = static_cast<int*>(a);
  }
  return base[dev] + 2 * (next.fetch_add(1) % kQueueSlots);
}

template <int D, bool C>
cudaError_t launch_persist_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const FwdParams& p, cudaStream_t stream) {
  using T = PTraits<D>;
  auto kern = fwd_persist_kernel<D, C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidValue;
  FwdParams pc = p;
  pc.n_units = p.n_mtiles * p.B * p.H;
  pc.tail = uniform_levels(C, p.vl, p.mk, false) ? 1 : order_tail(p.n_mtiles, p.B * p.H, p.G);
  pc.sched = queue_slot();
  if (pc.sched == nullptr) return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)min(pc.n_units, sms);  // one CTA per SM
  kern<<<grid, T::THREADS, T::SMEM, stream>>>(tq, tk, tv, pc);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_persist(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const FwdParams& p, cudaStream_t stream) {
  switch (d) {
    case 64: return causal ? launch_persist_t<64, true>(tq, tk, tv, p, stream) : launch_persist_t<64, false>(tq, tk, tv, p, stream);
    case 96: return causal ? launch_persist_t<96, true>(tq, tk, tv, p, stream) : launch_persist_t<96, false>(tq, tk, tv, p, stream);
    case 128:
      return causal ? launch_persist_t<128, true>(tq, tk, tv, p, stream) : launch_persist_t<128, false>(tq, tk, tv, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sdpa
