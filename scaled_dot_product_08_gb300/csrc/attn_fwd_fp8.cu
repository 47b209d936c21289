// attn_fwd_fp8.cu — forward of exact attention with FP8 (e4m3) tensor-core
// products on sm_103a, head_dim 64, 96 or 128.
//
// Method: the forward of attn_fwd.cu (page "Flash Attention原理", §三 tiling,
// §四 online softmax, §五 only O and the row statistic leave the chip), with
// both products on the FP8 tensor cores — the FlashAttention-3 idea the page
// describes in §六 and FAQ Q8 (FP8 tensor cores, per-tensor scales).  Q, K
// and V arrive as e4m3 with one dequantisation factor each (q = q8 * q_scale
// and so on); S = Q K^T accumulates in fp32 (tcgen05 kind::f8f6f4, K = 32 per
// instruction), the softmax runs in fp32 exactly as in the bf16 kernel, and
// P is rounded to e4m3 for the P V product.  P is computed as
// 2^(s - m + 4), so that small probabilities stay clear of e4m3's subnormal
// range (below 2^-6); the running max m is raised lazily, only when a tile
// max exceeds it by more than 4 (a factor 16), so P stays within 2^8, below
// e4m3's largest value 448.  The factor cancels in O = (P V) / l and is
// removed from lse.  O is written in bf16 (times v_scale), lse in
// float32.
//
// GB300 mapping: the bf16 forward's warp roles, barriers and tensor-memory
// plan, with e4m3 tiles of [128 rows x 128 bytes] (one 128-byte swizzle
// block per tile, half the bf16 bytes), so the K/V ring holds 10 stages.
// At d = 64 / 96 a row's d bytes fill the start of its 128-byte line and the
// TMA box fills the rest with zeros; Q K^T runs d / 32 K-steps and P V has
// N = d, so the padding costs shared memory, not MMA work:
//   warps 0-7  softmax (warpgroup s = query tile s of a unit)
//   warp  8    TMA producer (Q tiles, then K_j / V_j)
//   warp  9    MMA issuer
//   warps 10-11 idle
// Tensor memory: [0,128) S0, P0 (e4m3, 4 per column) over its first 32
// columns; [128,256) S1 / P1; [256,256+d) O0; [384,384+d) O1 (fp32).
// Two schedules of the (head, pair of query tiles) units, the same bits:
//   * fwd_fp8_kernel, one CTA per unit (d = 128);
//   * fwd_fp8_persist_kernel (d = 64, 96): the persistent schedule of
//     attn_fwd_persist.cu, one CTA per SM taking the units from a queue, the
//     producer running ahead into the next unit so that its first Q K^T
//     overlaps the current epilogue.  A/B, bit-identical: c3cf8 (d = 64)
//     228 -> 213 us; at d = 128 (c4f8) 278 -> 280 us, so d = 128 keeps one
//     CTA per unit.
#include <atomic>
#include <cmath>

#include <cuda_fp8.h>

#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {

namespace {

template <int D_>
struct F8 {
  static constexpr int D = D_;
  static constexpr int TILE_BYTES = 128 * 128;  // [128 rows x 128 e4m3]
  static constexpr int NSTAGE = 10;             // K/V ring depth
  static constexpr int KSTEPS = D / 32;         // K = 32 per e4m3 MMA
  // q_full[2] q_empty[2] kv_full[NSTAGE] kv_empty[NSTAGE] s_full[2]
  // p_full[2][2] o_full[2] unit_full[2] unit_empty[2] drain (the
  // persistent kernel's set; the one-CTA-per-unit kernel uses a subset)
  static constexpr int NBAR = 2 + 2 + 2 * NSTAGE + 2 + 4 + 2 + 2 + 2 + 1;
  static constexpr int MISC = 32;  // tmem slot, abort flag, unit ring
  static constexpr int SCRATCH_BYTES = D == 128 ? 8 * 4096 : 0;  // epilogue scratch, one 4 KB per softmax warp
  static constexpr int SMEM = 1024 + (2 + NSTAGE) * TILE_BYTES + SCRATCH_BYTES + NBAR * 8 + MISC;
  static constexpr int THREADS = 384;
};

// Arrivals on unit_empty: every thread that reads a ring entry (the MMA
// warp and both softmax warpgroups).
constexpr int kF8UnitReaders = 32 + 256;

// Instruction descriptor, kind::f8f6f4 with e4m3 A and B (format code 0) and
// an f32 accumulator; field positions as in idesc_bf16_f32.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N, bool b_mn_major) {
  return (1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f8_ss_p(uint32_t leader, uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(leader)
      : "memory");
}
__device__ __forceinline__ void mma_f8_ts_p(uint32_t leader, uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(leader)
      : "memory");
}

// Four floats to four e4m3 (round to nearest even, saturating), the first in
// the lowest byte: the K order of an 8-bit A operand in tensor memory.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using T = F8<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);

  const uint32_t sQ = base;                          // 2 query tiles
  const uint32_t sKV = base + 2 * T::TILE_BYTES;     // K/V ring
  const uint32_t sScr = sKV + T::NSTAGE * T::TILE_BYTES;  // d = 128: epilogue scratch, 4 KB per softmax warp
  const uint32_t sBar = sScr + T::SCRATCH_BYTES;
  const uint32_t bQ = sBar;                          // q_full[2]
  const uint32_t bKVf = sBar + 8u * 2;               // kv_full[NSTAGE]
  const uint32_t bKVe = bKVf + 8u * T::NSTAGE;       // kv_empty[NSTAGE]
  const uint32_t bS = bKVe + 8u * T::NSTAGE;         // s_full[2]
  const uint32_t bP = bS + 16u;                      // p_full[2][2] (tile, half of the keys)
  const uint32_t bO = bP + 32u;                      // o_full[2]
  const uint32_t bDrain = bO + 16u;
  uint8_t* const misc = gbase + (sBar - base) + 8 * T::NBAR;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(misc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work unit (work_unit): head-major, the heaviest causal query tiles of a
  // head first; the last heads level-major, for a short tail.
  int bh, lv;
  work_unit((int)blockIdx.x, p.n_mtiles, p.B * p.H, p.tail, bh, lv);
  const int mt = p.n_mtiles - 1 - lv;
  const int bhk = (bh / p.H) * p.Hkv + (bh % p.H) / p.G;
  int n0 = p.nkv, n1 = p.nkv;  // key tiles visited by query tile 0 / 1
  if (CAUSAL) {  // up to the tile holding the last row's last visible key, koff + 128 qi + 127
    n0 = min((p.koff + 256 * mt + 127) / 128 + 1, p.nkv);
    n1 = min((p.koff + 256 * mt + 255) / 128 + 1, p.nkv);
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bQ + 8u * s, 1);
      mbar_init(bS + 8u * s, 1);
      mbar_init(bP + 16u * s, 128);
      mbar_init(bP + 16u * s + 8u, 128);
      mbar_init(bO + 8u * s, 1);
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

  if (warp < 8) {
    setmaxnreg_inc<208>();
    reg_split_sync(384);
    // ------------------------------------------------------------ softmax
    const int s = warp >> 2;            // query tile of this warpgroup
    const int r = threadIdx.x & 127;    // row within the tile == TMEM lane
    const int qi = 2 * mt + s;          // global query tile index
    const int n = s ? n1 : n0;
    // Columns at or past lim0 - 128 j of key tile j are invisible to row r.
    const int lim0 = CAUSAL ? min(p.Nk, p.koff + qi * 128 + r + 1) : p.Nk;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + s * 128 + lane_off;
    const uint32_t tO = tmem + 256 + s * 128 + lane_off;
    const uint32_t barS = bS + 8u * s, barP = bP + 16u * s, barO = bO + 8u * s;
    const float c = p.scale_log2;  // softmax scale * log2 e * q_scale * k_scale
    float m = -1e30f, l = 0.f;     // running max (base 2) and sum of 2^(s - m + 4)
    bool ok = true;

    for (int j = 0; j < n; ++j) {
      ok = __all_sync(0xffffffffu, wait_bounded(wc, barS, j & 1, wait_site(0xc1 + s, j)));
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
      {
        const int lim = lim0 - j * 128;
        if (__any_sync(0xffffffffu, lim < 128)) {
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i >= lim) x[i] = -INFINITY;
        }
      }
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = x[k];
#pragma unroll
      for (int i = 8; i < 128; i += 2) mx[(i >> 1) & 7] = fmax3(mx[(i >> 1) & 7], x[i], x[i + 1]);
      const float tile_max = fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], fmax3(mx[4], mx[5], mx[6]), mx[7]));
      const float mc = tile_max * c;
      const bool raise = mc > m + 4.0f;  // always true on the first tile; keeps 2^(s - m + 4) <= 2^8
      float alpha = 1.f;
      if (raise) {
        alpha = ex2(m - mc);
        m = mc;
      }
      if (j > 0 && __any_sync(0xffffffffu, raise)) {
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
      // p = 2^(x c - m + 4) in [0, 256]; e4m3, four to a column; published
      // in two halves of 64 keys.
      const float2 c2 = make_float2(c, c), nm2 = make_float2(4.f - m, 4.f - m);
      float2 sum[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) sum[k] = make_float2(0.f, 0.f);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int i = 64 * h + 4 * e;
          const float2 t0 = ffma2(make_float2(x[i], x[i + 1]), c2, nm2);
          const float2 t1 = ffma2(make_float2(x[i + 2], x[i + 3]), c2, nm2);
          const float2 p0 = make_float2(ex2(t0.x), ex2(t0.y)), p1 = make_float2(ex2(t1.x), ex2(t1.y));
          sum[e & 3] = fadd2(sum[e & 3], fadd2(p0, p1));
          pk[e] = pack_e4m3x4(p0.x, p0.y, p1.x, p1.y);
        }
        tmem_st16(tS + 16 * h, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(barP + 8u * h);
      }
      const float2 s01 = fadd2(sum[0], sum[1]), s23 = fadd2(sum[2], sum[3]);
      l = l * alpha + ((s01.x + s23.x) + (s01.y + s23.y));
    }

    // ------------------------------------------------------------ epilogue
    // O = (P V) * v_scale / l in bf16, straight from registers to global
    // memory (a bf16 tile is twice an e4m3 tile, so there is no staging
    // buffer in the K/V ring while the other query tile still uses it).
    if (ok) ok = __all_sync(0xffffffffu, wait_bounded(wc, barO, 0, wait_site(0xc3 + s, 0)));
    if (ok) {
      tc_fence_after();
      const int row = qi * 128 + r;
      const float inv = l > 0.f ? p.o_scale / l : 0.f;
      if constexpr (D == 128) {
        // The warp's 32 rows, written a row slice per group of lanes
        // through the warp's shared-memory scratch (store_rows_staged):
        // whole lines per store.  (A/B with a shuffle transpose: d = 128
        // 285 -> 279 us on c4f8; at d = 64 it cost more than it saved,
        // 228 -> 234 us on c3cf8, so the other head dims store rows
        // directly.)
        const int wr0 = qi * 128 + 32 * (warp & 3);
        uint16_t* const wdst = p.o + ((size_t)bh * p.Nq + wr0) * D;
        int nvalid = min(32, p.Nq - wr0);
        if (nvalid > 0 && !ATTN_IN_RANGE(((size_t)bh * p.Nq + wr0 + nvalid) * D - 1, (size_t)p.B * p.H * p.Nq * D, p, 0x601))
          nvalid = 0;
        // Columns 32 cc .. 32 cc + 31 of this thread's row as four bf16 chunks.
        auto chunks = [&](int cc, uint4* ch) {
          uint32_t o[32];
          tmem_ld32(tO + cc * 32, o);
          tmem_wait_ld();
          reg_fence(o);
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
        for (int cc = 0; cc < D / 32; cc += 2) {
          uint4 ch[8];
          chunks(cc, ch);
          chunks(cc + 1, ch + 4);
          store_rows_staged<8>(ch, sScr + (uint32_t)warp * 4096u, wdst + cc * 32, D, nvalid);
        }
      } else {
        uint16_t* const orow = p.o + ((size_t)bh * p.Nq + row) * D;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + cc * 32, o);
          tmem_wait_ld();
          reg_fence(o);
          if (row < p.Nq && ATTN_IN_RANGE(((size_t)bh * p.Nq + row) * D + cc * 32 + 31, (size_t)p.B * p.H * p.Nq * D, p, 0x601)) {
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
      if (row < p.Nq && ATTN_IN_RANGE((size_t)bh * p.Nq + row, (size_t)p.B * p.H * p.Nq, p, 0x602))
        p.lse[(size_t)bh * p.Nq + row] = (m + log2f(l) - 4.f) * 0.69314718055994531f;
    }
    setmaxnreg_dec<168>();
  } else {
    setmaxnreg_dec<88>();
    reg_split_sync(384);
    if (warp == 8) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        for (int s = 0; s < 2; ++s) {
          mbar_expect_tx(bQ + 8u * s, T::TILE_BYTES);
          tma_load_3d(sQ + s * T::TILE_BYTES, &tmQ, bQ + 8u * s, 0, (2 * mt + s) * 128, bh);
        }
        bool ok = true;
        int t = 0;  // ring slot counter: K_j is slot 2j, V_j is slot 2j+1
        for (int j = 0; j < n1 && ok; ++j) {
          for (int w = 0; w < 2; ++w) {
            const int st = t % T::NSTAGE, rd = t / T::NSTAGE;
            if (rd > 0 && !(ok = wait_bounded(wc, bKVe + 8u * st, (rd - 1) & 1, wait_site(0xd1, t)))) break;
            if (blockIdx.x == 0 && p.debug_drop_p == t + 1) {  // test of the bounded waits only
              ++t;
              continue;
            }
            mbar_expect_tx(bKVf + 8u * st, T::TILE_BYTES);
            tma_load_3d(sKV + st * T::TILE_BYTES, (w == 0) ? &tmK : &tmV, bKVf + 8u * st, 0, j * 128, bhk);
            ++t;
          }
        }
        for (int s = 0; s < 2; ++s) wait_drain(bQ + 8u * s, 0, p.limit_ns);
        for (int i = 0; i < T::NSTAGE && i < t; ++i) {
          const int last = ((t - 1 - i) / T::NSTAGE) * T::NSTAGE + i;
          wait_drain(bKVf + 8u * i, (last / T::NSTAGE) & 1, p.limit_ns);
        }
      }
      __syncwarp();
    } else if (warp == 9) {
      // ------------------------------------------------------------ MMA issuer
      {
        const uint32_t leader = elect_one();
        constexpr uint32_t IQK = idesc_e4m3_f32(128, 128, false);  // S = Q K^T (both K-major)
        constexpr uint32_t IPV = idesc_e4m3_f32(128, D, true);     // O += P V (A in TMEM, V MN-major)
        const uint32_t tS0 = tmem, tS1 = tmem + 128, tO0 = tmem + 256, tO1 = tmem + 384;
        const uint64_t dQ0 = sdesc_sw128(sQ, 16, 1024), dQ1 = sdesc_sw128(sQ + T::TILE_BYTES, 16, 1024);
        const uint64_t dK0 = sdesc_sw128(sKV, 16, 1024);               // K slots (K-major)
        const uint64_t dV0 = sdesc_sw128(sKV, T::TILE_BYTES, 1024);    // V slots (MN-major; d = one 128-byte chunk)
        // S = Q K^T: K = 32 e4m3 (32 bytes) per instruction inside the 128-byte rows.
        auto qk = [&](uint32_t dS, uint64_t qd, uint64_t kd) {
#pragma unroll
          for (int kk = 0; kk < T::KSTEPS; ++kk)
            mma_f8_ss_p(leader, dS, sdesc_add(qd, kk * 32), sdesc_add(kd, kk * 32), IQK, kk > 0);
        };
        // O += P V over keys [64h, 64h + 64): two K steps of 32 keys; P's
        // K step kk is tensor-memory columns 8 kk .. 8 kk + 7, V's is rows
        // 32 kk .. 32 kk + 31 (4096 bytes).
        auto pv_half = [&](uint32_t dO, uint32_t p_tmem, uint64_t vd, bool acc, int h) {
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            const int kk = 2 * h + k2;
            mma_f8_ts_p(leader, dO, p_tmem + kk * 8, sdesc_add(vd, kk * 4096), IPV, (acc || kk > 0) ? 1u : 0u);
          }
        };
        auto wait_all = [&](uint32_t bar, uint32_t parity, int site) {
          return __all_sync(0xffffffffu, wait_bounded(wc, bar, parity, site));
        };
        bool ok = wait_all(bKVf, 0, wait_site(0xe1, 0)) && wait_all(bQ, 0, wait_site(0xe2, 0));
        if (ok) {
          tc_fence_after();
          qk(tS0, dQ0, dK0);
          mma_commit_p(leader, bS);
          ok = wait_all(bQ + 8u, 0, wait_site(0xe3, 0));
        }
        if (ok) {
          tc_fence_after();
          qk(tS1, dQ1, dK0);
          mma_commit_p(leader, bS + 8u);
          mma_commit_p(leader, bKVe);  // K_0 consumed
        }
        int t = 1;
        for (int j = 0; j < n1 && ok; ++j, t += 2) {
          const int sv = t % T::NSTAGE, sk = (t + 1) % T::NSTAGE;
          const bool next = j + 1 < n1;
          const uint64_t vd = sdesc_add(dV0, sv * T::TILE_BYTES), kd = sdesc_add(dK0, sk * T::TILE_BYTES);
          if (!(ok = wait_all(bKVf + 8u * sv, (t / T::NSTAGE) & 1, wait_site(0xe4, j)))) break;
          if (j < n0) {
            if (!(ok = wait_all(bP, j & 1, wait_site(0xe6, j)))) break;
            tc_fence_after();
            pv_half(tO0, tS0, vd, j > 0, 0);
            if (!(ok = wait_all(bP + 8u, j & 1, wait_site(0xe8, j)))) break;
            tc_fence_after();
            pv_half(tO0, tS0, vd, j > 0, 1);
            if (j + 1 < n0) {
              if (!(ok = wait_all(bKVf + 8u * sk, ((t + 1) / T::NSTAGE) & 1, wait_site(0xe5, j)))) break;
              tc_fence_after();
              qk(tS0, dQ0, kd);
              mma_commit_p(leader, bS);
            } else {
              mma_commit_p(leader, bO);
            }
          }
          if (!(ok = wait_all(bP + 16u, j & 1, wait_site(0xe7, j)))) break;
          tc_fence_after();
          pv_half(tO1, tS1, vd, j > 0, 0);
          if (!(ok = wait_all(bP + 24u, j & 1, wait_site(0xe9, j)))) break;
          tc_fence_after();
          pv_half(tO1, tS1, vd, j > 0, 1);
          if (next) {
            if (!(ok = wait_all(bKVf + 8u * sk, ((t + 1) / T::NSTAGE) & 1, wait_site(0xea, j)))) break;
            tc_fence_after();
            qk(tS1, dQ1, kd);
            mma_commit_p(leader, bS + 8u);
          } else {
            mma_commit_p(leader, bO + 8u);
          }
          mma_commit_p(leader, bKVe + 8u * sv);
          if (next) mma_commit_p(leader, bKVe + 8u * sk);
        }
        mma_commit_p(leader, bDrain);
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

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    fwd_fp8_persist_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using T = F8<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);

  const uint32_t sQ = base;                          // 2 query tiles
  const uint32_t sKV = base + 2 * T::TILE_BYTES;     // K/V ring
  const uint32_t sBar = sKV + T::NSTAGE * T::TILE_BYTES;
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
      mbar_init(bUe + 8u * s, kF8UnitReaders);
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
    ok = __all_sync(0xffffffffu, wait_bounded(wc, bUf + 8u * e, (k >> 1) & 1, wait_site(0xc5, k)));
    const int u = ok ? unit_ring[e] : -1;
    mbar_arrive(bUe + 8u * e);
    return u;
  };

  if (warp < 8) {
    setmaxnreg_inc<208>();
    reg_split_sync(384);
    // ------------------------------------------------------------ softmax
    // Warpgroup s takes query tile s of every unit (one thread per row).
    const int s = warp >> 2;
    const int r = threadIdx.x & 127;  // row within the tile == TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + s * 128 + lane_off;
    const uint32_t tO = tmem + 256 + s * 128 + lane_off;
    const uint32_t barS = bS + 8u * s, barP = bP + 16u * s, barO = bO + 8u * s;
    const float c = p.scale_log2;  // softmax scale * log2 e * q_scale * k_scale
    uint32_t ns = 0;               // S tiles of this query tile consumed so far, over all units
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int u = next_unit(k, ok);
      if (u < 0) break;
      int bh, mt;
      unit_of(u, bh, mt);
      const int qi = 2 * mt + s;  // global query tile index
      const int n = ntiles(mt, s);
      // Columns at or past lim0 - 128 j of key tile j are invisible to row r.
      const int lim0 = CAUSAL ? min(p.Nk, p.koff + qi * 128 + r + 1) : p.Nk;
      float m = -1e30f, l = 0.f;  // running max (base 2) and sum of 2^(s - m + 4)
      for (int j = 0; j < n; ++j, ++ns) {
        ok = __all_sync(0xffffffffu, wait_bounded(wc, barS, ns & 1, wait_site(0xc1 + s, j)));
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
        {
          const int lim = lim0 - j * 128;
          if (__any_sync(0xffffffffu, lim < 128)) {
#pragma unroll
            for (int i = 0; i < 128; ++i)
              if (i >= lim) x[i] = -INFINITY;
          }
        }
        float mx[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) mx[q] = x[q];
#pragma unroll
        for (int i = 8; i < 128; i += 2) mx[(i >> 1) & 7] = fmax3(mx[(i >> 1) & 7], x[i], x[i + 1]);
        const float tile_max = fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], fmax3(mx[4], mx[5], mx[6]), mx[7]));
        const float mc = tile_max * c;
        const bool raise = mc > m + 4.0f;  // always true on the first tile; keeps 2^(s - m + 4) <= 2^8
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
        // p = 2^(x c - m + 4) in [0, 256]; e4m3, four to a column; published
        // in two halves of 64 keys.
        const float2 c2 = make_float2(c, c), nm2 = make_float2(4.f - m, 4.f - m);
        float2 sum[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) sum[q] = make_float2(0.f, 0.f);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int i = 64 * h + 4 * e;
            const float2 t0 = ffma2(make_float2(x[i], x[i + 1]), c2, nm2);
            const float2 t1 = ffma2(make_float2(x[i + 2], x[i + 3]), c2, nm2);
            const float2 p0 = make_float2(ex2(t0.x), ex2(t0.y)), p1 = make_float2(ex2(t1.x), ex2(t1.y));
            sum[e & 3] = fadd2(sum[e & 3], fadd2(p0, p1));
            pk[e] = pack_e4m3x4(p0.x, p0.y, p1.x, p1.y);
          }
          tmem_st16(tS + 16 * h, pk);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(barP + 8u * h);
        }
        const float2 s01 = fadd2(sum[0], sum[1]), s23 = fadd2(sum[2], sum[3]);
        l = l * alpha + ((s01.x + s23.x) + (s01.y + s23.y));
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      // O = (P V) * v_scale / l in bf16 from registers to this row of O, and
      // lse.  The next unit's first P V, which overwrites O in tensor
      // memory, waits for this warpgroup's next P, published after these
      // loads.
      ok = __all_sync(0xffffffffu, wait_bounded(wc, barO, k & 1, wait_site(0xc3 + s, k)));
      if (!ok) break;
      tc_fence_after();
      const int row = qi * 128 + r;
      const float inv = l > 0.f ? p.o_scale / l : 0.f;
      uint16_t* const orow = p.o + ((size_t)bh * p.Nq + row) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + cc * 32, o);
        tmem_wait_ld();
        reg_fence(o);
        if (row < p.Nq && ATTN_IN_RANGE(((size_t)bh * p.Nq + row) * D + cc * 32 + 31, (size_t)p.B * p.H * p.Nq * D, p, 0x601)) {
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
      if (row < p.Nq && ATTN_IN_RANGE((size_t)bh * p.Nq + row, (size_t)p.B * p.H * p.Nq, p, 0x602))
        p.lse[(size_t)bh * p.Nq + row] = (m + log2f(l) - 4.f) * 0.69314718055994531f;
    }
    setmaxnreg_dec<168>();
  } else {
    setmaxnreg_dec<88>();
    reg_split_sync(384);
    if (warp == 8) {
      // ------------------------------------------------------------ unit queue and TMA producer
      // Takes the next unit from the queue, hands it to the other roles
      // through the unit ring, then loads its Q tiles (once the previous
      // unit's last Q K^T of that tile has read the buffer) and its K_j / V_j
      // into the ring, which runs on across units.
      if (lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        bool ok = true;
        int t = 0;   // ring slot counter over all units: K_j is slot t, V_j slot t + 1
        int nq = 0;  // units whose Q tiles were issued
        for (int k = 0; ok; ++k) {
          const int e = k & 1;
          // CTA b's first unit is unit b (no queue round trip before the first
          // loads); the counter hands out the rest, from gridDim.x on.
          int u = k == 0 ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(p.sched, 1);
          if (u >= p.n_units) u = -1;
          if (k >= 2 && !(ok = wait_bounded(wc, bUe + 8u * e, ((k - 2) >> 1) & 1, wait_site(0xd2, k)))) break;
          unit_ring[e] = u;
          mbar_arrive(bUf + 8u * e);  // (release: the entry is visible to the roles that wait for it)
          if (u < 0) break;
          int bh, mt;
          unit_of(u, bh, mt);
          const int bhk = (bh / p.H) * p.Hkv + (bh % p.H) / p.G;
          const int n1 = ntiles(mt, 1);
          for (int s = 0; s < 2 && ok; ++s) {
            if (k >= 1 && !(ok = wait_bounded(wc, bQe + 8u * s, (k - 1) & 1, wait_site(0xd3 + s, k)))) break;
            mbar_expect_tx(bQ + 8u * s, T::TILE_BYTES);
            tma_load_3d(sQ + s * T::TILE_BYTES, &tmQ, bQ + 8u * s, 0, (2 * mt + s) * 128, bh);
          }
          if (!ok) break;
          nq = k + 1;
          for (int j = 0; j < n1 && ok; ++j) {
            for (int w = 0; w < 2; ++w) {
              const int st = t % T::NSTAGE, rd = t / T::NSTAGE;
              if (rd > 0 && !(ok = wait_bounded(wc, bKVe + 8u * st, (rd - 1) & 1, wait_site(0xd1, t)))) break;
              if (u == 0 && p.debug_drop_p == 2 * j + w + 1) {  // test of the bounded waits only
                ++t;
                continue;
              }
              mbar_expect_tx(bKVf + 8u * st, T::TILE_BYTES);
              tma_load_3d(sKV + st * T::TILE_BYTES, (w == 0) ? &tmK : &tmV, bKVf + 8u * st, 0, j * 128, bhk);
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
      // The bf16 forward's schedule for each unit in turn; the ring slot
      // counter and the P barriers' phases run on across units.
      {
        const uint32_t leader = elect_one();
        constexpr uint32_t IQK = idesc_e4m3_f32(128, 128, false);  // S = Q K^T (both K-major)
        constexpr uint32_t IPV = idesc_e4m3_f32(128, D, true);     // O += P V (A in TMEM, V MN-major)
        const uint32_t tS0 = tmem, tS1 = tmem + 128, tO0 = tmem + 256, tO1 = tmem + 384;
        const uint64_t dQ0 = sdesc_sw128(sQ, 16, 1024), dQ1 = sdesc_sw128(sQ + T::TILE_BYTES, 16, 1024);
        const uint64_t dK0 = sdesc_sw128(sKV, 16, 1024);               // K slots (K-major)
        const uint64_t dV0 = sdesc_sw128(sKV, T::TILE_BYTES, 1024);    // V slots (MN-major; d = one 128-byte chunk)
        // S = Q K^T: K = 32 e4m3 (32 bytes) per instruction inside the 128-byte rows.
        auto qk = [&](uint32_t dS, uint64_t qd, uint64_t kd) {
#pragma unroll
          for (int kk = 0; kk < T::KSTEPS; ++kk)
            mma_f8_ss_p(leader, dS, sdesc_add(qd, kk * 32), sdesc_add(kd, kk * 32), IQK, kk > 0);
        };
        // O += P V over keys [64h, 64h + 64): two K steps of 32 keys; P's
        // K step kk is tensor-memory columns 8 kk .. 8 kk + 7, V's is rows
        // 32 kk .. 32 kk + 31 (4096 bytes).
        auto pv_half = [&](uint32_t dO, uint32_t p_tmem, uint64_t vd, bool acc, int h) {
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            const int kk = 2 * h + k2;
            mma_f8_ts_p(leader, dO, p_tmem + kk * 8, sdesc_add(vd, kk * 4096), IPV, (acc || kk > 0) ? 1u : 0u);
          }
        };
        auto wait_all = [&](uint32_t bar, uint32_t parity, int site) {
          return __all_sync(0xffffffffu, wait_bounded(wc, bar, parity, site));
        };
        bool ok = true;
        int tb = 0;                 // ring index of this unit's K_0
        uint32_t np0 = 0, np1 = 0;  // P tiles each softmax warpgroup has published so far
        for (int k = 0; ok; ++k) {
          const int u = next_unit(k, ok);
          if (u < 0) break;
          int bh, mt;
          unit_of(u, bh, mt);
          const int n0 = ntiles(mt, 0), n1 = ntiles(mt, 1);  // key tiles of query tiles 0 / 1 (n0 <= n1)
          const uint32_t qp = k & 1;
          const uint64_t dKf = sdesc_add(dK0, (tb % T::NSTAGE) * T::TILE_BYTES);
          if (!(ok = wait_all(bKVf + 8u * (tb % T::NSTAGE), (tb / T::NSTAGE) & 1, wait_site(0xe1, k)) &&
                     wait_all(bQ, qp, wait_site(0xe2, k))))
            break;
          tc_fence_after();
          qk(tS0, dQ0, dKf);
          mma_commit_p(leader, bS);
          if (n0 == 1) mma_commit_p(leader, bQe);  // Q tile 0 read for the last time
          if (!(ok = wait_all(bQ + 8u, qp, wait_site(0xe3, k)))) break;
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
            if (!(ok = wait_all(bKVf + 8u * sv, (t / T::NSTAGE) & 1, wait_site(0xe4, j)))) break;
            if (j < n0) {
              if (!(ok = wait_all(bP, np0 & 1, wait_site(0xe6, j)))) break;  // keys 0-63
              tc_fence_after();
              pv_half(tO0, tS0, vd, j > 0, 0);
              if (!(ok = wait_all(bP + 8u, np0 & 1, wait_site(0xe8, j)))) break;  // keys 64-127
              tc_fence_after();
              pv_half(tO0, tS0, vd, j > 0, 1);
              ++np0;
              if (j + 1 < n0) {
                if (!(ok = wait_all(bKVf + 8u * sk, ((t + 1) / T::NSTAGE) & 1, wait_site(0xe5, j)))) break;
                tc_fence_after();
                qk(tS0, dQ0, kd);
                mma_commit_p(leader, bS);
                if (j + 2 == n0) mma_commit_p(leader, bQe);
              } else {
                mma_commit_p(leader, bO);
              }
            }
            if (!(ok = wait_all(bP + 16u, np1 & 1, wait_site(0xe7, j)))) break;
            tc_fence_after();
            pv_half(tO1, tS1, vd, j > 0, 0);
            if (!(ok = wait_all(bP + 24u, np1 & 1, wait_site(0xe9, j)))) break;
            tc_fence_after();
            pv_half(tO1, tS1, vd, j > 0, 1);
            ++np1;
            if (next) {
              if (!(ok = wait_all(bKVf + 8u * sk, ((t + 1) / T::NSTAGE) & 1, wait_site(0xea, j)))) break;
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

// Queue slots (next unit, CTAs done), one per launch in flight (see
// attn_fwd_persist.cu).
constexpr int kF8QueueSlots = 256;
__device__ int g_fp8_queue[kF8QueueSlots][2];

int* fp8_queue_slot() {
  static std::atomic<unsigned> next{0};
  static int* base[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (base[dev] == nullptr) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_fp8_queue) != cudaSuccess) return nullptr;
    base[dev] = static_cast<int*>(a);
  }
  return base[dev] + 2 * (next.fetch_add(1) % kF8QueueSlots);
}

template <int D, bool C>
cudaError_t launch_fp8_persist_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                         cudaStream_t stream) {
  using F = F8<D>;
  auto kern = fwd_fp8_persist_kernel<D, C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, F::SMEM);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidValue;
  FwdParams pc = p;
  pc.n_units = p.n_mtiles * p.B * p.H;
  pc.tail = !C ? 1 : order_tail(p.n_mtiles, p.B * p.H, p.G);  // (non-causal: every level alike)
  pc.sched = fp8_queue_slot();
  if (pc.sched == nullptr) return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)min(pc.n_units, sms);  // one CTA per SM
  kern<<<grid, F::THREADS, F::SMEM, stream>>>(tq, tk, tv, pc);
  return cudaGetLastError();
}

template <int D, bool C>
cudaError_t launch_fp8_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                         cudaStream_t stream) {
  using F = F8<D>;
  auto kern = fwd_fp8_kernel<D, C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, F::SMEM);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)p.n_mtiles * (unsigned)(p.B * p.H);
  FwdParams pc = p;
  pc.tail = !C ? 1 : order_tail(p.n_mtiles, p.B * p.H, p.G);  // (non-causal: every level alike)
  kern<<<grid, F::THREADS, F::SMEM, stream>>>(tq, tk, tv, pc);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_fp8(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const FwdParams& p, cudaStream_t stream) {
  switch (d) {
    case 64:
      return causal ? launch_fp8_persist_t<64, true>(tq, tk, tv, p, stream) : launch_fp8_persist_t<64, false>(tq, tk, tv, p, stream);
    case 96:
      return causal ? launch_fp8_persist_t<96, true>(tq, tk, tv, p, stream) : launch_fp8_persist_t<96, false>(tq, tk, tv, p, stream);
    case 128:
      return causal ? launch_fp8_t<128, true>(tq, tk, tv, p, stream) : launch_fp8_t<128, false>(tq, tk, tv, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sdpa
