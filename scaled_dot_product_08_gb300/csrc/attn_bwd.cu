// attn_bwd.cu — backward pass of exact attention on sm_103a.
//
// Method (page "Flash Attention原理：分块计算与重计算，如何降低O(n^2)的显存占用",
// §五 and FAQ Q19): the forward kept only O and the per-row logsumexp; the
// backward recomputes each probability tile from them instead of reading a
// stored P, and applies the chain rule of softmax-then-matmul:
//     P  = exp(scale * Q K^T - lse)        (recomputed per tile)
//     dV = P^T dO,  dP = dO V^T,  D = rowsum(dO * O),
//     dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
//
// Three kernels on the caller's stream:
//   bwd_pre     -D = -rowsum(dO * O) (fp32), -lse2 = -lse * log2(e) (-inf on
//               the padding rows of each head), dQ accumulator := 0
//   bwd_main    one CTA per (key tile j, batch, K/V head); loops over the
//               GQA group's query heads and the query tiles i (i >= j when
//               causal).  dK_j and dV_j accumulate in tensor memory; dQ_i
//               contributions are added to a float32 accumulator in global
//               memory with TMA bulk reductions.
//   bwd_convert dQ accumulator -> bf16 dQ
//
// bwd_main warp roles (384 threads = 3 warpgroups):
//   warps 0-3   compute: S^T -> P^T (written to TMEM as the A operand of the
//               dV MMA), dP^T -> dS^T (written to shared memory, the A
//               operand of the dK and dQ MMAs); dK/dV epilogue
//   warps 4-7   dQ drain: TMEM -> shared memory -> TMA reduce-add
//   warp  8     TMA producer: K_j, V_j once; Q_i, dO_i, lse2_i, D_i per step
//   warp  9     MMA issuer (one thread)
//   warps 10-11 idle
// setmaxnreg: compute 240, drain 160, producer/MMA 104 registers per thread
// (128 * (240 + 160 + 104) = 384 * 168, the launch allocation).
// Tensor memory: [0,128) S^T / P^T, [128,256) dP^T / dQ_i, [256,256+d) dK,
// [384,384+d) dV.  All score tiles are 128 x 128 (keys x queries).
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {

// ------------------------------------------------------------------ preprocess
// One warp per (head, padded row).  Row i < N: stores -D = -(dO_i . O_i)
// (fp32) and -lse_i * log2(e).  Row i >= N: -D = 0 and -lse2 = -inf (so P = 0
// there).  The negated values let the grad kernel form P and dP - D with one
// packed FMA / add per pair.  Every row of the dQ accumulator is zeroed.
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdParams p) {
  const long long rows = (long long)p.B * p.H * p.Npad;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const long long bh = row / p.Npad;
  const int i = (int)(row % p.Npad);
  float4* acc = reinterpret_cast<float4*>(p.dq_acc + row * p.d);
  for (int c = lane; c < p.d / 4; c += 32) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  float dot = 0.f;
  if (i < p.N) {
    const size_t off = ((size_t)bh * p.N + i) * p.d;
    if (lane * 8 < p.d) {
      const uint4 o = *reinterpret_cast<const uint4*>(p.o + off + lane * 8);
      const uint4 g = *reinterpret_cast<const uint4*>(p.dout + off + lane * 8);
      const uint32_t ow[4] = {o.x, o.y, o.z, o.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[e]));
        const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[e]));
        dot = fmaf(of.x, gf.x, dot);
        dot = fmaf(of.y, gf.y, dot);
      }
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, s);
  }
  if (lane == 0) {
    p.dvec[row] = (i < p.N) ? -dot : 0.f;
    p.lse2[row] = (i < p.N) ? -p.lse[(size_t)bh * p.N + i] * 1.4426950408889634f : -INFINITY;
  }
}

// ------------------------------------------------------------------ convert
// dQ (bf16) = dQ accumulator (fp32) for the N real rows of each head.
__global__ void __launch_bounds__(256) bwd_convert_kernel(const BwdParams p) {
  const long long rows = (long long)p.B * p.H * p.N;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const long long bh = row / p.N;
  const int i = (int)(row % p.N);
  const float* src = p.dq_acc + ((size_t)bh * p.Npad + i) * p.d;
  uint16_t* dst = p.dq + (size_t)row * p.d;
  for (int c = lane * 4; c < p.d; c += 128) {
    const float4 a = *reinterpret_cast<const float4*>(src + c);
    uint2 w;
    w.x = pack_bf16(a.x, a.y);
    w.y = pack_bf16(a.z, a.w);
    *reinterpret_cast<uint2*>(dst + c) = w;
  }
}

// ------------------------------------------------------------------ main
template <int D>
struct BwdTraits {
  static constexpr int NB = (D + 63) / 64;
  static constexpr int BLOCK_BYTES = 128 * 128;
  static constexpr int TILE_BYTES = NB * BLOCK_BYTES;  // one [128 rows x d] bf16 tile
  static constexpr int KSTEPS = D / 16;
  static constexpr int DS_BYTES = 2 * BLOCK_BYTES;     // dS^T: 128 keys x 128 queries, any d
  static constexpr int VEC_BYTES = 1024;               // lse2[128] + D[128]
  static constexpr int NBAR = 1 + 2 + 2 + 1 + 1 + 1 + 1 + 1 + 1 + 1 + 1 + 1;
  // K, V, Q[2], dO[2], dS^T, then vectors, barriers, misc
  static constexpr int TILES_BYTES = 6 * TILE_BYTES + DS_BYTES;
  static constexpr int SMEM = TILES_BYTES + 2 * VEC_BYTES + NBAR * 8 + 16;
  static constexpr int THREADS = 384;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                    const __grid_constant__ CUtensorMap tmdQacc, const BwdParams p) {
  using T = BwdTraits<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = smem_u32(smem_raw);
  // The layout needs a 1024-byte aligned start (128-byte swizzle atoms); the
  // dynamic shared window starts there in practice.  Refuse to run otherwise.
  if (base & 1023u) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0, kDevMisaligned);
    return;
  }
  const uint32_t sK = base;
  const uint32_t sV = sK + T::TILE_BYTES;
  const uint32_t sQ = sV + T::TILE_BYTES;            // [2]
  const uint32_t sdO = sQ + 2 * T::TILE_BYTES;       // [2]
  const uint32_t sDS = sdO + 2 * T::TILE_BYTES;      // dS^T, bf16, [keys][queries]
  const uint32_t sVec = sDS + T::DS_BYTES;           // [2] x {lse2[128], D[128]}
  const uint32_t sBar = sVec + 2 * T::VEC_BYTES;
  const uint32_t bKV = sBar;
  const uint32_t bQf = bKV + 8;     // qdo_full[2]
  const uint32_t bQe = bQf + 16;    // qdo_empty[2]
  const uint32_t bS = bQe + 16;     // S^T ready
  const uint32_t bP = bS + 8;       // P^T in TMEM (128 arrivals)
  const uint32_t bDs = bP + 8;      // dS^T in smem (128 arrivals)
  const uint32_t bDqf = bDs + 8;    // dQ_i in TMEM
  const uint32_t bDqe = bDqf + 8;   // dQ_i drained (128 arrivals)
  const uint32_t bFin = bDqe + 8;   // every MMA done
  const uint32_t bDrain = bFin + 8;
  const uint32_t bDp = bDrain + 8;  // dP^T ready
  const uint32_t bStg = bDp + 8;    // dQ_i staged in shared memory (128 arrivals)
  uint8_t* const misc = smem_raw + (sBar - base) + 8 * T::NBAR;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  const float* const vec_g = reinterpret_cast<const float*>(smem_raw + (sVec - base));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkv = p.nq;
  const int bhk = blockIdx.x / nkv;           // b * Hkv + hk
  const int j = blockIdx.x % nkv;             // key tile (0 = most causal work)
  const int b = bhk / p.Hkv, hk = bhk % p.Hkv;
  const int i0 = CAUSAL ? j : 0;
  const int ni = p.nq - i0;                   // query tiles per head
  const int total = p.G * ni;                 // steps: (head in group) x (query tile)

  if (threadIdx.x == 0) {
    mbar_init(bKV, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bQf + 8u * s, 1);
      mbar_init(bQe + 8u * s, 1);
    }
    mbar_init(bS, 1);
    mbar_init(bDp, 1);
    mbar_init(bStg, 128);
    mbar_init(bP, 128);
    mbar_init(bDs, 128);
    mbar_init(bDqf, 1);
    mbar_init(bDqe, 128);
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

  if (warp < 4) {
    setmaxnreg_inc<240>();
    reg_split_sync(384);
    // -------------------------------------------------------------- compute
    const int r = threadIdx.x;  // key row within the tile == TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tS = tmem + lane_off, tdP = tmem + 128 + lane_off;
    const float c = p.scale_log2;
    const float2 c2 = make_float2(c, c);
    bool ok = true;
    for (int it = 0; it < total; ++it) {
      const int i = i0 + it % ni;
      const float* vl = vec_g + (it & 1) * (T::VEC_BYTES / 4);  // -lse2[128], then -D[128]
      // The lse2 / D vectors come from the bulk copy of this step: observe
      // its barrier (already complete by now) before reading them.
      ok = __all_sync(0xffffffffu, wait_bounded(wc, bQf + 8u * (it & 1), (it >> 1) & 1, wait_site(0x11, it)) &&
                                       wait_bounded(wc, bS, it & 1, wait_site(0x12, it)));
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
        for (int e = 0; e < 32; ++e) {
          x[e] = __uint_as_float(ra[e]);
          x[32 + e] = __uint_as_float(rb[e]);
          x[64 + e] = __uint_as_float(rc[e]);
          x[96 + e] = __uint_as_float(rd[e]);
        }
      }
      // P^T[r][q] = exp2(S^T * scale * log2e - lse2[q]); masked (key > query
      // on the diagonal tile) entries are exactly 0.
#pragma unroll
      for (int q4 = 0; q4 < 32; ++q4) {
        const float4 l4 = *reinterpret_cast<const float4*>(vl + 4 * q4);
        const float2 t0 = ffma2(make_float2(x[4 * q4 + 0], x[4 * q4 + 1]), c2, make_float2(l4.x, l4.y));
        const float2 t1 = ffma2(make_float2(x[4 * q4 + 2], x[4 * q4 + 3]), c2, make_float2(l4.z, l4.w));
        x[4 * q4 + 0] = ex2(t0.x);
        x[4 * q4 + 1] = ex2(t0.y);
        x[4 * q4 + 2] = ex2(t1.x);
        x[4 * q4 + 3] = ex2(t1.y);
      }
      if (CAUSAL && i == j) {
#pragma unroll
        for (int q = 0; q < 128; ++q)
          if (r > q) x[q] = 0.f;
      }
      // P^T as bf16 pairs: written to TMEM for the dV MMA and kept in
      // registers for dS.
      uint32_t pa[32], pb[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        pa[e] = pack_bf16(x[2 * e], x[2 * e + 1]);
        pb[e] = pack_bf16(x[64 + 2 * e], x[64 + 2 * e + 1]);
      }
      tmem_st32(tS, pa);
      tmem_st32(tS + 32, pb);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bP);
      // dS^T[r][q] = P^T[r][q] * (dP^T[r][q] - D[q]) -> bf16 -> smem (128-byte
      // swizzled rows: block q/64, 16-byte chunk (q%64)/8).  The softmax scale
      // is applied later, to dK in its epilogue and to dQ in the drain.
      ok = __all_sync(0xffffffffu, wait_bounded(wc, bDp, it & 1, wait_site(0x14, it)));
      if (!ok) break;
      tc_fence_after();
      uint32_t g0[32], g1[32], g2[32], g3[32];
      tmem_ld32(tdP + 0, g0);
      tmem_ld32(tdP + 32, g1);
      tmem_ld32(tdP + 64, g2);
      tmem_ld32(tdP + 96, g3);
      tmem_wait_ld();
      reg_fence(g0);
      reg_fence(g1);
      reg_fence(g2);
      reg_fence(g3);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const uint32_t* g = cc == 0 ? g0 : cc == 1 ? g1 : cc == 2 ? g2 : g3;
        const uint32_t* pk = (cc < 2) ? pa : pb;
        const float4* Dv = reinterpret_cast<const float4*>(vl + 128 + cc * 32);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t w[4];
          const float4 da = Dv[2 * q4], db = Dv[2 * q4 + 1];
          const float2 dd[4] = {make_float2(da.x, da.y), make_float2(da.z, da.w), make_float2(db.x, db.y),
                                make_float2(db.z, db.w)};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int q = q4 * 8 + 2 * e;  // column within this 32-column chunk
            const uint32_t pp = pk[((cc & 1) * 32 + q) >> 1];
            const float2 pf = make_float2(__uint_as_float(pp << 16), __uint_as_float(pp & 0xffff0000u));
            const float2 dpd = fadd2(make_float2(__uint_as_float(g[q]), __uint_as_float(g[q + 1])), dd[e]);
            const float2 ds = fmul2(pf, dpd);
            w[e] = pack_bf16(ds.x, ds.y);
          }
          st_shared_v4(sDS + (cc >> 1) * T::BLOCK_BYTES + sw128_offset(r, (cc & 1) * 4 + q4), w[0], w[1], w[2],
                       w[3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bDs);
    }
    // ------------------------------------------------------------ dK / dV out
    if (ok) ok = __all_sync(0xffffffffu, wait_bounded(wc, bFin, 0, wait_site(0x13, total)));
    const uint32_t stage_dv = sDS, stage_dk = sK;  // both free once every MMA is done
    if (ok) {
      tc_fence_after();
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t src = tmem + (which ? 256u : 384u) + lane_off;
        const uint32_t dst = which ? stage_dk : stage_dv;
        const float2 f2 = which ? make_float2(p.scale, p.scale) : make_float2(1.f, 1.f);  // dK = scale dS^T Q
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(src + cc * 32, o);
          tmem_wait_ld();
          reg_fence(o);
          const int blk = (cc * 32) / 64, ch0 = ((cc * 32) % 64) / 8;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 t = fmul2(make_float2(__uint_as_float(o[q4 * 8 + 2 * e]),
                                                 __uint_as_float(o[q4 * 8 + 2 * e + 1])), f2);
              w[e] = pack_bf16(t.x, t.y);
            }
            st_shared_v4(dst + blk * T::BLOCK_BYTES + sw128_offset(r, ch0 + q4), w[0], w[1], w[2], w[3]);
          }
        }
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128);
    if (ok && r == 0) {
      for (int cb = 0; cb < T::NB; ++cb) {
        tma_store_3d(&tmdV, stage_dv + cb * T::BLOCK_BYTES, cb * 64, j * 128, bhk);
        tma_store_3d(&tmdK, stage_dk + cb * T::BLOCK_BYTES, cb * 64, j * 128, bhk);
      }
      bulk_commit();
      bulk_wait_read_all();
    }
    setmaxnreg_dec<168>();
  } else if (warp < 8) {
    setmaxnreg_dec<160>();
    reg_split_sync(384);
    // -------------------------------------------------------------- dQ drain
    const int q = threadIdx.x - 128;  // query row within the tile == TMEM lane
    const uint32_t tQ = tmem + 128 + ((uint32_t)((warp - 4) * 32) << 16);
    const float2 sc2 = make_float2(p.scale, p.scale);  // dQ = scale dS K
    // dQ_i goes out through the step's Q / dO shared-memory stage, which is
    // idle once dQ_i is final (every MMA that read it has completed): fp32,
    // boxes of 32 columns x 128 rows with the 128-byte swizzle, added into
    // the accumulator by TMA reductions.  The stage is then handed back to
    // the producer (qdo_empty).
    constexpr int NBOX = D / 32;
    for (int it = 0; it < total; ++it) {
      const int h = hk * p.G + it / ni, i = i0 + it % ni;
      const int st = it & 1;
      if (!__all_sync(0xffffffffu, wait_bounded(wc, bDqf, it & 1, wait_site(0x21, it)))) break;
      tc_fence_after();
      uint32_t g[NBOX][32];
#pragma unroll
      for (int cc = 0; cc < NBOX; ++cc) tmem_ld32(tQ + cc * 32, g[cc]);
      tmem_wait_ld();
#pragma unroll
      for (int cc = 0; cc < NBOX; ++cc) reg_fence(g[cc]);
      tc_fence_before();
      mbar_arrive(bDqe);  // TMEM columns free for the next dP^T
#pragma unroll
      for (int cc = 0; cc < NBOX; ++cc) {
        const uint32_t box = (cc < T::NB) ? sQ + st * T::TILE_BYTES + cc * T::BLOCK_BYTES
                                          : sdO + st * T::TILE_BYTES + (cc - T::NB) * T::BLOCK_BYTES;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          const float2 a0 = fmul2(make_float2(__uint_as_float(g[cc][4 * c8]), __uint_as_float(g[cc][4 * c8 + 1])), sc2);
          const float2 a1 = fmul2(make_float2(__uint_as_float(g[cc][4 * c8 + 2]), __uint_as_float(g[cc][4 * c8 + 3])), sc2);
          st_shared_v4(box + sw128_offset(q, c8), __float_as_uint(a0.x), __float_as_uint(a0.y), __float_as_uint(a1.x),
                       __float_as_uint(a1.y));
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bStg);
      // One thread waits (bounded) for all 128 to have staged, then reduces.
      if (q == 0 && wait_bounded(wc, bStg, it & 1, wait_site(0x22, it))) {
        const int bh = b * p.H + h;
#pragma unroll
        for (int cc = 0; cc < NBOX; ++cc) {
          const uint32_t box = (cc < T::NB) ? sQ + st * T::TILE_BYTES + cc * T::BLOCK_BYTES
                                            : sdO + st * T::TILE_BYTES + (cc - T::NB) * T::BLOCK_BYTES;
          tma_reduce_add_3d(&tmdQacc, box, cc * 32, i * 128, bh);
        }
        bulk_commit();
        bulk_wait_read_all();
        mbar_arrive(bQe + 8u * st);
      }
    }
    if (q == 0) bulk_wait_all();  // every reduction has landed before the CTA exits
    setmaxnreg_inc<168>();
  } else {
    setmaxnreg_dec<104>();
    reg_split_sync(384);
    if (warp == 8) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmdO);
        mbar_expect_tx(bKV, 2 * T::TILE_BYTES);
        for (int cb = 0; cb < T::NB; ++cb) {
          tma_load_3d(sK + cb * T::BLOCK_BYTES, &tmK, bKV, cb * 64, j * 128, bhk);
          tma_load_3d(sV + cb * T::BLOCK_BYTES, &tmV, bKV, cb * 64, j * 128, bhk);
        }
        int issued = 0;
        for (int it = 0; it < total; ++it) {
          const int st = it & 1, rd = it >> 1;
          if (rd > 0 && !wait_bounded(wc, bQe + 8u * st, (rd - 1) & 1, wait_site(0x31, it))) break;
          const int h = hk * p.G + it / ni, i = i0 + it % ni;
          const int bh = b * p.H + h;
          const uint32_t bar = bQf + 8u * st;
          mbar_expect_tx(bar, 2 * T::TILE_BYTES + T::VEC_BYTES);
          for (int cb = 0; cb < T::NB; ++cb) {
            tma_load_3d(sQ + st * T::TILE_BYTES + cb * T::BLOCK_BYTES, &tmQ, bar, cb * 64, i * 128, bh);
            tma_load_3d(sdO + st * T::TILE_BYTES + cb * T::BLOCK_BYTES, &tmdO, bar, cb * 64, i * 128, bh);
          }
          const size_t voff = (size_t)bh * p.Npad + (size_t)i * 128;
          bulk_load(sVec + st * T::VEC_BYTES, p.lse2 + voff, 512, bar);
          bulk_load(sVec + st * T::VEC_BYTES + 512, p.dvec + voff, 512, bar);
          issued = it + 1;
        }
        // Every copy issued above has landed before the CTA may exit.
        wait_drain(bKV, 0, p.limit_ns);
        for (int st = 0; st < 2 && st < issued; ++st) {
          const int last = ((issued - 1 - st) / 2) * 2 + st;
          wait_drain(bQf + 8u * st, (last >> 1) & 1, p.limit_ns);
        }
      }
      __syncwarp();
    } else if (warp == 9) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t I_SS = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
        constexpr uint32_t I_TB = idesc_bf16_f32(128, D, false, true);     // dV (A in TMEM), dK
        constexpr uint32_t I_MM = idesc_bf16_f32(128, D, true, true);      // dQ (A = dS, MN-major)
        const uint32_t tS = tmem, tdP = tmem + 128, tdK = tmem + 256, tdV = tmem + 384;
        // D[128 x 128] = A[128 x d] * B[128 x d]^T with both K-major tiles.
        auto mma_kk = [&](uint32_t dst, uint32_t a_tile, uint32_t b_tile) {
#pragma unroll
          for (int kk = 0; kk < T::KSTEPS; ++kk) {
            const uint32_t off = (kk >> 2) * T::BLOCK_BYTES + (kk & 3) * 32;
            mma_ss(dst, sdesc_sw128(a_tile + off, 16, 1024), sdesc_sw128(b_tile + off, 16, 1024), I_SS, kk > 0);
          }
        };
        // Issue order per step i (stage st): dV(i), S^T(i+1), dK(i), dQ(i),
        // dP^T(i+1).  S^T(i+1) overwrites P^T(i) in TMEM only after dV(i),
        // which was issued first (MMAs from one thread run in order), so
        // the softmax of step i+1 overlaps the dK / dQ MMAs of step i.
        bool ok = wait_bounded(wc, bKV, 0, wait_site(0x41, 0)) &&
                  wait_bounded(wc, bQf, 0, wait_site(0x42, 0));
        if (ok) {
          tc_fence_after();
          mma_kk(tS, sK, sQ);  // S^T_0 = K Q_0^T
          mma_commit(bS);
          mma_kk(tdP, sV, sdO);  // dP^T_0 = V dO_0^T
          mma_commit(bDp);
        }
        for (int it = 0; it < total && ok; ++it) {
          const int st = it & 1, sn = st ^ 1;
          const bool nx = it + 1 < total;
          const uint32_t q_t = sQ + st * T::TILE_BYTES, do_t = sdO + st * T::TILE_BYTES;
          const uint32_t q_n = sQ + sn * T::TILE_BYTES, do_n = sdO + sn * T::TILE_BYTES;
          if (!(ok = wait_bounded(wc, bP, it & 1, wait_site(0x44, it)))) break;
          tc_fence_after();
          // dV += P^T dO_i: A = P^T (TMEM, bf16 pairs), B = dO_i (MN-major)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tdV, tS + kk * 8, sdesc_sw128(do_t + kk * 2048, T::BLOCK_BYTES, 1024), I_TB,
                   (it > 0 || kk > 0) ? 1u : 0u);
          if (nx) {
            if (!(ok = wait_bounded(wc, bQf + 8u * sn, ((it + 1) >> 1) & 1, wait_site(0x46, it)))) break;
            tc_fence_after();
            mma_kk(tS, sK, q_n);  // S^T_{i+1}
            mma_commit(bS);
          }
          if (!(ok = wait_bounded(wc, bDs, it & 1, wait_site(0x45, it)))) break;
          tc_fence_after();
          // dK += dS^T Q_i: A = dS^T (K-major over queries), B = Q_i (MN-major)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tdK, sdesc_sw128(sDS + (kk >> 2) * T::BLOCK_BYTES + (kk & 3) * 32, 16, 1024),
                   sdesc_sw128(q_t + kk * 2048, T::BLOCK_BYTES, 1024), I_TB, (it > 0 || kk > 0) ? 1u : 0u);
          // dQ_i = dS K_j: A = dS (queries contiguous: MN-major), B = K_j (MN-major)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tdP, sdesc_sw128(sDS + kk * 2048, T::BLOCK_BYTES, 1024),
                   sdesc_sw128(sK + kk * 2048, T::BLOCK_BYTES, 1024), I_MM, kk > 0 ? 1u : 0u);
          mma_commit(bDqf);  // the drain releases the Q / dO stage after staging dQ_i in it
          if (nx) {
            if (!(ok = wait_bounded(wc, bDqe, it & 1, wait_site(0x43, it)))) break;
            tc_fence_after();
            mma_kk(tdP, sV, do_n);  // dP^T_{i+1}
            mma_commit(bDp);
          }
        }
        if (ok) mma_commit(bFin);
        mma_commit(bDrain);  // fires once every MMA issued above has finished
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

size_t bwd_smem_bytes(int d) {
  switch (d) {
    case 64: return BwdTraits<64>::SMEM;
    case 96: return BwdTraits<96>::SMEM;
    case 128: return BwdTraits<128>::SMEM;
    default: return 0;
  }
}

template <int D, bool C>
static cudaError_t launch_main_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                                 const CUtensorMap& tdqa, const BwdParams& p, cudaStream_t stream) {
  auto kern = bwd_main_kernel<D, C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdTraits<D>::SMEM);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)p.nq * (unsigned)(p.B * p.Hkv);
  kern<<<grid, BwdTraits<D>::THREADS, BwdTraits<D>::SMEM, stream>>>(tq, tk, tv, tdo, tdk, tdv, tdqa, p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep(const BwdParams& p, cudaStream_t stream) {
  const long long rows = (long long)p.B * p.H * p.Npad;
  bwd_pre_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_grad(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                            const CUtensorMap& tdqa, const BwdParams& p, cudaStream_t stream) {
  switch (d) {
    case 64: return causal ? launch_main_t<64, true>(tq, tk, tv, tdo, tdk, tdv, tdqa, p, stream)
                           : launch_main_t<64, false>(tq, tk, tv, tdo, tdk, tdv, tdqa, p, stream);
    case 96: return causal ? launch_main_t<96, true>(tq, tk, tv, tdo, tdk, tdv, tdqa, p, stream)
                           : launch_main_t<96, false>(tq, tk, tv, tdo, tdk, tdv, tdqa, p, stream);
    case 128: return causal ? launch_main_t<128, true>(tq, tk, tv, tdo, tdk, tdv, tdqa, p, stream)
                            : launch_main_t<128, false>(tq, tk, tv, tdo, tdk, tdv, tdqa, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bwd_dq(const BwdParams& p, cudaStream_t stream) {
  const long long rows = (long long)p.B * p.H * p.N;
  bwd_convert_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace sdpa
