// attn_decode.cu — decode attention against a KV cache, split over the keys.
//
// Method: exact softmax(scale Q K^T) V for a block of Nq new queries per head
// against Nk cached keys/values (page "Flash Attention原理：分块计算与重计算，
// 如何降低O(n^2)的显存占用", FAQ on inference with a KV cache), computed in
// key chunks whose normalised partial outputs are combined with the
// two-block merge of §四 generalised to any number of blocks:
//     lse = ln sum_s exp(lse_s),   O = sum_s exp(lse_s - lse) O_s.
// Causal: query t of the block sits at position Nk - Nq + t (the new tokens
// end the sequence) and sees keys 0 .. Nk - Nq + t.
//
// A decode step reads every cached key and value once for the R = G * Nq
// query rows of their K/V head (the head's G query heads times the Nq new
// tokens), so it is bound by HBM bandwidth.  The two contractions are still
// dense (R x 128 keys x d per tile), and running them on the tensor cores
// keeps the instruction stream short enough for the SM to stream K/V at full
// bandwidth (an FMA-pipe version of this kernel issued ~3,400 warp
// instructions per 64 KB tile and reached ~20% of HBM bandwidth).
//
// Two kernels on the caller's stream:
//   decode_split  one CTA per (key chunk, batch * K/V head), 192 threads,
//                 two CTAs per SM (97 KB shared memory, 256 TMEM columns
//                 each), so one CTA's loads overlap the other's work:
//                   warps 0-3  softmax, one thread per query row (TMEM lane);
//                              rows >= R (up to 128 rows per K/V head are
//                              live) are padding and only keep the phases
//                   warp 4     TMA producer: the group's 128 query rows
//                              (rows >= R are whatever follows; their
//                              results are never read), then K_j, V_j
//                   warp 5     MMA issuer (one elected lane issues)
//                 Per 128-key tile j: S = Q K_j^T (TMEM, M = 128 query rows,
//                 N = 128 keys), online softmax in base 2 with a lazily
//                 raised running max (as in the forward kernel), P as bf16
//                 pairs over S, O += P V_j (A = P in TMEM).  The chunk's
//                 normalised O and its lse go to the workspace (lse = -inf,
//                 O = 0 when no key of the chunk is visible to the row).
//   decode_merge  one CTA per (batch, head, query): the lse-weighted merge
//                 of the chunks -> O (bf16) and lse.
// Tensor memory (256 columns per CTA): S / P [0,128), O [128,128+d).
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {

namespace {

constexpr int kDecThreads = 192;

template <int D>
struct DecTraits {
  static constexpr int NB = (D + 63) / 64;
  static constexpr int BLOCK_BYTES = 128 * 128;        // [128 rows x 64 columns] bf16, swizzled
  static constexpr int TILE_BYTES = NB * BLOCK_BYTES;  // one [128 rows x d] tile
  static constexpr int KSTEPS = D / 16;
  static constexpr int NBAR = 10;
  static constexpr int SMEM = 1024 + 3 * TILE_BYTES + NBAR * 8 + 16;  // Q, K, V
};

}  // namespace

// PAGED: the cache is paged (DecParams' page fields): per-sequence key
// counts, tiles gathered from the block table, and the rows of a last tile
// past the sequence zeroed before the P V product (their cache slots may
// hold anything, and 0 * NaN is NaN).
template <int D, bool CAUSAL, bool PAGED>
__global__ void __launch_bounds__(kDecThreads, 2)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const DecParams p) {
  using T = DecTraits<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t sQ = base, sK = sQ + T::TILE_BYTES, sV = sK + T::TILE_BYTES;
  const uint32_t sBar = sV + T::TILE_BYTES;
  const uint32_t bQ = sBar;          // Q loaded
  const uint32_t bKf = bQ + 8;       // K_j loaded (phase j)
  const uint32_t bKe = bKf + 8;      // K slot free: S_j done (phase j)
  const uint32_t bVf = bKe + 8;      // V_j loaded
  const uint32_t bVe = bVf + 8;      // V slot free: P V_j done
  const uint32_t bS = bVe + 8;       // S_j ready (phase j)
  const uint32_t bP = bS + 8;        // P_j in TMEM (128 arrivals)
  const uint32_t bO = bP + 8;        // the chunk's last P V done
  const uint32_t bDrain = bO + 8;
  uint8_t* const misc = gbase + (sBar - base) + 8 * T::NBAR;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, bhk = blockIdx.y;
  const int b = bhk / p.Hkv, hk = bhk % p.Hkv;
  const int R = p.G * p.Nq;                    // live query rows
  const int qrow0 = (b * p.H + hk * p.G) * p.Nq;  // first query row of the group in (B*H*Nq, d)
  // Cached keys of this batch element: Nk, or its sequence length (paged;
  // a length past the table's capacity is an error, reported and clamped).
  int nkb = p.Nk;
  if (PAGED) {
    nkb = p.seq_lens[b];
    if (nkb < 0 || nkb > p.Nk) {
      if (threadIdx.x == 0 && split == 0) atomicCAS(p.status, 0, kDevBadSeqlens);
      nkb = max(0, min(nkb, p.Nk));
    }
  }
  const int key0 = split * p.split_keys;
  const int key1 = min(nkb, key0 + p.split_keys);
  const int n = max(0, (key1 - key0 + 127) / 128);  // key tiles of this chunk (0: a chunk past the sequence)

  if (threadIdx.x == 0) {
    mbar_init(bQ, 1);
    mbar_init(bKf, 1);
    mbar_init(bKe, 1);
    mbar_init(bVf, 1);
    mbar_init(bVe, 1);
    mbar_init(bS, 1);
    mbar_init(bP, 128);
    mbar_init(bO, 1);
    mbar_init(bDrain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  const WaitCtx wc{abort_flag, p.status, p.limit_ns, p.info};

  if (warp < 4) {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x;            // query row == TMEM lane
    const bool live = r < R;
    const bool warp_live = warp * 32 < R;  // rows >= R only keep the phases
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tS = tmem + lane_off, tO = tmem + 128 + lane_off;
    const float c = p.scale_log2;
    // One past the last key this row may see: the chunk end, and for causal
    // rows position Nk - Nq + t (plus one).
    const int vis_end = CAUSAL ? min(key1, nkb - p.Nq + (live ? r % p.Nq : 0) + 1) : key1;
    float m = -INFINITY, l = 0.f;  // running max (scaled, base 2), running sum
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      ok = __all_sync(0xffffffffu, wait_bounded(wc, bS, j & 1, wait_site(0xc1, j)));
      if (!ok) break;
      tc_fence_after();
      if (warp_live) {
        const int kt = key0 + j * 128;                      // key of column 0
        const int lim = vis_end - kt;                       // columns >= lim are masked
        // Pass 1: row max over the tile (two loads of 64 columns).
        float mx = -INFINITY;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t xa[32], xb[32];
          tmem_ld32(tS + 64 * h, xa);
          tmem_ld32(tS + 64 * h + 32, xb);
          tmem_wait_ld();
          reg_fence(xa);
          reg_fence(xb);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int ca = 64 * h + i, cb = 64 * h + 32 + i;
            mx = fmax3(mx, ca < lim ? __uint_as_float(xa[i]) : -INFINITY, cb < lim ? __uint_as_float(xb[i]) : -INFINITY);
          }
        }
        const float mc = mx * c;
        float alpha = 1.f;
        if (mc > m + 8.0f) {  // raise the running max (always on the first live tile)
          alpha = (m == -INFINITY) ? 0.f : ex2(m - mc);
          m = mc;
        }
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // O <- alpha O for this warp's rows (P V_{j-1} finished before S_j).
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + cc * 32, o);
            tmem_wait_ld();
            reg_fence(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tO + cc * 32, o);
          }
        }
        // Pass 2: p = 2^(s*c - m) (0 where masked or while no key is visible)
        // as bf16 pairs over the first 64 columns of S, a quarter at a time:
        // quarter q reads S columns 32q .. 32q+31 and writes packed columns
        // 16q .. 16q+15, which earlier quarters have already read.
        const float mm = (m == -INFINITY) ? 0.f : m;
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t xa[32], pk[16];
          tmem_ld32(tS + 32 * q, xa);
          tmem_wait_ld();
          reg_fence(xa);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int i = 32 * q + 2 * e;
            const float p0 = (i < lim) ? ex2(__uint_as_float(xa[2 * e]) * c - mm) : 0.f;
            const float p1 = (i + 1 < lim) ? ex2(__uint_as_float(xa[2 * e + 1]) * c - mm) : 0.f;
            sum += p0 + p1;
            pk[e] = pack_bf16(p0, p1);
          }
          tmem_st16(tS + 16 * q, pk);
        }
        tmem_wait_st();
        l = l * alpha + sum;
      }
      tc_fence_before();
      mbar_arrive(bP);
    }
    // ------------------------------------------------------------ chunk out
    if (ok) ok = __all_sync(0xffffffffu, wait_bounded(wc, bO, 0, wait_site(0xc2, n)));
    if (ok && warp_live) {
      tc_fence_after();
      const size_t row = (size_t)qrow0 + r;  // == ((b * H + h) * Nq + t) for live rows
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + cc * 32, o);
        tmem_wait_ld();
        reg_fence(o);
        if (live && ATTN_IN_RANGE(((long long)row * p.nsplit + split) * D + cc * 32 + 31,
                                  (long long)p.B * p.H * p.Nq * p.nsplit * D, p, 0x501)) {
          // A row that saw no key of the chunk writes zeros, not 0 * O: a
          // chunk with no key tile at all (paged: past its sequence) never
          // ran a P V product, and its O columns hold whatever was there.
          float4* dst = reinterpret_cast<float4*>(p.o_part + (row * p.nsplit + split) * D + cc * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = l > 0.f ? make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                           __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      if (live && ATTN_IN_RANGE((long long)row * p.nsplit + split, (long long)p.B * p.H * p.Nq * p.nsplit, p, 0x502))
        p.lse_part[row * p.nsplit + split] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
  } else if (warp == 4) {
    // ------------------------------------------------------------ producer
    // Lane 0 waits for the free slots and arms the barriers; the K / V boxes
    // of a tile are issued by the warp's lanes (paged: lane i fetches the
    // i-th piece's page from the block table and loads it, so the table
    // lookups of a tile overlap instead of following one another).
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_expect_tx(bQ, T::TILE_BYTES);
      for (int cb = 0; cb < T::NB; ++cb) tma_load_3d(sQ + cb * T::BLOCK_BYTES, &tmQ, bQ, cb * 64, qrow0, 0);
    }
    int nk = 0, nv = 0;
    // One 128-key tile into [128 rows x d] at dst: a plain box, or (paged)
    // 128 / box_rows boxes, each box_rows tokens of one physical page.
    // Pages past the sequence, or table entries out of range, load from page
    // num_pages: out of the map's bounds, so the box reads as zeros (an
    // out-of-range entry the sequence needs is also reported).
    auto load_tile = [&](uint32_t dst, const CUtensorMap* m, uint32_t bar, int key) {
      if constexpr (!PAGED) {
        if (lane == 0)
          for (int cb = 0; cb < T::NB; ++cb) tma_load_3d(dst + cb * T::BLOCK_BYTES, m, bar, cb * 64, key, bhk);
      } else {
        for (int piece = lane; piece < 128 / p.box_rows; piece += 32) {
          const int kp = key + piece * p.box_rows;
          const int lp = kp / p.page_size, off = kp % p.page_size;
          int page = p.num_pages;
          if (kp < nkb && ATTN_IN_RANGE((size_t)b * p.max_pages + lp, (size_t)p.B * p.max_pages, p, 0x503)) {
            page = p.block_table[(size_t)b * p.max_pages + lp];
            if (page < 0 || page >= p.num_pages) {
              atomicCAS(p.status, 0, kDevBadSeqlens);
              page = p.num_pages;
            }
          }
          for (int cb = 0; cb < T::NB; ++cb)
            tma_load_4d(dst + cb * T::BLOCK_BYTES + piece * p.box_rows * 128, m, bar, cb * 64, hk, off, page);
        }
      }
    };
    for (int j = 0; j < n; ++j) {
      bool ok = true;
      if (lane == 0) {
        ok = j == 0 || wait_bounded(wc, bKe, (j - 1) & 1, wait_site(0xd1, j));
        if (ok) mbar_expect_tx(bKf, T::TILE_BYTES);
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;  // the barrier is armed before any box is issued
      load_tile(sK, &tmK, bKf, key0 + j * 128);
      nk = j + 1;
      if (lane == 0) {
        ok = j == 0 || wait_bounded(wc, bVe, (j - 1) & 1, wait_site(0xd2, j));
        if (ok) mbar_expect_tx(bVf, T::TILE_BYTES);
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      load_tile(sV, &tmV, bVf, key0 + j * 128);
      nv = j + 1;
    }
    // Every copy issued above has landed before the CTA may exit.
    if (lane == 0) {
      wait_drain(bQ, 0, p.limit_ns);
      if (nk > 0) wait_drain(bKf, (nk - 1) & 1, p.limit_ns);
      if (nv > 0) wait_drain(bVf, (nv - 1) & 1, p.limit_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ MMA issuer
    {
      const uint32_t leader = elect_one();
      constexpr uint32_t IQK = idesc_bf16_f32(128, 128, false, false);  // S = Q K^T (K-major x K-major)
      constexpr uint32_t IPV = idesc_bf16_f32(128, D, false, true);     // O += P V (A in TMEM, B MN-major)
      const uint32_t tS = tmem, tO = tmem + 128;
      const uint64_t dQ = sdesc_sw128(sQ, 16, 1024);
      const uint64_t dK = sdesc_sw128(sK, 16, 1024);
      const uint64_t dV = sdesc_sw128(sV, T::BLOCK_BYTES, 1024);
      auto wait_all = [&](uint32_t bar, uint32_t parity, int site) {
        return __all_sync(0xffffffffu, wait_bounded(wc, bar, parity, site));
      };
      bool ok = wait_all(bQ, 0, wait_site(0xe1, 0));
      for (int j = 0; j < n && ok; ++j) {
        if (!(ok = wait_all(bKf, j & 1, wait_site(0xe2, j)))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < T::KSTEPS; ++kk) {
          const uint32_t off = (kk >> 2) * T::BLOCK_BYTES + (kk & 3) * 32;
          mma_ss_p(leader, tS, sdesc_add(dQ, off), sdesc_add(dK, off), IQK, kk > 0);
        }
        mma_commit_p(leader, bS);
        mma_commit_p(leader, bKe);  // K_j consumed
        if (!(ok = wait_all(bP, j & 1, wait_site(0xe3, j)))) break;
        if (!(ok = wait_all(bVf, j & 1, wait_site(0xe4, j)))) break;
        if (PAGED) {
          // Rows of V past the sequence (the tail of its last page) hold
          // whatever the cache slot holds: zero them, P is 0 there.
          const int valid = nkb - (key0 + j * 128);
          if (valid < 128) {
            for (int e = lane; e < (128 - valid) * 8 * T::NB; e += 32) {
              const int row = valid + e / (8 * T::NB), cb = (e / 8) % T::NB, ch = e % 8;
              st_shared_v4(sV + cb * T::BLOCK_BYTES + row * 128 + ch * 16, 0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_p(leader, tO, tS + kk * 8, sdesc_add(dV, kk * 2048), IPV, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit_p(leader, bVe);  // V_j consumed (and P_j read)
      }
      if (ok) mma_commit_p(leader, bO);
      mma_commit_p(leader, bDrain);  // fires once every MMA issued above has finished
      wait_drain(bDrain, 0, p.limit_ns);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// One CTA of 128 threads per (batch, head, query) row: O = sum_s w_s O_s /
// sum_s w_s with w_s = exp(lse_s - max lse); lse = max + ln sum w (-inf and
// O = 0 if no chunk saw a visible key).  The chunks are dealt to the four
// warps so that a row with many chunks is read by many loads in flight;
// the warps' sums are combined in shared memory.  Lane l holds columns l,
// l + 32, ... (coalesced scalar loads, aligned for every d).
template <int D>
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecParams p) {
  __shared__ float red[4][D];
  __shared__ float wsum[4];
  __shared__ float wmax[4];
  const long long row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (!ATTN_IN_RANGE(row, (long long)p.B * p.H * p.Nq, p, 0x504)) return;  // (uniform over the block)
  const float* lp = p.lse_part + row * p.nsplit;
  float mx = -INFINITY;
  for (int s = threadIdx.x; s < p.nsplit; s += 128) mx = fmaxf(mx, lp[s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) wmax[warp] = mx;
  __syncthreads();
  mx = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
  constexpr int C = D / 32;  // columns per lane: lane + 32 c (coalesced scalar loads)
  float acc[C];
#pragma unroll
  for (int c = 0; c < C; ++c) acc[c] = 0.f;
  float tot = 0.f;
  if (mx != -INFINITY) {
#pragma unroll 4
    for (int s = warp; s < p.nsplit; s += 4) {
      const float w = __expf(lp[s] - mx);
      tot += w;
      const float* op = p.o_part + (row * p.nsplit + s) * D + lane;
#pragma unroll
      for (int c = 0; c < C; ++c) acc[c] = fmaf(w, op[32 * c], acc[c]);
    }
  }
#pragma unroll
  for (int c = 0; c < C; ++c) red[warp][lane + 32 * c] = acc[c];
  if (lane == 0) wsum[warp] = tot;
  __syncthreads();
  const float all = (wsum[0] + wsum[1]) + (wsum[2] + wsum[3]);
  const float inv = all > 0.f ? 1.f / all : 0.f;
  for (int c = threadIdx.x; c < D; c += 128) {
    const float v = ((red[0][c] + red[1][c]) + (red[2][c] + red[3][c])) * inv;
    p.o[row * D + c] = (uint16_t)(pack_bf16(v, 0.f) & 0xffffu);
  }
  if (threadIdx.x == 0) p.lse[row] = all > 0.f ? mx + logf(all) : -INFINITY;
}

size_t decode_smem_bytes(int d) {
  switch (d) {
    case 64: return DecTraits<64>::SMEM;
    case 96: return DecTraits<96>::SMEM;
    case 128: return DecTraits<128>::SMEM;
    default: return 0;
  }
}

template <int D, bool C, bool PG = false>
static cudaError_t launch_decode_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                   const DecParams& p, cudaStream_t stream) {
  auto kern = decode_split_kernel<D, C, PG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DecTraits<D>::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<dim3((unsigned)p.nsplit, (unsigned)(p.B * p.Hkv)), kDecThreads, DecTraits<D>::SMEM, stream>>>(tq, tk, tv, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const long long rows = (long long)p.B * p.H * p.Nq;
  decode_merge_kernel<D><<<(unsigned)rows, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const DecParams& p, cudaStream_t stream, bool paged) {
  if (paged) {
    switch (d) {
      case 64: return causal ? launch_decode_t<64, true, true>(tq, tk, tv, p, stream)
                             : launch_decode_t<64, false, true>(tq, tk, tv, p, stream);
      case 96: return causal ? launch_decode_t<96, true, true>(tq, tk, tv, p, stream)
                             : launch_decode_t<96, false, true>(tq, tk, tv, p, stream);
      case 128: return causal ? launch_decode_t<128, true, true>(tq, tk, tv, p, stream)
                              : launch_decode_t<128, false, true>(tq, tk, tv, p, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (d) {
    case 64: return causal ? launch_decode_t<64, true>(tq, tk, tv, p, stream)
                           : launch_decode_t<64, false>(tq, tk, tv, p, stream);
    case 96: return causal ? launch_decode_t<96, true>(tq, tk, tv, p, stream)
                           : launch_decode_t<96, false>(tq, tk, tv, p, stream);
    case 128: return causal ? launch_decode_t<128, true>(tq, tk, tv, p, stream)
                            : launch_decode_t<128, false>(tq, tk, tv, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sdpa
