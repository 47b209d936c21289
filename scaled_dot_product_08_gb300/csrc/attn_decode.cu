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
// The work reads every cached key and value once and does 4d flops per key
// and query row, so for the few query rows of a decode step it is bound by
// HBM bandwidth, not by the tensor cores: the arithmetic runs on the FMA
// pipes and the design effort goes into streaming K/V at full bandwidth.
//
// Two kernels on the caller's stream:
//   decode_split  one CTA per (key chunk, batch * K/V head), 256 threads.
//                 The R = G * Nq query rows of a K/V head (its G query heads
//                 times the Nq new tokens) share every K/V tile the CTA
//                 loads.  Thread 0 streams 128-key K and V tiles by TMA
//                 into a 2-stage ring (128-byte swizzle, so 16-byte reads of
//                 consecutive rows hit distinct banks); per tile:
//                   scores   one key per thread, R/2 query rows each, fp32 FMA
//                            against Q rows pre-scaled by scale * log2(e)
//                   softmax  one warp per query row: tile max, running max,
//                            rescale factor, exp2, row sum (online, §四)
//                   P V      each thread owns (query row, 8 columns) pairs for
//                            a subset of the tile's keys; partial sums stay in
//                            registers across tiles and are combined once
//                 and writes its chunk's normalised O and lse (natural log;
//                 -inf with O = 0 when every key of the chunk is masked).
//   decode_merge  one warp per (batch, head, query): the lse-weighted merge
//                 of the chunks -> O (bf16) and lse.
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {

namespace {

constexpr int kDecThreads = 256;
constexpr int kDecTileKeys = 128;

template <int D>
struct DecTraits {
  static constexpr int NB = (D + 63) / 64;
  static constexpr int BLOCK_BYTES = 128 * 128;        // [128 keys x 64 columns] bf16, swizzled
  static constexpr int TILE_BYTES = NB * BLOCK_BYTES;  // one [128 keys x d] tile
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;   // K and V
  static constexpr int QS_BYTES = kDecMaxRows * D * 4; // Q rows, fp32, pre-scaled
  static constexpr int PS_BYTES = kDecMaxRows * kDecTileKeys * 4;  // P of one tile, fp32
  static constexpr int STAT_BYTES = kDecMaxRows * 4 * 3;           // m, l, alpha per row
  static constexpr int SMEM = 1024 + 2 * STAGE_BYTES + QS_BYTES + PS_BYTES + STAT_BYTES + 64;
  // (query row, 8-column group) pairs each thread accumulates in P V
  static constexpr int MAX_PAIRS = (kDecMaxRows * (D / 8) + kDecThreads - 1) / kDecThreads;
};

// Column group c8 (8 bf16 columns) of row `row` of a swizzled [128 x d] tile.
__device__ __forceinline__ uint32_t dec_chunk(uint32_t tile, int row, int c8) {
  return tile + (uint32_t)(c8 >> 3) * (128u * 128u) + (uint32_t)row * 128u + ((uint32_t)((c8 & 7) ^ (row & 7)) << 4);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

}  // namespace

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const DecParams p) {
  using T = DecTraits<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t sStage = base;                              // [2] {K tile, V tile}
  float* const q_s = reinterpret_cast<float*>(gbase + 2 * T::STAGE_BYTES);            // [R][D]
  float* const p_s = reinterpret_cast<float*>(gbase + 2 * T::STAGE_BYTES + T::QS_BYTES);  // [R][128]
  float* const m_s = reinterpret_cast<float*>(gbase + 2 * T::STAGE_BYTES + T::QS_BYTES + T::PS_BYTES);
  float* const l_s = m_s + kDecMaxRows;
  float* const a_s = l_s + kDecMaxRows;
  const uint32_t sBar = smem_u32(a_s + kDecMaxRows);
  const uint32_t bFull = (sBar + 7u) & ~7u;                  // [2] stage loaded
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbase + (bFull - base) + 16);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, bhk = blockIdx.y;
  const int b = bhk / p.Hkv, hk = bhk % p.Hkv;
  const int R = p.G * p.Nq;                                  // query rows of this K/V head
  const int key0 = split * p.split_keys;
  const int key1 = min(p.Nk, key0 + p.split_keys);
  const int ntiles = (key1 - key0 + kDecTileKeys - 1) / kDecTileKeys;

  if (tid == 0) {
    mbar_init(bFull, 1);
    mbar_init(bFull + 8u, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Q rows of the group, fp32, pre-scaled into the base-2 domain.
  for (int e = tid; e < R * (D / 8); e += kDecThreads) {
    const int r = e / (D / 8), c8 = e % (D / 8);
    const int h = hk * p.G + r / p.Nq, t = r % p.Nq;
    const uint4 w = *reinterpret_cast<const uint4*>(p.q + (((size_t)b * p.H + h) * p.Nq + t) * D + c8 * 8);
    float* dst = q_s + r * D + c8 * 8;
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      dst[2 * k] = bf_lo(ws[k]) * p.scale_log2;
      dst[2 * k + 1] = bf_hi(ws[k]) * p.scale_log2;
    }
  }
  for (int r = tid; r < kDecMaxRows; r += kDecThreads) {
    m_s[r] = -INFINITY;
    l_s[r] = 0.f;
  }
  __syncthreads();
  const WaitCtx wc{abort_flag, p.status, p.limit_ns, p.info};

  auto issue = [&](int tile) {  // thread 0: K and V of `tile` into stage tile & 1
    const uint32_t st = sStage + (uint32_t)(tile & 1) * T::STAGE_BYTES, bar = bFull + 8u * (tile & 1);
    fence_proxy_async_smem();
    mbar_expect_tx(bar, T::STAGE_BYTES);
    const int row = key0 + tile * kDecTileKeys;
    for (int cb = 0; cb < T::NB; ++cb) {
      tma_load_3d(st + cb * T::BLOCK_BYTES, &tmK, bar, cb * 64, row, bhk);
      tma_load_3d(st + T::TILE_BYTES + cb * T::BLOCK_BYTES, &tmV, bar, cb * 64, row, bhk);
    }
  };
  int issued = 0;
  if (tid == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (; issued < ntiles && issued < 2; ++issued) issue(issued);
  }

  // P V ownership: pairs (row r, column group c8) in row-major order; with
  // fewer pairs than threads, the tile's keys are dealt to `kg` groups.
  const int npairs = R * (D / 8);
  const int kg = npairs >= kDecThreads ? 1 : min(16, kDecThreads / npairs);
  const int grp = npairs >= kDecThreads ? 0 : tid / npairs;
  const bool pv_active = npairs >= kDecThreads || tid < npairs * kg;
  float acc[T::MAX_PAIRS][8];
#pragma unroll
  for (int u = 0; u < T::MAX_PAIRS; ++u)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[u][c] = 0.f;

  bool ok = true;
  for (int tile = 0; tile < ntiles; ++tile) {
    const uint32_t st = sStage + (uint32_t)(tile & 1) * T::STAGE_BYTES;
    ok = __syncthreads_and(wait_bounded(wc, bFull + 8u * (tile & 1), (tile >> 1) & 1, wait_site(0xb1, tile)));
    if (!ok) break;
    const int kt0 = key0 + tile * kDecTileKeys;  // first key of the tile
    // ---- scores: key jj = tid % 128, rows rh, rh + 2, ...
    {
      const int jj = tid & (kDecTileKeys - 1), rh = tid >> 7;
      const int key = kt0 + jj;
      const bool key_ok = key < key1;
      for (int r0 = rh; r0 < R; r0 += 16) {  // up to 8 rows per pass
        float s[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) s[u] = 0.f;
#pragma unroll 4
        for (int c8 = 0; c8 < D / 8; ++c8) {
          const uint4 kw = lds128(dec_chunk(st, jj, c8));
          const float kf[8] = {bf_lo(kw.x), bf_hi(kw.x), bf_lo(kw.y), bf_hi(kw.y),
                               bf_lo(kw.z), bf_hi(kw.z), bf_lo(kw.w), bf_hi(kw.w)};
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int r = r0 + 2 * u;
            if (r < R) {
              const float4 qa = *reinterpret_cast<const float4*>(q_s + r * D + c8 * 8);
              const float4 qb = *reinterpret_cast<const float4*>(q_s + r * D + c8 * 8 + 4);
              s[u] = fmaf(qa.x, kf[0], s[u]);
              s[u] = fmaf(qa.y, kf[1], s[u]);
              s[u] = fmaf(qa.z, kf[2], s[u]);
              s[u] = fmaf(qa.w, kf[3], s[u]);
              s[u] = fmaf(qb.x, kf[4], s[u]);
              s[u] = fmaf(qb.y, kf[5], s[u]);
              s[u] = fmaf(qb.z, kf[6], s[u]);
              s[u] = fmaf(qb.w, kf[7], s[u]);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int r = r0 + 2 * u;
          if (r < R) {
            bool live = key_ok;
            if (CAUSAL) live = live && key <= p.Nk - p.Nq + r % p.Nq;
            p_s[r * kDecTileKeys + jj] = live ? s[u] : -INFINITY;
          }
        }
      }
    }
    __syncthreads();
    // ---- online softmax: one warp per row
    for (int r = warp; r < R; r += kDecThreads / 32) {
      float* row = p_s + r * kDecTileKeys;
      float v4[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) v4[k] = row[lane + 32 * k];
      float mx = fmaxf(fmaxf(v4[0], v4[1]), fmaxf(v4[2], v4[3]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_old = m_s[r];
      const float m_new = fmaxf(m_old, mx);
      // Rows with no live key so far keep m = -inf: every p is then 0.
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      float sum = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float e = ex2(v4[k] - m_use);
        row[lane + 32 * k] = e;
        sum += e;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (lane == 0) {
        const float alpha = (m_old == -INFINITY) ? 0.f : ex2(m_old - m_use);
        a_s[r] = alpha;
        l_s[r] = l_s[r] * alpha + sum;
        m_s[r] = m_new;
      }
    }
    __syncthreads();
    // ---- P V
    if (pv_active) {
#pragma unroll
      for (int u = 0; u < T::MAX_PAIRS; ++u) {
        const int pair = (npairs >= kDecThreads) ? tid + u * kDecThreads : tid % npairs;
        if ((npairs >= kDecThreads && pair < npairs) || (npairs < kDecThreads && u == 0)) {
          const int r = pair / (D / 8), c8 = pair % (D / 8);
          const float alpha = a_s[r];
#pragma unroll
          for (int c = 0; c < 8; ++c) acc[u][c] *= alpha;
          const float* prow = p_s + r * kDecTileKeys;
#pragma unroll 4
          for (int jj = grp; jj < kDecTileKeys; jj += kg) {
            const float pv = prow[jj];
            const uint4 vw = lds128(dec_chunk(st + T::TILE_BYTES, jj, c8));
            acc[u][0] = fmaf(pv, bf_lo(vw.x), acc[u][0]);
            acc[u][1] = fmaf(pv, bf_hi(vw.x), acc[u][1]);
            acc[u][2] = fmaf(pv, bf_lo(vw.y), acc[u][2]);
            acc[u][3] = fmaf(pv, bf_hi(vw.y), acc[u][3]);
            acc[u][4] = fmaf(pv, bf_lo(vw.z), acc[u][4]);
            acc[u][5] = fmaf(pv, bf_hi(vw.z), acc[u][5]);
            acc[u][6] = fmaf(pv, bf_lo(vw.w), acc[u][6]);
            acc[u][7] = fmaf(pv, bf_hi(vw.w), acc[u][7]);
          }
        }
      }
    }
    __syncthreads();  // stage tile & 1 and p_s are free again
    if (tid == 0 && issued < ntiles) issue(issued++);
  }
  if (tid == 0) {  // nothing of ours may still be landing in shared memory at exit
    // Tiles before the one the loop stopped at were consumed; at most the
    // last two issued can still be in flight.
    for (int t = issued - 2 > 0 ? issued - 2 : 0; t < issued; ++t)
      wait_drain(bFull + 8u * (t & 1), (t >> 1) & 1, p.limit_ns);
  }
  if (!ok) return;
  // ---- combine the key groups' partial sums (through p_s), normalise, store
  float* const red = p_s;  // [kg][npairs][8] when kg > 1
  if (kg > 1) {
    if (pv_active) {
#pragma unroll
      for (int c = 0; c < 8; ++c) red[(grp * npairs + (tid % npairs)) * 8 + c] = acc[0][c];
    }
    __syncthreads();
  }
  for (int u = 0; u < T::MAX_PAIRS; ++u) {
    const int pair = (npairs >= kDecThreads) ? tid + u * kDecThreads : tid;
    if (pair >= npairs || (npairs < kDecThreads && u > 0)) break;
    const int r = pair / (D / 8), c8 = pair % (D / 8);
    float o[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) o[c] = (kg > 1) ? 0.f : acc[u][c];
    if (kg > 1)
      for (int g2 = 0; g2 < kg; ++g2)
#pragma unroll
        for (int c = 0; c < 8; ++c) o[c] += red[(g2 * npairs + pair) * 8 + c];
    const float l = l_s[r];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int h = hk * p.G + r / p.Nq, t = r % p.Nq;
    const size_t row = ((size_t)b * p.H + h) * p.Nq + t;
    float4* dst = reinterpret_cast<float4*>(p.o_part + (row * p.nsplit + split) * D + c8 * 8);
    dst[0] = make_float4(o[0] * inv, o[1] * inv, o[2] * inv, o[3] * inv);
    dst[1] = make_float4(o[4] * inv, o[5] * inv, o[6] * inv, o[7] * inv);
    if (c8 == 0)
      p.lse_part[row * p.nsplit + split] = l > 0.f ? (m_s[r] + log2f(l)) * 0.69314718055994531f : -INFINITY;
  }
}

// One warp per (batch, head, query): O = sum_s w_s O_s / sum_s w_s with
// w_s = exp(lse_s - max lse); lse = max + ln sum w (-inf, O = 0 if no split
// saw a live key).
template <int D>
__global__ void __launch_bounds__(256) decode_merge_kernel(const DecParams p) {
  const long long rows = (long long)p.B * p.H * p.Nq;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* lp = p.lse_part + row * p.nsplit;
  float mx = -INFINITY;
  for (int s = lane; s < p.nsplit; s += 32) mx = fmaxf(mx, lp[s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  constexpr int C = D / 32;  // columns per lane
  float acc[C];
#pragma unroll
  for (int c = 0; c < C; ++c) acc[c] = 0.f;
  float tot = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < p.nsplit; ++s) {
      const float w = __expf(lp[s] - mx);
      tot += w;
      const float* op = p.o_part + (row * p.nsplit + s) * D;
#pragma unroll
      for (int c = 0; c < C; ++c) acc[c] = fmaf(w, op[lane + 32 * c], acc[c]);
    }
  }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  uint16_t* out = p.o + row * D;
#pragma unroll
  for (int c = 0; c < C; ++c) {
    const float v = acc[c] * inv;
    out[lane + 32 * c] = (uint16_t)(pack_bf16(v, 0.f) & 0xffffu);
  }
  if (lane == 0) p.lse[row] = tot > 0.f ? mx + logf(tot) : -INFINITY;
}

size_t decode_smem_bytes(int d) {
  switch (d) {
    case 64: return DecTraits<64>::SMEM;
    case 96: return DecTraits<96>::SMEM;
    case 128: return DecTraits<128>::SMEM;
    default: return 0;
  }
}

template <int D, bool C>
static cudaError_t launch_decode_t(const CUtensorMap& tk, const CUtensorMap& tv, const DecParams& p,
                                   cudaStream_t stream) {
  auto kern = decode_split_kernel<D, C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DecTraits<D>::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<dim3((unsigned)p.nsplit, (unsigned)(p.B * p.Hkv)), kDecThreads, DecTraits<D>::SMEM, stream>>>(tk, tv, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const long long rows = (long long)p.B * p.H * p.Nq;
  decode_merge_kernel<D><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode(int d, bool causal, const CUtensorMap& tk, const CUtensorMap& tv, const DecParams& p,
                          cudaStream_t stream) {
  switch (d) {
    case 64: return causal ? launch_decode_t<64, true>(tk, tv, p, stream) : launch_decode_t<64, false>(tk, tv, p, stream);
    case 96: return causal ? launch_decode_t<96, true>(tk, tv, p, stream) : launch_decode_t<96, false>(tk, tv, p, stream);
    case 128: return causal ? launch_decode_t<128, true>(tk, tv, p, stream)
                            : launch_decode_t<128, false>(tk, tv, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sdpa
