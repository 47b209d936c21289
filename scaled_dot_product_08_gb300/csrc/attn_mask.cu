// attn_mask.cu — packs a boolean attention mask into the bit layouts the
// masked kernel instances read.
//
// The mask is the boolean attn_mask of page "SDPA backend 与 FlashAttention"
// (§3; FAQ Q11 of "Flash Attention原理": an arbitrary boolean mask, handled
// inside the kernel rather than materialised as scores): shape
// (mask_b, mask_h, Nq, Nk) bytes, nonzero = the key takes part.  The kernels
// want one bit per (query, key): row bits (bit j % 32 of word j / 32 of a
// query row) for the forward and dQ kernels, whose threads own query rows,
// and transposed bits (bit i % 32 of word i / 32 of a key row) for the
// dK/dV kernel, whose threads own key rows.  A 128 x 128 tile of bits is
// 2 KB against 16 KB of mask bytes, so the kernels read an eighth of the
// mask per pass, with one 16- or 8-byte load per row and tile.  One byte per
// 128 x 128 tile classifies it (nothing visible / some / all), so that the
// kernels skip the tiles a sparse mask (documents, prefix-LM) hides.
#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {

namespace {

constexpr int kTile = 128;
constexpr int kPitchW = 33;  // shared row pitch in 32-bit words: row-wise and column-wise reads spread over the banks

// One CTA per (plane, 128-row query tile, 128-column key tile).  The tile's
// bytes go through shared memory.  A row word (32 keys of one query row) is
// built by one thread from eight 4-byte reads: __vsetne4 turns each byte
// into 0 / 1 and one multiply gathers the four into a nibble.  A transposed
// word (32 query rows of one key) is a warp ballot, lane l holding row
// 32 w + l; each lane reads four keys at once, so one read feeds four
// ballots.
__global__ void __launch_bounds__(256) mask_pack_kernel(const uint8_t* __restrict__ mask, int Nq, int Nk,
                                                        uint32_t* __restrict__ bits, int words,
                                                        uint32_t* __restrict__ bits_t, int words_t,
                                                        uint8_t* __restrict__ flags) {
  __shared__ uint32_t tile_w[kTile * kPitchW];
  __shared__ int any_vis, all_vis;
  uint8_t* tile = reinterpret_cast<uint8_t*>(tile_w);
  constexpr int kPitch = 4 * kPitchW;
  const int nqt = (Nq + kTile - 1) / kTile, nkt = (Nk + kTile - 1) / kTile;
  const int kt = (int)(blockIdx.x % nkt);
  const int qt = (int)((blockIdx.x / nkt) % nqt);
  const int plane = (int)(blockIdx.x / ((unsigned)nkt * nqt));
  const uint8_t* src = mask + (size_t)plane * Nq * Nk;
  if ((Nk & 15) == 0 && (reinterpret_cast<uintptr_t>(mask) & 15) == 0) {
    // 16 bytes per load (rows start 16-byte aligned); four 4-byte stores
    // into the padded shared rows.  Bytes keep their values: only their
    // being nonzero is read below.
    for (int e = threadIdx.x; e < kTile * kTile / 16; e += blockDim.x) {
      const int r = e / (kTile / 16), c16 = e % (kTile / 16);
      const int qi = qt * kTile + r, kj = kt * kTile + c16 * 16;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (qi < Nq && kj < Nk) v = *reinterpret_cast<const uint4*>(src + (size_t)qi * Nk + kj);
      uint32_t* dst = tile_w + r * kPitchW + c16 * 4;
      dst[0] = v.x;
      dst[1] = v.y;
      dst[2] = v.z;
      dst[3] = v.w;
    }
  } else {
    for (int e = threadIdx.x; e < kTile * kTile; e += blockDim.x) {
      const int r = e / kTile, c = e % kTile;
      const int qi = qt * kTile + r, kj = kt * kTile + c;
      tile[r * kPitch + c] = (qi < Nq && kj < Nk) ? (src[(size_t)qi * Nk + kj] != 0) : 0;
    }
  }
  if (threadIdx.x == 0) {
    any_vis = 0;
    all_vis = 1;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int kvalid = min(kTile, Nk - kt * kTile);  // key columns that exist
  const int qvalid = min(kTile, Nq - qt * kTile);  // query rows that exist
  bool any = false, all = true;
  // Row words: thread e handles (row e / 4, word e % 4), every thread the
  // same number of times.
  for (int e = threadIdx.x; e < kTile * 4; e += blockDim.x) {
    const int r = e >> 2, w = e & 3;
    const uint32_t* rw = tile_w + r * kPitchW + 8 * w;
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // bytes b0..b3 of nz are 0 / 1; the product puts b_k at bit 24 + k
      // and every cross term below bit 24 or above bit 31
      const uint32_t nz = __vsetne4(rw[i], 0u);
      word |= ((nz * 0x01020408u) >> 24) << (4 * i);
    }
    if (r < qvalid) {
      const int nb = min(32, max(0, kvalid - 32 * w));
      const uint32_t valid = nb == 32 ? 0xffffffffu : ((1u << nb) - 1u);
      any |= (word & valid) != 0;
      all &= (word & valid) == valid;
      bits[((size_t)plane * Nq + qt * kTile + r) * words + kt * 4 + w] = word;
    }
  }
  if (flags != nullptr) {
    // The tile's class for skipping: 0 = nothing visible, 1 = some, 2 = all.
    any = __any_sync(0xffffffffu, any);
    all = __all_sync(0xffffffffu, all);
    if (lane == 0 && any) atomicOr(&any_vis, 1);
    if (lane == 0 && !all) atomicAnd(&all_vis, 0);
    __syncthreads();
    if (threadIdx.x == 0)
      flags[((size_t)plane * nqt + qt) * nkt + kt] = (uint8_t)(any_vis == 0 ? 0 : (all_vis ? 2 : 1));
  }
  if (bits_t != nullptr) {
    // (row block w, keys 4 g .. 4 g + 3): four transposed words per item.
    for (int wg = warp; wg < 4 * (kTile / 4); wg += nw) {
      const int w = wg / (kTile / 4), g = wg % (kTile / 4);
      const uint32_t nz = __vsetne4(tile_w[(32 * w + lane) * kPitchW + g], 0u);
      uint32_t mine = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t word = __ballot_sync(0xffffffffu, (nz >> (8 * k)) & 1u);
        if (lane == k) mine = word;
      }
      const int c = 4 * g + lane;
      if (lane < 4 && kt * kTile + c < Nk)
        bits_t[((size_t)plane * Nk + kt * kTile + c) * words_t + qt * 4 + w] = mine;
    }
  }
}

// The additive mask's transpose, (planes, Nq, Nk) -> (planes, Nk, Nq), for
// the dK/dV kernel, whose threads own key rows: 32 x 32 blocks through
// shared memory (pitch 33 elements: the column reads hit distinct banks).
// T: float (float32 mask) or uint16_t (bf16 bits, moved unchanged).
template <typename T>
__global__ void __launch_bounds__(256) bias_transpose_kernel(const T* __restrict__ bias, int Nq, int Nk,
                                                             T* __restrict__ bias_t) {
  __shared__ T blk[32][33];
  const int tk = (Nk + 31) / 32;
  const int kb = (int)(blockIdx.x % tk), qb = (int)(blockIdx.x / tk);
  const size_t plane = blockIdx.y;
  const T* src = bias + plane * Nq * Nk;
  T* dst = bias_t + plane * Nq * Nk;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int rr = ty; rr < 32; rr += 8) {
    const int qi = qb * 32 + rr, kj = kb * 32 + tx;
    if (qi < Nq && kj < Nk) blk[rr][tx] = src[(size_t)qi * Nk + kj];
  }
  __syncthreads();
  for (int rr = ty; rr < 32; rr += 8) {
    const int kj = kb * 32 + rr, qi = qb * 32 + tx;
    if (qi < Nq && kj < Nk) dst[(size_t)kj * Nq + qi] = blk[tx][rr];
  }
}

}  // namespace

cudaError_t launch_bias_transpose(const void* bias, bool bf16, int planes, int Nq, int Nk, void* bias_t,
                                  cudaStream_t stream) {
  const unsigned blocks = (unsigned)((Nq + 31) / 32) * (unsigned)((Nk + 31) / 32);
  if (bf16)
    bias_transpose_kernel<uint16_t><<<dim3(blocks, (unsigned)planes), 256, 0, stream>>>(
        static_cast<const uint16_t*>(bias), Nq, Nk, static_cast<uint16_t*>(bias_t));
  else
    bias_transpose_kernel<float><<<dim3(blocks, (unsigned)planes), 256, 0, stream>>>(
        static_cast<const float*>(bias), Nq, Nk, static_cast<float*>(bias_t));
  return cudaGetLastError();
}

cudaError_t launch_mask_pack(const uint8_t* mask, int mask_b, int mask_h, int Nq, int Nk, uint32_t* bits, int words,
                             uint32_t* bits_t, int words_t, uint8_t* flags, cudaStream_t stream) {
  const unsigned tiles = (unsigned)((Nq + kTile - 1) / kTile) * (unsigned)((Nk + kTile - 1) / kTile);
  mask_pack_kernel<<<tiles * (unsigned)(mask_b * mask_h), 256, 0, stream>>>(mask, Nq, Nk, bits, words, bits_t,
                                                                            words_t, flags);
  return cudaGetLastError();
}

}  // namespace sdpa
