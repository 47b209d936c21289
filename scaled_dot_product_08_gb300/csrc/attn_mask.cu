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
constexpr int kPitch = 132;  // shared row pitch in bytes: column reads spread over the banks

// One CTA per (plane, 128-row query tile, 128-column key tile).  The tile's
// bytes go through shared memory; each 32-bit word is then one warp ballot
// (lane l supplies element 32 w + l), over a row for the row bits and over a
// column for the transposed bits.
__global__ void __launch_bounds__(256) mask_pack_kernel(const uint8_t* __restrict__ mask, int Nq, int Nk,
                                                        uint32_t* __restrict__ bits, int words,
                                                        uint32_t* __restrict__ bits_t, int words_t,
                                                        uint8_t* __restrict__ flags) {
  __shared__ uint8_t tile[kTile * kPitch];
  __shared__ int any_vis, all_vis;
  const int nqt = (Nq + kTile - 1) / kTile, nkt = (Nk + kTile - 1) / kTile;
  const int kt = (int)(blockIdx.x % nkt);
  const int qt = (int)((blockIdx.x / nkt) % nqt);
  const int plane = (int)(blockIdx.x / ((unsigned)nkt * nqt));
  const uint8_t* src = mask + (size_t)plane * Nq * Nk;
  for (int e = threadIdx.x; e < kTile * kTile; e += blockDim.x) {
    const int r = e / kTile, c = e % kTile;
    const int qi = qt * kTile + r, kj = kt * kTile + c;
    tile[r * kPitch + c] = (qi < Nq && kj < Nk) ? (src[(size_t)qi * Nk + kj] != 0) : 0;
  }
  if (threadIdx.x == 0) {
    any_vis = 0;
    all_vis = 1;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  // Columns of word w that exist (keys < Nk).
  const int kvalid = min(kTile, Nk - kt * kTile);
  bool any = false, all = true;
  for (int rw = warp; rw < kTile * 4; rw += nw) {
    const int r = rw >> 2, w = rw & 3;
    const uint32_t word = __ballot_sync(0xffffffffu, tile[r * kPitch + 32 * w + lane] != 0);
    if (qt * kTile + r < Nq) {
      const int nb = min(32, max(0, kvalid - 32 * w));
      const uint32_t valid = nb == 32 ? 0xffffffffu : ((1u << nb) - 1u);
      any |= (word & valid) != 0;
      all &= (word & valid) == valid;
      if (lane == 0) bits[((size_t)plane * Nq + qt * kTile + r) * words + kt * 4 + w] = word;
    }
  }
  if (flags != nullptr) {
    // The tile's class for skipping: 0 = nothing visible, 1 = some, 2 = all.
    if (lane == 0 && any) atomicOr(&any_vis, 1);
    if (lane == 0 && !all) atomicAnd(&all_vis, 0);
    __syncthreads();
    if (threadIdx.x == 0)
      flags[((size_t)plane * nqt + qt) * nkt + kt] = (uint8_t)(any_vis == 0 ? 0 : (all_vis ? 2 : 1));
  }
  if (bits_t != nullptr) {
    for (int cw = warp; cw < kTile * 4; cw += nw) {
      const int c = cw >> 2, w = cw & 3;
      const uint32_t word = __ballot_sync(0xffffffffu, tile[(32 * w + lane) * kPitch + c] != 0);
      if (lane == 0 && kt * kTile + c < Nk)
        bits_t[((size_t)plane * Nk + kt * kTile + c) * words_t + qt * 4 + w] = word;
    }
  }
}

}  // namespace

cudaError_t launch_mask_pack(const uint8_t* mask, int mask_b, int mask_h, int Nq, int Nk, uint32_t* bits, int words,
                             uint32_t* bits_t, int words_t, uint8_t* flags, cudaStream_t stream) {
  const unsigned tiles = (unsigned)((Nq + kTile - 1) / kTile) * (unsigned)((Nk + kTile - 1) / kTile);
  mask_pack_kernel<<<tiles * (unsigned)(mask_b * mask_h), 256, 0, stream>>>(mask, Nq, Nk, bits, words, bits_t,
                                                                            words_t, flags);
  return cudaGetLastError();
}

}  // namespace sdpa
