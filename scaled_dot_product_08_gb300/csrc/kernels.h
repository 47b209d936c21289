// kernels.h — internal launch interface between the C ABI (attn_api.cu) and
// the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace sdpa {

// Packed variable-length batch (cu_seqlens): sequence b owns query rows
// cu_q[b] .. cu_q[b+1]-1 and key rows cu_k[b] .. cu_k[b+1]-1 of a
// (total, heads, d) tensor.  cu_q == nullptr: the dense (B, heads, N, d) batch.
struct VarlenArgs {
  const int* cu_q;
  const int* cu_k;
  int total_q, total_k;  // packed rows (the bound every offset is checked against)
};

// Masks beyond causal (the masked kernel instances only).  Query row i sits
// at position Nk - Nq + i; key j is visible to it when
//   j >= pos - wl (wl >= 0),  j <= pos + wr (wr >= 0; causal sets wr = 0),
//   j < key_len[b] (key_len != nullptr),  and its bit is set (bits != nullptr).
// bits: (planes, Nq, words) uint32, bit j % 32 of word j / 32 of a query row;
// bits_t: (planes, Nk, words_t), bit i % 32 of word i / 32 of a key row;
// words / words_t are multiples of 4 (one 16-byte group per 128 columns).
// plane = (mask_b > 1 ? b : 0) * mask_h + (mask_h > 1 ? h : 0).
// flags: (planes, ceil(Nq/128), ceil(Nk/128)) bytes, one per 128 x 128 tile:
// 0 = no visible entry (the tile is skipped), 1 = some, 2 = all.
struct MaskArgs {
  int wl, wr;
  const int* key_len;
  const uint32_t* bits;
  const uint32_t* bits_t;
  int words, words_t;
  int mask_b, mask_h;
  const uint8_t* flags;
  int ftq, ftk;  // query and key tiles per plane in flags
  // Additive mask (float32, or bf16 when bias_bf16; added to the scaled
  // scores): (bias_b, bias_h, Nq, Nk) as given, and its (bias_b * bias_h,
  // Nk, Nq) transpose in the same type for the dK/dV kernel (backward only);
  // inv_scale = 1 / scale, so that x + b * inv_scale, scaled, is scale x + b.
  const void* bias;
  const void* bias_t;
  int bias_b, bias_h;
  float inv_scale;
  int bias_bf16;
};

// Most key tiles a masked forward / dQ CTA can list for skipping (its
// shared-memory list of uint16 tile indices), and most (head, query tile)
// steps a masked dK / dV CTA can list (uint32 entries).  Beyond these the
// kernels visit every tile of their range without skipping.
constexpr int kMaxTileList = 880;
constexpr int kMaxStepList = 8192;

// Forward kernel arguments (tensor maps are passed separately).
struct FwdParams {
  float* lse;            // (B, H, Nq) float32
  int B, H, Hkv, G;      // G = H / Hkv
  int Nq, Nk;            // query rows, key/value rows per head
  int koff;              // causal: query row i sits at position koff + i (Nk - Nq)
  int n_mtiles;          // ceil(Nq / 256): one CTA = two 128-row query tiles
  int nkv;               // ceil(Nk / 128): key/value tiles
  float scale_log2;      // scale * log2(e)
  int* status;           // device status word
  unsigned long long limit_ns;  // bounded-wait limit
  int* info;             // first-timeout record (4 ints)
  VarlenArgs vl;         // varlen: Nq / Nk above are the longest sequences
  uint16_t* o;           // varlen: O base, for the rows of a sequence's last tile; FP8: O base
  MaskArgs mk;           // masked instances only
  float o_scale;         // FP8: V's dequantisation factor, applied to O
  int debug_drop1;       // 0; n > 0 only in a test of the bounded waits: CTA 0's producer skips ring load n - 1
  int tail;              // heads in the level-major tail of the CTA order (work_unit); set by the launcher
  int debug_plant;       // 0; 1 only in a test of the debug build's checks: CTA 0 offsets its lse store out of range
  int* sched;            // persistent forward: this launch's queue (next unit, CTAs done); set by its launcher
  int n_units;           // persistent forward: units in the launch
  int debug_drop_p;      // 0; n > 0 only in a test of the bounded waits: the persistent forward skips unit 0's ring load n - 1
                         // (the FP8 forward: the same, or CTA 0's, for the one-CTA-per-unit kernel)
};

// Backward arguments.
struct BwdParams {
  const uint16_t* o;     // (B, H, N, d) bf16
  const uint16_t* dout;  // (B, H, N, d) bf16
  const float* lse;      // (B, H, N)
  float* dvec;           // (B, H, Npad) float32 workspace: -D = -rowsum(dO * O)
  float* lse2;           // (B, H, Npad) float32 workspace: -lse * log2(e), -inf on padding rows
  int rows_in_dq;        // 1: the dQ kernel forms -D and -lse2 from o, dout, lse and writes them
  int B, H, Hkv, N, Npad, G, d;  // N: query rows per head (Npad: rounded up to 128)
  int nq;                // ceil(N / 128): query tiles
  int Nk, nkv;           // key/value rows per head, ceil(Nk / 128) key tiles
  int koff;              // causal: query row i sits at position koff + i (Nk - N)
  float scale;           // softmax scale
  float scale_log2;      // scale * log2(e)
  int* status;
  unsigned long long limit_ns;
  int* info;
  VarlenArgs vl;         // varlen: N / Nk above are the longest sequences
  int vec_stride;        // varlen: workspace floats per head (see varlen_vec_offset)
  uint16_t* dq;          // varlen: output bases, for the rows of a sequence's last tile
  uint16_t* dk;
  uint16_t* dv;
  MaskArgs mk;           // masked instances only
  int debug_drop1;       // 0; n > 0 only in a test of the bounded waits: CTA 0's producer skips ring load n - 1
  int tail;              // heads in the level-major tail of the CTA order (work_unit); set by each launcher
  int debug_plant;       // 0; 2 only in a test of the debug build's checks: CTA 0 of the dQ kernel offsets its row-vector store out of range
  int* sched;            // persistent dQ and dK/dV kernels: this launch's queue (next unit, CTAs done); set by its launcher
  int n_units;           // persistent dQ and dK/dV kernels: units in the launch
  int debug_drop_p;      // 0; n > 0 only in a test of the bounded waits: the persistent dK/dV kernel skips unit 0's
                         // Q load n - 1, the persistent dQ kernel its K load n - 1
};

// CTA order of the forward, dQ and dK/dV launches.  A launch's CTAs cover
// (head, level) work units, level 0 the heaviest (the longest causal walk).
// Head-major order keeps the CTAs in flight on few heads, whose streamed
// operands (K and V; Q and dO for dK/dV) are read once from HBM and then
// from L2, but it ends on the heaviest unit of the last head and the other
// SMs idle meanwhile.  So the last `tail` heads go level-major instead: all
// their level-0 units, then all level-1 units, and so on, and the launch
// ends on its lightest units.  tail = 1 is head-major order throughout.
__host__ __device__ __forceinline__ void work_unit(int cta, int nlev, int nheads, int tail, int& head, int& level) {
  const int lead = (nheads - tail) * nlev;  // CTAs of the head-major part
  if (cta < lead) {
    head = cta / nlev;
    level = cta - head * nlev;
  } else {
    const int c = cta - lead;
    level = c / tail;
    head = nheads - tail + (c - level * tail);
  }
}

// Every level of a launch does the same work (no causal edge, window, key
// lengths, tile mask or packed batch): the tail gains nothing there, and
// head-major order keeps each head's CTAs together in L2.
inline bool uniform_levels(bool causal, const VarlenArgs& vl, const MaskArgs& mk, bool masked) {
  return !causal && vl.cu_q == nullptr &&
         (!masked || (mk.wl < 0 && mk.wr < 0 && mk.key_len == nullptr && mk.flags == nullptr));
}

// The level-major tail: whole groups of `group` heads (those that share K
// and V), enough for about three waves of CTAs on this device's SMs, or all
// heads.
inline int order_tail(int nlev, int nheads, int group) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 152;
  int t = (3 * sms + nlev - 1) / (nlev > 0 ? nlev : 1);
  t = (t + group - 1) / group * group;
  return t < nheads ? (t > 0 ? t : 1) : nheads;
}

// Decode (split over the keys) arguments.
constexpr int kDecMaxRows = 128;  // G * Nq query rows per K/V head (one 128-row MMA tile)
struct DecParams {
  const uint16_t* q;     // (B, H, Nq, d) bf16
  uint16_t* o;           // (B, H, Nq, d) bf16
  float* lse;            // (B, H, Nq)
  float* o_part;         // (B, H, Nq, nsplit, d) float32 workspace
  float* lse_part;       // (B, H, Nq, nsplit) float32 workspace
  int B, H, Hkv, G, Nq, Nk;
  int nsplit, split_keys;  // key chunks: [s * split_keys, min(Nk, (s + 1) * split_keys))
  float scale_log2;
  int* status;
  unsigned long long limit_ns;
  int* info;
  // Paged KV cache (the paged instance): K / V as (num_pages, page_size, Hkv,
  // d), batch element b's logical page i in physical page block_table[b *
  // max_pages + i], seq_lens[b] cached keys; a 128-key tile is loaded as
  // 128 / box_rows boxes of box_rows = min(page_size, 128) tokens.
  const int* block_table;
  const int* seq_lens;
  int page_size, max_pages, num_pages, box_rows;
};

// Device status value for cu_seqlens that are out of range (a sequence longer
// than the stated maximum, decreasing offsets, or past the packed length).
constexpr int kDevBadSeqlens = 9;

// Predicate checks of the debug build (-DATTN_DEBUG).  ATTN_IN_RANGE(i, n,
// params, site) guards a plain global load or store whose element index i
// a kernel computes: in the debug build it is 0 <= i < n, and a failure
// records kDevCheckFailed in the device status word and, if it is the first
// failure on the device, (site << 16, CTA, thread, i) in the record that
// attn_get_timeout_info reads; the caller then skips the access.  No trap,
// no assert: the launch completes and the context stays usable.  In the
// release build the macro is `true` and its arguments are not evaluated.
constexpr int kDevCheckFailed = 10;
#ifdef ATTN_DEBUG
__device__ __noinline__ inline bool check_failed(int* status, int* info, int site, long long i) {
  if (atomicCAS(status, 0, kDevCheckFailed) == 0 && info != nullptr) {
    info[0] = site << 16;
    info[1] = (int)(blockIdx.x + gridDim.x * blockIdx.y);
    info[2] = (int)threadIdx.x;
    info[3] = (int)(i < -2147483647ll ? -2147483647ll : i > 2147483647ll ? 2147483647ll : i);
  }
  return false;
}
__device__ __forceinline__ bool in_range(long long i, long long n, int* status, int* info, int site) {
  return (i >= 0 && i < n) ? true : check_failed(status, info, site, i);
}
#define ATTN_IN_RANGE(i, n, prm, site) \
  ::sdpa::in_range((long long)(i), (long long)(n), (prm).status, (prm).info, (site))
constexpr bool kDebugChecks = true;
#else
#define ATTN_IN_RANGE(i, n, prm, site) true
constexpr bool kDebugChecks = false;
#endif

// Floats in each of the backward's row-vector arrays (-D, -lse2).
__host__ __device__ inline size_t vec_floats(const BwdParams& p) {
  return p.vl.cu_q != nullptr ? (size_t)p.H * p.vec_stride : (size_t)p.B * p.H * p.Npad;
}

// Varlen backward workspace: per head, sequence b's row vectors start at
// float offset varlen_vec_offset(cu_q[b], b) (16-byte aligned) and span
// ceil(Nq_b / 128) * 128 floats, the rows past Nq_b holding the padding
// values.  Regions of consecutive sequences never overlap; every region ends
// below varlen_vec_stride(total_q, B) floats.
__host__ __device__ inline long long varlen_vec_offset(long long q0, long long b) {
  return ((q0 + 132 * b) + 3) / 4 * 4;
}
__host__ __device__ inline long long varlen_vec_stride(long long total_q, long long B) {
  return varlen_vec_offset(total_q, B) + 128;
}

#ifdef __CUDACC__
// floor(a / 128) for any sign of a.
__device__ __forceinline__ int floor_div128(int a) { return a >= 0 ? a / 128 : -((127 - a) / 128); }

// Mask plane of batch b, head h.
__device__ __forceinline__ int mask_plane(const MaskArgs& mk, int b, int h) {
  return (mk.mask_b > 1 ? b : 0) * mk.mask_h + (mk.mask_h > 1 ? h : 0);
}
__device__ __forceinline__ int bias_plane(const MaskArgs& mk, int b, int h) {
  return (mk.bias_b > 1 ? b : 0) * mk.bias_h + (mk.bias_h > 1 ? h : 0);
}

// n (<= CNT) consecutive values of an additive mask, element `off` of the
// array at `base` on, as float (float32 storage, or bf16 when BF16); the
// rest of out[] is 0.  vec: the values start 16-byte aligned and n is a
// multiple of 16 bytes' worth (4 float32, 8 bf16), so 16-byte loads are used.
template <int CNT, bool BF16>
__device__ __forceinline__ void load_bias_row(const void* base, size_t off, int n, bool vec, float (&out)[CNT]) {
#pragma unroll
  for (int i = 0; i < CNT; ++i) out[i] = 0.f;
  if constexpr (BF16) {
    const uint16_t* r = static_cast<const uint16_t*>(base) + off;
    if (vec) {
#pragma unroll
      for (int i = 0; i < CNT; i += 8) {
        if (i < n) {
          const uint4 u = __ldg(reinterpret_cast<const uint4*>(r + i));
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            out[i + 2 * e] = __uint_as_float(w[e] << 16);
            out[i + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
          }
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < CNT; ++i)
        if (i < n) out[i] = __uint_as_float((uint32_t)__ldg(r + i) << 16);
    }
  } else {
    const float* r = static_cast<const float*>(base) + off;
    if (vec) {
#pragma unroll
      for (int i = 0; i < CNT; i += 4) {
        if (i < n) {
          const float4 v = __ldg(reinterpret_cast<const float4*>(r + i));
          out[i] = v.x;
          out[i + 1] = v.y;
          out[i + 2] = v.z;
          out[i + 3] = v.w;
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < CNT; ++i)
        if (i < n) out[i] = __ldg(r + i);
    }
  }
}
// Whether rows of length `len` of an additive mask array at `base` start
// 16-byte aligned (element size 2 for bf16, else 4).
__device__ __forceinline__ bool bias_rows_vec(const void* base, int len, bool bf16) {
  return (reinterpret_cast<uintptr_t>(base) & 15) == 0 && (len & (bf16 ? 7 : 3)) == 0;
}

// One sequence of a (possibly packed) batch as a kernel sees it.
struct SeqView {
  int q0, nq;  // first query row in the tensor map, query rows
  int k0, nk;  // first key row, key rows
  bool ok;     // offsets consistent with the packed lengths and maxima
};
__device__ __forceinline__ SeqView seq_view(const VarlenArgs& vl, int b, int Nq, int Nk) {
  SeqView v{0, Nq, 0, Nk, true};
  if (vl.cu_q != nullptr) {
    v.q0 = vl.cu_q[b];
    v.nq = vl.cu_q[b + 1] - v.q0;
    v.k0 = vl.cu_k[b];
    v.nk = vl.cu_k[b + 1] - v.k0;
    v.ok = v.q0 >= 0 && v.nq >= 0 && v.nq <= Nq && v.q0 <= vl.total_q - v.nq && v.k0 >= 0 && v.nk >= 0 &&
           v.nk <= Nk && v.k0 <= vl.total_k - v.nk;
  }
  return v;
}
#endif

// Shared-memory bytes of each kernel instance (for validation and launch).
size_t fwd_smem_bytes(int d);
size_t bwd_smem_bytes(int d);
size_t bwd_dq_smem_bytes(int d);
size_t decode_smem_bytes(int d);

// masked: the instance that applies p.mk (causal then enters as wr = 0).
// tb (masked, bf16 additive mask only): a map over the mask as (planes, Nq,
// Nk) bf16 with boxes of 128 rows x 64 columns, 128-byte swizzle; given, the
// kernel stages the mask's tiles by TMA instead of per-thread loads.
// The dense forward (no mask, no packed batch) as a persistent kernel; O is
// written through p.o, laid out as (B, H, Nq, d).
cudaError_t launch_fwd_persist(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const FwdParams& p, cudaStream_t stream);
cudaError_t launch_fwd(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdParams& p, cudaStream_t stream, bool masked = false,
                       const CUtensorMap* tb = nullptr);

// FP8 (e4m3) forward, head_dim d in {64, 96, 128}, dense (B, H, N, d) e4m3
// Q, K, V (maps of bytes, boxes of 128 x 128 bytes zero-filled past d), O
// bf16 through p.o; p.scale_log2 carries q_scale * k_scale.
cudaError_t launch_fwd_fp8(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const FwdParams& p, cudaStream_t stream);

cudaError_t launch_bwd_prep(const BwdParams& p, cudaStream_t stream);
// The dK/dV kernel of the dense backward (no mask, no packed batch) as a
// persistent kernel; dK and dV are written through p.dk and p.dv.
cudaError_t launch_bwd_grad_persist(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                    const CUtensorMap& tv, const CUtensorMap& tdo, const BwdParams& p,
                                    cudaStream_t stream);
// The dQ kernel of the dense backward (no mask, no packed batch) as a
// persistent kernel; dQ is written through p.dq, and with p.rows_in_dq the
// row vectors are formed from p.o, p.dout and p.lse.
cudaError_t launch_bwd_dq_persist(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                  const CUtensorMap& tv, const CUtensorMap& tdo, const BwdParams& p,
                                  cudaStream_t stream);
// tbt (masked, bf16 additive mask, no boolean mask): a map over the mask's
// transpose (planes, Nk, Nq) with boxes of 128 rows x 64 columns, 128-byte
// swizzle; given, the dK/dV kernel stages its tiles by TMA.
cudaError_t launch_bwd_grad(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                            const BwdParams& p, cudaStream_t stream, bool masked = false,
                            const CUtensorMap* tbt = nullptr);
// `to` (a map over O laid out as Q) is read only when p.rows_in_dq is set.
cudaError_t launch_bwd_dq(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& to, const BwdParams& p,
                          cudaStream_t stream, bool masked = false);
// Writes the (planes, Nk, Nq) transpose of a (planes, Nq, Nk) additive mask,
// float32 or bf16 (the dK/dV kernel reads it by key row).
cudaError_t launch_bias_transpose(const void* bias, bool bf16, int planes, int Nq, int Nk, void* bias_t,
                                  cudaStream_t stream);
// Packs a boolean (mask_b, mask_h, Nq, Nk) byte mask into the row and
// transposed bit layouts of MaskArgs (bits_t may be null: row bits only).
cudaError_t launch_mask_pack(const uint8_t* mask, int mask_b, int mask_h, int Nq, int Nk, uint32_t* bits,
                             int words, uint32_t* bits_t, int words_t, uint8_t* flags, cudaStream_t stream);
// paged: tk / tv are 4-D maps over (d, Hkv, page_size, num_pages).
cudaError_t launch_decode(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const DecParams& p, cudaStream_t stream, bool paged = false);

}  // namespace sdpa
