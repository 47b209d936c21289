// kernels.h — internal launch interface between the C ABI (attn_api.cu) and
// the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace sdpa {

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
};

// Backward arguments.
struct BwdParams {
  const uint16_t* o;     // (B, H, N, d) bf16
  const uint16_t* dout;  // (B, H, N, d) bf16
  const float* lse;      // (B, H, N)
  float* dvec;           // (B, H, Npad) float32 workspace: -D = -rowsum(dO * O)
  float* lse2;           // (B, H, Npad) float32 workspace: -lse * log2(e), -inf on padding rows
  int B, H, Hkv, N, Npad, G, d;  // N: query rows per head (Npad: rounded up to 128)
  int nq;                // ceil(N / 128): query tiles
  int Nk, nkv;           // key/value rows per head, ceil(Nk / 128) key tiles
  int koff;              // causal: query row i sits at position koff + i (Nk - N)
  float scale;           // softmax scale
  float scale_log2;      // scale * log2(e)
  int* status;
  unsigned long long limit_ns;
  int* info;
};

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
};

// Shared-memory bytes of each kernel instance (for validation and launch).
size_t fwd_smem_bytes(int d);
size_t bwd_smem_bytes(int d);
size_t bwd_dq_smem_bytes(int d);
size_t decode_smem_bytes(int d);

cudaError_t launch_fwd(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdParams& p, cudaStream_t stream);

cudaError_t launch_bwd_prep(const BwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd_grad(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                            const BwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd_dq(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParams& p, cudaStream_t stream);
cudaError_t launch_decode(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const DecParams& p, cudaStream_t stream);

}  // namespace sdpa
