// attn_noalloc.cu — attn_bwd_noalloc: the backward pass for callers that
// cannot allocate device memory.
//
// attn_bwd needs a caller-supplied float32 workspace (two per-row vectors,
// D = rowsum(dO * O) and the logsumexp in base 2).  Some callers cannot provide one: code that runs
// where cudaMalloc is not allowed or not wanted, such as a custom allocator
// that must not recurse into itself, a runtime that has already handed all
// device memory to its own pool, or a plug-in ABI that passes only tensor
// pointers.  For them this file keeps the workspace in a fixed,
// statically sized device array that is part of the library image, so the
// call itself allocates nothing.
//
// The array is kSdpaNoallocScratchBytes (64 MiB) per GPU.  Every GPU that
// loads the library holds it until the process exits.  All calls share it:
// two calls whose kernels overlap on the GPU (on different streams, or from
// different host threads) race on it and give wrong results.
//
// The array's device address is looked up once per device and kept for the
// life of the process, so the library supports the primary context only: a
// cudaDeviceReset (or a non-primary driver context) makes the kept address
// stale.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/attn.h"

namespace {

constexpr size_t kSdpaNoallocScratchBytes = 64ull << 20;
constexpr int kMaxNoallocDevices = 64;

// The scratch.  In host code this name is only a host-side stand-in for the
// symbol, not a device address: the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kSdpaNoallocScratchBytes];

void* g_scratch_ptr[kMaxNoallocDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch on the current device, looked up once per
// device (with that device current).
attn_status_t scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxNoallocDevices) return ATTN_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" {

// attn_bwd's checks (arguments, then the device), in attn_api.cu.
attn_status_t sdpa_bwd_check_args(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                  const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int N,
                                  int d, float scale, int causal);

attn_status_t attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                               const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int N, int d,
                               float scale, int causal, void* stream) {
  const size_t need = attn_bwd_workspace_size(B, H, Hkv, N, d);
  if (need == 0) return ATTN_ERR_UNSUPPORTED_SHAPE;
  if (need > kSdpaNoallocScratchBytes) return ATTN_ERR_WORKSPACE;  // shape too large for the fixed scratch
  // Every other invalid argument, and an unsupported device, get attn_bwd's
  // own status before the scratch is looked up.
  attn_status_t s = sdpa_bwd_check_args(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, N, d, scale, causal);
  if (s != ATTN_OK) return s;
  void* scratch = nullptr;
  s = scratch_address(&scratch);
  if (s != ATTN_OK) return s;
  // attn_bwd's first kernel (dQ) writes both row vectors of every row
  // before the dK/dV kernel reads them, so a call that completes without a
  // timeout reads nothing an earlier call left in the scratch.  After a
  // timeout (ATTN_ERR_TIMEOUT from attn_get_device_status) some row vectors
  // may be an earlier call's, so dK and dV of that call must be discarded.
  return attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, scratch, kSdpaNoallocScratchBytes, B, H, Hkv, N, d, scale,
                  causal, stream);
}

}  // extern "C"
