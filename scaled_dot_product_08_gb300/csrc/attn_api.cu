// attn_api.cu — the C ABI declared in include/attn.h: argument validation,
// TMA tensor-map construction, device checks, the device status word and the
// bounded-wait self-test.  No computation happens here; every step of the
// attention path runs in the kernels of attn_fwd.cu / attn_bwd.cu.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/attn.h"
#include "kernels.h"
#include "ptx.cuh"

#define ATTN_TRY_INNER(x)               \
  do {                                  \
    attn_status_t _s = (x);             \
    if (_s != ATTN_OK) return _s;       \
  } while (0)

namespace {

constexpr int kMaxDevices = 64;

// Limit of each on-chip wait: 2 s, or SDPA08_WAIT_LIMIT_MS milliseconds
// (1 .. 60000) when that environment variable is set at the first call.
unsigned long long wait_limit_ns() {
  static unsigned long long lim = [] {
    unsigned long long v = 2000000000ull;
    if (const char* e = std::getenv("SDPA08_WAIT_LIMIT_MS")) {
      const long ms = std::strtol(e, nullptr, 10);
      if (ms >= 1 && ms <= 60000) v = (unsigned long long)ms * 1000000ull;
    }
    return v;
  }();
  return lim;
}

// The dropped-load test hook (attn_debug_drop_load): armed for one launch of
// one kernel, then cleared.  kernel: 0 forward, 1 dQ, 2 dK/dV, and the
// persistent kernels 3 forward, 4 dK/dV, 5 dQ; 6 the FP8 forward.
std::mutex g_debug_mu;
int g_debug_kernel = -1, g_debug_drop1 = 0;
unsigned long long g_debug_limit_ns = 0;

// Applies (and clears) the hook when it is armed for `kernel`.
void take_debug(int kernel, int* drop1, unsigned long long* limit_ns) {
  std::lock_guard<std::mutex> lk(g_debug_mu);
  if (g_debug_kernel != kernel) return;
  *drop1 = g_debug_drop1;
  *limit_ns = g_debug_limit_ns;
  g_debug_kernel = -1;
}

// The planted-index test hook of the debug build (attn_debug_plant_index):
// armed for one launch of one kernel (0 forward, 1 dQ), then cleared.
int g_plant_kernel = -1;

// Sets *plant = value (and clears the hook) when it is armed for `kernel`.
void take_plant(int kernel, int* plant, int value) {
  std::lock_guard<std::mutex> lk(g_debug_mu);
  if (g_plant_kernel != kernel) return;
  *plant = value;
  g_plant_kernel = -1;
}

// Written by kernels when a bounded wait gives up (0 = fine), and where the
// first such timeout happened.
__device__ int g_status_word;
__device__ int g_timeout_info[4];

struct DeviceInfo {
  bool probed = false;
  bool supported = false;
  int* status = nullptr;  // device address of g_status_word
  int* info = nullptr;    // device address of g_timeout_info
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Probes the current device once: compute capability 10.3 and the device
// address of the status word (cudaGetSymbolAddress, with that device current).
attn_status_t current_device(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.probed) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    di.supported = (major == 10 && minor == 3);
    if (di.supported) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return ATTN_ERR_CUDA;
      di.status = static_cast<int*>(p);
      if (cudaGetSymbolAddress(&p, g_timeout_info) != cudaSuccess) return ATTN_ERR_CUDA;
      di.info = static_cast<int*>(p);
    }
    di.probed = true;
  }
  if (!di.supported) return ATTN_ERR_UNSUPPORTED_DEVICE;
  *out = &di;
  return ATTN_OK;
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link-time dependency on libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D map over a dense bf16 (rows = B*heads, N, d) tensor: box of 64 columns
// (128 bytes) x 128 rows x 1 head, 128-byte swizzle.  Rows past N and
// columns past d read as zero and are never written.
bool make_map_bf16(CUtensorMap* m, const void* ptr, int d, int N, long long heads) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * (cuuint64_t)N};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over a packed (total, heads, d) bf16 tensor (sequences one after
// another, token-major): dims (d, total, heads), so a box of 128 rows x 1
// head is 128 consecutive tokens of one head, and the kernels address it
// exactly like the dense map (row, plane = head).
bool make_map_bf16_packed(CUtensorMap* m, const void* ptr, int d, long long total, int heads) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)total, (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)heads * d * 2, (cuuint64_t)d * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// e4m3 (B*heads, N, d) as planes of [N x d] bytes; boxes of 128 rows x 128
// bytes, the bytes past d read as zeros.
bool make_map_e4m3(CUtensorMap* m, const void* ptr, int d, int N, long long heads) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)d, (cuuint64_t)d * (cuuint64_t)N};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks shared by forward and backward.
attn_status_t check_shape(int B, int H, int Hkv, int N, int d) {
  if (B < 1 || H < 1 || Hkv < 1 || N < 1) return ATTN_ERR_UNSUPPORTED_SHAPE;
  if (d != 64 && d != 96 && d != 128) return ATTN_ERR_UNSUPPORTED_SHAPE;
  if (H % Hkv != 0) return ATTN_ERR_UNSUPPORTED_SHAPE;
  const long long bh = (long long)B * H;
  const long long ntile = (N + 255) / 256;
  if (bh > (1ll << 30) || (long long)N > (1ll << 30) || bh * ntile > 0x7fffffffll ||
      bh * ((N + 127) / 128) > 0x7fffffffll)
    return ATTN_ERR_UNSUPPORTED_SHAPE;
  return ATTN_OK;
}

attn_status_t check_scale_flag(float scale, int causal) {
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

// Every pointer must be non-null and 16-byte aligned (checked on the host,
// for all pointers, before any CUDA call) and must be device memory.
attn_status_t check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p == nullptr) return ATTN_ERR_INVALID_ARG;
  for (const void* p : ps)
    if (!aligned16(p)) return ATTN_ERR_MISALIGNED;
  for (const void* p : ps) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_INVALID_ARG;
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return ATTN_ERR_INVALID_ARG;
  }
  return ATTN_OK;
}

// cu_seqlens arrays: non-null, int32-aligned device memory.
attn_status_t check_offsets_ptrs(const int* a, const int* b) {
  for (const int* p : {a, b}) {
    if (p == nullptr) return ATTN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(p) & 3u) return ATTN_ERR_MISALIGNED;
  }
  for (const int* p : {a, b}) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_INVALID_ARG;
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return ATTN_ERR_INVALID_ARG;
  }
  return ATTN_OK;
}

// Shape checks of a packed batch: B sequences of at most max_q query and
// max_k key rows, total_q / total_k rows in all.
attn_status_t check_varlen_shape(int B, int H, int Hkv, int total_q, int total_k, int max_q, int max_k, int d) {
  ATTN_TRY_INNER(check_shape(B, H, Hkv, max_q, d));
  ATTN_TRY_INNER(check_shape(B, H, Hkv, max_k, d));
  if (total_q < 1 || total_k < 1) return ATTN_ERR_UNSUPPORTED_SHAPE;
  if ((long long)total_q > (long long)B * max_q || (long long)total_k > (long long)B * max_k)
    return ATTN_ERR_UNSUPPORTED_SHAPE;  // some sequence would be longer than its maximum
  if ((long long)total_q * H > (1ll << 31) || (long long)total_k * Hkv > (1ll << 31)) return ATTN_ERR_UNSUPPORTED_SHAPE;
  if ((long long)H * d * 128 >= (1ll << 32)) return ATTN_ERR_UNSUPPORTED_SHAPE;  // 32-bit tile row offsets
  if (sdpa::varlen_vec_stride(total_q, B) >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED_SHAPE;
  return ATTN_OK;
}

__global__ void selftest_wait_kernel(int* status, int* info, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    sdpa::mbar_init(sdpa::smem_u32(&bar), 1);
    abort_flag = 0;
    sdpa::fence_mbar_init();
  }
  __syncthreads();
  const sdpa::WaitCtx wc{&abort_flag, status, limit_ns, info};
  // Nothing ever arrives on `bar`: every thread must give up and return.
  (void)sdpa::wait_bounded(wc, sdpa::smem_u32(&bar), 0, sdpa::wait_site(0x01, 0));
  __syncthreads();
}

}  // namespace

#define ATTN_TRY(x)                     \
  do {                                  \
    attn_status_t _s = (x);             \
    if (_s != ATTN_OK) return _s;       \
  } while (0)

extern "C" {

int attn_abi_version(void) { return 3; }

const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED_SHAPE: return "ATTN_ERR_UNSUPPORTED_SHAPE";
    case ATTN_ERR_UNSUPPORTED_DEVICE: return "ATTN_ERR_UNSUPPORTED_DEVICE";
    case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
    case ATTN_ERR_LAUNCH: return "ATTN_ERR_LAUNCH";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_CHECK: return "ATTN_ERR_CHECK";
  }
  return "ATTN_ERR_UNKNOWN";
}

// Forward over Nq query rows and Nk key rows per head (Nq == Nk for
// attn_fwd); causal rows sit at positions Nk - Nq + i.
static attn_status_t fwd_common(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                int Hkv, int Nq, int Nk, int d, float scale, int causal, void* stream) {
  ATTN_TRY(check_shape(B, H, Hkv, Nq, d));
  ATTN_TRY(check_shape(B, H, Hkv, Nk, d));
  ATTN_TRY(check_scale_flag(scale, causal));
  if (causal && Nq > Nk) return ATTN_ERR_UNSUPPORTED_SHAPE;  // a causal row would see no key
  ATTN_TRY(check_ptrs({q, k, v, o, lse}));
  DeviceInfo* di = nullptr;
  ATTN_TRY(current_device(&di));

  CUtensorMap tq, tk, tv, to;
  if (!make_map_bf16(&tq, q, d, Nq, (long long)B * H) || !make_map_bf16(&tk, k, d, Nk, (long long)B * Hkv) ||
      !make_map_bf16(&tv, v, d, Nk, (long long)B * Hkv) || !make_map_bf16(&to, o, d, Nq, (long long)B * H))
    return ATTN_ERR_CUDA;

  sdpa::FwdParams p;
  memset(&p, 0, sizeof(p));
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.G = H / Hkv;
  p.Nq = Nq;
  p.Nk = Nk;
  p.koff = causal ? Nk - Nq : 0;
  p.n_mtiles = (Nq + 255) / 256;
  p.nkv = (Nk + 127) / 128;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = di->status;
  p.limit_ns = wait_limit_ns();
  p.info = di->info;
  take_debug(0, &p.debug_drop1, &p.limit_ns);
  take_debug(3, &p.debug_drop_p, &p.limit_ns);
  take_plant(0, &p.debug_plant, 1);
  p.o = static_cast<uint16_t*>(o);  // (the persistent kernel writes O directly)
  cudaError_t e = sdpa::launch_fwd(d, causal != 0, tq, tk, tv, to, p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv,
                       int N, int d, float scale, int causal, void* stream) {
  return fwd_common(q, k, v, o, lse, B, H, Hkv, N, N, d, scale, causal, stream);
}

attn_status_t attn_fwd_cross(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                             int Hkv, int Nq, int Nk, int d, float scale, int causal, void* stream) {
  return fwd_common(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, scale, causal, stream);
}

attn_status_t attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                              const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H, int Hkv, int total_q,
                              int total_k, int max_seqlen_q, int max_seqlen_k, int d, float scale, int causal,
                              void* stream) {
  ATTN_TRY(check_varlen_shape(B, H, Hkv, total_q, total_k, max_seqlen_q, max_seqlen_k, d));
  ATTN_TRY(check_scale_flag(scale, causal));
  ATTN_TRY(check_ptrs({q, k, v, o, lse}));
  ATTN_TRY(check_offsets_ptrs(cu_seqlens_q, cu_seqlens_k));
  DeviceInfo* di = nullptr;
  ATTN_TRY(current_device(&di));

  CUtensorMap tq, tk, tv, to;
  if (!make_map_bf16_packed(&tq, q, d, total_q, H) || !make_map_bf16_packed(&tk, k, d, total_k, Hkv) ||
      !make_map_bf16_packed(&tv, v, d, total_k, Hkv) || !make_map_bf16_packed(&to, o, d, total_q, H))
    return ATTN_ERR_CUDA;

  sdpa::FwdParams p;
  memset(&p, 0, sizeof(p));
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.G = H / Hkv;
  p.Nq = max_seqlen_q;
  p.Nk = max_seqlen_k;
  p.n_mtiles = (max_seqlen_q + 255) / 256;
  p.nkv = (max_seqlen_k + 127) / 128;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = di->status;
  p.limit_ns = wait_limit_ns();
  p.info = di->info;
  p.vl.cu_q = cu_seqlens_q;
  p.vl.cu_k = cu_seqlens_k;
  p.vl.total_q = total_q;
  p.vl.total_k = total_k;
  p.o = static_cast<uint16_t*>(o);
  cudaError_t e = sdpa::launch_fwd(d, causal != 0, tq, tk, tv, to, p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

size_t attn_bwd_workspace_size(int B, int H, int Hkv, int N, int d) {
  if (check_shape(B, H, Hkv, N, d) != ATTN_OK) return 0;
  const size_t npad = (size_t)((N + 127) / 128) * 128;
  const size_t rows = (size_t)B * H * npad;
  return rows * 4 * 2;  // -D and -lse*log2(e) per (head, padded row), float32
}

// Workspace carve-up shared by the three backward stages: [-D | -lse2], one
// float per (head, padded query row).  Nq query rows, Nk key rows; causal
// query row i sits at position Nk - Nq + i.
static void bwd_params(sdpa::BwdParams* p, void* workspace, int B, int H, int Hkv, int Nq, int Nk, int d,
                       float scale, int causal, const DeviceInfo* di) {
  const int npad = ((Nq + 127) / 128) * 128;
  const size_t rows = (size_t)B * H * npad;
  memset(p, 0, sizeof(*p));
  p->dvec = static_cast<float*>(workspace);
  p->lse2 = p->dvec + rows;
  p->B = B;
  p->H = H;
  p->Hkv = Hkv;
  p->N = Nq;
  p->Npad = npad;
  p->G = H / Hkv;
  p->d = d;
  p->nq = (Nq + 127) / 128;
  p->Nk = Nk;
  p->nkv = (Nk + 127) / 128;
  p->koff = causal ? Nk - Nq : 0;
  p->scale = scale;
  p->scale_log2 = scale * 1.4426950408889634f;
  p->status = di->status;
  p->limit_ns = wait_limit_ns();
  p->info = di->info;
}

static attn_status_t check_workspace(void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int N, int d) {
  if (workspace == nullptr || workspace_bytes < attn_bwd_workspace_size(B, H, Hkv, N, d)) return ATTN_ERR_WORKSPACE;
  return ATTN_OK;
}

static attn_status_t check_bwd_shape(int B, int H, int Hkv, int Nq, int Nk, int d, int causal) {
  ATTN_TRY(check_shape(B, H, Hkv, Nq, d));
  ATTN_TRY(check_shape(B, H, Hkv, Nk, d));
  if (causal == 1 && Nq > Nk) return ATTN_ERR_UNSUPPORTED_SHAPE;  // a causal row would see no key
  return ATTN_OK;
}

static attn_status_t bwd_prep_x(const void* o, const float* lse, const void* dout, void* workspace,
                                size_t workspace_bytes, int B, int H, int Hkv, int Nq, int d, void* stream) {
  ATTN_TRY(check_shape(B, H, Hkv, Nq, d));
  ATTN_TRY(check_workspace(workspace, workspace_bytes, B, H, Hkv, Nq, d));
  ATTN_TRY(check_ptrs({o, lse, dout, workspace}));
  DeviceInfo* di = nullptr;
  ATTN_TRY(current_device(&di));
  sdpa::BwdParams p;
  bwd_params(&p, workspace, B, H, Hkv, Nq, Nq, d, 1.f, 0, di);
  p.o = static_cast<const uint16_t*>(o);
  p.dout = static_cast<const uint16_t*>(dout);
  p.lse = lse;
  return sdpa::launch_bwd_prep(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

static attn_status_t bwd_grad_x(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv,
                                void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int Nq, int Nk, int d,
                                float scale, int causal, void* stream) {
  ATTN_TRY(check_scale_flag(scale, causal));
  ATTN_TRY(check_bwd_shape(B, H, Hkv, Nq, Nk, d, causal));
  ATTN_TRY(check_workspace(workspace, workspace_bytes, B, H, Hkv, Nq, d));
  ATTN_TRY(check_ptrs({q, k, v, dout, dk, dv, workspace}));
  DeviceInfo* di = nullptr;
  ATTN_TRY(current_device(&di));
  CUtensorMap tq, tk, tv, tdo, tdk, tdv;
  if (!make_map_bf16(&tq, q, d, Nq, (long long)B * H) || !make_map_bf16(&tk, k, d, Nk, (long long)B * Hkv) ||
      !make_map_bf16(&tv, v, d, Nk, (long long)B * Hkv) || !make_map_bf16(&tdo, dout, d, Nq, (long long)B * H) ||
      !make_map_bf16(&tdk, dk, d, Nk, (long long)B * Hkv) || !make_map_bf16(&tdv, dv, d, Nk, (long long)B * Hkv))
    return ATTN_ERR_CUDA;
  sdpa::BwdParams p;
  bwd_params(&p, workspace, B, H, Hkv, Nq, Nk, d, scale, causal, di);
  p.dk = static_cast<uint16_t*>(dk);
  p.dv = static_cast<uint16_t*>(dv);
  take_debug(2, &p.debug_drop1, &p.limit_ns);
  take_debug(4, &p.debug_drop_p, &p.limit_ns);
  cudaError_t e = sdpa::launch_bwd_grad(d, causal != 0, tq, tk, tv, tdo, tdk, tdv, p,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

static attn_status_t bwd_dq_x(const void* q, const void* k, const void* v, const void* dout, void* dq, void* workspace,
                              size_t workspace_bytes, int B, int H, int Hkv, int Nq, int Nk, int d, float scale,
                              int causal, void* stream) {
  ATTN_TRY(check_scale_flag(scale, causal));
  ATTN_TRY(check_bwd_shape(B, H, Hkv, Nq, Nk, d, causal));
  ATTN_TRY(check_workspace(workspace, workspace_bytes, B, H, Hkv, Nq, d));
  ATTN_TRY(check_ptrs({q, k, v, dout, dq, workspace}));
  DeviceInfo* di = nullptr;
  ATTN_TRY(current_device(&di));
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (!make_map_bf16(&tq, q, d, Nq, (long long)B * H) || !make_map_bf16(&tk, k, d, Nk, (long long)B * Hkv) ||
      !make_map_bf16(&tv, v, d, Nk, (long long)B * Hkv) || !make_map_bf16(&tdo, dout, d, Nq, (long long)B * H) ||
      !make_map_bf16(&tdq, dq, d, Nq, (long long)B * H))
    return ATTN_ERR_CUDA;
  sdpa::BwdParams p;
  bwd_params(&p, workspace, B, H, Hkv, Nq, Nk, d, scale, causal, di);
  p.dq = static_cast<uint16_t*>(dq);
  take_debug(1, &p.debug_drop1, &p.limit_ns);
  take_debug(5, &p.debug_drop_p, &p.limit_ns);
  cudaError_t e =
      sdpa::launch_bwd_dq(d, causal != 0, tq, tk, tv, tdo, tdq, tq, p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

// The dQ stage that forms and writes the row vectors itself (from o, lse,
// dout): replaces prep + dq, and grad runs after it.
static attn_status_t bwd_dq_rows_x(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                   const void* dout, void* dq, void* workspace, size_t workspace_bytes, int B, int H,
                                   int Hkv, int Nq, int Nk, int d, float scale, int causal, void* stream) {
  ATTN_TRY(check_scale_flag(scale, causal));
  ATTN_TRY(check_bwd_shape(B, H, Hkv, Nq, Nk, d, causal));
  ATTN_TRY(check_workspace(workspace, workspace_bytes, B, H, Hkv, Nq, d));
  ATTN_TRY(check_ptrs({q, k, v, o, lse, dout, dq, workspace}));
  DeviceInfo* di = nullptr;
  ATTN_TRY(current_device(&di));
  CUtensorMap tq, tk, tv, tdo, tdq, to;
  if (!make_map_bf16(&tq, q, d, Nq, (long long)B * H) || !make_map_bf16(&tk, k, d, Nk, (long long)B * Hkv) ||
      !make_map_bf16(&tv, v, d, Nk, (long long)B * Hkv) || !make_map_bf16(&tdo, dout, d, Nq, (long long)B * H) ||
      !make_map_bf16(&tdq, dq, d, Nq, (long long)B * H) || !make_map_bf16(&to, o, d, Nq, (long long)B * H))
    return ATTN_ERR_CUDA;
  sdpa::BwdParams p;
  bwd_params(&p, workspace, B, H, Hkv, Nq, Nk, d, scale, causal, di);
  p.dq = static_cast<uint16_t*>(dq);
  p.lse = lse;
  p.o = static_cast<const uint16_t*>(o);  // (the persistent kernel reads O and dO rows directly)
  p.dout = static_cast<const uint16_t*>(dout);
  p.rows_in_dq = 1;
  take_debug(1, &p.debug_drop1, &p.limit_ns);
  take_debug(5, &p.debug_drop_p, &p.limit_ns);
  take_plant(1, &p.debug_plant, 2);
  cudaError_t e = sdpa::launch_bwd_dq(d, causal != 0, tq, tk, tv, tdo, tdq, to, p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

static attn_status_t bwd_all(const void* q, const void* k, const void* v, const void* o, const float* lse,
                             const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                             int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal, void* stream) {
  // Validate everything up front so that nothing is launched on a bad call.
  ATTN_TRY(check_scale_flag(scale, causal));
  ATTN_TRY(check_bwd_shape(B, H, Hkv, Nq, Nk, d, causal));
  ATTN_TRY(check_workspace(workspace, workspace_bytes, B, H, Hkv, Nq, d));
  ATTN_TRY(check_ptrs({q, k, v, o, lse, dout, dq, dk, dv, workspace}));
  ATTN_TRY(bwd_dq_rows_x(q, k, v, o, lse, dout, dq, workspace, workspace_bytes, B, H, Hkv, Nq, Nk, d, scale, causal,
                         stream));
  return bwd_grad_x(q, k, v, dout, dk, dv, workspace, workspace_bytes, B, H, Hkv, Nq, Nk, d, scale, causal, stream);
}

attn_status_t attn_bwd_prep(const void* o, const float* lse, const void* dout, void* workspace,
                            size_t workspace_bytes, int B, int H, int Hkv, int N, int d, void* stream) {
  return bwd_prep_x(o, lse, dout, workspace, workspace_bytes, B, H, Hkv, N, d, stream);
}

attn_status_t attn_bwd_grad(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv,
                            void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int N, int d,
                            float scale, int causal, void* stream) {
  return bwd_grad_x(q, k, v, dout, dk, dv, workspace, workspace_bytes, B, H, Hkv, N, N, d, scale, causal, stream);
}

attn_status_t attn_bwd_dq(const void* q, const void* k, const void* v, const void* dout, void* dq, void* workspace,
                          size_t workspace_bytes, int B, int H, int Hkv, int N, int d, float scale, int causal,
                          void* stream) {
  return bwd_dq_x(q, k, v, dout, dq, workspace, workspace_bytes, B, H, Hkv, N, N, d, scale, causal, stream);
}

attn_status_t attn_bwd_dq_rows(const void* q, const void* k, const void* v, const void* o, const float* lse,
                               const void* dout, void* dq, void* workspace, size_t workspace_bytes, int B, int H,
                               int Hkv, int Nq, int Nk, int d, float scale, int causal, void* stream) {
  return bwd_dq_rows_x(q, k, v, o, lse, dout, dq, workspace, workspace_bytes, B, H, Hkv, Nq, Nk, d, scale, causal,
                       stream);
}

// Everything attn_bwd checks except the workspace, the device included, in
// the same order (attn_bwd_noalloc runs it before it looks up its scratch).
// Internal to the library: hidden from its exported symbols.
__attribute__((visibility("hidden"))) attn_status_t sdpa_bwd_check_args(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                  const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int N,
                                  int d, float scale, int causal) {
  ATTN_TRY(check_scale_flag(scale, causal));
  ATTN_TRY(check_bwd_shape(B, H, Hkv, N, N, d, causal));
  ATTN_TRY(check_ptrs({q, k, v, o, lse, dout, dq, dk, dv}));
  DeviceInfo* di = nullptr;
  return current_device(&di);
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                       int B, int H, int Hkv, int N, int d, float scale, int causal, void* stream) {
  return bwd_all(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, H, Hkv, N, N, d, scale, causal,
                 stream);
}

attn_status_t attn_bwd_grad_cross(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv,
                                  void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int Nq, int Nk,
                                  int d, float scale, int causal, void* stream) {
  return bwd_grad_x(q, k, v, dout, dk, dv, workspace, workspace_bytes, B, H, Hkv, Nq, Nk, d, scale, causal, stream);
}

attn_status_t attn_bwd_dq_cross(const void* q, const void* k, const void* v, const void* dout, void* dq,
                                void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int Nq, int Nk,
                                int d, float scale, int causal, void* stream) {
  return bwd_dq_x(q, k, v, dout, dq, workspace, workspace_bytes, B, H, Hkv, Nq, Nk, d, scale, causal, stream);
}

attn_status_t attn_bwd_cross(const void* q, const void* k, const void* v, const void* o, const float* lse,
                             const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                             int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal, void* stream) {
  return bwd_all(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, H, Hkv, Nq, Nk, d, scale, causal,
                 stream);
}

size_t attn_bwd_varlen_workspace_size(int B, int H, int Hkv, int total_q, int d) {
  if (check_shape(B, H, Hkv, 1, d) != ATTN_OK || total_q < 1) return 0;
  return (size_t)H * (size_t)sdpa::varlen_vec_stride(total_q, B) * 4 * 2;  // -D and -lse2 per head, float32
}

// Everything the three varlen backward stages share: validation, tensor
// maps and kernel arguments.  Maps for arguments a stage does not use are
// built over placeholders that stay valid (they are never read).
struct VarlenBwd {
  CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv, to;
  sdpa::BwdParams p;
};

static attn_status_t varlen_bwd_setup(VarlenBwd* w, const void* q, const void* k, const void* v, const void* o,
                                      const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                      const int* cu_q, const int* cu_k, void* workspace, size_t workspace_bytes,
                                      int B, int H, int Hkv, int total_q, int total_k, int max_q, int max_k, int d,
                                      float scale, int causal) {
  ATTN_TRY(check_varlen_shape(B, H, Hkv, total_q, total_k, max_q, max_k, d));
  ATTN_TRY(check_scale_flag(scale, causal));
  if (workspace == nullptr || workspace_bytes < attn_bwd_varlen_workspace_size(B, H, Hkv, total_q, d))
    return ATTN_ERR_WORKSPACE;
  ATTN_TRY(check_ptrs({q, k, v, o, lse, dout, dq, dk, dv, workspace}));
  ATTN_TRY(check_offsets_ptrs(cu_q, cu_k));
  DeviceInfo* di = nullptr;
  ATTN_TRY(current_device(&di));
  if (!make_map_bf16_packed(&w->tq, q, d, total_q, H) || !make_map_bf16_packed(&w->tk, k, d, total_k, Hkv) ||
      !make_map_bf16_packed(&w->tv, v, d, total_k, Hkv) || !make_map_bf16_packed(&w->tdo, dout, d, total_q, H) ||
      !make_map_bf16_packed(&w->tdq, dq, d, total_q, H) || !make_map_bf16_packed(&w->tdk, dk, d, total_k, Hkv) ||
      !make_map_bf16_packed(&w->tdv, dv, d, total_k, Hkv) || !make_map_bf16_packed(&w->to, o, d, total_q, H))
    return ATTN_ERR_CUDA;
  sdpa::BwdParams& p = w->p;
  memset(&p, 0, sizeof(p));
  p.o = static_cast<const uint16_t*>(o);
  p.dout = static_cast<const uint16_t*>(dout);
  p.lse = lse;
  p.vec_stride = (int)sdpa::varlen_vec_stride(total_q, B);
  p.dvec = static_cast<float*>(workspace);
  p.lse2 = p.dvec + (size_t)H * p.vec_stride;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.N = max_q;
  p.G = H / Hkv;
  p.d = d;
  p.nq = (max_q + 127) / 128;
  p.Nk = max_k;
  p.nkv = (max_k + 127) / 128;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = di->status;
  p.limit_ns = wait_limit_ns();
  p.info = di->info;
  p.vl.cu_q = cu_q;
  p.vl.cu_k = cu_k;
  p.vl.total_q = total_q;
  p.vl.total_k = total_k;
  p.dq = static_cast<uint16_t*>(dq);
  p.dk = static_cast<uint16_t*>(dk);
  p.dv = static_cast<uint16_t*>(dv);
  return ATTN_OK;
}

enum : unsigned { kStagePrep = 1, kStageGrad = 2, kStageDq = 4, kStageDqRows = 8, kStagesAll = 15 };

static attn_status_t varlen_bwd_run(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                    const void* dout, void* dq, void* dk, void* dv, const int* cu_q, const int* cu_k,
                                    void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int total_q,
                                    int total_k, int max_q, int max_k, int d, float scale, int causal, void* stream,
                                    unsigned stages) {
  VarlenBwd w;
  ATTN_TRY(varlen_bwd_setup(&w, q, k, v, o, lse, dout, dq, dk, dv, cu_q, cu_k, workspace, workspace_bytes, B, H,
                            Hkv, total_q, total_k, max_q, max_k, d, scale, causal));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((stages & kStagePrep) && sdpa::launch_bwd_prep(w.p, st) != cudaSuccess) return ATTN_ERR_LAUNCH;
  if (stages & kStageDqRows) {
    sdpa::BwdParams pr = w.p;
    pr.rows_in_dq = 1;
    if (sdpa::launch_bwd_dq(d, causal != 0, w.tq, w.tk, w.tv, w.tdo, w.tdq, w.to, pr, st) != cudaSuccess)
      return ATTN_ERR_LAUNCH;
  }
  if ((stages & kStageGrad) &&
      sdpa::launch_bwd_grad(d, causal != 0, w.tq, w.tk, w.tv, w.tdo, w.tdk, w.tdv, w.p, st) != cudaSuccess)
    return ATTN_ERR_LAUNCH;
  if ((stages & kStageDq) &&
      sdpa::launch_bwd_dq(d, causal != 0, w.tq, w.tk, w.tv, w.tdo, w.tdq, w.to, w.p, st) != cudaSuccess)
    return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}

attn_status_t attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                              const void* dout, void* dq, void* dk, void* dv, const int* cu_seqlens_q,
                              const int* cu_seqlens_k, void* workspace, size_t workspace_bytes, int B, int H,
                              int Hkv, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d,
                              float scale, int causal, void* stream) {
  return varlen_bwd_run(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, workspace, workspace_bytes,
                        B, H, Hkv, total_q, total_k, max_seqlen_q, max_seqlen_k, d, scale, causal, stream,
                        kStageDqRows | kStageGrad);
}

attn_status_t attn_bwd_varlen_stages(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                     const void* dout, void* dq, void* dk, void* dv, const int* cu_seqlens_q,
                                     const int* cu_seqlens_k, void* workspace, size_t workspace_bytes, int B, int H,
                                     int Hkv, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d,
                                     float scale, int causal, unsigned stages, void* stream) {
  if (stages == 0 || (stages & ~kStagesAll) != 0) return ATTN_ERR_INVALID_ARG;
  return varlen_bwd_run(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, workspace, workspace_bytes,
                        B, H, Hkv, total_q, total_k, max_seqlen_q, max_seqlen_k, d, scale, causal, stream, stages);
}

// ------------------------------------------------------------------ FP8
attn_status_t attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv,
                           int Nq, int Nk, int d, float scale, float q_scale, float k_scale, float v_scale, int causal,
                           void* stream) {
  ATTN_TRY(check_shape(B, H, Hkv, Nq, d));
  ATTN_TRY(check_shape(B, H, Hkv, Nk, d));
  ATTN_TRY(check_scale_flag(scale, causal));
  for (float f : {q_scale, k_scale, v_scale})
    if (!std::isfinite(f) || !(f > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale * q_scale * k_scale * 1.4426950408889634f)) return ATTN_ERR_INVALID_ARG;
  if (causal && Nq > Nk) return ATTN_ERR_UNSUPPORTED_SHAPE;
  ATTN_TRY(check_ptrs({q, k, v, o, lse}));
  DeviceInfo* di = nullptr;
  ATTN_TRY(current_device(&di));
  CUtensorMap tq, tk, tv;
  if (!make_map_e4m3(&tq, q, d, Nq, (long long)B * H) || !make_map_e4m3(&tk, k, d, Nk, (long long)B * Hkv) ||
      !make_map_e4m3(&tv, v, d, Nk, (long long)B * Hkv))
    return ATTN_ERR_CUDA;
  sdpa::FwdParams p;
  memset(&p, 0, sizeof(p));
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.G = H / Hkv;
  p.Nq = Nq;
  p.Nk = Nk;
  p.koff = causal ? Nk - Nq : 0;
  p.n_mtiles = (Nq + 255) / 256;
  p.nkv = (Nk + 127) / 128;
  p.scale_log2 = scale * q_scale * k_scale * 1.4426950408889634f;
  p.o_scale = v_scale;
  p.o = static_cast<uint16_t*>(o);
  p.status = di->status;
  p.limit_ns = wait_limit_ns();
  p.info = di->info;
  take_debug(6, &p.debug_drop_p, &p.limit_ns);
  return sdpa::launch_fwd_fp8(d, causal != 0, tq, tk, tv, p, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_LAUNCH;
}

// ------------------------------------------------------------------ masks
// Bit-array geometry of a mask (see MaskArgs): words per query row and per
// key row, planes, and the byte sizes of the two arrays.
struct MaskGeom {
  int words, words_t, planes;
  size_t bits_bytes, bits_t_bytes, flags_bytes;
  int bias_planes;
  size_t bias_t_bytes;  // the additive mask's transpose (backward only)
};

static MaskGeom mask_geom(int Nq, int Nk, const attn_mask_t* m) {
  MaskGeom g{((Nk + 127) / 128) * 4, ((Nq + 127) / 128) * 4, 0, 0, 0, 0, 0, 0};
  if (m != nullptr && m->mask != nullptr) {
    g.planes = m->mask_batch * m->mask_heads;
    g.bits_bytes = (size_t)g.planes * Nq * g.words * 4;
    g.bits_t_bytes = (size_t)g.planes * Nk * g.words_t * 4;
    g.flags_bytes = ((size_t)g.planes * (g.words_t / 4) * (g.words / 4) + 15) / 16 * 16;
  }
  if (m != nullptr && m->bias != nullptr) {
    g.bias_planes = m->bias_batch * m->bias_heads;
    g.bias_t_bytes = ((size_t)g.bias_planes * Nq * Nk * (m->bias_bf16 ? 2 : 4) + 15) / 16 * 16;
  }
  return g;
}

static attn_status_t check_mask(int B, int H, int Nq, int Nk, const attn_mask_t* m) {
  if (m == nullptr) return ATTN_ERR_INVALID_ARG;
  if (m->window_left < -1 || m->window_right < -1) return ATTN_ERR_INVALID_ARG;
  if (m->key_lengths != nullptr) {
    if (reinterpret_cast<uintptr_t>(m->key_lengths) & 3u) return ATTN_ERR_MISALIGNED;
  }
  if (m->mask != nullptr) {
    if ((m->mask_batch != 1 && m->mask_batch != B) || (m->mask_heads != 1 && m->mask_heads != H))
      return ATTN_ERR_INVALID_ARG;
    const MaskGeom g = mask_geom(Nq, Nk, m);
    // The kernels index the bit arrays with 32-bit word indices.
    if ((long long)g.planes * Nq * g.words >= 0xffffffffll || (long long)g.planes * Nk * g.words_t >= 0xffffffffll)
      return ATTN_ERR_UNSUPPORTED_SHAPE;
  }
  if (m->bias != nullptr) {
    if ((m->bias_batch != 1 && m->bias_batch != B) || (m->bias_heads != 1 && m->bias_heads != H))
      return ATTN_ERR_INVALID_ARG;
    if (m->bias_bf16 != 0 && m->bias_bf16 != 1) return ATTN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(m->bias) & (m->bias_bf16 ? 1u : 3u)) return ATTN_ERR_MISALIGNED;
    if (m->bias_batch * m->bias_heads > 65535) return ATTN_ERR_UNSUPPORTED_SHAPE;  // planes on the grid's y
  }
  return ATTN_OK;
}

static attn_status_t check_mask_ptrs(const attn_mask_t* m) {
  for (const void* p : {static_cast<const void*>(m->key_lengths), static_cast<const void*>(m->mask),
                        static_cast<const void*>(m->bias)}) {
    if (p == nullptr) continue;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_INVALID_ARG;
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return ATTN_ERR_INVALID_ARG;
  }
  return ATTN_OK;
}

// Kernel mask arguments; the bit arrays (when there is a mask) at `bits` and
// `bits_t`, and the additive mask's transpose at `bias_t` (backward), inside
// the caller's workspace.  Causal enters as wr = 0.
static sdpa::MaskArgs mask_args(const attn_mask_t* m, int Nq, int Nk, int causal, float scale, uint32_t* bits,
                                uint32_t* bits_t, uint8_t* flags, void* bias_t) {
  const MaskGeom g = mask_geom(Nq, Nk, m);
  sdpa::MaskArgs a;
  a.bias = m->bias;
  a.bias_t = m->bias != nullptr ? bias_t : nullptr;
  a.bias_b = m->bias != nullptr ? m->bias_batch : 1;
  a.bias_h = m->bias != nullptr ? m->bias_heads : 1;
  a.bias_bf16 = m->bias != nullptr ? m->bias_bf16 : 0;
  a.inv_scale = 1.f / scale;
  a.flags = m->mask != nullptr ? flags : nullptr;
  a.ftq = g.words_t / 4;
  a.ftk = g.words / 4;
  a.wl = m->window_left;
  a.wr = causal ? 0 : m->window_right;
  a.key_len = m->key_lengths;
  a.bits = m->mask != nullptr ? bits : nullptr;
  a.bits_t = m->mask != nullptr ? bits_t : nullptr;
  a.words = g.words;
  a.words_t = g.words_t;
  a.mask_b = m->mask != nullptr ? m->mask_batch : 1;
  a.mask_h = m->mask != nullptr ? m->mask_heads : 1;
  return a;
}

size_t attn_masked_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d, const attn_mask_t* mask,
                                  int backward) {
  if (check_shape(B, H, Hkv, Nq, d) != ATTN_OK || check_shape(B, H, Hkv, Nk, d) != ATTN_OK ||
      check_mask(B, H, Nq, Nk, mask) != ATTN_OK)
    return 0;
  const MaskGeom g = mask_geom(Nq, Nk, mask);
  if (!backward) return g.bits_bytes + g.flags_bytes;
  return attn_bwd_workspace_size(B, H, Hkv, Nq, d) + g.bits_bytes + g.bits_t_bytes + g.flags_bytes + g.bias_t_bytes;
}

attn_status_t attn_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                              int Hkv, int Nq, int Nk, int d, float scale, int causal, const attn_mask_t* mask,
                              void* workspace, size_t workspace_bytes, void* stream) {
  ATTN_TRY(check_shape(B, H, Hkv, Nq, d));
  ATTN_TRY(check_shape(B, H, Hkv, Nk, d));
  ATTN_TRY(check_scale_flag(scale, causal));
  ATTN_TRY(check_mask(B, H, Nq, Nk, mask));
  const MaskGeom g = mask_geom(Nq, Nk, mask);
  if (g.bits_bytes > 0 && (workspace == nullptr || workspace_bytes < g.bits_bytes + g.flags_bytes))
    return ATTN_ERR_WORKSPACE;
  ATTN_TRY(check_ptrs({q, k, v, o, lse}));
  if (g.bits_bytes > 0) ATTN_TRY(check_ptrs({workspace}));
  ATTN_TRY(check_mask_ptrs(mask));
  DeviceInfo* di = nullptr;
  ATTN_TRY(current_device(&di));
  CUtensorMap tq, tk, tv, to;
  if (!make_map_bf16(&tq, q, d, Nq, (long long)B * H) || !make_map_bf16(&tk, k, d, Nk, (long long)B * Hkv) ||
      !make_map_bf16(&tv, v, d, Nk, (long long)B * Hkv) || !make_map_bf16(&to, o, d, Nq, (long long)B * H))
    return ATTN_ERR_CUDA;
  sdpa::FwdParams p;
  memset(&p, 0, sizeof(p));
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.G = H / Hkv;
  p.Nq = Nq;
  p.Nk = Nk;
  p.n_mtiles = (Nq + 255) / 256;
  p.nkv = (Nk + 127) / 128;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = di->status;
  p.limit_ns = wait_limit_ns();
  p.info = di->info;
  // Workspace: [row bits | tile flags].
  uint32_t* bits = static_cast<uint32_t*>(workspace);
  uint8_t* flags = static_cast<uint8_t*>(workspace) + g.bits_bytes;
  p.mk = mask_args(mask, Nq, Nk, causal, scale, bits, nullptr, flags, nullptr);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (mask->mask != nullptr &&
      sdpa::launch_mask_pack(static_cast<const uint8_t*>(mask->mask), mask->mask_batch, mask->mask_heads, Nq, Nk,
                             bits, g.words, nullptr, 0, flags, st) != cudaSuccess)
    return ATTN_ERR_LAUNCH;
  // A bf16 additive mask whose rows are whole 16-byte units arrives by TMA
  // (a map over its planes of [Nq x Nk]); any other goes through per-thread loads.
  CUtensorMap tb;
  const bool staged = mask->bias != nullptr && mask->bias_bf16 && Nk % 8 == 0 && aligned16(mask->bias);
  if (staged && !make_map_bf16(&tb, mask->bias, Nk, Nq, (long long)p.mk.bias_b * p.mk.bias_h)) return ATTN_ERR_CUDA;
  return sdpa::launch_fwd(d, false, tq, tk, tv, to, p, st, true, staged ? &tb : nullptr) == cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_LAUNCH;
}

attn_status_t attn_bwd_masked_stages(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                     const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int Nq,
                                     int Nk, int d, float scale, int causal, const attn_mask_t* mask, void* workspace,
                                     size_t workspace_bytes, unsigned stages, void* stream) {
  if (stages == 0 || (stages & ~kStagesAll) != 0) return ATTN_ERR_INVALID_ARG;
  ATTN_TRY(check_shape(B, H, Hkv, Nq, d));
  ATTN_TRY(check_shape(B, H, Hkv, Nk, d));
  ATTN_TRY(check_scale_flag(scale, causal));
  ATTN_TRY(check_mask(B, H, Nq, Nk, mask));
  const size_t need = attn_masked_workspace_size(B, H, Hkv, Nq, Nk, d, mask, 1);
  if (workspace == nullptr || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  ATTN_TRY(check_ptrs({q, k, v, o, lse, dout, dq, dk, dv, workspace}));
  ATTN_TRY(check_mask_ptrs(mask));
  DeviceInfo* di = nullptr;
  ATTN_TRY(current_device(&di));
  CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv, to;
  if (!make_map_bf16(&tq, q, d, Nq, (long long)B * H) || !make_map_bf16(&tk, k, d, Nk, (long long)B * Hkv) ||
      !make_map_bf16(&tv, v, d, Nk, (long long)B * Hkv) || !make_map_bf16(&tdo, dout, d, Nq, (long long)B * H) ||
      !make_map_bf16(&tdq, dq, d, Nq, (long long)B * H) || !make_map_bf16(&tdk, dk, d, Nk, (long long)B * Hkv) ||
      !make_map_bf16(&tdv, dv, d, Nk, (long long)B * Hkv) || !make_map_bf16(&to, o, d, Nq, (long long)B * H))
    return ATTN_ERR_CUDA;
  // Workspace: [row vectors | row bits | transposed bits | tile flags |
  // additive mask transposed].
  const MaskGeom g = mask_geom(Nq, Nk, mask);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* bits = reinterpret_cast<uint32_t*>(ws + attn_bwd_workspace_size(B, H, Hkv, Nq, d));
  uint32_t* bits_t = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(bits) + g.bits_bytes);
  uint8_t* flags = reinterpret_cast<uint8_t*>(bits_t) + g.bits_t_bytes;
  void* bias_t = flags + g.flags_bytes;
  sdpa::BwdParams p;
  bwd_params(&p, workspace, B, H, Hkv, Nq, Nk, d, scale, causal, di);
  p.o = static_cast<const uint16_t*>(o);
  p.dout = static_cast<const uint16_t*>(dout);
  p.lse = lse;
  p.mk = mask_args(mask, Nq, Nk, causal, scale, bits, bits_t, flags, bias_t);
  p.dq = static_cast<uint16_t*>(dq);  // outputs whose tiles nothing attends to are zeroed in place
  p.dk = static_cast<uint16_t*>(dk);
  p.dv = static_cast<uint16_t*>(dv);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The mask is packed (and the additive mask transposed) once, by the
  // first of stages 1 and 8 that runs.
  if ((stages & (kStagePrep | kStageDqRows)) && mask->mask != nullptr &&
      sdpa::launch_mask_pack(static_cast<const uint8_t*>(mask->mask), mask->mask_batch, mask->mask_heads, Nq, Nk,
                             bits, g.words, bits_t, g.words_t, flags, st) != cudaSuccess)
    return ATTN_ERR_LAUNCH;
  if ((stages & (kStagePrep | kStageDqRows)) && mask->bias != nullptr &&
      sdpa::launch_bias_transpose(mask->bias, mask->bias_bf16 != 0, g.bias_planes, Nq, Nk, bias_t, st) !=
          cudaSuccess)
    return ATTN_ERR_LAUNCH;
  if ((stages & kStagePrep) && sdpa::launch_bwd_prep(p, st) != cudaSuccess) return ATTN_ERR_LAUNCH;
  if (stages & kStageDqRows) {
    sdpa::BwdParams pr = p;
    pr.rows_in_dq = 1;
    if (sdpa::launch_bwd_dq(d, false, tq, tk, tv, tdo, tdq, to, pr, st, true) != cudaSuccess) return ATTN_ERR_LAUNCH;
  }
  // A bf16 additive mask without a boolean mask reaches the dK/dV kernel by
  // TMA when the rows of its transpose are whole 16-byte units.
  CUtensorMap tbt;
  const bool staged_t = mask->bias != nullptr && mask->bias_bf16 && mask->mask == nullptr && Nq % 8 == 0;
  if (staged_t && !make_map_bf16(&tbt, bias_t, Nq, Nk, (long long)g.bias_planes)) return ATTN_ERR_CUDA;
  if ((stages & kStageGrad) &&
      sdpa::launch_bwd_grad(d, false, tq, tk, tv, tdo, tdk, tdv, p, st, true, staged_t ? &tbt : nullptr) != cudaSuccess)
    return ATTN_ERR_LAUNCH;
  if ((stages & kStageDq) && sdpa::launch_bwd_dq(d, false, tq, tk, tv, tdo, tdq, to, p, st, true) != cudaSuccess)
    return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}

attn_status_t attn_bwd_masked(const void* q, const void* k, const void* v, const void* o, const float* lse,
                              const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int Nq, int Nk,
                              int d, float scale, int causal, const attn_mask_t* mask, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return attn_bwd_masked_stages(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, Nq, Nk, d, scale, causal, mask,
                                workspace, workspace_bytes, kStageDqRows | kStageGrad, stream);
}

// Key chunks of the decode kernel, a pure function of the shape (so the
// workspace size needs no device query): chunks of whole 128-key tiles,
// about 1216 CTAs in all (four waves of two CTAs on each of 152 SMs) when
// the cache is long enough.
static void decode_plan(int B, int Hkv, int Nk, int* nsplit, int* split_keys) {
  const int tiles = (Nk + 127) / 128;
  const long long bh = (long long)B * Hkv;
  const long long want = (1216 + bh - 1) / bh;
  const int ns0 = (int)std::min<long long>(tiles, want);
  const int per = (tiles + ns0 - 1) / ns0;  // tiles per chunk
  *nsplit = (tiles + per - 1) / per;
  *split_keys = per * 128;
}

static attn_status_t check_decode_shape(int B, int H, int Hkv, int Nq, int Nk, int d) {
  if (B < 1 || H < 1 || Hkv < 1 || Nq < 1 || Nk < 1 || Nq > Nk) return ATTN_ERR_UNSUPPORTED_SHAPE;
  if (d != 64 && d != 96 && d != 128) return ATTN_ERR_UNSUPPORTED_SHAPE;
  if (H % Hkv != 0 || (long long)(H / Hkv) * Nq > sdpa::kDecMaxRows) return ATTN_ERR_UNSUPPORTED_SHAPE;
  if ((long long)B * H * Nq > (1ll << 31) / 8 || (long long)B * Hkv > 65535) return ATTN_ERR_UNSUPPORTED_SHAPE;
  return ATTN_OK;
}

size_t attn_decode_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d) {
  if (check_decode_shape(B, H, Hkv, Nq, Nk, d) != ATTN_OK) return 0;
  int nsplit = 0, split_keys = 0;
  decode_plan(B, Hkv, Nk, &nsplit, &split_keys);
  const size_t rows = (size_t)B * H * Nq * (size_t)nsplit;
  return rows * (size_t)d * 4 + rows * 4;  // partial O, then partial lse
}

attn_status_t attn_decode(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                          size_t workspace_bytes, int B, int H, int Hkv, int Nq, int Nk, int d, float scale,
                          int causal, void* stream) {
  ATTN_TRY(check_decode_shape(B, H, Hkv, Nq, Nk, d));
  ATTN_TRY(check_scale_flag(scale, causal));
  if (workspace == nullptr || workspace_bytes < attn_decode_workspace_size(B, H, Hkv, Nq, Nk, d))
    return ATTN_ERR_WORKSPACE;
  ATTN_TRY(check_ptrs({q, k, v, o, lse, workspace}));
  DeviceInfo* di = nullptr;
  ATTN_TRY(current_device(&di));
  CUtensorMap tq, tk, tv;  // q as one (B*H*Nq) x d matrix: a K/V head's query rows are contiguous
  if (!make_map_bf16(&tq, q, d, B * H * Nq, 1) || !make_map_bf16(&tk, k, d, Nk, (long long)B * Hkv) ||
      !make_map_bf16(&tv, v, d, Nk, (long long)B * Hkv))
    return ATTN_ERR_CUDA;
  sdpa::DecParams p;
  memset(&p, 0, sizeof(p));
  decode_plan(B, Hkv, Nk, &p.nsplit, &p.split_keys);
  const size_t rows = (size_t)B * H * Nq * (size_t)p.nsplit;
  p.q = static_cast<const uint16_t*>(q);
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.o_part = static_cast<float*>(workspace);
  p.lse_part = p.o_part + rows * (size_t)d;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.G = H / Hkv;
  p.Nq = Nq;
  p.Nk = Nk;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = di->status;
  p.limit_ns = wait_limit_ns();
  p.info = di->info;
  cudaError_t e = sdpa::launch_decode(d, causal != 0, tq, tk, tv, p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

// ------------------------------------------------------------------ paged decode
static attn_status_t check_paged(int B, int page_size, int num_pages, int max_pages) {
  if (page_size < 16 || page_size % 16 != 0) return ATTN_ERR_UNSUPPORTED_SHAPE;
  if (page_size < 128 ? (128 % page_size != 0) : (page_size % 128 != 0)) return ATTN_ERR_UNSUPPORTED_SHAPE;
  if (num_pages < 1 || max_pages < 1) return ATTN_ERR_UNSUPPORTED_SHAPE;
  if ((long long)page_size * max_pages > (1ll << 30) || (long long)B * max_pages > (1ll << 31))
    return ATTN_ERR_UNSUPPORTED_SHAPE;
  return ATTN_OK;
}

size_t attn_decode_paged_workspace_size(int B, int H, int Hkv, int Nq, int page_size, int max_pages, int d) {
  if (check_paged(B, page_size, 1, max_pages) != ATTN_OK) return 0;
  return attn_decode_workspace_size(B, H, Hkv, Nq, page_size * max_pages, d);
}

attn_status_t attn_decode_paged(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                                const int* block_table, const int* seq_lens, void* workspace,
                                size_t workspace_bytes, int B, int H, int Hkv, int Nq, int page_size, int num_pages,
                                int max_pages, int d, float scale, int causal, void* stream) {
  ATTN_TRY(check_paged(B, page_size, num_pages, max_pages));
  const int Nk = page_size * max_pages;  // the most keys a sequence can hold
  ATTN_TRY(check_decode_shape(B, H, Hkv, Nq, Nk, d));
  ATTN_TRY(check_scale_flag(scale, causal));
  if (workspace == nullptr || workspace_bytes < attn_decode_workspace_size(B, H, Hkv, Nq, Nk, d))
    return ATTN_ERR_WORKSPACE;
  ATTN_TRY(check_ptrs({q, k_cache, v_cache, o, lse, workspace}));
  ATTN_TRY(check_offsets_ptrs(block_table, seq_lens));
  DeviceInfo* di = nullptr;
  ATTN_TRY(current_device(&di));
  // Cache maps: 4-D over (d, Hkv, page_size, num_pages), box 64 x 1 x
  // min(page_size, 128) x 1 (one page's tokens of one head).
  EncodeTiledFn enc = encode_fn();
  if (!enc) return ATTN_ERR_CUDA;
  CUtensorMap tq, tk, tv;
  if (!make_map_bf16(&tq, q, d, B * H * Nq, 1)) return ATTN_ERR_CUDA;
  const int box_rows = std::min(page_size, 128);
  for (int t = 0; t < 2; ++t) {
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)Hkv, (cuuint64_t)page_size, (cuuint64_t)num_pages};
    cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)Hkv * d * 2, (cuuint64_t)page_size * Hkv * d * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    if (enc(t == 0 ? &tk : &tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(t == 0 ? k_cache : v_cache),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return ATTN_ERR_CUDA;
  }
  sdpa::DecParams p;
  memset(&p, 0, sizeof(p));
  decode_plan(B, Hkv, Nk, &p.nsplit, &p.split_keys);
  const size_t rows = (size_t)B * H * Nq * (size_t)p.nsplit;
  p.q = static_cast<const uint16_t*>(q);
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.o_part = static_cast<float*>(workspace);
  p.lse_part = p.o_part + rows * (size_t)d;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.G = H / Hkv;
  p.Nq = Nq;
  p.Nk = Nk;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = di->status;
  p.limit_ns = wait_limit_ns();
  p.info = di->info;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.page_size = page_size;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.box_rows = box_rows;
  cudaError_t e = sdpa::launch_decode(d, causal != 0, tq, tk, tv, p, static_cast<cudaStream_t>(stream), true);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

attn_status_t attn_get_device_status(void* stream) {
  DeviceInfo* di = nullptr;
  ATTN_TRY(current_device(&di));
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  int host = 0;
  if (cudaMemcpyFromSymbol(&host, g_status_word, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  if (host != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  if (host == 0) return ATTN_OK;
  if (host == sdpa::kDevTimeout) return ATTN_ERR_TIMEOUT;
  if (host == sdpa::kDevBadSeqlens) return ATTN_ERR_INVALID_ARG;
  if (host == sdpa::kDevCheckFailed) return ATTN_ERR_CHECK;
  return ATTN_ERR_CUDA;
}

attn_status_t attn_get_timeout_info(int info[4], void* stream) {
  if (info == nullptr) return ATTN_ERR_INVALID_ARG;
  DeviceInfo* di = nullptr;
  ATTN_TRY(current_device(&di));
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  if (cudaMemcpyFromSymbol(info, g_timeout_info, 4 * sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  const int zero[4] = {0, 0, 0, 0};
  if (cudaMemcpyToSymbol(g_timeout_info, zero, sizeof(zero)) != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

attn_status_t attn_selftest_wait_timeout(unsigned int timeout_us, void* stream) {
  DeviceInfo* di = nullptr;
  ATTN_TRY(current_device(&di));
  if (timeout_us == 0 || timeout_us > 5000000u) return ATTN_ERR_INVALID_ARG;
  selftest_wait_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(di->status, di->info,
                                                                         (unsigned long long)timeout_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

attn_status_t attn_debug_drop_load(int kernel, int load_index, unsigned int limit_us) {
  if (kernel < 0 || kernel > 6 || load_index < 0 || load_index > (1 << 20)) return ATTN_ERR_INVALID_ARG;
  if (limit_us < 1000u || limit_us > 60000000u) return ATTN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_debug_mu);
  g_debug_kernel = kernel;
  g_debug_drop1 = load_index + 1;
  g_debug_limit_ns = (unsigned long long)limit_us * 1000ull;
  return ATTN_OK;
}

int attn_debug_build(void) { return sdpa::kDebugChecks ? 1 : 0; }

attn_status_t attn_debug_plant_index(int kernel) {
  if (!sdpa::kDebugChecks || kernel < 0 || kernel > 1) return ATTN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_debug_mu);
  g_plant_kernel = kernel;
  return ATTN_OK;
}

}  // extern "C"
