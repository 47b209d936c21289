// ptx.cuh — thin inline-PTX wrappers for the sm_103a features the attention
// kernels use: mbarriers, TMA tensor copies, tcgen05 MMAs into tensor memory
// (TMEM), TMEM loads/stores, and the bounded waits that let a kernel stop
// with an error status instead of hanging.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

namespace sdpa {

// Device status word values (host maps them to attn_status_t).
constexpr int kDevTimeout = 7;      // a bounded wait ran out
constexpr int kDevMisaligned = 8;   // dynamic shared memory not 1024-byte aligned

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// True once the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared state for bounded waits: a CTA-wide abort flag in shared memory and
// the device status word in global memory.
struct WaitCtx {
  volatile int* abort_flag;  // shared memory
  int* status;               // global memory
  uint64_t limit_ns;
  int* info;                 // global memory: where the first timeout happened
};

// Wait-site codes recorded with a timeout: (site << 16) | (loop step & 0xffff).
__device__ __forceinline__ int wait_site(int site, int step) { return (site << 16) | (step & 0xffff); }

// Waits for phase `parity` of `bar`.  Gives up when another role of the CTA
// has aborted, or when `limit_ns` has passed, in which case it raises the
// CTA abort flag, records a timeout in the status word and, for the first
// timeout on the device, where it happened (site, block, thread, waited us).
// Returns false when the caller must stop.
__device__ __forceinline__ bool wait_bounded(const WaitCtx& w, uint32_t bar, uint32_t parity, int site = 0) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (true) {
    if (mbar_try(bar, parity)) return true;
    if ((++it & 15u) == 0) {
      if (*w.abort_flag) return false;
      if (globaltimer_ns() - t0 > w.limit_ns) {
        *w.abort_flag = 1;
        if (atomicCAS(w.status, 0, kDevTimeout) == 0 && w.info != nullptr) {
          w.info[0] = site;
          w.info[1] = (int)blockIdx.x;
          w.info[2] = (int)threadIdx.x;
          w.info[3] = (int)((globaltimer_ns() - t0) / 1000);
        }
        return false;
      }
    }
  }
}

// Used only after an abort: waits (bounded, ignoring the abort flag) for an
// asynchronous operation this thread issued, e.g. a TMA load still in
// flight, so that the CTA never exits with copies targeting its memory.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// --------------------------------------------------------------- TMA (bulk)
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int c0, int c1, int c2,
                                            int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
// Asks L2 for a box of a tensor map (no shared memory written, no barrier):
// the later load of the same box then finds it there.
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* m, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
// Element-wise add of a shared-memory box into global memory through the
// tensor map (the reduction is performed by the memory system, per line).
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* m, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
// Plain (untiled) bulk copy global -> shared; both addresses 16-B aligned,
// size a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]; bf16 x bf16 -> f32, shape from idesc.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem].
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Predicated forms for a warp that runs the issue loop converged: only the
// lane with `leader` != 0 (from elect_one) issues; descriptor arithmetic stays
// warp-uniform, so it needs no per-MMA moves into uniform registers.
__device__ __forceinline__ uint32_t elect_one() {
  uint32_t pred;
  asm volatile("{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}" : "=r"(pred));
  return pred;
}
__device__ __forceinline__ void mma_ss_p(uint32_t leader, uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(leader)
      : "memory");
}
__device__ __forceinline__ void mma_ts_p(uint32_t leader, uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(leader)
      : "memory");
}
__device__ __forceinline__ void mma_commit_p(uint32_t leader, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %1, 0;\n\t"
      "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}\n" ::"r"(bar),
      "r"(leader)
      : "memory");
}
// A shared-memory descriptor moved by `bytes` (start-address field only;
// addresses stay below 2^18, so the 14-bit field never carries).
__host__ __device__ constexpr uint64_t sdesc_add(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }

// Arrive once on `bar` when every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Instruction descriptor, kind::f16 with bf16 A/B and f32 accumulator.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format
//   (1 = bf16), 15 A major (1 = MN), 16 B major (1 = MN), 17-22 N>>3,
//   24-28 M>>4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor for the 128-byte swizzle layout written by
// TMA with CU_TENSOR_MAP_SWIZZLE_128B (rows of 128 bytes, 8-row / 1024-byte
// swizzle atoms, atoms 1024-byte aligned).
//   bits 0-13 start>>4, 16-29 leading byte offset>>4, 32-45 stride byte
//   offset>>4, 46-47 version (1), 61-63 layout (2 = 128-byte swizzle).
// K-major operand: LBO unused, SBO = 1024 (8-row group stride); a K step of
//   16 bf16 inside a 128-byte row advances the start address by 32 bytes.
// MN-major operand: LBO = byte stride between 64-element MN chunks,
//   SBO = 1024 (stride between 8-row K groups).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// TMEM loads/stores: 32 lanes x 32 consecutive 32-bit columns; thread t of a
// warp gets lane (base + t).  Results are valid only after tmem_wait_ld().
#define SDPA_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), \
                   "=r"(r[i + 6]), "=r"(r[i + 7])
#define SDPA_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), \
                   "r"(r[i + 6]), "r"(r[i + 7])
#define SDPA_P8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), "+r"(r[i + 5]), \
                   "+r"(r[i + 6]), "+r"(r[i + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : SDPA_R8(0), SDPA_R8(8), SDPA_R8(16), SDPA_R8(24)
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : SDPA_R8(0), SDPA_R8(8)
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      SDPA_W8(0), SDPA_W8(8), SDPA_W8(16), SDPA_W8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      SDPA_W8(0), SDPA_W8(8)
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), SDPA_W8(0)
               : "memory");
}
// One 32-bit column of the warp's 32 lanes (lane base + t for thread t).
__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr) : "memory");
  return r;
}
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Ties registers written by a tcgen05.ld to a point after tmem_wait_ld(), so
// the compiler cannot move their uses above the wait.
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
  asm volatile("" : SDPA_P8(0), SDPA_P8(8), SDPA_P8(16), SDPA_P8(24));
}
__device__ __forceinline__ void reg_fence(uint32_t (&r)[16]) { asm volatile("" : SDPA_P8(0), SDPA_P8(8)); }

#undef SDPA_R8
#undef SDPA_W8
#undef SDPA_P8

// Re-balances registers between warpgroups (all threads of a warpgroup).
// setmaxnreg.inc waits until other warps have released registers, and it
// waits forever if they never do.  A kernel whose idle warps give registers
// back with dec and later take them again with inc must therefore make every
// inc at the start complete before any warp can run its closing inc:
// reg_split_sync() after the opening setmaxnreg of every warpgroup does that.
constexpr uint32_t kRegSplitBarrier = 15;
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void reg_split_sync(uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(kRegSplitBarrier), "r"(nthreads) : "memory");
}

// ------------------------------------------------- Blackwell fp32 pair math
// Three-input maximum and packed fp32x2 FMA / add / multiply (sm_100+): one
// instruction does the work of two (or, for max, halves a reduction chain).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// ------------------------------------------------------------- misc helpers
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void named_bar_arrive(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Same with the barrier id and count as immediates (no register held for
// them; in register-tight code a register operand cost a spill).
template <int ID, int N>
__device__ __forceinline__ void named_bar_arrive_c() {
  asm volatile("bar.arrive %0, %1;" ::"n"(ID), "n"(N) : "memory");
}
template <int ID, int N>
__device__ __forceinline__ void named_bar_sync_c() {
  asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(N) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ float4 ld_shared_v4f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a tile of
// 128-byte rows stored with the 128-byte swizzle (chunk index XOR row%8).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}
__device__ __forceinline__ uint4 ld_shared_v4u(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Rows [0, nrows) of a [128 x D] bf16 tile staged in shared memory with the
// 128-byte swizzle (blocks of [128 rows x 64 columns], 16 KB apart) go to
// global memory with plain 16-byte stores: row r to dst + r * row_stride
// elements.  For tiles whose remaining rows belong to someone else (the last
// tile of a packed sequence), where a TMA store of the whole box would write
// them.  Thread t of nt takes chunks t, t + nt, ...  128 * row_stride must
// fit in 32 bits (the host checks heads * d * 128 < 2^32).
// Rows [0, nrows) of a [rows x D] bf16 tile (row stride row_stride
// elements) set to zero by the whole CTA.  Out of line: it runs only for
// outputs that nothing attends to (in packed batches), and inlined it would
// take registers from the kernels' main loops.
template <int D>
__device__ __noinline__ void zero_rows_bf16(uint16_t* dst, uint32_t row_stride, int nrows) {
  for (int c = threadIdx.x; c < nrows * (D / 8); c += blockDim.x)
    *reinterpret_cast<uint4*>(dst + ((uint32_t)(c / (D / 8)) * row_stride + (c % (D / 8)) * 8)) = make_uint4(0, 0, 0, 0);
}
// The same for two tiles with one row layout (dK and dV).
template <int D>
__device__ __noinline__ void zero_rows2_bf16(uint16_t* a, uint16_t* b, uint32_t row_stride, int nrows) {
  for (int c = threadIdx.x; c < nrows * (D / 8); c += blockDim.x) {
    const uint32_t e = (uint32_t)(c / (D / 8)) * row_stride + (c % (D / 8)) * 8;
    *reinterpret_cast<uint4*>(a + e) = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(b + e) = make_uint4(0, 0, 0, 0);
  }
}

template <int D>
__device__ __forceinline__ void store_rows_sw128(uint32_t stage, uint16_t* dst, uint32_t row_stride, int nrows,
                                                 int t, int nt) {
  constexpr uint32_t CH = D / 8;  // 16-byte chunks per row
#pragma unroll 1
  for (int c = t; c < nrows * (int)CH; c += nt) {
    const uint32_t row = (uint32_t)c / CH, ch = (uint32_t)c % CH;
    const uint4 v = ld_shared_v4u(stage + (ch >> 3) * 16384u + sw128_offset(row, ch & 7));
    *reinterpret_cast<uint4*>(dst + (row * row_stride + ch * 8)) = v;
  }
}

// The same store through a per-warp 4 KB shared-memory scratch instead of
// shuffles: each lane writes its row's NCH chunks at a 128-byte pitch (chunk
// c of row l at slot c ^ (l % 8), so that a warp's writes of one chunk fall
// on all banks), then reads back chunk L % NCH of row (32 / NCH) s + L / NCH
// for s = 0 .. NCH - 1 and stores it: each store instruction again covers
// 32 / NCH whole row slices.  Costs 2 NCH shared-memory accesses per lane
// where the shuffle transpose costs about 24 NCH instructions.  Rows at or
// past nvalid are not written.  Every lane of the warp takes part; the
// scratch is free again when it returns.
template <int NCH>
__device__ __forceinline__ void store_rows_staged(const uint4 (&x)[NCH], uint32_t scr, uint16_t* dst, size_t stride,
                                                  int nvalid) {
  static_assert(NCH == 4 || NCH == 8, "chunks per row");
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = 0; c < NCH; ++c)
    st_shared_v4(scr + (uint32_t)lane * 128u + ((uint32_t)(c ^ (lane & 7)) << 4), x[c].x, x[c].y, x[c].z, x[c].w);
  __syncwarp();
  const int c = lane % NCH;
#pragma unroll
  for (int s = 0; s < NCH; ++s) {
    const int r = (32 / NCH) * s + lane / NCH;
    const uint4 v = ld_shared_v4u(scr + (uint32_t)r * 128u + ((uint32_t)(c ^ (r & 7)) << 4));
    if (r < nvalid) *reinterpret_cast<uint4*>(dst + (size_t)r * stride + 8 * c) = v;
  }
  __syncwarp();
}

// Writes 16-byte chunks that the lanes of a warp hold one row each (lane l:
// row l of the warp's 32 rows, x[k] = columns 8k .. 8k + 7 of a slice that
// starts at dst for row 0; row r at dst + r * stride elements) so that every
// store instruction covers whole slices of 32 / NCH rows, rather than 32
// pieces of 32 rows: an NCH x NCH transpose of the chunks inside each group
// of NCH lanes (log2 NCH stages: lanes whose bit m differs swap the chunks
// whose bit m differs from theirs), after which lane g NCH + j holds chunk j
// of rows g NCH + s in x[s].  Rows at or past nvalid are not written.  Every
// lane of the warp takes part.
template <int NCH>
__device__ __forceinline__ void store_rows_transposed(uint4 (&x)[NCH], uint16_t* dst, size_t stride, int nvalid) {
  static_assert(NCH == 2 || NCH == 4 || NCH == 8, "chunks per row");
  const int lane = threadIdx.x & 31, li = lane & (NCH - 1);
#pragma unroll
  for (int m = NCH / 2; m >= 1; m >>= 1) {
    const bool hi = (li & m) != 0;
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
      if (k & m) continue;
      const uint4 out = hi ? x[k] : x[k | m];
      uint4 in;
      in.x = __shfl_xor_sync(0xffffffffu, out.x, m);
      in.y = __shfl_xor_sync(0xffffffffu, out.y, m);
      in.z = __shfl_xor_sync(0xffffffffu, out.z, m);
      in.w = __shfl_xor_sync(0xffffffffu, out.w, m);
      if (hi)
        x[k] = in;
      else
        x[k | m] = in;
    }
  }
  const int g = lane / NCH;
#pragma unroll
  for (int s = 0; s < NCH; ++s) {
    const int r = g * NCH + s;
    if (r < nvalid) *reinterpret_cast<uint4*>(dst + (size_t)r * stride + 8 * li) = x[s];
  }
}

}  // namespace sdpa
