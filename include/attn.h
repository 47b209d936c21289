/*
 * attn.h — C ABI of a GB300 (sm_103a) library for exact scaled-dot-product
 * attention, computed FlashAttention-style.
 *
 * What is computed (page "Flash Attention原理：分块计算与重计算，如何降低O(n^2)的
 * 显存占用", §一 and §四):
 *     S = scale * Q K^T            (n x n per head; causal: S_ij = -inf for j > i)
 *     P = softmax(S) row-wise      (max-subtracted, exact)
 *     O = P V
 * The n x n matrices S and P are never written to device memory: the forward
 * pass tiles Q, K and V through shared memory and tensor memory with a running
 * row max and row sum (the online softmax of §四) and stores only O and one
 * per-row statistic (§五 keeps m and l; here lse = m + ln l, natural log of
 * the scaled, masked scores).  The backward pass recomputes P tile by tile
 * from lse (§五, "recomputation") and returns dQ, dK, dV.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Element type: bf16 (IEEE bfloat16) for Q, K, V, O, dO, dQ, dK, dV;
 *    float32 for lse.  Accumulation is float32.
 *  - Layout: dense row-major (B, H, N, d) for Q, O, dO, dQ and (B, Hkv, N, d)
 *    for K, V, dK, dV (the (batch, num_heads, seq_len, head_dim) layout of the
 *    page above, §一); lse is (B, H, N).  Strides are implied by the shape.
 *  - Grouped-query attention: Hkv must divide H; query head h reads K/V head
 *    h / (H / Hkv) (contiguous groups).  Hkv == H is ordinary multi-head.
 *  - Supported head_dim d: 64, 96, 128.  Any N >= 1.  Queries and keys share
 *    positions 0..N-1; the causal mask hides key j from query i when j > i.
 *  - All pointers are DEVICE pointers owned by the caller, 16-byte aligned.
 *    The library never allocates or frees device memory and keeps no pointer
 *    after a call returns.
 *  - stream: a cudaStream_t (NULL = legacy default stream).  Work is enqueued
 *    asynchronously; a return of ATTN_OK means the arguments were valid and
 *    the kernels were launched, not that they have finished.
 *  - Errors are returned, never hidden: there is no fallback path.  A bad
 *    argument returns an error before anything is launched.  A device-side
 *    wait that runs past its time limit makes the kernel stop early and
 *    record ATTN_ERR_TIMEOUT in a device status word, which
 *    attn_get_device_status() reports.
 *  - Device: a GPU of compute capability 10.3 (GB300); others give
 *    ATTN_ERR_UNSUPPORTED_DEVICE.
 */
#ifndef SDPA08_ATTN_H
#define SDPA08_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,        /* null pointer, non-finite scale, bad flag   */
  ATTN_ERR_UNSUPPORTED_SHAPE = 2,  /* d not in {64,96,128}, H % Hkv != 0, size < 1 or too large */
  ATTN_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not compute capability 10.3 */
  ATTN_ERR_MISALIGNED = 4,         /* a pointer is not 16-byte aligned            */
  ATTN_ERR_WORKSPACE = 5,          /* workspace missing or smaller than required  */
  ATTN_ERR_LAUNCH = 6,             /* the CUDA launch itself failed               */
  ATTN_ERR_TIMEOUT = 7,            /* a device-side wait ran out (reported by attn_get_device_status) */
  ATTN_ERR_CUDA = 8,               /* another CUDA runtime/driver error           */
  ATTN_ERR_CHECK = 9               /* debug build only: an in-kernel index check failed (reported by attn_get_device_status) */
} attn_status_t;

/*
 * Forward pass.  Page "Flash Attention原理", §三 (tiling), §四 (online softmax),
 * §五 (store only per-row statistics).
 *   q    [in]  bf16 (B, H, N, d)
 *   k, v [in]  bf16 (B, Hkv, N, d)
 *   o    [out] bf16 (B, H, N, d)          O = softmax(scale*QK^T [+mask]) V
 *   lse  [out] float32 (B, H, N)          ln sum_j exp(scale*q_i.k_j) over unmasked j
 *   scale      softmax scale (1/sqrt(d) for standard attention); finite and > 0
 *   causal     0 or 1
 * Outputs must not overlap inputs.
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int H, int Hkv, int N, int d, float scale, int causal,
                       void* stream);

/*
 * Forward with Nq query rows and Nk key/value rows per head (cross
 * attention; chunked prefill of Nq new tokens against a cache of Nk).  The
 * SDPA call of page "SDPA backend 与 FlashAttention" (§3) takes query and key
 * sequences of their own lengths; the pages fix no causal alignment for
 * Nq != Nk, and the one taken is that of a block of new tokens ending the
 * sequence: query row i sits at position Nk - Nq + i and sees keys
 * 0 .. Nk - Nq + i (top-left and bottom-right agree when Nq == Nk).
 *   q, o [in/out] bf16 (B, H, Nq, d);  k, v [in] bf16 (B, Hkv, Nk, d)
 *   lse  [out] float32 (B, H, Nq)
 * causal requires Nq <= Nk (otherwise ATTN_ERR_UNSUPPORTED_SHAPE).
 * attn_fwd(..., N, ...) is attn_fwd_cross(..., N, N, ...).
 */
attn_status_t attn_fwd_cross(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                             void* stream);

/*
 * Bytes of device workspace attn_bwd needs for this shape: two float32
 * per-row vectors (D = rowsum(dO * O) and lse in base 2), each padded to a
 * multiple of 128 rows per head, i.e. 8 * B * H * ceil(N/128) * 128 bytes.
 * Returns 0 for an invalid shape.
 */
size_t attn_bwd_workspace_size(int B, int H, int Hkv, int N, int d);

/*
 * Backward pass.  Page "Flash Attention原理", §五 (recompute P from the stored
 * statistic instead of keeping S and P) and FAQ Q19 (gradients by the chain
 * rule); the gradients are those of softmax-then-matmul:
 *   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - rowsum(dO * O)),
 *   dQ = scale dS K,  dK = scale dS^T Q   (dK, dV summed over a GQA group).
 *   q, k, v, o [in] as in attn_fwd;  lse [in] float32 (B, H, N) from attn_fwd
 *   dout [in]  bf16 (B, H, N, d)  gradient of the loss w.r.t. O
 *   dq   [out] bf16 (B, H, N, d);  dk, dv [out] bf16 (B, Hkv, N, d)
 *   workspace  device buffer of at least attn_bwd_workspace_size() bytes,
 *              owned by the caller; its contents on entry are ignored and on
 *              return are unspecified.  It must not overlap any other argument.
 */
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dout,
                       void* dq, void* dk, void* dv,
                       void* workspace, size_t workspace_bytes,
                       int B, int H, int Hkv, int N, int d, float scale, int causal,
                       void* stream);

/*
 * The stages of the backward, for callers that schedule (or time) them
 * separately.  Same arguments, layouts and workspace as attn_bwd.  The
 * workspace's row vectors (D = rowsum(dO * O) and lse in base 2) must be
 * complete before grad or dq starts:
 *   attn_bwd_prep     the row vectors into the workspace  (reads o, lse, dout)
 *   attn_bwd_grad     one pass per key tile: recomputes P^T and dS^T tile by
 *                     tile; writes dK, dV; reads the row vectors
 *                                                       (reads q, k, v, dout)
 *   attn_bwd_dq       one pass per query tile: recomputes P and dS tile by
 *                     tile; writes dq; reads the row vectors
 *                                                       (reads q, k, v, dout)
 *   attn_bwd_dq_rows  attn_bwd_dq that forms each query tile's row vectors
 *                     itself (from o, lse, dout) and writes them into the
 *                     workspace: it replaces prep + dq, and grad runs after
 *                     it.  attn_bwd is attn_bwd_dq_rows then attn_bwd_grad.
 *                     Nq query rows and Nk key rows (Nq == Nk for attn_bwd's
 *                     shapes; attn_bwd_cross's otherwise); workspace of
 *                     attn_bwd_workspace_size(B, H, Hkv, Nq, d) bytes.
 * Every output element has exactly one writer (no atomics), so the results
 * are the same on every run; D summed by prep and by dq_rows may differ in
 * its last bits (another order of the same float32 additions).
 */
attn_status_t attn_bwd_prep(const void* o, const float* lse, const void* dout,
                            void* workspace, size_t workspace_bytes,
                            int B, int H, int Hkv, int N, int d, void* stream);
attn_status_t attn_bwd_grad(const void* q, const void* k, const void* v, const void* dout,
                            void* dk, void* dv, void* workspace, size_t workspace_bytes,
                            int B, int H, int Hkv, int N, int d, float scale, int causal,
                            void* stream);
attn_status_t attn_bwd_dq(const void* q, const void* k, const void* v, const void* dout,
                          void* dq, void* workspace, size_t workspace_bytes,
                          int B, int H, int Hkv, int N, int d, float scale, int causal,
                          void* stream);
attn_status_t attn_bwd_dq_rows(const void* q, const void* k, const void* v, const void* o,
                               const float* lse, const void* dout, void* dq,
                               void* workspace, size_t workspace_bytes,
                               int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                               void* stream);

/*
 * Backward of attn_fwd_cross: Nq query rows, Nk key/value rows per head,
 * the same causal alignment (query row i sees keys 0 .. Nk - Nq + i) and the
 * same gradients as attn_bwd.
 *   q, o, dout [in] bf16 (B, H, Nq, d);  lse [in] float32 (B, H, Nq)
 *   k, v [in] bf16 (B, Hkv, Nk, d)
 *   dq [out] bf16 (B, H, Nq, d);  dk, dv [out] bf16 (B, Hkv, Nk, d)
 *   workspace  at least attn_bwd_workspace_size(B, H, Hkv, Nq, d) bytes
 * causal requires Nq <= Nk (otherwise ATTN_ERR_UNSUPPORTED_SHAPE).  Nothing
 * is launched when any check fails.  attn_bwd(..., N, ...) is
 * attn_bwd_cross(..., N, N, ...).
 */
attn_status_t attn_bwd_cross(const void* q, const void* k, const void* v, const void* o,
                             const float* lse, const void* dout,
                             void* dq, void* dk, void* dv,
                             void* workspace, size_t workspace_bytes,
                             int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                             void* stream);

/*
 * The grad and dq stages of attn_bwd_cross, for callers that schedule them
 * separately (the prep stage is attn_bwd_prep with N = Nq; attn_bwd_dq_rows
 * takes Nq and Nk itself).  Arguments and ordering rules as for
 * attn_bwd_grad / attn_bwd_dq, with the shapes of attn_bwd_cross.
 */
attn_status_t attn_bwd_grad_cross(const void* q, const void* k, const void* v, const void* dout,
                                  void* dk, void* dv, void* workspace, size_t workspace_bytes,
                                  int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                                  void* stream);
attn_status_t attn_bwd_dq_cross(const void* q, const void* k, const void* v, const void* dout,
                                void* dq, void* workspace, size_t workspace_bytes,
                                int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                                void* stream);

/*
 * Decode against a paged KV cache.  Page "Flash Attention原理", FAQ Q12 and
 * Q13: at inference the KV cache is combined with PagedAttention, which
 * keeps each sequence's cached keys and values in fixed-size pages found
 * through a block table.  The attention is attn_decode's, over the cached
 * keys of each batch element:
 *   k_cache, v_cache [in] bf16 (num_pages, page_size, Hkv, d): physical
 *            pages of page_size tokens, heads interleaved per token
 *   block_table [in] DEVICE int32 (B, max_pages): logical page i of batch
 *            element b is physical page block_table[b * max_pages + i];
 *            entries past a sequence's last page are never read
 *   seq_lens [in] DEVICE int32 (B): cached keys of each batch element
 *            (the Nk of attn_decode, the new tokens included), at most
 *            page_size * max_pages
 *   q, o, lse, workspace, scale, causal as attn_decode (causal: query t of
 *            batch element b at position seq_lens[b] - Nq + t)
 * page_size: a multiple of 16 that divides 128, or a multiple of 128.
 * Table entries a sequence needs that are out of [0, num_pages), or lengths
 * past the capacity, are read as zero keys and make
 * attn_get_device_status() return ATTN_ERR_INVALID_ARG.
 */
size_t attn_decode_paged_workspace_size(int B, int H, int Hkv, int Nq, int page_size, int max_pages, int d);
attn_status_t attn_decode_paged(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                                const int* block_table, const int* seq_lens,
                                void* workspace, size_t workspace_bytes,
                                int B, int H, int Hkv, int Nq, int page_size, int num_pages, int max_pages,
                                int d, float scale, int causal, void* stream);

/*
 * Forward with FP8 (e4m3) tensor-core products, head_dim 64, 96 or 128.  Page "Flash
 * Attention原理" (§六 and FAQ Q8: FlashAttention-3 runs attention on FP8
 * tensor cores).  Q, K and V are e4m3 (1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits; no infinities) with one dequantisation factor each: the
 * attention is that of q = q8 * q_scale, k = k8 * k_scale, v = v8 * v_scale.
 * S accumulates in float32; the softmax is float32; P is rounded to e4m3 for
 * the P V product, which makes O approximate to about e4m3's precision
 * (3 mantissa bits) while lse keeps float32 accuracy.
 *   q [in]  e4m3 bytes (B, H, Nq, d);  k, v [in] e4m3 bytes (B, Hkv, Nk, d)
 *   o [out] bf16 (B, H, Nq, d);  lse [out] float32 (B, H, Nq)
 *   scale   softmax scale; q_scale, k_scale, v_scale finite and > 0
 * Causal alignment and the Nq > Nk rule as attn_fwd_cross.  d outside
 * {64, 96, 128} gives ATTN_ERR_UNSUPPORTED_SHAPE.
 */
attn_status_t attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int Hkv, int Nq, int Nk, int d, float scale,
                           float q_scale, float k_scale, float v_scale, int causal, void* stream);

/*
 * Masks beyond is_causal (page "SDPA backend 与 FlashAttention" §3: the
 * boolean attn_mask of the SDPA call; "Flash Attention原理" FAQ Q11: padding
 * and arbitrary boolean masks handled inside the kernel).  Query row i sits
 * at position pos = Nk - Nq + i (i itself when Nq == Nk); key j takes part in
 * row i when all of these hold:
 *   causal (the call's flag)     j <= pos
 *   window_left  >= 0            j >= pos - window_left
 *   window_right >= 0            j <= pos + window_right   (a sliding window)
 *   key_lengths != NULL          j < key_lengths[b]        (padding mask;
 *                                values are clamped to [0, Nk])
 *   mask != NULL                 mask[b'][h'][i][j] != 0, with b' = b (or 0
 *                                when mask_batch == 1), h' = h (or 0 when
 *                                mask_heads == 1)
 * -1 leaves a window side open.  An additive mask (SDPA's float attn_mask)
 * adds bias[b''][h''][i][j] (broadcast over bias_batch, bias_heads as for
 * mask) to the scaled score of every (i, j) the conditions above keep:
 * softmax over j of scale * q_i . k_j + bias[i][j].  Its entries are finite
 * or -inf (-inf hides the key); +inf and NaN are not allowed.  The bias gets
 * no gradient.  A row no key passes (or whose bias is -inf at every key it
 * may see) gets O = 0, lse = -inf and dQ = 0; keys no row sees get
 * dK = dV = 0.
 *   key_lengths  DEVICE int32 (B), 4-byte aligned, or NULL
 *   mask         DEVICE bytes (mask_batch, mask_heads, Nq, Nk), dense
 *                row-major, any alignment, or NULL
 *   bias         DEVICE float32 (bias_bf16 == 0) or bf16 (bias_bf16 == 1)
 *                (bias_batch, bias_heads, Nq, Nk), dense row-major, aligned
 *                to its element size, or NULL (bias_batch, bias_heads and
 *                bias_bf16 are then ignored).  A bf16 bias is SDPA's float
 *                attn_mask in the query's dtype: half the bytes to read,
 *                the same arithmetic on the values it holds.  Any other
 *                bias_bf16 value gives ATTN_ERR_INVALID_ARG.
 */
typedef struct {
  int window_left;
  int window_right;
  const int* key_lengths;
  const unsigned char* mask;
  int mask_batch;   /* 1 or B */
  int mask_heads;   /* 1 or H */
  const void* bias; /* float32, or bf16 when bias_bf16 */
  int bias_batch;   /* 1 or B */
  int bias_heads;   /* 1 or H */
  int bias_bf16;    /* 0: float32 bias, 1: bf16 bias */
} attn_mask_t;

/*
 * Workspace bytes of attn_fwd_masked (backward = 0) or attn_bwd_masked
 * (backward = 1): the bit-packed mask (one bit per (query, key), plus its
 * transpose for the backward) and, for the backward, attn_bwd's row vectors.
 * 0 when the forward needs none (no boolean mask) or the shape is invalid.
 */
size_t attn_masked_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d, const attn_mask_t* mask,
                                  int backward);

/*
 * Forward and backward under the masks above; layouts as attn_fwd_cross /
 * attn_bwd_cross (Nq query rows, Nk key rows; Nq == Nk for self-attention).
 * Unlike attn_fwd_cross, causal with Nq > Nk is accepted (the first rows see
 * no key).  The workspace is owned by the caller (at least
 * attn_masked_workspace_size bytes, 16-byte aligned; NULL allowed when that
 * size is 0).  attn_bwd_masked_stages runs a subset of the backward's
 * stages, as attn_bwd_varlen_stages (1: prep and mask packing, 8: dQ with
 * the row vectors and mask packing, 2: dK / dV, 4: dQ); attn_bwd_masked runs
 * 8 then 2.
 */
attn_status_t attn_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                              const attn_mask_t* mask, void* workspace, size_t workspace_bytes,
                              void* stream);
attn_status_t attn_bwd_masked(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout,
                              void* dq, void* dk, void* dv,
                              int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                              const attn_mask_t* mask, void* workspace, size_t workspace_bytes,
                              void* stream);
attn_status_t attn_bwd_masked_stages(const void* q, const void* k, const void* v, const void* o,
                                     const float* lse, const void* dout,
                                     void* dq, void* dk, void* dv,
                                     int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                                     const attn_mask_t* mask, void* workspace, size_t workspace_bytes,
                                     unsigned stages, void* stream);

/*
 * Packed variable-length batch.  Page "Flash Attention原理", FAQ Q10:
 * sequences of different lengths are packed into one batch, delimited by
 * cumulative offsets (cu_seqlens), so no padding is computed.  Sequence b
 * owns query rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key rows
 * cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1 and attends only within itself.
 *   q, o   [in/out] bf16 (total_q, H, d)   packed, token-major
 *   k, v   [in]     bf16 (total_k, Hkv, d)
 *   lse    [out]    float32 (H, total_q)
 *   cu_seqlens_q, cu_seqlens_k  [in] DEVICE int32 arrays of B + 1 offsets:
 *          0 = cu[0] <= cu[1] <= ... <= cu[B] = total (4-byte aligned)
 *   max_seqlen_q, max_seqlen_k  upper bounds of the sequence lengths (they
 *          size the launch)
 * Causal: per sequence, query row i sits at position Nk_b - Nq_b + i and
 * sees keys 0 .. Nk_b - Nq_b + i.  Sequences may be empty, and Nq_b > Nk_b
 * is allowed: a row that sees no key gets O = 0 and lse = -inf (the result
 * of softmax over an empty set taken as zero weight everywhere).
 * The offsets are read on the device: inconsistent ones (decreasing, past
 * total, or longer than the stated maximum) skip the affected sequences and
 * make attn_get_device_status() return ATTN_ERR_INVALID_ARG.  Requires
 * total_q, total_k >= 1 and H * d * 128 < 2^32.
 */
attn_status_t attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                              const int* cu_seqlens_q, const int* cu_seqlens_k,
                              int B, int H, int Hkv, int total_q, int total_k,
                              int max_seqlen_q, int max_seqlen_k, int d, float scale, int causal,
                              void* stream);

/*
 * Bytes of device workspace attn_bwd_varlen needs: two float32 row vectors
 * per head, each sequence's rows in a 16-byte aligned region padded to a
 * multiple of 128, i.e. 8 * H * (round_up(total_q + 132 * B, 4) + 128).
 * Returns 0 for an invalid shape.
 */
size_t attn_bwd_varlen_workspace_size(int B, int H, int Hkv, int total_q, int d);

/*
 * Backward of attn_fwd_varlen: the gradients of attn_bwd per sequence, in
 * the packed layouts of attn_fwd_varlen (dq like q, dk / dv like k / v).
 * Keys that no query sees (an empty query sequence) get dK = dV = 0; rows
 * that saw no key get dQ = 0.  Same offset checks as attn_fwd_varlen.
 */
attn_status_t attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout,
                              void* dq, void* dk, void* dv,
                              const int* cu_seqlens_q, const int* cu_seqlens_k,
                              void* workspace, size_t workspace_bytes,
                              int B, int H, int Hkv, int total_q, int total_k,
                              int max_seqlen_q, int max_seqlen_k, int d, float scale, int causal,
                              void* stream);

/*
 * The stages of attn_bwd_varlen, for callers that schedule (or time) them
 * separately: `stages` is a non-zero OR of 1 (prep: D and lse in base 2 into
 * the workspace), 8 (dq_rows: dQ, forming and writing those row vectors),
 * 2 (grad: dK, dV) and 4 (dq: dQ from the row vectors), run in that order;
 * other bits are ATTN_ERR_INVALID_ARG.  The ordering rules of attn_bwd_prep /
 * _grad / _dq / _dq_rows apply: the row vectors are complete before grad or
 * dq starts.  attn_bwd_varlen runs 8 then 2.  Other arguments as
 * attn_bwd_varlen (all pointers are checked whether or not the stage reads
 * them).
 */
attn_status_t attn_bwd_varlen_stages(const void* q, const void* k, const void* v, const void* o,
                                     const float* lse, const void* dout,
                                     void* dq, void* dk, void* dv,
                                     const int* cu_seqlens_q, const int* cu_seqlens_k,
                                     void* workspace, size_t workspace_bytes,
                                     int B, int H, int Hkv, int total_q, int total_k,
                                     int max_seqlen_q, int max_seqlen_k, int d, float scale, int causal,
                                     unsigned stages, void* stream);

/*
 * Decode: attention of Nq new queries per head against a cache of Nk keys
 * and values (a KV cache), computed in key chunks that are merged by their
 * logsumexp.  Page "Flash Attention原理", FAQ on inference (the KV cache moves
 * the work into decode steps, profiled apart from prefill); the merge is the
 * two-block merge of §四 applied to any number of chunks.
 *   q    [in]  bf16 (B, H, Nq, d)     the new queries
 *   k, v [in]  bf16 (B, Hkv, Nk, d)   the cache; every position is valid
 *   o    [out] bf16 (B, H, Nq, d)     softmax(scale * q K^T [+ mask]) V
 *   lse  [out] float32 (B, H, Nq)     natural-log logsumexp of each query's
 *                                     scaled, masked scores
 *   causal     0: each query sees all Nk keys.  1: query t (0-based) of the
 *              block sits at position Nk - Nq + t, i.e. the new tokens end
 *              the sequence, and sees keys 0 .. Nk - Nq + t.
 *   workspace  device buffer of at least attn_decode_workspace_size() bytes,
 *              owned by the caller; its contents on entry are ignored.
 * Limits: 1 <= Nq <= Nk; (H / Hkv) * Nq <= 128 query rows per K/V head;
 * d in {64, 96, 128}.  Two kernels run on `stream` (chunk pass, merge); the
 * chunk count depends only on the shape.  Bound by the HBM read of K and V.
 */
size_t attn_decode_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d);
attn_status_t attn_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                          void* workspace, size_t workspace_bytes,
                          int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                          void* stream);

/*
 * Synchronises `stream`, then returns (and clears) the device status word
 * that the kernels set when a bounded wait runs out: ATTN_OK or
 * ATTN_ERR_TIMEOUT (ATTN_ERR_INVALID_ARG for device-side offsets found out
 * of range, ATTN_ERR_CHECK for a failed index check of the debug build);
 * ATTN_ERR_CUDA if the synchronisation itself failed.
 */
attn_status_t attn_get_device_status(void* stream);

/*
 * Where the first bounded wait that ran out since the last call happened,
 * for diagnosing ATTN_ERR_TIMEOUT: info[0] = (wait site << 16) | loop step,
 * info[1] = CTA index, info[2] = thread index, info[3] = microseconds waited;
 * all zero if no wait ran out.  In the debug build the first failed index
 * check (ATTN_ERR_CHECK) fills the same record when it comes first:
 * info[0] = check site << 16, info[3] = the offending element index
 * (clamped to the int range).  Synchronises `stream`, then clears the record.
 * Each wait is limited to 2 s, or to SDPA08_WAIT_LIMIT_MS milliseconds
 * (1..60000) if that environment variable is set when the library is first
 * used on a device.
 */
attn_status_t attn_get_timeout_info(int info[4], void* stream);

/* Human-readable name of a status code (static storage; never NULL). */
const char* attn_status_string(attn_status_t s);

/* ABI version of this header (incremented on incompatible changes; 3: attn_mask_t.bias_bf16). */
int attn_abi_version(void);

/*
 * Self-test of the bounded-wait machinery: launches one CTA whose threads
 * wait, with a limit of `timeout_us` microseconds, on an on-chip barrier that
 * nothing ever signals.  The kernel must give up, record ATTN_ERR_TIMEOUT
 * and exit, leaving the context usable.  Returns ATTN_OK if launched; read
 * the outcome with attn_get_device_status().  The pages have no counterpart;
 * this exists so the failure-detection path can be tested without faulting
 * or hanging a GPU.
 */
attn_status_t attn_selftest_wait_timeout(unsigned int timeout_us, void* stream);

/*
 * Test hook for the failure-detection path of the production kernels (off
 * unless called; the pages have no counterpart).  Arms one launch: the next
 * launch of `kernel` from this process (0: the launch-per-unit forward
 * kernel, which then serves attn_fwd / attn_fwd_cross for that launch; 1:
 * the dQ kernel, attn_bwd's first stage; 2: the dK/dV kernel, its second;
 * 3: the persistent forward kernel, which serves attn_fwd / attn_fwd_cross
 * otherwise; 4: the persistent dK/dV kernel, which serves the dense second
 * stage otherwise, kernel 2 being the launch-per-unit one; 5: the persistent
 * dQ kernel, which serves the dense first stage otherwise, kernel 1 being
 * the launch-per-unit one; 6: the FP8 forward, attn_fwd_fp8) runs with
 * every on-chip wait limited to `limit_us` microseconds, and in its first
 * CTA (kernels 3, 4, 5, and 6 at head_dim 64 / 96: the CTA that takes the
 * first work unit) the TMA producer does not issue its `load_index`-th ring
 * load of that unit (forward and FP8 forward: K_0, V_0, K_1, ...; dQ: the
 * same; dK/dV: the query tiles Q_i with their row vectors; persistent dQ:
 * the key tiles K_0, K_1, ...).  The consumers of that load then wait in
 * vain: the first wait to run out records ATTN_ERR_TIMEOUT in the device
 * status word (attn_get_device_status) and where it gave up
 * (attn_get_timeout_info), and every role of that CTA stops and exits, so
 * the context stays usable; the other CTAs complete normally.
 * The outputs of that launch are not valid.  The hook is cleared by the
 * launch it applies to.
 *   load_index: 0 .. 2^20; limit_us: 1000 .. 60,000,000.  Other values give
 *   ATTN_ERR_INVALID_ARG (and arm nothing).
 */
attn_status_t attn_debug_drop_load(int kernel, int load_index, unsigned int limit_us);

/*
 * attn_bwd for callers that cannot allocate device memory.  The pages have no
 * counterpart; this is a property of the library, not of the method.
 *
 * Some callers have no way to provide attn_bwd's workspace: code running
 * where cudaMalloc is not allowed (inside a custom allocator, or a runtime
 * that owns the whole device memory pool) or a plug-in interface that passes
 * only tensor pointers.  This entry point computes exactly what attn_bwd
 * computes, with the same arguments minus the workspace, using instead a
 * fixed 64 MiB scratch array compiled into the library.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *   - Limit: shapes whose attn_bwd_workspace_size() exceeds 64 MiB
 *     (67108864 bytes) are rejected with ATTN_ERR_WORKSPACE; use attn_bwd
 *     with a caller workspace for those.  (That allows
 *     B*H*ceil(N/128)*128 <= 8,388,608 padded rows, e.g. B=8, H=16,
 *     N=65536.)
 *   - Memory: every GPU that loads the library holds the 64 MiB until the
 *     process exits.
 *   - Set-up: the first call on a device looks up the array's device address
 *     with that device current; make that first call before any stream
 *     capture.  The address is kept for the life of the process, so only
 *     the device's primary context is supported, and no cudaDeviceReset
 *     between calls.
 *   - Errors: arguments and the device are checked as attn_bwd checks them,
 *     with the same status values, before the array is looked up.  After a
 *     call whose kernels timed out (ATTN_ERR_TIMEOUT from
 *     attn_get_device_status), dK and dV may come from an earlier call's
 *     row vectors and must be discarded.
 *   - Sharing: all calls use the same array, which keeps the last call's
 *     contents (each call rewrites what it reads).  Calls whose work
 *     overlaps on the GPU (different streams, or different host threads
 *     without ordering) race on the array and give wrong results; order
 *     them on one stream.
 */
attn_status_t attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                               const float* lse, const void* dout,
                               void* dq, void* dk, void* dv,
                               int B, int H, int Hkv, int N, int d, float scale, int causal,
                               void* stream);

/*
 * 1 when this library was built with the index checks of the debug build
 * (-DATTN_DEBUG), 0 for the release build.  The pages have no counterpart:
 * compute-sanitizer is not available on the target machines, and these
 * checks stand in for its bounds checking.  In the debug build every plain
 * global load and store whose element index a kernel computes (row vectors,
 * lse, mask bits, the additive mask, packed-batch rows, decode partials,
 * block-table entries) first checks that index against the extent implied
 * by the call's arguments; a failed check records ATTN_ERR_CHECK
 * (attn_get_device_status) and where it failed (attn_get_timeout_info),
 * and the access is skipped (or, for a copy whose barrier expects its
 * bytes, read from an in-range place), so the launch still completes and
 * the context stays usable.  TMA copies need no check: the hardware clips
 * them to the tensor map.
 */
int attn_debug_build(void);

/*
 * Test hook of the debug build (the pages have no counterpart): arms one
 * launch, like attn_debug_drop_load, in which the first CTA computes an
 * element index past the end of an output array, so that the index checks
 * must catch it.  kernel 0: the forward kernel's lse store (attn_fwd and the
 * calls built on it); 1: the dQ kernel's row-vector store into the workspace
 * (attn_bwd's first stage; the dK/dV results of that call are then
 * undefined).  The check records ATTN_ERR_CHECK and skips the store.
 * Returns ATTN_ERR_INVALID_ARG for another kernel value and in the release
 * build, where nothing is armed.
 */
attn_status_t attn_debug_plant_index(int kernel);

#ifdef __cplusplus
}
#endif

#endif /* SDPA08_ATTN_H */
