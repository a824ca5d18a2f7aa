/*
 * fa_gb300.h -- C ABI of the exact IO-aware attention library for GB300 (sm_103a).
 *
 * The operation (all entry points below compute pieces of it):
 *
 *   O = softmax(s * Q K^T) V,  per (batch, head), s = `scale`,
 *
 * evaluated tile by tile with the online-softmax recurrence: a running max
 * m, a running sum l and an unnormalised accumulator, rescaled by
 * exp(m_old - m_new) whenever m grows ("FlashAttention 为什么不需要存下注意力矩阵",
 * jefxiong.cn, section 3.2; "FlashAttention V1 技术深度解析", spark.aweffr.cn,
 * section 3.2).  The forward pass writes only O and the per-row log-sum-exp
 * LSE = m + ln l; the backward pass recomputes every tile of P on chip from
 * LSE (same tutorial, section 3.3) -- no N x N matrix is ever written to
 * device memory.  Under the causal mask, key j is visible to query i iff
 * j <= i, and key tiles that are entirely masked are skipped (same tutorial,
 * section 3.2 and 4.5).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers are DEVICE pointers owned by the caller; the library never
 *   allocates or frees device memory and keeps no pointer after returning.
 *   Every device pointer must be 16-byte aligned.
 * - Q, K, V, O, dO, dQ, dK, dV are contiguous [B, H, N, d] arrays of the
 *   16-bit type `dtype` (FA_FP16 or FA_BF16).  LSE and D are contiguous
 *   [B, H, N] float32 arrays.  LSE is in natural-log units of the scaled
 *   scores: LSE_i = ln sum_j exp(s * q_i . k_j).
 * - Supported: d in {64, 96, 128, 256} (split-KV decoding: 64, 128, 256; block masks: not
 *   256); N >= 1
 *   (any N: tails are masked); B, H >= 1 with B*H*N*d < 2^31; scale finite
 *   and > 0.  d = 96 runs the d = 128 kernels with features 96-127 read as
 *   zero and never stored.
 * - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *   enqueue work on it and return; nothing is written to host memory and
 *   the host never waits.
 * - Return value: FA_OK, or FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED before
 *   anything is launched, or FA_ERR_CUDA if a launch failed.  A kernel that
 *   finds a pipeline wait exceeding ~2 s gives up, returns, and latches
 *   FA_ERR_TIMEOUT in a device status word that fa_device_status() reports.
 * - No exceptions cross this interface; all entry points are thread-safe
 *   (they keep no mutable host state).
 * - Outputs must not alias inputs.
 * - Packed variable-length batches (fa_*_varlen): see the block before
 *   fa_forward_varlen.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,
  FA_ERR_UNSUPPORTED = 2,
  FA_ERR_CUDA = 3,
  FA_ERR_TIMEOUT = 4,
  FA_ERR_WORKSPACE = 5,
  FA_ERR_SCRATCH_TOO_SMALL = 6,
  FA_ERR_SEQLENS = 7
} fa_status;

typedef enum { FA_FP16 = 0, FA_BF16 = 1 } fa_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char* fa_status_string(int status);

/*
 * Forward pass.  Writes O [B,H,N,d] (dtype) and LSE [B,H,N] (float32).
 * Exact softmax attention by the online-softmax recurrence (tutorial
 * section 3.2); LSE = m + ln l is the only extra output kept for the
 * backward pass (tutorial section 3.2, last remark, and section 3.3).
 * q, k, v: inputs; o, lse: outputs, fully overwritten.
 */
fa_status fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                     int d, int dtype, int causal, float scale, void* stream);

/*
 * Block-sparse forward: fa_forward with whole 128 x 128 (query, key) blocks
 * removed.  The tutorial's section 06 generalises the causal whole-block skip
 * to any sparsity pattern; kept blocks are computed exactly as in
 * fa_forward, removed blocks are never loaded or multiplied.
 * block_mask: DEVICE pointer to uint8 [mask_heads, T, T], T = ceil(N/128),
 * row-major; nonzero = keep the block (query block i, key block j).
 * mask_heads: 1 (one mask for every head) or B*H (one per head, in [B,H]
 * order).  `causal` still applies inside kept blocks.  A query row that keeps
 * no key at all gets O = 0 and LSE = -inf.  Errors: FA_ERR_INVALID_ARG for a
 * null mask or a mask_heads other than 1 or B*H; otherwise as fa_forward.
 */
fa_status fa_forward_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse,
                                 const uint8_t* block_mask, int mask_heads, int B, int H, int N, int d, int dtype,
                                 int causal, float scale, void* stream);

/*
 * Bytes of device workspace fa_backward needs: D (B*H*N float32) followed by
 * the float32 dQ accumulator (B*H*N*d float32), each 256-byte aligned.
 * Linear in N.  Returns 0 for invalid sizes.
 */
size_t fa_backward_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass (tutorial section 3.3): with G = dO and P recomputed tile by
 * tile as exp(s * Q K^T - LSE),
 *   dS = P * (G V^T - D),  D_i = sum_c dO_ic O_ic  ( = rowsum(P * (G V^T)) ),
 *   dQ = s dS K,  dK = s dS^T Q,  dV = P^T G.
 * Two strategies for dQ, both exact (chosen per call, see below):
 *   - split (d in {64, 96, 128} without dropout: dense layouts with or
 *     without a block mask, packed batches): fa_backward_preprocess with
 *     dq_accum = NULL, fa_backward_dk_dv, fa_backward_dq (with a block mask:
 *     fa_backward_dk_dv_blocksparse, fa_backward_dq_blocksparse; packed:
 *     fa_backward_dk_dv_varlen, fa_backward_dq_varlen) -- dQ by a kernel of
 *     its own that recomputes P and dP, no float32 accumulator;
 *   - accumulated (d = 256, dropout): fa_backward_preprocess,
 *     fa_backward_dkdv, fa_backward_dq_convert -- dQ partials added into a
 *     float32 accumulator by the dK / dV kernel.
 *     (fa_backward_dk_dv_dropout / fa_backward_dq_dropout run dropout on the
 *     split kernels for callers without room for the accumulator.)
 * All stages run in order on `stream`.  `workspace` must hold
 * fa_backward_workspace_size(B,H,N,d) bytes (else FA_ERR_WORKSPACE); its
 * contents on entry do not matter and are overwritten.
 * o and lse are the forward outputs for the same q, k, v, causal and scale.
 */
fa_status fa_backward(const void* q, const void* k, const void* v, const void* o, const void* dO,
                      const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, int dtype,
                      int causal, float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Block-sparse backward: fa_backward for the forward of
 * fa_forward_blocksparse with the same block_mask / mask_heads / causal.
 * Products of removed blocks are skipped; a key block kept by no query block
 * gets dK = dV = 0, a query row with no visible key gets dQ = 0.
 */
fa_status fa_backward_blocksparse(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                  const float* lse, void* dq, void* dk, void* dv, const uint8_t* block_mask,
                                  int mask_heads, int B, int H, int N, int d, int dtype, int causal, float scale,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * Attention dropout ("FlashAttention 为什么不需要存下注意力矩阵", section 05: the
 * kernel stores no dropout mask, only the seed and offset of a Philox
 * counter-based generator, and the backward pass regenerates the mask).
 *
 * The dropout acts on the normalised probabilities: O = (P * Z / (1 - p')) V
 * with Z the keep mask and p' = t / 256, t = round(p_drop * 256) (p_drop is
 * quantised to 2^-8); lse is still the log-sum-exp of the undropped scores.
 * Z is drawn with Philox4x32-10 (Salmon et al., SC 2011): entry (head
 * bh = b*H + h, query i, key j) uses counter (j / 16, i, bh, offset) and key
 * (seed & 0xffffffff, seed >> 32); byte j % 4 (least significant first) of
 * word (j / 4) % 4 of the output gives an 8-bit draw, and the entry is kept
 * iff draw >= t.  The same (p_drop, seed, offset) must be
 * passed to the backward call; a new offset (or seed) gives a new mask.
 * p_drop must be in [0, 1) and not round to 1, else FA_ERR_INVALID_ARG;
 * p_drop rounding to 0 computes plain attention.  Dense attention only
 * (no block mask).  Other arguments, errors and layouts as fa_forward /
 * fa_backward / fa_backward_dkdv.
 */
fa_status fa_forward_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                             int d, int dtype, int causal, float scale, float p_drop, uint64_t seed,
                             uint32_t offset, void* stream);
fa_status fa_backward_dropout(const void* q, const void* k, const void* v, const void* o, const void* dO,
                              const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, int dtype,
                              int causal, float scale, float p_drop, uint64_t seed, uint32_t offset, void* workspace,
                              size_t workspace_bytes, void* stream);
fa_status fa_backward_dkdv_dropout(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                                   const float* delta, float* dq_accum, void* dk, void* dv, int B, int H, int N,
                                   int d, int dtype, int causal, float scale, float p_drop, uint64_t seed,
                                   uint32_t offset, void* stream);
/*
 * The split backward with dropout, d in {64, 96, 128}: no float32 dQ
 * accumulator, at the price of drawing the keep mask in both kernels
 * (fa_backward_dropout, which accumulates dQ, is faster).  With Z the
 * regenerated keep mask and c = 256 / (256 - t),
 *   dV = c (P * Z)^T dO,  dS = P * (c Z * (dO V^T) - D),  dK = s dS^T Q,
 *   dQ = s dS K,
 * D = rowsum(dO * O) from fa_backward_preprocess(o, dO, delta, NULL, ...).
 * fa_backward_dk_dv_dropout writes dk, dv; fa_backward_dq_dropout writes dq
 * (no workspace).  Dropout arguments as fa_forward_dropout, the rest as
 * fa_backward_dk_dv / fa_backward_dq; d = 256 gives FA_ERR_UNSUPPORTED.
 */
fa_status fa_backward_dk_dv_dropout(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                                    const float* delta, void* dk, void* dv, int B, int H, int N, int d, int dtype,
                                    int causal, float scale, float p_drop, uint64_t seed, uint32_t offset,
                                    void* stream);
fa_status fa_backward_dq_dropout(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                                 const float* delta, void* dq, int B, int H, int N, int d, int dtype, int causal,
                                 float scale, float p_drop, uint64_t seed, uint32_t offset, void* stream);

/*
 * The keep mask the dropout entry points use, written out: keep is a device
 * buffer of BH * Nq * Nk bytes ([BH, Nq, Nk], 1 = kept, 0 = dropped).  For
 * inspection and tests; the attention entry points never store it.
 */
fa_status fa_dropout_keep_mask(uint8_t* keep, int BH, int Nq, int Nk, float p_drop, uint64_t seed, uint32_t offset,
                               void* stream);

/*
 * Self-test of failure detection: launches one thread that waits, with the
 * bounded pipeline wait every kernel uses, on a barrier nothing ever
 * completes.  The wait gives up after ~2 s and latches FA_ERR_TIMEOUT, so the
 * next fa_device_status() returns FA_ERR_TIMEOUT (and clears it) while the
 * context stays usable.  No counterpart in the pages: it checks that a stuck
 * pipeline ends and is reported instead of hanging the GPU.
 */
fa_status fa_selftest_wait_timeout(void* stream);

/*
 * Stage 1 of the backward pass: D_i = sum_c dO_ic * O_ic in float32 (the
 * row-sum shortcut for rowsum(P * (dO V^T)), which holds because O = P V),
 * and dq_accum := 0.  delta: [B,H,N] float32 out; dq_accum: [B,H,N,d]
 * float32 out, or NULL (only D is computed; the split backward needs no
 * accumulator).
 */
fa_status fa_backward_preprocess(const void* o, const void* dO, float* delta, float* dq_accum, int B, int H,
                                 int N, int d, int dtype, void* stream);

/*
 * Stage 2: for every key tile, recompute S^T and P^T per query tile from
 * LSE, form dP^T = V dO^T and dS^T = P^T * (dP^T - D), accumulate
 * dV = P^T dO and dK = s dS^T Q on chip and write them (dtype), and add the
 * per-tile dQ partials dS K (unscaled, float32) into dq_accum with atomics.
 * Causal: query tiles entirely above the diagonal are skipped.
 */
fa_status fa_backward_dkdv(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                           const float* delta, float* dq_accum, void* dk, void* dv, int B, int H, int N, int d,
                           int dtype, int causal, float scale, void* stream);

/*
 * Stage 2 of fa_backward_blocksparse: fa_backward_dkdv restricted to the
 * kept blocks of block_mask (same mask arguments and errors as
 * fa_forward_blocksparse).  A key block kept by no query block gets
 * dK = dV = 0 and adds nothing to dq_accum.
 */
fa_status fa_backward_dkdv_blocksparse(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                                       const float* delta, float* dq_accum, void* dk, void* dv,
                                       const uint8_t* block_mask, int mask_heads, int B, int H, int N, int d,
                                       int dtype, int causal, float scale, void* stream);

/* Stage 3: dq = scale * dq_accum, rounded to dtype. */
fa_status fa_backward_dq_convert(const float* dq_accum, void* dq, int B, int H, int N, int d, int dtype,
                                 float scale, void* stream);

/*
 * The split backward (tutorial section 3.3 with the dQ sum done apart from
 * dK and dV), after fa_backward_preprocess(o, dO, delta, NULL, ...):
 *
 * fa_backward_dk_dv: for every 128-key tile, loop over the 128-query tiles
 * that see it, recompute S^T, P^T = exp(s K Q^T - LSE) and dP^T = V dO^T on
 * chip, form dS^T = P^T * (dP^T - D), accumulate dV = P^T dO and
 * dK = s dS^T Q on chip and write dk, dv (dtype).  No dQ work.
 *
 * fa_backward_dq: for every 128-query tile, loop over the key tiles it sees,
 * recompute S, P and dP, form dS = P * (dP - D), accumulate dQ = s dS K on
 * chip and write dq (dtype).  Writes nothing else; needs no workspace.
 *
 * Both: dense [B, H, N, d] tensors, d in {64, 96, 128} (256 gives
 * FA_ERR_UNSUPPORTED), lse and delta [B, H, N] float32 inputs (the forward's
 * LSE and the preprocess stage's D); causal: tiles entirely above the
 * diagonal are skipped.  Errors as fa_backward_dkdv, before any launch.
 */
fa_status fa_backward_dk_dv(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                            const float* delta, void* dk, void* dv, int B, int H, int N, int d, int dtype, int causal,
                            float scale, void* stream);
fa_status fa_backward_dq(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                         const float* delta, void* dq, int B, int H, int N, int d, int dtype, int causal, float scale,
                         void* stream);

/*
 * The split backward restricted to the kept blocks of block_mask (the
 * whole-block skip of the tutorial's section 06 applied to both kernels;
 * mask arguments and errors as fa_forward_blocksparse, the rest as
 * fa_backward_dk_dv / fa_backward_dq).  fa_backward_dk_dv_blocksparse: a key
 * block kept by no query block gets dK = dV = 0.  fa_backward_dq_blocksparse:
 * a query block that keeps no key block gets dQ = 0.
 */
fa_status fa_backward_dk_dv_blocksparse(const void* q, const void* k, const void* v, const void* dO,
                                        const float* lse, const float* delta, void* dk, void* dv,
                                        const uint8_t* block_mask, int mask_heads, int B, int H, int N, int d,
                                        int dtype, int causal, float scale, void* stream);
fa_status fa_backward_dq_blocksparse(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                                     const float* delta, void* dq, const uint8_t* block_mask, int mask_heads, int B,
                                     int H, int N, int d, int dtype, int causal, float scale, void* stream);

/*
 * Packed variable-length batches.  B sequences of different lengths laid end
 * to end in token-major tensors: q, o, dq are [total_q, H, d] and k, v, dk, dv
 * are [total_k, H, d] (16-bit, contiguous); lse is [total_q, H] float32 (the
 * same flat order as the rows of q).  cu_seqlens_q and cu_seqlens_k are
 * device int32 arrays of B + 1 offsets: sequence b owns query rows
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key rows cu_seqlens_k[b] ..
 * cu_seqlens_k[b+1]-1 (cu[0] = 0, non-decreasing, cu[B] = total).  Each
 * sequence is an independent attention problem ("FlashAttention 为什么不需要存下
 * 注意力矩阵", section 3, applied per sequence); under the causal mask the
 * diagonal is aligned bottom-right: query i of a sequence with Nq queries and
 * Nk keys sees key j iff j <= i + Nk - Nq, and a query that sees no key (and
 * every query of a sequence with no key) gets O = 0 and LSE = -inf, and dQ = 0.
 * max_seqlen_q / max_seqlen_k (host ints) bound the per-sequence lengths and
 * size the grid.  The offsets are read on the device only: a sequence whose
 * range leaves [0, total] or exceeds the maxima is skipped and FA_ERR_SEQLENS
 * is latched for fa_device_status().  p_drop, seed, offset: dropout as for
 * fa_forward_dropout (p_drop = 0: none), with the query index counted within
 * its sequence and bh = b * H + h.  The backward workspace holds
 * fa_backward_varlen_workspace_size(total_q, H, d) bytes (256-byte aligned).
 */
fa_status fa_forward_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                            const int* cu_seqlens_k, int B, int H, int max_seqlen_q, int max_seqlen_k, int total_q,
                            int total_k, int d, int dtype, int causal, float scale, float p_drop, uint64_t seed,
                            uint32_t offset, void* stream);
size_t fa_backward_varlen_workspace_size(int total_q, int H, int d);
fa_status fa_backward_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO,
                             const float* lse, void* dq, void* dk, void* dv, const int* cu_seqlens_q,
                             const int* cu_seqlens_k, int B, int H, int max_seqlen_q, int max_seqlen_k, int total_q,
                             int total_k, int d, int dtype, int causal, float scale, float p_drop, uint64_t seed,
                             uint32_t offset, void* workspace, size_t workspace_bytes, void* stream);
/*
 * Stage 2 of fa_backward_varlen (the dK/dV kernel alone).  Stages 1 and 3 are
 * fa_backward_preprocess and fa_backward_dq_convert called with B = 1, H = 1,
 * N = total_q * H: they treat the packed rows as one flat [rows, d] array.
 * delta [total_q, H] and dq_accum [total_q, H, d] float32 as in the workspace
 * of fa_backward_varlen (delta first, dq_accum at the next 256-byte boundary).
 */
fa_status fa_backward_dkdv_varlen(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                                  const float* delta, float* dq_accum, void* dk, void* dv, const int* cu_seqlens_q,
                                  const int* cu_seqlens_k, int B, int H, int max_seqlen_q, int max_seqlen_k,
                                  int total_q, int total_k, int d, int dtype, int causal, float scale, float p_drop,
                                  uint64_t seed, uint32_t offset, void* stream);
/*
 * The split backward of a packed batch (what fa_backward_varlen runs at
 * d in {64, 96, 128} without dropout), after fa_backward_preprocess(o, dO,
 * delta, NULL, 1, 1, total_q * H, d, ...): fa_backward_dk_dv_varlen writes
 * dk, dv; fa_backward_dq_varlen writes dq (each needs no workspace).  As
 * fa_backward_dk_dv / fa_backward_dq per sequence, with the layouts,
 * offsets and bottom-right causal mask of fa_backward_varlen; d = 256 gives
 * FA_ERR_UNSUPPORTED.
 */
fa_status fa_backward_dk_dv_varlen(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                                   const float* delta, void* dk, void* dv, const int* cu_seqlens_q,
                                   const int* cu_seqlens_k, int B, int H, int max_seqlen_q, int max_seqlen_k,
                                   int total_q, int total_k, int d, int dtype, int causal, float scale, void* stream);
fa_status fa_backward_dq_varlen(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                                const float* delta, void* dq, const int* cu_seqlens_q, const int* cu_seqlens_k, int B,
                                int H, int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int d, int dtype,
                                int causal, float scale, void* stream);

/*
 * Split-KV forward for few queries against many keys (decoding).
 * q, o: [B,H,Nq,d]; k, v: [B,H,Nk,d]; lse: [B,H,Nq] float32 (natural log, as
 * fa_forward).  Same result as fa_forward on a rectangular problem: the key
 * range of every head is cut into `num_splits` chunks, each chunk yields its
 * normalised output and log-sum-exp with the online-softmax recurrence
 * (tutorial section 3.2), and the chunks are merged exactly by
 * LSE = log sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s.
 * Causal: the queries are the last Nq of the Nk positions, so key j is
 * visible to query i iff j <= i + Nk - Nq (requires Nq <= Nk).
 * num_splits = 0 picks a count that fills the GPU; otherwise 1..1024.
 * workspace: fa_decode_workspace_size(B,H,Nq,Nk,d,num_splits) bytes of
 * device memory (partial outputs), contents irrelevant on entry.
 * Supported: d in {64, 128, 256}, fp16/bf16, B*H <= 65535, Nq, Nk >= 1.
 */
size_t fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits);
fa_status fa_forward_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                            int Nq, int Nk, int d, int dtype, int causal, float scale, int num_splits,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * Split-KV decoding with grouped queries: Hq query heads share Hkv K / V heads
 * (Hq a multiple of Hkv; query head h reads K / V head h / (Hq / Hkv)).
 * q, o: [B,Hq,Nq,d]; k, v: [B,Hkv,Nk,d]; lse: [B,Hq,Nq] float32.  Every query
 * head gets what fa_forward_decode gives it against its K / V head (causal:
 * query i of every head at position i + Nk - Nq), but each K / V chunk is read
 * once for all the query heads that share it.  workspace:
 * fa_decode_gqa_workspace_size(B,Hq,Hkv,Nq,Nk,d,num_splits) bytes (0 for
 * invalid sizes).  Hq not a multiple of Hkv, or Hq, Hkv < 1, gives
 * FA_ERR_INVALID_ARG; other arguments and errors as fa_forward_decode (which
 * is this call with Hq = Hkv = H).
 */
size_t fa_decode_gqa_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d, int num_splits);
fa_status fa_forward_decode_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                int Hkv, int Nq, int Nk, int d, int dtype, int causal, float scale, int num_splits,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * Size of the fixed device scratch array used by fa_backward_noalloc.
 */
#define FA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * fa_backward without a workspace argument, for callers that cannot
 * allocate device memory (plugins inside a framework that owns every
 * allocation, allocation-free serving paths, callers that only hold raw
 * input/output pointers).  The pages have no counterpart: this is a
 * deployment convenience, computing exactly what fa_backward computes.
 * The D vector and the fp32 dQ accumulator live in a static device array of
 * FA_NOALLOC_SCRATCH_BYTES (32 MiB) that every GPU loading the library keeps
 * until the process exits.  Problems with fa_backward_workspace_size() larger
 * than that return FA_ERR_SCRATCH_TOO_SMALL before any launch; any other
 * invalid argument gets the status fa_backward returns for it, checked
 * first and before any CUDA call.  The first
 * call on a device looks up the array's address with that device current;
 * make it before any stream capture starts.  All calls share the array:
 * calls that overlap on the GPU race and must be serialised.  Each call
 * rewrites D and zeroes the accumulator, so stale contents do not matter.
 * Other arguments, ownership and errors: as fa_backward.
 */
fa_status fa_backward_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                              const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                              int dtype, int causal, float scale, void* stream);

/*
 * Waits for all work queued on `stream`, then returns and clears the device
 * status word of the library on the current device: FA_OK, FA_ERR_TIMEOUT if
 * a kernel gave up waiting since the last call, or FA_ERR_CUDA if the
 * stream reports an error.  The only entry point that blocks the host.
 */
fa_status fa_device_status(void* stream);

/*
 * Work counters, for checking which score tiles the kernels compute.  The
 * tiled algorithm ("FlashAttention 为什么不需要存下注意力矩阵", jefxiong.cn,
 * section 04.5: a tile lying wholly above the causal diagonal is skipped)
 * visits T(T+1)/2 of the T x T square tiles under the causal mask, and the
 * block-sparse variant only the kept blocks.  Every forward and dK/dV kernel
 * adds the score blocks it computed, in units of 64 query rows x 64 keys
 * (a 128 x 128 tile counts 4), to one of two 64-bit device counters: the
 * forward kernels to *fwd_blocks, the dK/dV kernels to *bwd_blocks (a
 * score block recomputed by both feature halves at d = 256 counts once).
 * Tiles cover whole tile shapes, so at a ragged tail a partial tile counts
 * in full.  Waits for all work queued on `stream`, stores both counters
 * through the host pointers (either may be NULL) and zeroes them if `reset`
 * is nonzero.  Blocks the host.  Errors: FA_ERR_CUDA if the stream or a copy
 * fails.
 */
fa_status fa_score_blocks(void* stream, unsigned long long* fwd_blocks, unsigned long long* bwd_blocks, int reset);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
