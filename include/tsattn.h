/*
 * tsattn.h -- C ABI of the attention block on GB300 (sm_103a).
 *
 * Operation.  For every batch b and head h,
 *
 *     O[b,h] = softmax(scale * Q[b,h] K[b,h]^T) V[b,h]
 *
 * with Q (Sq x D), K and V (Sk x D) and O (Sq x D), the softmax taken over
 * the keys a query row may see: all of them, or, with `causal`, keys
 * t <= i + Sk - Sq for query row i (a row that sees no key is zero).  This
 * is the per-device block of the FlashMLA example of the TileScale README
 * (section "Example of FlashMLA"): blocks of query rows loop over key /
 * value blocks, S = Q K^T on the tensor cores, a running row maximum and
 * row sums (online softmax with base-2 exponentials), the weights cast to
 * the 16-bit input format and O += P V on the tensor cores, O divided by
 * the row sums at the end.  The example's multi-GPU context parallelism
 * and its MLA split of the query into a latent and a rotary part are not
 * part of tsattn_forward: there Q K^T runs over one head dimension D.
 * tsattn_mla_decode below is the MLA decode shape.
 *
 * Formats.  Q, K, V and O are all fp16 or all bf16 (TSGEMM_F16 /
 * TSGEMM_BF16 of tsgemm.h); D = 128.  Scores, the softmax and the O
 * accumulator are fp32; the weights are rounded to the input format before
 * they multiply V; O is rounded to nearest, ties to even.
 *
 * Memory.  Q, K, V, O are device pointers of the current device, 16-byte
 * aligned, laid out [B][H][S][D] row-major (D contiguous); O must not
 * overlap Q, K or V.  Nothing is allocated.
 *
 * Errors.  Argument errors are returned before anything is launched:
 * TSGEMM_ERR_INVALID_ARG (sizes < 1, null or overlapping pointers, a
 * non-finite scale), TSGEMM_ERR_ALIGNMENT, TSGEMM_ERR_UNSUPPORTED (D other
 * than 128, another dtype, a device other than compute capability 10.3),
 * TSGEMM_ERR_CUDA (a failed CUDA call or launch).
 * Every device wait is bounded (1 s); an expired wait writes
 * TSGEMM_ERR_TIMEOUT to `status` (a device int, cleared on `stream` before
 * the launch) or, when `status` is NULL, to a word of the library that
 * tsattn_status() reads and clears after the caller has synchronised.
 */
#ifndef TSATTN_H
#define TSATTN_H

#include <stdint.h>

#include "tsgemm.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Enqueue the attention forward pass on `stream` (a cudaStream_t; NULL is
 * the legacy default stream).  Asynchronous. */
TSGEMM_API tsgemm_status_t tsattn_forward(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int32_t D,
                                          tsgemm_dtype_t dtype, float scale, int32_t causal,
                                          const void* Q, const void* K, const void* V, void* O,
                                          int* status, void* stream);

/* tsattn_forward with test-only flags (TSGEMM_DEBUG_SKIP_FIRST_LOAD: the
 * first CTA leaves its first key/value block unloaded, so a bounded wait
 * runs out) and the limit of every device wait in milliseconds (0: 1 s). */
TSGEMM_API tsgemm_status_t tsattn_forward_ex(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int32_t D,
                                             tsgemm_dtype_t dtype, float scale, int32_t causal,
                                             const void* Q, const void* K, const void* V, void* O,
                                             int* status, void* stream, int32_t debug_flags,
                                             int32_t timeout_ms);

/* ---- MLA decode --------------------------------------------------------
 *
 * The decode shape of the same block in the FlashMLA example of the
 * TileScale README (section "Example of FlashMLA"): one query token per
 * sequence, every query head of a batch against one shared latent cache
 * that is both key and value.  For batch b and head h,
 *
 *     s[t]   = scale * (Q[b,h] . KV[b,t] + Q_pe[b,h] . K_pe[b,t])
 *     O[b,h] = sum_t softmax(s)[t] * KV[b,t]
 *
 * over the keys t = 0 .. Skv - 1, with Q (H x dim) and Q_pe (H x pe_dim)
 * per batch, the latent cache KV (Skv x dim) and its rotary part K_pe
 * (Skv x pe_dim) per batch, and O (H x dim): scores 576 deep, values 512
 * wide.  dim must be 512 and pe_dim 64 (the example's latent and rotary
 * widths); any H >= 1 and Skv >= 1.
 *
 * Formats and numerics as for tsattn_forward: all tensors fp16 or all
 * bf16; scores (the latent and rotary parts summed in fp32), the softmax
 * and the accumulator are fp32; weights are rounded to the input format
 * before they multiply KV; O is rounded to nearest, ties to even.
 *
 * Memory.  Row-major device pointers of the current device, 16-byte
 * aligned: Q [B][H][dim], Q_pe [B][H][pe_dim], KV [B][Skv][dim], K_pe
 * [B][Skv][pe_dim], O [B][H][dim]; O must not overlap an input.  Nothing is
 * allocated.  Each batch's 128-head block runs on a pair of CTAs (a 2 x 1
 * cluster) that split the value columns and the score contraction and
 * exchange partial scores through distributed shared memory.
 *
 * Errors as for tsattn_forward (TSGEMM_ERR_UNSUPPORTED for dim != 512 or
 * pe_dim != 64); a timeout goes to `status`, or, when it is NULL, to the
 * word tsattn_status() reads. */
TSGEMM_API tsgemm_status_t tsattn_mla_decode(int64_t B, int64_t H, int64_t Skv, int32_t dim, int32_t pe_dim,
                                             tsgemm_dtype_t dtype, float scale, const void* Q, const void* Q_pe,
                                             const void* KV, const void* K_pe, void* O, int* status, void* stream);

/* tsattn_mla_decode with test-only flags (TSGEMM_DEBUG_SKIP_FIRST_LOAD: the
 * first pair's first CTA leaves its first key block unloaded), the limit of
 * every device wait in milliseconds (0: 1 s), and the number of key blocks
 * (64 keys each) the loader asks for in L2 ahead of the one it loads (0:
 * none; at most 64). */
TSGEMM_API tsgemm_status_t tsattn_mla_decode_ex(int64_t B, int64_t H, int64_t Skv, int32_t dim, int32_t pe_dim,
                                                tsgemm_dtype_t dtype, float scale, const void* Q,
                                                const void* Q_pe, const void* KV, const void* K_pe, void* O,
                                                int* status, void* stream, int32_t debug_flags, int32_t timeout_ms,
                                                int32_t prefetch_blocks);

/* The library's own status word of the current device (used when
 * tsattn_forward or tsattn_mla_decode is given status = NULL): TSGEMM_OK or
 * TSGEMM_ERR_TIMEOUT.  Reading it clears it.  Synchronise the stream
 * first. */
TSGEMM_API tsgemm_status_t tsattn_status(void);

#ifdef __cplusplus
}
#endif

#endif /* TSATTN_H */
