/*
 * gqa_prefill.h -- chunked causal prefill attention (libgqa_decode.so).
 *
 * A block of T new tokens per sequence on top of a KV cache that already holds the
 * sequence's earlier tokens ("ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)",
 * section 5.4, PREFILL with no sequence parallelism: the prompt is resident, the query is
 * a chunk of T_q tokens, and causality decides per (query block, KV tile) pair whether a
 * tile is wholly past, partial (triangular mask) or wholly future (skipped)).  Each chunk
 * token first gets the decode prologue -- per-head QK RMSNorm, then RoPE at its position,
 * k (post-RoPE) and v (raw) appended to the cache ("Qwen3-14B Optimization", section 2.1
 * Shape 4 and section 3.3) -- and then attends to every cached token and to the chunk's
 * tokens up to and including itself.  The G query heads of a KV head share one operand,
 * as in decode (section 5.4 "GQA batches the group's query heads along the same axis").
 *
 * Conventions are those of gqa_decode.h (bf16 as 16-bit storage, dense row-major device
 * tensors, bf16 tensors 16-byte aligned and int32 ones 4-byte aligned, asynchronous on
 * `stream`, argument errors before any launch, device-side index errors as GQA_DEVERR_*
 * bits).  The call allocates nothing and keeps no state between calls besides the
 * kernels' one-time shared-memory configuration per device.
 */
#ifndef GQA_PREFILL_H_
#define GQA_PREFILL_H_

#include "gqa_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Shapes and layout of one prefill call. */
typedef struct gqa_prefill_desc {
    int batch;            /* B sequences, 1..GQA_MAX_BATCH */
    int num_q_heads;      /* H_q */
    int num_kv_heads;     /* H_kv; H_q % H_kv == 0 and G = H_q / H_kv <= 16 */
    int head_dim;         /* d; must be 128 */
    int chunk_len;        /* T: new tokens per sequence, 1 <= T <= max_seq_len */
    int block_size;       /* 64: paged cache [num_cache_blocks, 64, H_kv, d] with a page table;
                             0: contiguous cache [B, max_seq_len, H_kv, d] */
    int max_seq_len;      /* per-sequence capacity in tokens; the page table has
                             ceil(max_seq_len / 64) entries per sequence */
    int num_cache_blocks; /* paged: 64-token blocks in each cache pool (>= 1); else ignored */
    int device;           /* CUDA device ordinal the call runs on */
} gqa_prefill_desc_t;

/*
 * gqa_prefill_attn -- one chunk of causal prefill: prologue, cache append, attention.
 *   desc       geometry (read during the call only)
 *   q_new      [B, T, H_q, d]  bf16 device   chunk queries (pre-norm, pre-RoPE)
 *   k_new      [B, T, H_kv, d] bf16 device   chunk keys (pre-norm, pre-RoPE)
 *   v_new      [B, T, H_kv, d] bf16 device   chunk values
 *   k_cache, v_cache           bf16 device   as in gqa_decode_attn; rows of positions
 *                                            s_b .. s_b + T - 1 are written (s_b = q_start[b])
 *   page_table [B, ceil(max_seq_len/64)] int32 device, or NULL when contiguous; every page
 *                                            the chunk writes must belong to its sequence alone
 *   q_start    [B] int32 device   s_b: position of the chunk's first token; the cache holds
 *                                 the sequence's tokens 0 .. s_b - 1 (0 <= s_b and
 *                                 s_b + T <= max_seq_len)
 *   q_norm_w, k_norm_w [d] bf16 device, or NULL for no QK-norm on q / on k
 *   rope_theta RoPE base (> 0); frequencies theta^(-2i/d), half-split pairs (i, i + d/2)
 *   eps        RMSNorm epsilon (>= 0)
 *   out        [B, T, H_q, d] bf16 device   out[b, i, h] = softmax over keys t <= s_b + i of
 *                                           q_rot[b, i, h] . K_t / sqrt(d), applied to V_t;
 *                                           query head h reads KV head h / G.  Between the
 *                                           call's two kernels `out` holds the rotated queries,
 *                                           so it must not alias any input.
 *   device_errors optional device pointer to a uint32 the kernels OR GQA_DEVERR_* bits into
 *                 (the caller owns and clears it); NULL discards them.  A chunk outside
 *                 [0, max_seq_len) (GQA_DEVERR_POSITION for s_b < 0, GQA_DEVERR_SEQLEN for
 *                 s_b + T > max_seq_len) appends nothing and gives zeros for its output; a
 *                 page id outside the pool appends nothing there and reads that page as zeros;
 *                 GQA_DEVERR_LAUNCH: the attention kernel's shared memory was not 1024-byte
 *                 aligned, and it did no work (not expected on any supported device).
 *   stream     cudaStream_t as void*
 * Launches two kernels (three when the last round of query tiles is cut into KV parts,
 * the third merging their partials) with programmatic stream serialization: the prologue kernel (one
 * CTA per chunk token) reads q/k/v_new, q_start and the page table before it waits for the
 * preceding kernel in the stream, and writes `out` and the cache only after; so the kernel
 * launched immediately before the call must not write those inputs if it triggers
 * programmatic completion early.  The attention kernel waits for the prologue kernel.
 * Errors: GQA_ERR_INVALID_ARG (NULL desc or tensor, page_table given for a contiguous cache
 * or missing for a paged one, misaligned tensor, bad sizes, rope_theta <= 0, eps < 0 or not
 * finite), GQA_ERR_UNSUPPORTED (head_dim != 128, H_q % H_kv != 0, G > 16, block_size other
 * than 0 or 64, more than 2^31 cache rows, (H_q + 2 H_kv) x 256 B above 200 KiB), GQA_ERR_CUDA
 * (set-up or launch failure).
 */
gqa_status_t gqa_prefill_attn(const gqa_prefill_desc_t *desc,
                              const void *q_new, const void *k_new, const void *v_new,
                              void *k_cache, void *v_cache, const int32_t *page_table,
                              const int32_t *q_start,
                              const void *q_norm_w, const void *k_norm_w,
                              float rope_theta, float eps, void *out,
                              uint32_t *device_errors, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GQA_PREFILL_H_ */
