/*
 * gqa_q4.h -- the decode step over a 4-bit KV cache (libgqa_decode.so).
 *
 * The cache format of "Qwen3-14B Optimization", section 2.3 (TurboQuant): each cache row
 * (one token, one KV head, d = 128) holds 4-bit Lloyd-Max codebook indices, two per byte --
 * byte c holds idx[c + 64] * 16 + idx[c] -- and is dequantized by gather -> renormalize ->
 * scale -> unrotate.  The page gives neither the codebook, the rotation nor the scale
 * format; this library reads them as:
 *   codebook  16 bf16 levels, ascending (the caller's; gqa_q4_codebook gives the Lloyd-Max
 *             levels of a standard normal variable, Lloyd's algorithm / Max 1960);
 *   rotation  R = H D / sqrt(d): the Sylvester Walsh-Hadamard matrix H times a diagonal of
 *             the caller's +-1 signs D;
 *   scale     one fp32 per row: sigma = ||x|| / ||c[idx]||, so that the row dequantizes to
 *             x^ = sigma R^T c[idx];
 *   quantize  t = sqrt(d) R x / ||x||, idx_i = the level nearest to t_i (the lower one on a
 *             tie, i.e. idx_i = the number of midpoints between consecutive levels below
 *             t_i); a zero row gets sigma = 0.
 * The step is gqa_decode_attn's with the cache in this format: the new token's k row
 * (post QK-norm and RoPE) and v row are quantized and appended; attention reads the
 * dequantized rows.  Conventions (layouts, ownership, asynchrony, device error word) are
 * gqa_decode.h's; the plan is a gqa_plan_create plan of the same geometry.
 */
#ifndef GQA_Q4_H_
#define GQA_Q4_H_

#include "gqa_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

/* The 16 Lloyd-Max reconstruction levels of N(0, 1), ascending, rounded to bf16 (host,
 * synchronous, no device work).  Returns GQA_ERR_INVALID_ARG for a NULL pointer. */
gqa_status_t gqa_q4_codebook(uint16_t *levels_bf16);

/*
 * gqa_decode_attn_q4 -- the decode step over a 4-bit cache.
 *   plan                    a plan of this geometry (its workspace holds the rotated queries
 *                           and the partials)
 *   q_new, k_new, v_new     as gqa_decode_attn (bf16 device)
 *   k_idx, v_idx            uint8 device [rows, H_kv, 64] packed indices, rows as for the bf16
 *                           cache (num_cache_blocks * 64 paged, B * max_seq_len contiguous);
 *                           row positions[b] of sequence b is written
 *   k_scale, v_scale        float device [rows, H_kv] sigma of each row; written likewise
 *   page_table, seq_lens, positions, q_norm_w, k_norm_w, rope_theta, eps   as gqa_decode_attn
 *   rot_signs               int8 device [128], each +1 or -1 (the diagonal D of R)
 *   codebook                bf16 device [16] levels, ascending
 *   out                     bf16 device [B, H_q, 128]
 * The plan's form decides the launches (gqa_plan_cluster_size): in the single-launch form
 * one kernel per step (a cluster per (sequence, KV head); the rotated queries and the new
 * rows computed in it, the partials merged and rotated back on chip; the new rows, and
 * `out`, written only after the preceding kernel has completed); in the split-KV form three
 * (prologue: rotated queries and the appended rows; split-KV attention on the index tiles;
 * combine and unrotation).  Programmatic stream serialization as for gqa_decode_attn: the
 * first kernel reads its inputs and the RoPE table before it waits on the preceding
 * kernel (the split form's prologue also writes the rotated queries and the new rows, and
 * waits at its end), so the same rule holds -- the kernel launched immediately before the
 * call must not write the call's inputs if it triggers programmatic completion early;
 * after a RoPE table rebuild the first kernel is launched in plain stream order.  Errors: those of gqa_decode_attn; k_idx, v_idx 16-byte aligned,
 * scales and signs 4-byte aligned, else GQA_ERR_INVALID_ARG.
 */
gqa_status_t gqa_decode_attn_q4(const gqa_plan_t *plan,
                                const void *q_new, const void *k_new, const void *v_new,
                                uint8_t *k_idx, uint8_t *v_idx, float *k_scale, float *v_scale,
                                const int32_t *page_table, const int32_t *seq_lens,
                                const int32_t *positions, const void *q_norm_w, const void *k_norm_w,
                                const int8_t *rot_signs, const void *codebook,
                                float rope_theta, float eps, void *out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GQA_Q4_H_ */
