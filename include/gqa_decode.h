/*
 * gqa_decode.h -- C ABI of the GB300 fused GQA decode-attention library (libgqa_decode.so).
 *
 * One decode step for one new token per sequence:
 *   1. prologue: per-head QK RMSNorm, then RoPE at the token's position, on q and k;
 *      k (post-RoPE) and v (raw) are appended to the bf16 KV cache at that position
 *      ("Qwen3-14B Optimization", section 2.1 Shape 4 and "Then: buy it" / #796, where
 *      QK-norm and RoPE are folded into the attention kernel; section 3.3 for the folded
 *      norm reciprocal and the lo/hi RoPE halves; "ADR-0060: AHBM GQA Fused Attention
 *      Kernel (Llama3-70B)", section 0.5.1 preconditions P2-P4: K cached post-RoPE,
 *      V raw, the new row seen by attention).
 *   2. split-KV attention: the G = H_q / H_kv query heads that share a KV head are
 *      stacked into one tile (ADR-0060 section 5.2, M-fold), the KV cache is streamed in
 *      64-token tiles with an online softmax (ADR-0060 section 3), and each split writes
 *      an unnormalised (m, l, O) partial (ADR-0060 sections 0.5.4 and 4).
 *   3. combine: the log-sum-exp merge of the partials, normalised once (ADR-0060
 *      section 4, merge()).
 * Steps 1 and 2 run in one kernel (the prologue folded into the attention kernel, as
 * the pages do).  The plan picks one of two forms for step 3 ("Qwen3-14B Optimization",
 * section 2.1 "Then: buy it": delete a boundary; ADR-0060 section 9 item 5: short
 * contexts are dominated by the reduce):
 *   - split-KV + combine: the batch's KV tiles are cut into one contiguous range per SM
 *     (ADR-0060 section 2.1) whatever the sequence boundaries, the partials go to the
 *     workspace and a second kernel merges them.  For batches with many (sequence, KV
 *     head) segments or long ones.
 *   - single launch: one thread-block cluster of C CTAs per (sequence, KV head); the C
 *     CTAs split its tiles, and their partials are merged on chip (shared memory, then
 *     distributed shared memory across the cluster), so the step is one kernel.  For
 *     batches whose segments fit the SMs C at a time with short to mid-length contexts.
 *
 * Conventions shared by every entry point
 *   - bf16 tensors are passed as pointers to 16-bit storage (IEEE bfloat16 bits).
 *   - Device pointers must be device-accessible on the plan's device; all device
 *     tensors are dense, row-major, with the shapes stated; bf16 tensors 16-byte aligned,
 *     int32 ones 4-byte aligned (else GQA_ERR_INVALID_ARG, before anything is launched).
 *   - The caller owns every tensor.  The library writes only `out` (or the host
 *     output buffer), the B new cache rows, and its own plan workspace.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL is the
 *     legacy default stream) and never synchronise, except the functions documented
 *     as synchronous.  Two calls that share a plan must not run concurrently (they
 *     share the plan's workspace); order them on one stream.
 *   - Kernels are launched with programmatic stream serialization: a kernel may start
 *     while the previous kernel on the stream drains.  The split-KV attention kernel reads
 *     its inputs (q/k/v_new, seq_lens, positions, page table, norm weights, the cache)
 *     before it waits (griddepcontrol.wait) on that kernel, and writes the workspace
 *     only after; the combine reads only seq_lens before it waits.  The single-launch
 *     kernel reads the same inputs before it waits, and writes the cache, the workspace
 *     and `out` only after; it lets the next kernel launch once its cache rows are
 *     appended (and fenced).  So the kernel launched immediately
 *     before a step must not write the step's inputs if it triggers programmatic
 *     completion early (kernels launched without programmatic dependent launch, the
 *     usual case, never do).  After a RoPE table rebuild the attention kernel is launched
 *     in plain stream order.
 *   - The first call with a given rope_theta (and the first after a different one)
 *     also launches, on the same stream, the build of the plan's RoPE tables:
 *     cos/sin(p * theta^(-2i/d)) for every p < max_seq_len in binary64 and rounded to
 *     binary32 (max_seq_len x 1.5 KiB).
 *     Make that first call before capturing the step in a CUDA graph.
 *   - Argument errors are reported before anything is launched.  Index errors that can
 *     only be seen on the device do not fault; the kernels set a bit in the plan's
 *     device error word (gqa_plan_device_errors) and contain the damage to the offending
 *     sequence: a seq_len outside [1, max_seq_len] gives zeros for its output; a position
 *     outside [0, seq_len) appends nothing and attends with a zero query; a page id
 *     outside the pool reads that page as zeros and appends nothing there.
 *
 * Supported geometry: head_dim == 128, H_q % H_kv == 0, 1 <= G <= 16, batch <= 1024,
 * paged cache with 64-token blocks or a contiguous per-sequence cache.
 */
#ifndef GQA_DECODE_H_
#define GQA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GQA_HEAD_DIM 128
#define GQA_BLOCK_SIZE 64
#define GQA_MAX_GROUP 16
#define GQA_MAX_BATCH 1024

typedef enum gqa_status {
    GQA_OK = 0,
    GQA_ERR_INVALID_ARG = 1,   /* a NULL pointer, a bad size, or an inconsistent argument */
    GQA_ERR_UNSUPPORTED = 2,   /* a geometry outside the supported set above */
    GQA_ERR_CUDA = 3,          /* a CUDA runtime call or a kernel launch failed */
    GQA_ERR_WORKSPACE = 4,     /* the plan's workspace could not be allocated */
    GQA_ERR_SCRATCH_LIMIT = 5  /* gqa_decode_attn_static: the geometry needs more workspace
                                  than the library's fixed scratch (GQA_STATIC_SCRATCH_BYTES) */
} gqa_status_t;

/* Bits of the device error word (gqa_plan_device_errors). */
#define GQA_DEVERR_POSITION 0x1u  /* positions[b] outside [0, seq_lens[b]) */
#define GQA_DEVERR_SEQLEN 0x2u    /* seq_lens[b] outside [1, max_seq_len] */
#define GQA_DEVERR_PAGE 0x4u      /* a page-table entry outside [0, num_cache_blocks) */
#define GQA_DEVERR_TIMEOUT 0x8u   /* a pipeline wait gave up (the kernel returned early) */
#define GQA_DEVERR_LAUNCH 0x10u   /* a launch assumption did not hold (the kernel did no work) */

/* Shapes and layout a plan is built for. */
typedef struct gqa_plan_desc {
    int batch;            /* B, 1..GQA_MAX_BATCH */
    int num_q_heads;      /* H_q */
    int num_kv_heads;     /* H_kv; H_q % H_kv == 0 and G = H_q / H_kv <= 16 */
    int head_dim;         /* d; must be 128 */
    int block_size;       /* 64: paged cache [num_cache_blocks, 64, H_kv, d] with a page table;
                             0: contiguous cache [B, max_seq_len, H_kv, d], no page table */
    int max_seq_len;      /* per-sequence capacity in tokens (>= 1); the page table has
                             ceil(max_seq_len / 64) entries per sequence */
    int num_cache_blocks; /* paged: number of 64-token blocks in each cache pool (>= 1);
                             ignored (may be 0) when contiguous */
    int num_workers;      /* CTAs of the split-KV kernel; 0 lets the planner choose */
    int device;           /* CUDA device ordinal the plan and its calls run on */
    int cluster_size;     /* the step's form: 0 lets the planner choose; -1 asks for the
                             split-KV kernel + combine; 1 .. 16 asks for the single-launch
                             form with that many CTAs per (sequence, KV head) cluster
                             (GQA_ERR_UNSUPPORTED if the device cannot launch it).  A
                             non-zero num_workers with cluster_size 0 also means split-KV. */
    int ordered_start;    /* 0: a step's first kernel may start while the kernel before it
                             on the stream drains, so consecutive steps overlap; non-zero:
                             it is launched in plain stream order (the initial setting of
                             gqa_plan_set_ordered_start, which see).  The planner sizes the
                             clusters for the setting. */
} gqa_plan_desc_t;

typedef struct gqa_plan gqa_plan_t; /* opaque; owns the workspace (rotated q, fp32 partials) */

/*
 * gqa_plan_create -- the split planner.  Validates the geometry, chooses the step's form
 * and its splits (ADR-0060 sections 5.3 and 9 item 5: short contexts want few splits,
 * long contexts many) and allocates the workspace once, so no call allocates.
 *   - The single-launch form, for up to two waves of segments (B * H_kv <= 2 x SMs).
 *     Its cluster size C (2 .. 16, at most the longest segment's tile count,
 *     B * H_kv * C <= SMs; else C = 1) is the largest for which the device holds at once
 *     the clusters of: with overlapping steps (ordered_start 0) and short segments (a CTA
 *     streams at most two rings of tiles), two consecutive steps (2 B * H_kv clusters), so
 *     that the next step's CTAs start as this one finishes; with overlapping steps and long
 *     segments, one and a half steps, else one; with ordered starts (a step runs alone),
 *     one step, the most CTAs streaming.  Provided the B * H_kv * C CTAs can stream the
 *     cache (at least 48 of them, or one per tile).
 *   - Otherwise split-KV + combine: the whole batch's T KV tiles are cut into one
 *     contiguous range per worker (ADR-0060 section 2.1 contiguous-block placement); the
 *     fewest workers that keep the longest range at ceil(T / SMs) tiles.
 * gqa_plan_describe gives these choices for any device description, without a GPU.
 * The scope table's scalar form gqa_plan_create(batch, num_q_heads, num_kv_heads,
 * head_dim, block_size, max_seq_len, seq_lens_host, device, &plan) is this call with those
 * fields in `desc` (plus the cache pool size, which the tensor maps need, and the two
 * overrides); its gqa_plan_num_splits is declared below.  The workspace holds a copy of the rotated
 * queries, the fp32 (m, l, O) partials ((B*H_kv + workers) * 6 * G rows of 130 floats),
 * the RoPE tables (max_seq_len x 1.5 KiB), the first tiles each worker streamed at the
 * last call (contiguous caches: prefetched into L2 at the start of the next call) and
 * staging buffers for gqa_decode_attn_host.
 *   desc          : geometry (copied).
 *   seq_lens_host : optional host array [B] of expected lengths, used to choose the form,
 *                   the worker count and the cluster size, and to order the segments
 *                   longest first when the clusters come in more than one wave; NULL
 *                   plans for B sequences of max_seq_len tokens.  Other lengths at call
 *                   time are computed correctly, only possibly with a worse choice.
 *   plan          : receives the new plan.
 * Errors: GQA_ERR_INVALID_ARG, GQA_ERR_UNSUPPORTED, GQA_ERR_CUDA, GQA_ERR_WORKSPACE.
 * Synchronous (allocates device memory).
 */
gqa_status_t gqa_plan_create(const gqa_plan_desc_t *desc, const int32_t *seq_lens_host,
                             gqa_plan_t **plan);

/*
 * gqa_plan_describe -- the planner's choices for a geometry on a described device, with
 * no device work (for tests and tooling): the split-KV worker count, the step's form
 * (cluster size, 0 for split-KV + combine) and the splits of the longest segment, as
 * gqa_plan_create would make them.
 *   desc, seq_lens_host : as for gqa_plan_create (desc->device is not used).
 *   num_sms             : the device's SM count (>= 1).
 *   cluster_capacity    : [16] how many clusters of 1, 2, ..., 16 single-launch CTAs the
 *                         device holds at once (0: that size cannot be launched).
 *   num_workers, cluster_size, num_splits : outputs; any may be NULL.
 * Errors: those of gqa_plan_create's validation; GQA_ERR_UNSUPPORTED when a forced
 * cluster size has capacity 0.
 */
gqa_status_t gqa_plan_describe(const gqa_plan_desc_t *desc, const int32_t *seq_lens_host,
                               int num_sms, const int *cluster_capacity, int *num_workers,
                               int *cluster_size, int *num_splits);

/*
 * gqa_plan_set_ordered_start -- with `ordered` non-zero, the first kernel of each step on
 * this plan (gqa_decode_attn, gqa_decode_attn_host, gqa_attention_splitkv,
 * gqa_decode_attn_q4) is launched in plain stream order: it starts only once the kernel
 * before it on the stream has completed and its writes are visible, and so may follow a
 * caller kernel that triggers programmatic completion early while writing the step's
 * inputs (the precondition above).  The kernels within a step keep their programmatic
 * dependent launches; consecutive steps no longer overlap, so the plan switches to the
 * cluster size the planner takes for a step that runs alone (unless the plan was created
 * with an explicit cluster_size or num_workers).  0 restores the overlapped start and its
 * cluster size.  Returns GQA_ERR_INVALID_ARG for a NULL plan.  Not synchronised with calls
 * in flight: set it between steps.
 */
gqa_status_t gqa_plan_set_ordered_start(gqa_plan_t *plan, int ordered);

/* Frees the plan and its workspace (synchronous). NULL is accepted. */
gqa_status_t gqa_plan_destroy(gqa_plan_t *plan);

/* Number of split-KV workers (CTAs) of the plan's split-KV kernel (the split-KV form, and
 * gqa_attention_splitkv in either form); 0 for a NULL plan. */
int gqa_plan_num_workers(const gqa_plan_t *plan);

/* Number of KV splits of the longest (sequence, KV head) segment as planned: the cluster
 * size in the single-launch form (at most the segment's tile count), else the number of
 * split-KV workers whose ranges cover that segment.  0 for a NULL plan. */
int gqa_plan_num_splits(const gqa_plan_t *plan);

/* The step's form: the cluster size C of the single-launch form, or 0 for split-KV +
 * combine; 0 for a NULL plan. */
int gqa_plan_cluster_size(const gqa_plan_t *plan);

/* Bytes of device workspace the plan owns; 0 for a NULL plan. */
size_t gqa_plan_workspace_bytes(const gqa_plan_t *plan);

/*
 * gqa_decode_attn -- the whole decode step: prologue, split-KV attention, combine.
 *   q_new      [B, H_q, d]  bf16 device   new-token queries (pre-norm, pre-RoPE)
 *   k_new      [B, H_kv, d] bf16 device   new-token keys (pre-norm, pre-RoPE)
 *   v_new      [B, H_kv, d] bf16 device   new-token values
 *   k_cache, v_cache        bf16 device   paged [num_cache_blocks, 64, H_kv, d] or
 *                                         contiguous [B, max_seq_len, H_kv, d]; the row for
 *                                         token t of sequence b is
 *                                         page_table[b][t / 64] * 64 + t % 64 (paged) or
 *                                         b * max_seq_len + t (contiguous).  Modified in
 *                                         place at token positions[b] only.
 *   page_table [B, ceil(max_seq_len/64)] int32 device, or NULL when contiguous
 *   seq_lens   [B] int32 device   L_b = tokens to attend to, including the new one
 *   positions  [B] int32 device   p_b = RoPE position and cache slot of the new token,
 *                                 0 <= p_b < L_b (a decode step has p_b = L_b - 1)
 *   q_norm_w, k_norm_w [d] bf16 device, or NULL for no QK-norm on q / on k
 *   rope_theta RoPE base (> 0); frequencies theta^(-2i/d), half-split pairs (i, i + d/2)
 *   eps        RMSNorm epsilon (>= 0)
 *   out        [B, H_q, d] bf16 device   softmax(q k^T / sqrt(d)) v per query head,
 *                                        query head h reading KV head h / G
 *   stream     cudaStream_t as void*
 * Errors: GQA_ERR_INVALID_ARG (NULL plan or tensor, page_table given for a contiguous
 * plan or missing for a paged one, rope_theta <= 0, eps < 0 or not finite),
 * GQA_ERR_CUDA (launch failure).
 */
gqa_status_t gqa_decode_attn(const gqa_plan_t *plan,
                             const void *q_new, const void *k_new, const void *v_new,
                             void *k_cache, void *v_cache, const int32_t *page_table,
                             const int32_t *seq_lens, const int32_t *positions,
                             const void *q_norm_w, const void *k_norm_w,
                             float rope_theta, float eps, void *out, void *stream);

/*
 * gqa_decode_attn_host -- the same step with the per-step inputs and the output in host
 * memory: q_new, k_new, v_new, seq_lens, positions are read from host buffers and `out`
 * is written to a host buffer.  When all six are page-locked (cudaHostAlloc /
 * cudaHostRegister; mapped into the device's address space) and 16-byte aligned, the
 * kernels read and write them in place over the host link (NVLink-C2C on Grace-Blackwell)
 * with no copies; otherwise each goes through one cudaMemcpyAsync on `stream` into or out
 * of the plan's staging area.  The KV caches, the page table and the norm weights stay
 * device-resident (model state).  Shapes as for gqa_decode_attn.  The host buffers must
 * stay unchanged, and the output is valid, only once `stream` has been synchronised.
 * Errors as for gqa_decode_attn.
 */
gqa_status_t gqa_decode_attn_host(const gqa_plan_t *plan,
                                  const void *q_new_host, const void *k_new_host,
                                  const void *v_new_host,
                                  void *k_cache, void *v_cache, const int32_t *page_table,
                                  const int32_t *seq_lens_host, const int32_t *positions_host,
                                  const void *q_norm_w, const void *k_norm_w,
                                  float rope_theta, float eps, void *out_host, void *stream);

/*
 * The two launches of the split-KV form of gqa_decode_attn, separately, for callers that
 * schedule them themselves (and for step-level tests and timing); they run the split-KV
 * form (the plan's worker count) whichever form gqa_decode_attn takes.  They communicate
 * through the plan's workspace and must be issued in this order on one stream; arguments
 * are those of gqa_decode_attn, and so are the errors.
 *   gqa_attention_splitkv: the prologue and the split-KV attention in one kernel.  Its
 *     consumer warps apply QK-norm + RoPE to the new queries (into registers, with a copy
 *     to the workspace), append the new k (QK-norm + RoPE) and v rows to the cache, and
 *     run the split-KV attention over the cache, writing fp32 partials.  It reads its
 *     inputs and streams KV tiles before the preceding kernel in the stream has finished
 *     (it waits for that kernel only before writing the workspace's partials), so the
 *     inputs must not be written by an immediately preceding kernel that triggers
 *     programmatic completion early; the page holding a sequence's new token must belong
 *     to that sequence alone.
 *   gqa_combine: merges the partials into `out`.
 */
gqa_status_t gqa_attention_splitkv(const gqa_plan_t *plan, const void *q_new,
                                   const void *k_new, const void *v_new,
                                   void *k_cache, void *v_cache, const int32_t *page_table,
                                   const int32_t *seq_lens, const int32_t *positions,
                                   const void *q_norm_w, const void *k_norm_w,
                                   float rope_theta, float eps, void *stream);
gqa_status_t gqa_combine(const gqa_plan_t *plan, const int32_t *seq_lens, void *out,
                         void *stream);

/*
 * gqa_plan_read_q_rot -- copies the rotated, bf16-rounded queries of the last step out of
 * the workspace into host memory as [B, H_q, d] bf16 (rows of sequences with an invalid
 * length or position are left as they were).  Synchronous (waits for the device).  For
 * tests and debugging.
 */
gqa_status_t gqa_plan_read_q_rot(const gqa_plan_t *plan, uint16_t *q_rot_host);

/*
 * gqa_plan_device_errors -- reads the plan's device error word (GQA_DEVERR_* bits set by
 * any call since the last clear) into *flags, and clears it when `clear` is non-zero.
 * Synchronous: waits for all work on the plan's device.
 */
gqa_status_t gqa_plan_device_errors(const gqa_plan_t *plan, uint32_t *flags, int clear);

/*
 * gqa_partition_describe -- host-side view of how the split-KV kernel cuts a batch into
 * worker ranges (for tests and tooling; no device work).  Given B lengths, H_kv and the
 * worker count W, writes for every worker w its half-open range of global tile indices
 * [worker_range[2w], worker_range[2w+1]), where tiles are numbered sequence-major, then
 * KV head, then 64-token tile.  Returns the total number of tiles, or -1 on bad input.
 */
long long gqa_partition_describe(const int32_t *seq_lens_host, int batch, int num_kv_heads,
                                 int max_seq_len, int num_workers, long long *worker_range);

/*
 * gqa_decode_attn_static -- the decode step of gqa_decode_attn without a plan and without
 * allocating anything.  The source pages define no such call: it exists for callers that
 * may not allocate device memory at the point of the step -- a serving loop that has
 * handed all free HBM to its own KV pool, a runtime that forbids a library from owning
 * device memory, or a step that must not take the allocator's implicit synchronisation.
 *
 * The workspace (RoPE tables, rotated queries, fp32 partials) lives in one
 * array of GQA_STATIC_SCRATCH_BYTES (32 MiB) of static device memory inside the library,
 * one copy per device, which exists for as long as the library is loaded.  Its layout is
 * that of a plan's workspace without the host staging buffers:
 *   max_seq_len * 1.5 KiB                       RoPE tables (binary64 and binary32, first)
 * + B * H_q * 256 B                             rotated queries
 * + (B * H_kv + W) * 6 * G * 520 B              fp32 (m, l, O) partials
 * each rounded up to 256 bytes, plus 256; W = desc->num_workers, or when 0 the planner's
 * count (as gqa_plan_create) for B * H_kv * ceil(max_seq_len / 64) tiles.  A geometry that needs more is rejected
 * with GQA_ERR_SCRATCH_LIMIT before anything is launched; use a plan for it.  (For example
 * B = 32, H_q = 40, H_kv = 8, max_seq_len = 8192 needs about 18 MiB; max_seq_len = 131072
 * does not fit whatever the batch.)
 *
 *   desc       the geometry, as for gqa_plan_create (desc->device is the device the call
 *              runs on); it is read during the call only.
 *   q_new ... out, stream    as for gqa_decode_attn.
 *   device_errors            optional device pointer to a uint32 the kernels OR the
 *              GQA_DEVERR_* bits into; the caller owns it and clears it.  NULL sends them
 *              to a word in the scratch that nothing reads.
 *
 * Set-up: the first call on a device (per process) looks up the scratch array's device
 * address (cudaGetSymbolAddress, with that device current), which may load the library's
 * device code, and raises the kernels' shared-memory limits.  Make that first call before
 * any stream capture, e.g. once at start-up.  Each call with a rope_theta or a max_seq_len
 * other than the last call's on the device first rebuilds the RoPE tables in the scratch
 * on `stream` (max_seq_len x 1.5 KiB of writes).
 *
 * Sharing: every call on a device uses the same scratch.  Nothing in it has to start at
 * zero (each region is written by the call before it is read), but calls that overlap on
 * the device -- on different streams, or from threads that do not order their streams --
 * race on it and give wrong results.  Order all calls of a device on one stream (or
 * through events).  Host-side bookkeeping is guarded by a mutex.
 *
 * Errors: those of gqa_plan_create (GQA_ERR_INVALID_ARG, GQA_ERR_UNSUPPORTED) and of
 * gqa_decode_attn, GQA_ERR_SCRATCH_LIMIT, and GQA_ERR_CUDA when the set-up fails.
 */
#define GQA_STATIC_SCRATCH_BYTES (32u << 20)
gqa_status_t gqa_decode_attn_static(const gqa_plan_desc_t *desc,
                                    const void *q_new, const void *k_new, const void *v_new,
                                    void *k_cache, void *v_cache, const int32_t *page_table,
                                    const int32_t *seq_lens, const int32_t *positions,
                                    const void *q_norm_w, const void *k_norm_w,
                                    float rope_theta, float eps, void *out,
                                    uint32_t *device_errors, void *stream);

/* Static description of a status code. */
const char *gqa_status_string(gqa_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* GQA_DECODE_H_ */
