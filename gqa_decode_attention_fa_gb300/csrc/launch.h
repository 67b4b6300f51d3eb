// Internal launchers shared by the kernel files and the C-ABI layer (not part of the ABI).
#pragma once

#include <utility>

#include "gqa_common.cuh"
#include "../../include/gqa_prefill.h"
#include "../../include/gqa_q4.h"

namespace gqa {

cudaError_t launch_rope_table(const RopeTableParams &p, cudaStream_t stream);

// Launches `kernel`, with programmatic stream serialization when `pdl` is set (it may
// begin while the previous kernel in the stream finishes; the kernels order themselves
// with griddepcontrol.wait), else in plain stream order.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                      Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
  return launch_ex(true, kernel, grid, block, smem, stream, std::forward<Args>(args)...);
}

// Dynamic shared memory the split-KV kernel needs for a group padded to npad rows.
size_t attn_smem_bytes(int npad, int batch);
// Raises the kernel's dynamic shared-memory limit on the current device to what a launch
// of the largest supported batch needs.  The limit is per function, not per plan, so it
// never depends on one plan's batch: a plan made later for a smaller batch must not lower
// it under an earlier plan's launches.
cudaError_t attn_configure(int npad);
// The split-KV attention kernel.  It reads the caller's inputs and the RoPE table before
// waiting on the preceding kernel, so it is launched in plain stream order (`pdl` false)
// when the preceding kernel may write any of them (a RoPE table rebuild).
cudaError_t launch_attention(const CUtensorMap &tmK, const CUtensorMap &tmV, const AttnParams &p, int npad,
                             int num_workers, bool pdl, cudaStream_t stream);
// The single-launch form of the step: B * H_kv clusters of p.csize CTAs, writing p.out.
cudaError_t launch_attention_cluster(const CUtensorMap &tmK, const CUtensorMap &tmV, const AttnParams &p, int npad,
                                     bool pdl, cudaStream_t stream);
// How many clusters of `csize` CTAs of the single-launch kernel can be resident at once
// on the current device (0: that cluster size cannot be launched).  attn_configure(npad)
// must have run on the device first.
int attn_cluster_capacity(int npad, int csize);
// The step's form: the cluster size of the single-launch form, or 0 for split-KV +
// combine.  `forced` is the caller's choice (gqa_plan_desc_t.cluster_size: 0 lets this
// planner choose, -1 asks for split-KV + combine, else that cluster size); capacity[c - 1]
// is how many clusters of c CTAs the device holds at once (c = 1 .. 16); max_seg_tiles is the tile count
// of the longest (sequence, KV head) segment; `ordered`: consecutive steps do not overlap
// (gqa_plan_desc_t.ordered_start).  Returns -1 when a forced cluster size cannot be
// launched.
int plan_step_form(int forced, int num_workers, int num_sms, const int *capacity, long long num_segments,
                   long long max_seg_tiles, long long total_tiles, bool ordered);

// The combine: split 0 runs one CTA per (sequence, KV head) segment, split 4, 2 or 1 that
// many CTAs per query head; combine_split picks it from the geometry and worker count.
int combine_split(int batch, int num_q_heads, int num_kv_heads, int num_workers, int num_sms);
cudaError_t launch_combine(const CombineParams &p, int split, cudaStream_t stream);

// Tiled bf16 tensor map with 128-byte swizzling over `rank` dimensions (innermost first;
// `strides` in bytes for dimensions 1..rank-1), no interleave, zero fill out of bounds.
bool encode_bf16_map(CUtensorMap *m, int rank, const void *base, const cuuint64_t *dims, const cuuint64_t *strides,
                     const cuuint32_t *box);
// K or V cache viewed as [rows][H_kv][128] bf16; box = 64 dims x 1 head x 64 tokens.
bool make_cache_map(CUtensorMap *m, const void *base, int Hkv, long long rows);

// The decode step over a 4-bit KV cache (attention_q4.cu; include/gqa_q4.h).
struct Q4PrologueParams {
  const int32_t *seq_lens, *positions, *page_table;
  const uint16_t *q_new, *k_new, *v_new;    // [B,Hq,d], [B,Hkv,d], [B,Hkv,d]
  const uint16_t *q_norm_w, *k_norm_w;      // [d] or null
  const float2 *rope_tab32;                 // [max_seq][64] (cos, sin), binary32
  const int8_t *signs;                      // [d] +-1
  const uint16_t *codebook;                 // [16] bf16 levels, ascending
  uint16_t *q_hi, *q_lo;                    // [B,Hq,d] rotated queries, bf16 hi + lo
  uint8_t *k_idx, *v_idx;                   // [rows,Hkv,d/2] packed indices
  float *k_scale, *v_scale;                 // [rows,Hkv]
  uint32_t *err;
  int B, Hq, Hkv, paged, max_seq, max_blocks, num_blocks;
  float eps;
};
struct Q4AttnParams {
  const int32_t *seq_lens, *page_table;
  const uint16_t *q_hi, *q_lo;
  const float *k_scale, *v_scale;
  const uint16_t *codebook;
  float *part_o, *part_ml;
  uint32_t *err;
  int B, Hq, Hkv, G, paged, max_seq, max_blocks, num_blocks;
  float scale_log2;
};
// The single-launch form of the 4-bit step (attention_q4.cu): prologue, attention and the
// merge with unrotation in one kernel, a cluster of csize CTAs per (sequence, KV head).
struct Q4ClusterParams {
  const int32_t *seq_lens, *positions, *page_table;
  const uint16_t *q_new, *k_new, *v_new;    // [B,Hq,d], [B,Hkv,d], [B,Hkv,d]
  const uint16_t *q_norm_w, *k_norm_w;      // [d] or null
  const float2 *rope_tab32;                 // [max_seq][64] (cos, sin), binary32
  const int8_t *signs;                      // [d] +-1
  const uint16_t *codebook;                 // [16] bf16 levels, ascending
  uint8_t *k_idx, *v_idx;                   // [rows,Hkv,d/2] packed indices
  float *k_scale, *v_scale;                 // [rows,Hkv]
  uint16_t *out;                            // [B,Hq,d]
  uint32_t *err;
  int B, Hq, Hkv, G, paged, max_seq, max_blocks, num_blocks, csize;
  float eps, scale_log2;
  const int32_t *seg_order;                 // cluster i streams segment seg_order[i], or i when null
};
cudaError_t q4_configure();
cudaError_t launch_q4_cluster(const CUtensorMap &tmK, const CUtensorMap &tmV, const Q4ClusterParams &p, int npad,
                              bool pdl, cudaStream_t stream);
// The 4-bit step's prologue reads the caller's inputs and the RoPE table before it waits on
// the preceding kernel, so it is launched in plain stream order (`pdl` false) after a
// RoPE table rebuild.
cudaError_t launch_q4_prologue(const Q4PrologueParams &p, bool pdl, cudaStream_t stream);
cudaError_t launch_q4_attention(const CUtensorMap &tmK, const CUtensorMap &tmV, const Q4AttnParams &p, int npad,
                                int num_workers, cudaStream_t stream);
cudaError_t launch_q4_combine(const CombineParams &p, const int8_t *signs, cudaStream_t stream);
// Tiled uint8 tensor map over `rank` dimensions, no swizzle (see encode_bf16_map).
bool encode_u8_map(CUtensorMap *m, int rank, const void *base, const cuuint64_t *dims, const cuuint64_t *strides,
                   const cuuint32_t *box);

// Runs the calling thread on `dev` for the guard's lifetime.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
      ok = false;
      prev = -1;
      return;
    }
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

// Workspace of one decode step run without a plan: byte offsets of its regions from a
// 256-byte-aligned base.  The RoPE table comes first, so that its place does not depend on
// the batch geometry and a table built by one call stays usable by the next.
struct StepLayout {
  int G = 0, npad = 0, W = 0, max_blocks = 0, combine_split = 1, csize = 0, spec_tiles = 0;
  long long num_rows = 0;
  size_t tab_bytes = 0, off_q = 0, off_o = 0, off_ml = 0, off_err = 0, total = 0;
};

// Checks `d` as gqa_plan_create does (except the device index) and lays out its workspace;
// the worker count is d.num_workers, else one per SM up to B * H_kv * ceil(max_seq/64),
// and the step's form is planned for B sequences of max_seq_len tokens.  Needs the
// device current and attn_configure run on it.
gqa_status_t step_layout(const gqa_plan_desc_t &d, int num_sms, StepLayout *lay);

// One decode step (split-KV attention with the prologue folded in -> combine) on the
// workspace at `base`, laid out by `lay`, on the current device.  `err` is the device
// error word the kernels OR into; `table_ready` says the table at `base` already holds
// cos/sin for rope_theta at every position below d.max_seq_len (else the call rebuilds it
// first).
gqa_status_t run_step_at(const gqa_plan_desc_t &d, const StepLayout &lay, void *base, uint32_t *err,
                         bool table_ready, const void *q, const void *k, const void *v, void *kc, void *vc,
                         const int32_t *pt, const int32_t *sl, const int32_t *pos, const void *qw, const void *kw,
                         float theta, float eps, void *out, cudaStream_t stream);

// Gives the combine and table kernels the attention kernel's shared-memory
// carveout, so that consecutive kernels of a step never make an SM switch configuration.
cudaError_t configure_small_kernels();

}  // namespace gqa
