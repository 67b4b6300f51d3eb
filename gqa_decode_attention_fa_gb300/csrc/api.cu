// C ABI of libgqa_decode.so: plan (split planner + workspace), argument validation, tensor
// maps and the launch sequence split-KV attention (with the prologue folded in) -> combine.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <vector>
#include <cmath>
#include <mutex>
#include <new>

#include "launch.h"

using namespace gqa;

struct gqa_plan {
  gqa_plan_desc_t desc;
  int G = 0, npad = 0, W = 0, num_sms = 0, max_blocks = 0, combine_split = 1;
  int csize = 0;   // single-launch form: CTAs per (sequence, KV head) cluster; 0: split-KV + combine
  int spec_tiles = 0;  // tiles of the longest segment as planned
  // launch the first kernel of a step in plain stream order (it then starts only once the
  // preceding kernel has completed), for callers whose preceding kernels trigger early
  bool ordered_first = false;
  // the planner's form and splits for overlapping [0] and ordered [1] starts, and whether
  // the single-launch clusters then outnumber what the device holds at once
  int csize_by_start[2] = {0, 0}, nsplit_by_start[2] = {0, 0};
  bool waves_by_start[2] = {false, false};
  int32_t *seg_order = nullptr;  // [B H_kv] segments by planned tile count, longest first
  int nsplit = 0;  // KV splits of the longest (sequence, KV head) segment
  long long num_rows = 0;
  void *ws = nullptr;
  size_t ws_bytes = 0;
  uint16_t *q_rot = nullptr;
  uint16_t *q4_hi = nullptr, *q4_lo = nullptr;  // rotated queries of the 4-bit-cache step
  float *part_o = nullptr, *part_ml = nullptr;
  uint32_t *err = nullptr;
  int2 *spec = nullptr;  // [W][kStages] first tiles of each worker at the previous launch
  uint16_t *st_q = nullptr, *st_k = nullptr, *st_v = nullptr, *st_out = nullptr;
  int32_t *st_sl = nullptr, *st_pos = nullptr;
  // [max_seq_len][64] double-word (cos_hi, sin_hi, cos_lo, sin_lo) for tab_theta, followed
  // by the same rounded to binary32 ([max_seq_len][64] float2)
  float4 *rope_tab = nullptr;
  mutable bool tab_valid = false;
  mutable float tab_theta = 0.f;
  // tensor maps of the cache pairs seen, most recent kMapCache of them (a model's layers
  // each bring their own pair; encoding one is a driver call on every step otherwise)
  static constexpr int kMapCache = 128;
  struct CacheMaps {
    const void *k = nullptr, *v = nullptr;
    CUtensorMap tk, tv;
  };
  mutable std::mutex tm_mu;
  mutable CacheMaps tm[kMapCache];
  mutable int tm_next = 0, tm_last = 0;
};

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

}  // namespace

bool gqa::encode_bf16_map(CUtensorMap *m, int rank, const void *base, const cuuint64_t *dims,
                          const cuuint64_t *strides, const cuuint32_t *box) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || rank < 1 || rank > 5) return false;
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void *>(base), dims,
             strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool gqa::encode_u8_map(CUtensorMap *m, int rank, const void *base, const cuuint64_t *dims,
                        const cuuint64_t *strides, const cuuint32_t *box) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || rank < 1 || rank > 5) return false;
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<cuuint32_t>(rank), const_cast<void *>(base), dims, strides,
             box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The box is 64 dims (128 B, the 128-byte swizzle span) x 1 head x 64 tokens.
bool gqa::make_cache_map(CUtensorMap *m, const void *base, int Hkv, long long rows) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(Hkv),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2, static_cast<cuuint64_t>(Hkv) * kHeadDim * 2};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kTile)};
  return encode_bf16_map(m, 3, base, dims, strides, box);
}

namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Bytes of the two RoPE tables of a max_seq-token capacity.
size_t rope_tables_bytes(int max_seq) {
  return align256(static_cast<size_t>(max_seq) * (kHeadDim / 2) * (sizeof(float4) + sizeof(float2)));
}
const float2 *rope_tab32_of(const gqa_plan_t *plan) {
  return reinterpret_cast<const float2 *>(plan->rope_tab + static_cast<size_t>(plan->desc.max_seq_len) * 64);
}

// The split-KV form's worker count.  A worker streams its tiles at a rate that does not
// grow with fewer workers once the SMs are all busy, so the step takes about as long as
// the longest worker's range: use the fewest workers that keep the longest range at its
// minimum, ceil(T / SMs) tiles -- fewer workers also mean fewer partials to combine.
// Measured on one 4096-token sequence of 8 KV heads (512 tiles, four a worker at most):
// 128 workers 8.0 us a step, 152 workers 8.8 us (more partials, the same longest range).
int plan_workers(int num_sms, long long total_tiles) {
  if (total_tiles < 1) return 1;
  const long long per = (total_tiles + num_sms - 1) / num_sms;  // the longest range's minimum
  return static_cast<int>((total_tiles + per - 1) / per);
}

}  // namespace

int gqa::plan_step_form(int forced, int num_workers, int num_sms, const int *capacity, long long nseg,
                        long long max_seg_tiles, long long total_tiles, bool ordered) {
  auto cap = [&](int c) { return capacity[c - 1]; };
  if (forced < 0) return 0;
  if (forced > 0) return cap(forced) >= 1 ? forced : -1;
  if (num_workers > 0) return 0;           // an explicit worker count asks for the split-KV form
  if (nseg > 2LL * num_sms) return 0;      // more than two waves of one-CTA segments
  // The largest cluster size (a tile for every CTA, at most one CTA per SM) whose clusters
  // the device holds at once for `need2` steps' worth of segments (need2 / 2 steps), or 1.
  auto largest = [&](long long need2) {
    for (int c = 16; c >= 2; --c)
      if (c <= max_seg_tiles && nseg * c <= num_sms && 2LL * cap(c) >= need2 * nseg) return c;
    return 1;
  };
  int best;
  if (ordered) {
    best = largest(2);  // a step runs alone: the most CTAs streaming
  } else {
    // Steps overlap.  Short segments (a CTA streams at most two rings of tiles; the step
    // is latency-bound): room for two consecutive steps, so that the next step's CTAs
    // start as this one finishes.  Long segments (bandwidth-bound): room for one and a half
    // steps, else one -- more CTAs streaming while part of the next step already runs.
    // Measured on GB300 (15 clusters of 8 fit, 13 of 10, 23 of 6), 8 segments: a 4k step
    // 5.35 us with clusters of 6, 5.56 with 10, 5.85 with 8; 8k / 16k / 128k contexts
    // 7.82 / 12.1 / 75.5 us with 10, against 7.98 / 13.0 / 78.6 with 6.
    const int c2 = largest(4);
    const long long per_cta = (max_seg_tiles + c2 - 1) / c2;
    if (c2 > 1 && per_cta <= 2LL * kStages) {
      best = c2;
    } else {
      best = largest(3);
      if (best == 1) best = largest(2);
    }
  }
  if (best == 1 && cap(1) < 1) return 0;
  // Enough CTAs to stream: 48 SMs nearly saturate HBM (6.85 TB/s measured on a 128k
  // sequence, about 140 GB/s each), or one CTA per tile already.
  if (nseg * best < 48 && nseg * best < total_tiles) return 0;
  return best;
}

namespace {

// Workers whose tile ranges touch the longest segment of a batch (the split form), for
// gqa_plan_num_splits.
int split_count(const int32_t *lens, int B, int Hkv, int max_seq, int W) {
  long long T = 0, best_nt = -1, best_begin = 0;
  for (int b = 0; b < B; ++b) {
    long long L = lens ? lens[b] : max_seq;
    L = L < 1 ? 1 : (L > max_seq ? max_seq : L);
    const long long nt = (L + kTile - 1) / kTile;
    if (nt > best_nt) best_nt = nt, best_begin = T;
    T += Hkv * nt;
  }
  return worker_of(T, W, best_begin + best_nt - 1) - worker_of(T, W, best_begin) + 1;
}

bool finite_pos(float x) { return isfinite(x) && x > 0.f; }

// Is host pointer h page-locked memory mapped into the device's address space, 16-byte
// aligned?  Then *d is its device address.  (Asked on every call: a cached answer could
// outlive the allocation it describes.)
bool mapped_host(const void *h, void **d) {
  cudaPointerAttributes a;
  *d = nullptr;
  if (cudaPointerGetAttributes(&a, h) == cudaSuccess && a.type == cudaMemoryTypeHost && a.devicePointer &&
      (reinterpret_cast<uintptr_t>(a.devicePointer) & 15) == 0)
    *d = a.devicePointer;
  else
    cudaGetLastError();
  return *d != nullptr;
}

bool valid_cluster_size(int c) { return c >= -1 && c <= 16; }

// The kernels read and write whole 16-byte chunks of the bf16 tensors (and bulk-prefetch
// them), and 4-byte words of the int32 ones; NULL passes (optional tensors).
bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool device_args_aligned(const void *q, const void *k, const void *v, const void *kc, const void *vc,
                         const void *qw, const void *kw, const int32_t *pt, const int32_t *sl, const int32_t *pos) {
  return aligned(q, 16) && aligned(k, 16) && aligned(v, 16) && aligned(kc, 16) && aligned(vc, 16) &&
         aligned(qw, 16) && aligned(kw, 16) && aligned(pt, 4) && aligned(sl, 4) && aligned(pos, 4);
}

gqa_status_t check_step_args(const gqa_plan_t *plan, const void *q, const void *k, const void *v, const void *kc,
                             const void *vc, const int32_t *pt, const int32_t *sl, const int32_t *pos,
                             float theta, float eps, const void *out) {
  if (!plan || !q || !k || !v || !kc || !vc || !sl || !pos || !out) return GQA_ERR_INVALID_ARG;
  const bool paged = plan->desc.block_size > 0;
  if (paged != (pt != nullptr)) return GQA_ERR_INVALID_ARG;
  if (!finite_pos(theta) || !isfinite(eps) || eps < 0.f) return GQA_ERR_INVALID_ARG;
  return GQA_OK;
}

// The tensor maps of a cache pair: looked up among the pairs seen recently (searching
// from the last hit, as successive layers come in order), else encoded into the oldest
// slot.  A map describes only an address and the plan's geometry, so a cached one stays
// right for that address.
gqa_status_t cache_maps(const gqa_plan_t *plan, const void *kc, const void *vc, CUtensorMap *tk, CUtensorMap *tv) {
  std::lock_guard<std::mutex> lk(plan->tm_mu);
  constexpr int N = gqa_plan::kMapCache;
  for (int i = 0; i < N; ++i) {
    const gqa_plan::CacheMaps &e = plan->tm[(plan->tm_last + i) % N];
    if (e.k == kc && e.v == vc && kc) {
      plan->tm_last = (plan->tm_last + i) % N;
      *tk = e.tk;
      *tv = e.tv;
      return GQA_OK;
    }
  }
  gqa_plan::CacheMaps &e = plan->tm[plan->tm_next];
  e.k = e.v = nullptr;
  if (!make_cache_map(&e.tk, kc, plan->desc.num_kv_heads, plan->num_rows) ||
      !make_cache_map(&e.tv, vc, plan->desc.num_kv_heads, plan->num_rows))
    return GQA_ERR_CUDA;
  e.k = kc;
  e.v = vc;
  plan->tm_last = plan->tm_next;
  plan->tm_next = (plan->tm_next + 1) % N;
  *tk = e.tk;
  *tv = e.tv;
  return GQA_OK;
}

// (Re)builds the plan's RoPE table for `theta` on `stream` when it holds another theta;
// *rebuilt says whether it launched the build.
gqa_status_t ensure_rope_table(const gqa_plan_t *plan, float theta, cudaStream_t stream, bool *rebuilt) {
  *rebuilt = false;
  if (plan->tab_valid && plan->tab_theta == theta) return GQA_OK;
  RopeTableParams t;
  t.rope_dw = plan->rope_tab;
  t.rope_tab32 = const_cast<float2 *>(rope_tab32_of(plan));
  t.max_seq = plan->desc.max_seq_len;
  for (int i = 0; i < kHeadDim / 2; ++i)
    t.inv_freq[i] = pow(static_cast<double>(theta), -2.0 * i / static_cast<double>(kHeadDim));
  plan->tab_valid = false;
  if (launch_rope_table(t, stream) != cudaSuccess) return GQA_ERR_CUDA;
  plan->tab_valid = true;
  plan->tab_theta = theta;
  *rebuilt = true;
  return GQA_OK;
}

// The attention launch: the split-KV kernel (partials for gqa_combine) when `single_out`
// is null, else the single-launch form writing the step's output there.
gqa_status_t run_attention(const gqa_plan_t *plan, const void *q, const void *k, const void *v, void *kc, void *vc,
                           const int32_t *pt, const int32_t *sl, const int32_t *pos, const void *qw, const void *kw,
                           float theta, float eps, cudaStream_t stream, bool host_inputs = false,
                           void *single_out = nullptr) {
  if (!device_args_aligned(q, k, v, kc, vc, qw, kw, pt, sl, pos)) return GQA_ERR_INVALID_ARG;
  bool rebuilt = false;
  gqa_status_t st = ensure_rope_table(plan, theta, stream, &rebuilt);
  if (st != GQA_OK) return st;
  CUtensorMap tk, tv;
  st = cache_maps(plan, kc, vc, &tk, &tv);
  if (st != GQA_OK) return st;
  AttnParams p;
  memset(&p, 0, sizeof p);
  p.seq_lens = sl;
  p.page_table = pt;
  p.positions = pos;
  p.q_new = static_cast<const uint16_t *>(q);
  p.k_new = static_cast<const uint16_t *>(k);
  p.v_new = static_cast<const uint16_t *>(v);
  p.k_cache = static_cast<uint16_t *>(kc);
  p.v_cache = static_cast<uint16_t *>(vc);
  p.q_norm_w = static_cast<const uint16_t *>(qw);
  p.k_norm_w = static_cast<const uint16_t *>(kw);
  p.rope_dw = plan->rope_tab;
  p.rope_tab32 = rope_tab32_of(plan);
  p.q_rot = plan->q_rot;
  p.part_o = plan->part_o;
  p.part_ml = plan->part_ml;
  p.err = plan->err;
  p.inputs_in_host_memory = host_inputs ? 1 : 0;
  p.spec = plan->desc.block_size > 0 ? nullptr : plan->spec;
  p.B = plan->desc.batch;
  p.Hq = plan->desc.num_q_heads;
  p.Hkv = plan->desc.num_kv_heads;
  p.G = plan->G;
  p.paged = plan->desc.block_size > 0;
  p.max_seq = plan->desc.max_seq_len;
  p.max_blocks = plan->max_blocks;
  p.num_blocks = plan->desc.num_cache_blocks;
  p.eps = static_cast<double>(eps);
  p.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(kHeadDim)));
  cudaError_t e;
  if (single_out) {
    p.out = static_cast<uint16_t *>(single_out);
    p.csize = plan->csize;
    p.spec_tiles = plan->spec_tiles;
    p.spec = nullptr;
    // Segments longest first when the clusters come in more than one wave and the steps do
    // not overlap (measured on the ragged batch: 104.7 -> 94.0 us a step; with overlapping
    // steps the next step's clusters already fill the last wave's idle SMs, and the order
    // measured 1 % slower there).
    p.seg_order = plan->ordered_first && plan->waves_by_start[1] ? plan->seg_order : nullptr;
    e = launch_attention_cluster(tk, tv, p, plan->npad, !rebuilt && !plan->ordered_first, stream);
  } else {
    e = launch_attention(tk, tv, p, plan->npad, plan->W, !rebuilt && !plan->ordered_first, stream);
  }
  return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

gqa_status_t run_combine(const gqa_plan_t *plan, const int32_t *sl, void *out, cudaStream_t stream) {
  if (!aligned(out, 16) || !aligned(sl, 4)) return GQA_ERR_INVALID_ARG;
  CombineParams p;
  memset(&p, 0, sizeof p);
  p.seq_lens = sl;
  p.part_o = plan->part_o;
  p.part_ml = plan->part_ml;
  p.out = static_cast<uint16_t *>(out);
  p.B = plan->desc.batch;
  p.Hq = plan->desc.num_q_heads;
  p.Hkv = plan->desc.num_kv_heads;
  p.G = plan->G;
  p.W = plan->W;
  p.max_seq = plan->desc.max_seq_len;
  return launch_combine(p, plan->combine_split, stream) == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

gqa_status_t run_step(const gqa_plan_t *plan, const void *q, const void *k, const void *v, void *kc, void *vc,
                      const int32_t *pt, const int32_t *sl, const int32_t *pos, const void *qw, const void *kw,
                      float theta, float eps, void *out, cudaStream_t stream, bool host_inputs = false) {
  if (!aligned(out, 16)) return GQA_ERR_INVALID_ARG;  // checked before anything is launched
  gqa_status_t st = run_attention(plan, q, k, v, kc, vc, pt, sl, pos, qw, kw, theta, eps, stream, host_inputs,
                                  plan->csize > 0 ? out : nullptr);
  if (st != GQA_OK || plan->csize > 0) return st;
  return run_combine(plan, sl, out, stream);
}

// Checks a geometry (all but the device index).
gqa_status_t check_desc(const gqa_plan_desc_t &d) {
  if (d.batch < 1 || d.num_q_heads < 1 || d.num_kv_heads < 1 || d.max_seq_len < 1 || d.num_workers < 0 ||
      d.block_size < 0 || !valid_cluster_size(d.cluster_size))
    return GQA_ERR_INVALID_ARG;
  if (d.head_dim != GQA_HEAD_DIM || d.num_q_heads % d.num_kv_heads != 0 ||
      d.num_q_heads / d.num_kv_heads > GQA_MAX_GROUP || d.batch > GQA_MAX_BATCH ||
      (d.block_size != 0 && d.block_size != GQA_BLOCK_SIZE))
    return GQA_ERR_UNSUPPORTED;
  const bool paged = d.block_size > 0;
  if (paged && d.num_cache_blocks < 1) return GQA_ERR_INVALID_ARG;
  const long long max_blocks = (d.max_seq_len + kTile - 1) / kTile;
  const long long num_rows = paged ? static_cast<long long>(d.num_cache_blocks) * kTile
                                   : static_cast<long long>(d.batch) * d.max_seq_len;
  if (num_rows > 0x7fffffffLL - kTile) return GQA_ERR_UNSUPPORTED;
  if (static_cast<long long>(d.batch) * d.num_kv_heads * max_blocks > 0x7fffffffLL) return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}

// The planner's decisions for a checked geometry on a device with `num_sms` SMs that can
// hold capacity[c - 1] clusters of c single-launch CTAs at once (c = 1 .. 16): the split-KV worker count,
// the step's form, the splits of the longest segment and the combine's shape.  Lengths
// come from seq_lens_host (clamped to [1, max_seq_len]) or are max_seq_len.
struct PlanChoice {
  int W = 0, csize = 0, nsplit = 0, combine_split = 0, max_seg_tiles = 0;
};
gqa_status_t plan_choose(const gqa_plan_desc_t &d, const int32_t *seq_lens_host, int num_sms, const int *capacity,
                         PlanChoice *out) {
  long long total_tiles = 0, max_seg_tiles = 0;
  for (int b = 0; b < d.batch; ++b) {
    long long L = seq_lens_host ? seq_lens_host[b] : d.max_seq_len;
    if (L < 1) L = 1;
    if (L > d.max_seq_len) L = d.max_seq_len;
    total_tiles += d.num_kv_heads * ((L + kTile - 1) / kTile);
    max_seg_tiles = std::max(max_seg_tiles, (L + kTile - 1) / kTile);
  }
  PlanChoice c;
  c.W = d.num_workers > 0 ? d.num_workers : plan_workers(num_sms, total_tiles);
  c.combine_split = combine_split(d.batch, d.num_q_heads, d.num_kv_heads, c.W, num_sms);
  c.csize = plan_step_form(d.cluster_size, d.num_workers, num_sms, capacity,
                           static_cast<long long>(d.batch) * d.num_kv_heads, max_seg_tiles, total_tiles,
                           d.ordered_start != 0);
  if (c.csize < 0) return GQA_ERR_UNSUPPORTED;
  c.max_seg_tiles = static_cast<int>(max_seg_tiles);
  c.nsplit = c.csize > 0 ? static_cast<int>(std::min<long long>(c.csize, max_seg_tiles))
                         : split_count(seq_lens_host, d.batch, d.num_kv_heads, d.max_seq_len, c.W);
  *out = c;
  return GQA_OK;
}

// The current device's cluster capacities for a group size, clusters of 1 .. 16 CTAs
// (attn_configure first).
void device_capacity(int npad, int (&cap)[16]) {
  for (int k = 0; k < 16; ++k) cap[k] = attn_cluster_capacity(npad, k + 1);
}

}  // namespace

namespace gqa {

gqa_status_t step_layout(const gqa_plan_desc_t &d, int num_sms, StepLayout *lay) {
  gqa_status_t st = check_desc(d);
  if (st != GQA_OK) return st;
  const bool paged = d.block_size > 0;
  const long long B = d.batch, Hkv = d.num_kv_heads;
  const long long max_blocks = (d.max_seq_len + kTile - 1) / kTile;
  StepLayout l;
  l.G = d.num_q_heads / d.num_kv_heads;
  l.npad = l.G <= 8 ? 8 : 16;
  l.max_blocks = static_cast<int>(max_blocks);
  l.num_rows = paged ? static_cast<long long>(d.num_cache_blocks) * kTile : B * d.max_seq_len;
  int cap[16];
  device_capacity(l.npad, cap);
  PlanChoice pc;
  st = plan_choose(d, nullptr, num_sms, cap, &pc);
  if (st != GQA_OK) return st;
  l.W = pc.W;
  l.combine_split = pc.combine_split;
  l.csize = pc.csize;
  l.spec_tiles = pc.max_seg_tiles;
  const long long slots = B * Hkv + l.W;
  l.tab_bytes = rope_tables_bytes(d.max_seq_len);
  l.off_q = l.tab_bytes;
  l.off_o = l.off_q + align256(B * d.num_q_heads * kHeadDim * 2);
  l.off_ml = l.off_o + align256(slots * kConsumerWarps * l.G * kHeadDim * 4);
  l.off_err = l.off_ml + align256(slots * kConsumerWarps * l.G * 2 * 4);
  l.total = l.off_err + 256;
  *lay = l;
  return GQA_OK;
}

gqa_status_t run_step_at(const gqa_plan_desc_t &d, const StepLayout &lay, void *base, uint32_t *err,
                         bool table_ready, const void *q, const void *k, const void *v, void *kc, void *vc,
                         const int32_t *pt, const int32_t *sl, const int32_t *pos, const void *qw, const void *kw,
                         float theta, float eps, void *out, cudaStream_t stream) {
  if (!base || !err) return GQA_ERR_INVALID_ARG;
  gqa_plan_t plan;
  plan.desc = d;
  plan.G = lay.G;
  plan.npad = lay.npad;
  plan.W = lay.W;
  plan.max_blocks = lay.max_blocks;
  plan.combine_split = lay.combine_split;
  plan.csize = lay.csize;
  plan.spec_tiles = lay.spec_tiles;
  plan.num_rows = lay.num_rows;
  plan.ordered_first = d.ordered_start != 0;
  char *c = static_cast<char *>(base);
  plan.rope_tab = reinterpret_cast<float4 *>(c);
  plan.q_rot = reinterpret_cast<uint16_t *>(c + lay.off_q);
  plan.part_o = reinterpret_cast<float *>(c + lay.off_o);
  plan.part_ml = reinterpret_cast<float *>(c + lay.off_ml);
  plan.err = err;
  plan.tab_valid = table_ready;
  plan.tab_theta = theta;
  gqa_status_t st = check_step_args(&plan, q, k, v, kc, vc, pt, sl, pos, theta, eps, out);
  if (st != GQA_OK) return st;
  return run_step(&plan, q, k, v, kc, vc, pt, sl, pos, qw, kw, theta, eps, out, stream);
}

}  // namespace gqa

extern "C" {

gqa_status_t gqa_plan_create(const gqa_plan_desc_t *desc, const int32_t *seq_lens_host, gqa_plan_t **plan) {
  if (!desc || !plan) return GQA_ERR_INVALID_ARG;
  *plan = nullptr;
  const gqa_plan_desc_t &d = *desc;
  gqa_status_t st = check_desc(d);
  if (st != GQA_OK) return st;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) return GQA_ERR_CUDA;
  if (d.device < 0 || d.device >= ndev) return GQA_ERR_INVALID_ARG;

  DeviceGuard guard(d.device);
  if (!guard.ok) return GQA_ERR_CUDA;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d.device) != cudaSuccess) return GQA_ERR_CUDA;
  const int npad = d.num_q_heads / d.num_kv_heads <= 8 ? 8 : 16;
  if (attn_configure(npad) != cudaSuccess) {
    cudaGetLastError();
    return GQA_ERR_CUDA;
  }
  int cap[16];
  device_capacity(npad, cap);
  PlanChoice pc, pc_other;
  st = plan_choose(d, seq_lens_host, sms, cap, &pc);
  if (st != GQA_OK) return st;
  gqa_plan_desc_t d_other = d;
  d_other.ordered_start = d.ordered_start ? 0 : 1;
  st = plan_choose(d_other, seq_lens_host, sms, cap, &pc_other);
  if (st != GQA_OK) return st;

  gqa_plan_t *p = new (std::nothrow) gqa_plan_t();
  if (!p) return GQA_ERR_WORKSPACE;
  p->desc = d;
  p->G = d.num_q_heads / d.num_kv_heads;
  p->npad = npad;
  p->num_sms = sms;
  p->max_blocks = static_cast<int>((d.max_seq_len + kTile - 1) / kTile);
  p->num_rows = d.block_size > 0 ? static_cast<long long>(d.num_cache_blocks) * kTile
                                  : static_cast<long long>(d.batch) * d.max_seq_len;
  p->W = pc.W;
  p->combine_split = pc.combine_split;
  p->csize = pc.csize;
  p->nsplit = pc.nsplit;
  p->spec_tiles = pc.max_seg_tiles;
  p->ordered_first = d.ordered_start != 0;
  const int mine = p->ordered_first ? 1 : 0;
  p->csize_by_start[mine] = pc.csize, p->nsplit_by_start[mine] = pc.nsplit;
  p->csize_by_start[1 - mine] = pc_other.csize, p->nsplit_by_start[1 - mine] = pc_other.nsplit;
  // Launch order of the single-launch clusters when they outnumber what the device holds at
  // once: longest planned segment first, so that the last clusters to start are short ones
  // (a greedy longest-processing-time schedule; any order is correct).
  const long long nseg = static_cast<long long>(d.batch) * d.num_kv_heads;
  for (int m = 0; m < 2; ++m) {
    const int c = p->csize_by_start[m];
    p->waves_by_start[m] = seq_lens_host != nullptr && c > 0 && nseg > cap[c - 1];
  }

  const long long B = d.batch, Hq = d.num_q_heads, Hkv = d.num_kv_heads;
  const long long slots = B * Hkv + p->W;
  const size_t sz_q = align256(B * Hq * kHeadDim * 2);
  const size_t sz_o = align256(slots * kConsumerWarps * p->G * kHeadDim * 4);
  const size_t sz_ml = align256(slots * kConsumerWarps * p->G * 2 * 4);
  const size_t sz_err = 256;
  const size_t sz_sq = align256(B * Hq * kHeadDim * 2), sz_skv = align256(B * Hkv * kHeadDim * 2);
  const size_t sz_si = align256(B * 4);
  const size_t sz_tab = rope_tables_bytes(d.max_seq_len);
  const size_t sz_spec = align256(static_cast<size_t>(p->W) * kStages * sizeof(int2));
  const size_t sz_order = align256(static_cast<size_t>(nseg) * sizeof(int32_t));
  p->ws_bytes =
      sz_q + sz_o + sz_ml + sz_err + 2 * sz_sq + 2 * sz_skv + 2 * sz_si + sz_tab + sz_spec + 2 * sz_q + sz_order;
  if (cudaMalloc(&p->ws, p->ws_bytes) != cudaSuccess) {
    cudaGetLastError();
    delete p;
    return GQA_ERR_WORKSPACE;
  }
  char *c = static_cast<char *>(p->ws);
  p->q_rot = reinterpret_cast<uint16_t *>(c); c += sz_q;
  p->part_o = reinterpret_cast<float *>(c); c += sz_o;
  p->part_ml = reinterpret_cast<float *>(c); c += sz_ml;
  p->err = reinterpret_cast<uint32_t *>(c); c += sz_err;
  p->st_q = reinterpret_cast<uint16_t *>(c); c += sz_sq;
  p->st_out = reinterpret_cast<uint16_t *>(c); c += sz_sq;
  p->st_k = reinterpret_cast<uint16_t *>(c); c += sz_skv;
  p->st_v = reinterpret_cast<uint16_t *>(c); c += sz_skv;
  p->st_sl = reinterpret_cast<int32_t *>(c); c += sz_si;
  p->st_pos = reinterpret_cast<int32_t *>(c); c += sz_si;
  p->rope_tab = reinterpret_cast<float4 *>(c); c += sz_tab;
  p->spec = reinterpret_cast<int2 *>(c); c += sz_spec;
  p->q4_hi = reinterpret_cast<uint16_t *>(c); c += sz_q;
  p->q4_lo = reinterpret_cast<uint16_t *>(c); c += sz_q;
  p->seg_order = reinterpret_cast<int32_t *>(c); c += sz_order;
  std::vector<int32_t> order(static_cast<size_t>(nseg));
  {
    std::vector<long long> seg_tiles(static_cast<size_t>(nseg));
    for (long long sgi = 0; sgi < nseg; ++sgi) {
      long long L = seq_lens_host ? seq_lens_host[sgi / d.num_kv_heads] : d.max_seq_len;
      L = L < 1 ? 1 : (L > d.max_seq_len ? d.max_seq_len : L);
      seg_tiles[static_cast<size_t>(sgi)] = (L + kTile - 1) / kTile;
      order[static_cast<size_t>(sgi)] = static_cast<int32_t>(sgi);
    }
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
      return seg_tiles[static_cast<size_t>(a)] > seg_tiles[static_cast<size_t>(b)];
    });
  }
  if (cudaMemset(p->ws, 0, p->ws_bytes) != cudaSuccess || cudaMemset(p->spec, 0xff, sz_spec) != cudaSuccess ||
      cudaMemcpy(p->seg_order, order.data(), order.size() * sizeof(int32_t), cudaMemcpyHostToDevice) !=
          cudaSuccess ||
      q4_configure() != cudaSuccess ||
      configure_small_kernels() != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    cudaFree(p->ws);
    delete p;
    return GQA_ERR_CUDA;
  }
  *plan = p;
  return GQA_OK;
}

gqa_status_t gqa_plan_destroy(gqa_plan_t *plan) {
  if (!plan) return GQA_OK;
  DeviceGuard guard(plan->desc.device);
  cudaError_t e = cudaFree(plan->ws);
  delete plan;
  return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

gqa_status_t gqa_plan_describe(const gqa_plan_desc_t *desc, const int32_t *seq_lens_host, int num_sms,
                               const int *cluster_capacity, int *num_workers, int *cluster_size, int *num_splits) {
  if (!desc || !cluster_capacity || num_sms < 1) return GQA_ERR_INVALID_ARG;
  gqa_status_t st = check_desc(*desc);
  if (st != GQA_OK) return st;
  PlanChoice pc;
  st = plan_choose(*desc, seq_lens_host, num_sms, cluster_capacity, &pc);
  if (st != GQA_OK) return st;
  if (num_workers) *num_workers = pc.W;
  if (cluster_size) *cluster_size = pc.csize;
  if (num_splits) *num_splits = pc.nsplit;
  return GQA_OK;
}

gqa_status_t gqa_plan_set_ordered_start(gqa_plan_t *plan, int ordered) {
  if (!plan) return GQA_ERR_INVALID_ARG;
  plan->ordered_first = ordered != 0;
  // the planner's form for the new setting (the workspace holds either form's partials)
  plan->csize = plan->csize_by_start[plan->ordered_first ? 1 : 0];
  plan->nsplit = plan->nsplit_by_start[plan->ordered_first ? 1 : 0];
  return GQA_OK;
}

int gqa_plan_num_workers(const gqa_plan_t *plan) { return plan ? plan->W : 0; }

int gqa_plan_num_splits(const gqa_plan_t *plan) { return plan ? plan->nsplit : 0; }

int gqa_plan_cluster_size(const gqa_plan_t *plan) { return plan ? plan->csize : 0; }

size_t gqa_plan_workspace_bytes(const gqa_plan_t *plan) { return plan ? plan->ws_bytes : 0; }

gqa_status_t gqa_decode_attn(const gqa_plan_t *plan, const void *q_new, const void *k_new, const void *v_new,
                             void *k_cache, void *v_cache, const int32_t *page_table, const int32_t *seq_lens,
                             const int32_t *positions, const void *q_norm_w, const void *k_norm_w, float rope_theta,
                             float eps, void *out, void *stream) {
  gqa_status_t st = check_step_args(plan, q_new, k_new, v_new, k_cache, v_cache, page_table, seq_lens, positions,
                                    rope_theta, eps, out);
  if (st != GQA_OK) return st;
  DeviceGuard guard(plan->desc.device);
  if (!guard.ok) return GQA_ERR_CUDA;
  return run_step(plan, q_new, k_new, v_new, k_cache, v_cache, page_table, seq_lens, positions, q_norm_w, k_norm_w,
                  rope_theta, eps, out, static_cast<cudaStream_t>(stream));
}

gqa_status_t gqa_decode_attn_host(const gqa_plan_t *plan, const void *q_new_host, const void *k_new_host,
                                  const void *v_new_host, void *k_cache, void *v_cache, const int32_t *page_table,
                                  const int32_t *seq_lens_host, const int32_t *positions_host, const void *q_norm_w,
                                  const void *k_norm_w, float rope_theta, float eps, void *out_host, void *stream) {
  gqa_status_t st = check_step_args(plan, q_new_host, k_new_host, v_new_host, k_cache, v_cache, page_table,
                                    seq_lens_host, positions_host, rope_theta, eps, out_host);
  if (st != GQA_OK) return st;
  DeviceGuard guard(plan->desc.device);
  if (!guard.ok) return GQA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Page-locked host buffers are mapped into the device's address space: the kernels then
  // read the inputs and write the output through the host link directly (NVLink-C2C on a
  // Grace-Blackwell node), with no staging copies.  Other host memory is copied through
  // the plan's staging buffers.
  const void *hp[6] = {q_new_host, k_new_host, v_new_host, seq_lens_host, positions_host, out_host};
  void *dp[6];
  bool mapped = true;
  for (int i = 0; i < 6 && mapped; ++i) mapped = mapped_host(hp[i], &dp[i]);
  if (mapped)
    return run_step(plan, dp[0], dp[1], dp[2], k_cache, v_cache, page_table, static_cast<const int32_t *>(dp[3]),
                    static_cast<const int32_t *>(dp[4]), q_norm_w, k_norm_w, rope_theta, eps, dp[5], s, true);
  const size_t B = plan->desc.batch, Hq = plan->desc.num_q_heads, Hkv = plan->desc.num_kv_heads;
  const size_t bq = B * Hq * kHeadDim * 2, bkv = B * Hkv * kHeadDim * 2, bi = B * 4;
  if (cudaMemcpyAsync(plan->st_q, q_new_host, bq, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(plan->st_k, k_new_host, bkv, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(plan->st_v, v_new_host, bkv, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(plan->st_sl, seq_lens_host, bi, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(plan->st_pos, positions_host, bi, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return GQA_ERR_CUDA;
  st = run_step(plan, plan->st_q, plan->st_k, plan->st_v, k_cache, v_cache, page_table, plan->st_sl, plan->st_pos,
                q_norm_w, k_norm_w, rope_theta, eps, plan->st_out, s);
  if (st != GQA_OK) return st;
  if (cudaMemcpyAsync(out_host, plan->st_out, bq, cudaMemcpyDeviceToHost, s) != cudaSuccess) return GQA_ERR_CUDA;
  return GQA_OK;
}

gqa_status_t gqa_attention_splitkv(const gqa_plan_t *plan, const void *q_new, const void *k_new, const void *v_new,
                                   void *k_cache, void *v_cache, const int32_t *page_table, const int32_t *seq_lens,
                                   const int32_t *positions, const void *q_norm_w, const void *k_norm_w,
                                   float rope_theta, float eps, void *stream) {
  if (!plan || !q_new || !k_new || !v_new || !k_cache || !v_cache || !seq_lens || !positions)
    return GQA_ERR_INVALID_ARG;
  if ((plan->desc.block_size > 0) != (page_table != nullptr)) return GQA_ERR_INVALID_ARG;
  if (!finite_pos(rope_theta) || !isfinite(eps) || eps < 0.f) return GQA_ERR_INVALID_ARG;
  DeviceGuard guard(plan->desc.device);
  if (!guard.ok) return GQA_ERR_CUDA;
  return run_attention(plan, q_new, k_new, v_new, k_cache, v_cache, page_table, seq_lens, positions, q_norm_w,
                       k_norm_w, rope_theta, eps, static_cast<cudaStream_t>(stream));
}

gqa_status_t gqa_combine(const gqa_plan_t *plan, const int32_t *seq_lens, void *out, void *stream) {
  if (!plan || !seq_lens || !out) return GQA_ERR_INVALID_ARG;
  DeviceGuard guard(plan->desc.device);
  if (!guard.ok) return GQA_ERR_CUDA;
  return run_combine(plan, seq_lens, out, static_cast<cudaStream_t>(stream));
}

gqa_status_t gqa_plan_read_q_rot(const gqa_plan_t *plan, uint16_t *q_rot_host) {
  if (!plan || !q_rot_host) return GQA_ERR_INVALID_ARG;
  DeviceGuard guard(plan->desc.device);
  if (!guard.ok) return GQA_ERR_CUDA;
  const size_t bytes = static_cast<size_t>(plan->desc.batch) * plan->desc.num_q_heads * kHeadDim * 2;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(q_rot_host, plan->q_rot, bytes, cudaMemcpyDeviceToHost) != cudaSuccess)
    return GQA_ERR_CUDA;
  return GQA_OK;
}

gqa_status_t gqa_plan_device_errors(const gqa_plan_t *plan, uint32_t *flags, int clear) {
  if (!plan || !flags) return GQA_ERR_INVALID_ARG;
  DeviceGuard guard(plan->desc.device);
  if (!guard.ok) return GQA_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(flags, plan->err, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return GQA_ERR_CUDA;
  if (clear && (cudaMemset(plan->err, 0, sizeof(uint32_t)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess))
    return GQA_ERR_CUDA;
  return GQA_OK;
}

long long gqa_partition_describe(const int32_t *seq_lens_host, int batch, int num_kv_heads, int max_seq_len,
                                 int num_workers, long long *worker_range) {
  if (!seq_lens_host || !worker_range || batch < 1 || num_kv_heads < 1 || max_seq_len < 1 || num_workers < 1)
    return -1;
  long long T = 0;
  for (int b = 0; b < batch; ++b) T += static_cast<long long>(num_kv_heads) * tiles_of(seq_lens_host[b], max_seq_len);
  for (int w = 0; w < num_workers; ++w) {
    worker_range[2 * w] = worker_begin(T, num_workers, w);
    worker_range[2 * w + 1] = worker_begin(T, num_workers, w + 1);
  }
  return T;
}

const char *gqa_status_string(gqa_status_t status) {
  switch (status) {
    case GQA_OK: return "ok";
    case GQA_ERR_INVALID_ARG: return "invalid argument";
    case GQA_ERR_UNSUPPORTED: return "unsupported geometry";
    case GQA_ERR_CUDA: return "CUDA error";
    case GQA_ERR_WORKSPACE: return "workspace allocation failed";
    case GQA_ERR_SCRATCH_LIMIT: return "geometry needs more than the fixed static scratch";
  }
  return "unknown status";
}

}  // extern "C"

// ------------------------------------------------------------------------ 4-bit KV cache

extern "C" gqa_status_t gqa_q4_codebook(uint16_t *levels_bf16) {
  if (!levels_bf16) return GQA_ERR_INVALID_ARG;
  // Lloyd's algorithm for the 16-level quantizer of N(0,1): cell boundaries at the midpoints
  // of adjacent levels, each level moved to the mean of N(0,1) over its cell,
  //   E[X | a < X < b] = (pdf(a) - pdf(b)) / (cdf(b) - cdf(a)),
  // until no level moves.
  constexpr int kLv = 16;
  const double inv_sqrt2pi = 0.3989422804014327;
  auto pdf = [&](double x) { return std::isinf(x) ? 0.0 : inv_sqrt2pi * exp(-0.5 * x * x); };
  auto cdf = [](double x) { return 0.5 * erfc(-x * 0.7071067811865476); };
  double lv[kLv];
  for (int j = 0; j < kLv; ++j) lv[j] = 3.0 * (2.0 * j + 1.0 - kLv) / kLv;
  for (int it = 0; it < 200000; ++it) {
    double edge[kLv + 1];
    edge[0] = -INFINITY;
    edge[kLv] = INFINITY;
    for (int j = 1; j < kLv; ++j) edge[j] = 0.5 * (lv[j - 1] + lv[j]);
    double step = 0.0;
    for (int j = 0; j < kLv; ++j) {
      const double mass = cdf(edge[j + 1]) - cdf(edge[j]);
      const double mean = (pdf(edge[j]) - pdf(edge[j + 1])) / mass;
      step = std::max(step, fabs(mean - lv[j]));
      lv[j] = mean;
    }
    if (step < 1e-15) break;
  }
  for (int j = 0; j < kLv; ++j) {
    const __nv_bfloat16 b = __float2bfloat16_rn(static_cast<float>(lv[j]));
    memcpy(&levels_bf16[j], &b, sizeof(uint16_t));
  }
  return GQA_OK;
}

extern "C" gqa_status_t gqa_decode_attn_q4(const gqa_plan_t *plan, const void *q_new, const void *k_new,
                                           const void *v_new, uint8_t *k_idx, uint8_t *v_idx, float *k_scale,
                                           float *v_scale, const int32_t *page_table, const int32_t *seq_lens,
                                           const int32_t *positions, const void *q_norm_w, const void *k_norm_w,
                                           const int8_t *rot_signs, const void *codebook, float rope_theta, float eps,
                                           void *out, void *stream) {
  if (!plan || !q_new || !k_new || !v_new || !k_idx || !v_idx || !k_scale || !v_scale || !seq_lens || !positions ||
      !rot_signs || !codebook || !out)
    return GQA_ERR_INVALID_ARG;
  const bool paged = plan->desc.block_size > 0;
  if (paged != (page_table != nullptr)) return GQA_ERR_INVALID_ARG;
  if (!finite_pos(rope_theta) || !isfinite(eps) || eps < 0.f) return GQA_ERR_INVALID_ARG;
  if (!aligned(q_new, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_idx, 16) ||
      !aligned(v_idx, 16) || !aligned(q_norm_w, 16) || !aligned(k_norm_w, 16) || !aligned(out, 16) ||
      !aligned(k_scale, 4) || !aligned(v_scale, 4) || !aligned(rot_signs, 4) || !aligned(codebook, 2) ||
      !aligned(page_table, 4) || !aligned(seq_lens, 4) || !aligned(positions, 4))
    return GQA_ERR_INVALID_ARG;
  const gqa_plan_desc_t &d = plan->desc;
  DeviceGuard guard(d.device);
  if (!guard.ok) return GQA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool rebuilt = false;
  gqa_status_t st = ensure_rope_table(plan, rope_theta, s, &rebuilt);
  if (st != GQA_OK) return st;
  // index tiles: [rows][H_kv][64 bytes], box = 64 bytes x 1 head x 64 tokens
  CUtensorMap tk, tv;
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(d.num_kv_heads), static_cast<cuuint64_t>(plan->num_rows)};
  const cuuint64_t strides[2] = {64, static_cast<cuuint64_t>(d.num_kv_heads) * 64};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kTile)};
  if (!encode_u8_map(&tk, 3, k_idx, dims, strides, box) || !encode_u8_map(&tv, 3, v_idx, dims, strides, box))
    return GQA_ERR_CUDA;

  if (plan->csize > 0) {  // the single-launch form
    Q4ClusterParams cp;
    memset(&cp, 0, sizeof cp);
    cp.seq_lens = seq_lens;
    cp.positions = positions;
    cp.page_table = page_table;
    cp.q_new = static_cast<const uint16_t *>(q_new);
    cp.k_new = static_cast<const uint16_t *>(k_new);
    cp.v_new = static_cast<const uint16_t *>(v_new);
    cp.q_norm_w = static_cast<const uint16_t *>(q_norm_w);
    cp.k_norm_w = static_cast<const uint16_t *>(k_norm_w);
    cp.rope_tab32 = rope_tab32_of(plan);
    cp.signs = rot_signs;
    cp.codebook = static_cast<const uint16_t *>(codebook);
    cp.k_idx = k_idx;
    cp.v_idx = v_idx;
    cp.k_scale = k_scale;
    cp.v_scale = v_scale;
    cp.out = static_cast<uint16_t *>(out);
    cp.err = plan->err;
    cp.B = d.batch;
    cp.Hq = d.num_q_heads;
    cp.Hkv = d.num_kv_heads;
    cp.G = plan->G;
    cp.paged = paged ? 1 : 0;
    cp.max_seq = d.max_seq_len;
    cp.max_blocks = plan->max_blocks;
    cp.num_blocks = paged ? d.num_cache_blocks : 0;
    cp.csize = plan->csize;
    // Segments longest first whenever the clusters come in more than one wave (the 4-bit
    // step is bound by its arithmetic, so the last wave's imbalance counts with overlapping
    // steps too: the ragged batch 64.0 -> 59.9 us, 91.6 -> 71.9 us with ordered starts).
    cp.seg_order = plan->waves_by_start[plan->ordered_first ? 1 : 0] ? plan->seg_order : nullptr;
    cp.eps = eps;
    cp.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(kHeadDim)));
    return launch_q4_cluster(tk, tv, cp, plan->npad, !rebuilt && !plan->ordered_first, s) == cudaSuccess ? GQA_OK
                                                                                                    : GQA_ERR_CUDA;
  }

  Q4PrologueParams pp;
  memset(&pp, 0, sizeof pp);
  pp.seq_lens = seq_lens;
  pp.positions = positions;
  pp.page_table = page_table;
  pp.q_new = static_cast<const uint16_t *>(q_new);
  pp.k_new = static_cast<const uint16_t *>(k_new);
  pp.v_new = static_cast<const uint16_t *>(v_new);
  pp.q_norm_w = static_cast<const uint16_t *>(q_norm_w);
  pp.k_norm_w = static_cast<const uint16_t *>(k_norm_w);
  pp.rope_tab32 = rope_tab32_of(plan);
  pp.signs = rot_signs;
  pp.codebook = static_cast<const uint16_t *>(codebook);
  pp.q_hi = plan->q4_hi;
  pp.q_lo = plan->q4_lo;
  pp.k_idx = k_idx;
  pp.v_idx = v_idx;
  pp.k_scale = k_scale;
  pp.v_scale = v_scale;
  pp.err = plan->err;
  pp.B = d.batch;
  pp.Hq = d.num_q_heads;
  pp.Hkv = d.num_kv_heads;
  pp.paged = paged ? 1 : 0;
  pp.max_seq = d.max_seq_len;
  pp.max_blocks = plan->max_blocks;
  pp.num_blocks = paged ? d.num_cache_blocks : 0;
  pp.eps = eps;
  if (launch_q4_prologue(pp, !rebuilt && !plan->ordered_first, s) != cudaSuccess) return GQA_ERR_CUDA;

  Q4AttnParams ap;
  memset(&ap, 0, sizeof ap);
  ap.seq_lens = seq_lens;
  ap.page_table = page_table;
  ap.q_hi = plan->q4_hi;
  ap.q_lo = plan->q4_lo;
  ap.k_scale = k_scale;
  ap.v_scale = v_scale;
  ap.codebook = static_cast<const uint16_t *>(codebook);
  ap.part_o = plan->part_o;
  ap.part_ml = plan->part_ml;
  ap.err = plan->err;
  ap.B = d.batch;
  ap.Hq = d.num_q_heads;
  ap.Hkv = d.num_kv_heads;
  ap.G = plan->G;
  ap.paged = pp.paged;
  ap.max_seq = d.max_seq_len;
  ap.max_blocks = plan->max_blocks;
  ap.num_blocks = pp.num_blocks;
  ap.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(kHeadDim)));
  if (launch_q4_attention(tk, tv, ap, plan->npad, plan->W, s) != cudaSuccess) return GQA_ERR_CUDA;

  CombineParams cp;
  memset(&cp, 0, sizeof cp);
  cp.seq_lens = seq_lens;
  cp.part_o = plan->part_o;
  cp.part_ml = plan->part_ml;
  cp.out = static_cast<uint16_t *>(out);
  cp.B = d.batch;
  cp.Hq = d.num_q_heads;
  cp.Hkv = d.num_kv_heads;
  cp.G = plan->G;
  cp.W = plan->W;
  cp.max_seq = d.max_seq_len;
  if (launch_q4_combine(cp, rot_signs, s) != cudaSuccess) return GQA_ERR_CUDA;
  return GQA_OK;
}
