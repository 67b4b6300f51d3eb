// Chunked causal prefill attention on the 5th-generation tensor core (sm_103a).
//
// What it computes ("ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)", section 5.4,
// PREFILL with no sequence parallelism): sequence b receives a chunk of T new tokens at
// positions s_b .. s_b + T - 1 (s_b = q_start[b]) on top of a cache that holds positions
// [0, s_b).  Each chunk token gets the decode prologue -- QK RMSNorm, RoPE at its position,
// k and v appended to the cache ("Qwen3-14B Optimization", section 2.1 Shape 4 and
// section 3.3) -- and then attends causally: query token p sees keys 0 .. p.  The G query
// heads of a KV head share one operand (section 5.4: "GQA batches the group's query heads
// along the same axis as decode").
//
// Two kernels, and a third when query tiles are cut into KV parts:
//  * prefill_rope_kernel: one CTA per chunk token.  cos/sin of the token's position in
//    binary64, the rotated queries (binary32, rounded once to bf16) written to `out`, which
//    holds them until the attention kernel has read them, and the appended k row
//    (double-word arithmetic, rounded to bf16 as the exact value rounds) and v row.
//  * prefill_attn_kernel: one CTA per (sequence, KV head, block of Tt = 128 / G chunk
//    tokens); its 128-row M tile stacks those tokens' G heads.  A TMA warp streams 64-token
//    K tiles into a 2-stage ring and V tiles into a 3-stage one (a K tile is released once
//    S has used it, a V tile after P V); an MMA warp issues
//    S = Q K^T (M = 128, N = 64, K = 128) into tensor memory (two S buffers) and
//    O += P V (N = 128, K = 64) into a tensor-memory accumulator, P read from tensor
//    memory; four softmax warps own one row each per thread (tensor-memory lane = row),
//    apply the causal mask of the tile classes -- KV tiles wholly after the block's last
//    query are never loaded, the others are masked per row (key <= query position) -- run
//    the online softmax and store P over S as bf16 hi + lo, both multiplied into O, so
//    that rounding P costs no accuracy.  Two CTAs share an SM (about 97 KB of shared
//    memory and 256 tensor-memory columns each), so one CTA's softmax overlaps the
//    other's tensor work.  The running maximum is raised lazily: O in
//    tensor memory is rescaled only when a row's maximum grows by more than 2^8, so P stays
//    below 256 and most tiles need no rescale.
//  * prefill_merge_kernel: the KV parts of the cut query tiles (see the work items below)
//    leave fp32 partials; one CTA per (cut tile, 16 dims) merges them after the attention
//    kernel (M = max m_k, out = sum_k 2^(m_k - M) O_k / sum_k 2^(m_k - M) l_k).
#include <math.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "launch.h"
#include "rowmath.cuh"
#include "tc05.cuh"

namespace gqa {

namespace {

constexpr int kPfKStages = 2;                   // K ring depth (a K tile is released once S has used it)
constexpr int kPfVStages = 3;                   // V ring depth (a V tile is released after P V)
constexpr int kPfSoftmaxWarps = 4;              // one row per thread, 128 rows
constexpr int kPfThreads = 32 * (kPfSoftmaxWarps + 2);  // + TMA warp + MMA warp
constexpr int kPfProducerWarp = kPfSoftmaxWarps;
constexpr int kPfMmaWarp = kPfSoftmaxWarps + 1;
constexpr int kPfCtasPerSm = 2;                 // two CTAs share an SM: their softmax warps interleave
constexpr int kPfRows = 128;                    // M of every MMA
// Tensor memory per CTA: two S buffers (64 fp32 columns each; after the softmax has read
// S it stores P there as bf16 pairs, hi in the first 32 columns, lo in the next 32) and
// the O accumulator (128 columns).  Two CTAs fill the SM's 512 columns.
constexpr uint32_t kPfTmemCols = 256;
constexpr uint32_t kTmemO = 128;
constexpr float kRescaleLog2 = 8.f;             // lazy rescale threshold (P <= 2^8)

constexpr int kQBytes = 2 * kPfRows * kHalfRowBytes;     // 32 KiB: two 64-dim panels
constexpr int kKvTileBytes = 2 * kHalfTileBytes;          // 16 KiB: a K or V tile's two 64-dim halves
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;
constexpr int kOffV = kOffK + kPfKStages * kKvTileBytes;
constexpr int kOffBar = kOffV + kPfVStages * kKvTileBytes;
// barriers: q_full, k_full[2], k_empty[2], v_full[3], v_empty[3], s_full[2], p_full[2],
// o_done, drain
constexpr int kNumBars = 1 + 2 * kPfKStages + 2 * kPfVStages + 2 + 2 + 1 + 1;
// The dynamic shared memory is declared 1024-byte aligned (the 128-byte swizzle needs it);
// the kernel checks it rather than reserving slack, so that two CTAs fit an SM.
constexpr int kSmemBytes = kOffBar + 8 * kNumBars + 16;
constexpr int kPfMaxSlots = 320;                // split-tile partials the static scratch holds
constexpr int kPfMaxSplit = 6;                  // KV parts of one split query tile
// A partial is column-major, [130][128 rows] floats: O columns, then m, then l, so that the
// softmax warps (thread = row) write and read it in coalesced 128-byte lines.
constexpr int kPartFloats = (kHeadDim + 2) * kPfRows;
// The prologue holds a token's H_q + 2 H_kv rows in shared memory (256 B each).
constexpr int kRopeMaxSmem = 200 * 1024;
static_assert(kPfCtasPerSm * (kSmemBytes + 1024) <= 228 * 1024, "two prefill CTAs must share an SM");
static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kKvTileBytes % 1024 == 0, "swizzled tiles 1024-aligned");
static_assert(kPfCtasPerSm * kPfTmemCols <= 512, "tensor memory of the co-resident CTAs");

}  // namespace

struct PrefillParams {
  const uint16_t *q_new;       // [B, T, Hq, d]
  const uint16_t *k_new;       // [B, T, Hkv, d]
  const uint16_t *v_new;       // [B, T, Hkv, d]
  uint16_t *k_cache, *v_cache;
  const int32_t *page_table;   // [B, max_blocks] or null
  const int32_t *q_start;      // [B]
  const uint16_t *q_norm_w, *k_norm_w;
  uint16_t *out;               // [B, T, Hq, d]: rotated queries, then the attention output
  uint32_t *err;
  int B, T, Hq, Hkv, G, Tt, nqb;
  int paged, max_seq, max_blocks, num_blocks;
  float eps, scale_log2;
  double inv_freq[kHeadDim / 2];
  // Work items (CTAs): ndp whole query tiles, then ntail tiles cut into ksplit KV parts
  // each; a cut tile's parts leave fp32 partials in part[ntail * ksplit][kPartFloats],
  // which prefill_merge_kernel merges.
  int ndp, ntail, ksplit;
  float *part;
};

namespace {

__device__ __forceinline__ bool chunk_ok(const PrefillParams &p, int s) {
  return s >= 0 && static_cast<long long>(s) + p.T <= p.max_seq;
}

// Cache row of token position pos of sequence b, or -1 when its page id is out of range.
__device__ __forceinline__ long long cache_row_of(const PrefillParams &p, int b, int pos) {
  if (!p.paged) return static_cast<long long>(b) * p.max_seq + pos;
  const int pg = p.page_table[static_cast<long long>(b) * p.max_blocks + pos / kTile];
  if (pg < 0 || pg >= p.num_blocks) return -1;
  return static_cast<long long>(pg) * kTile + (pos & (kTile - 1));
}

}  // namespace

// ------------------------------------------------------------------------------ prologue
// One CTA per chunk token (blockIdx.x = b * T + i).  The token's query, key and value rows
// are contiguous in q/k/v_new, so one bulk copy each brings them into shared memory while
// the CTA computes cos/sin of the token's position; then warp w rotates rows w, w + 8, ...
// of the H_q query heads followed by the H_kv key heads (lane l holds dims 2l, 2l + 1,
// 2l + 64, 2l + 65) from shared memory.  The inputs are read before the wait on the
// preceding kernel; `out` and the cache are written after it.
__global__ void __launch_bounds__(256, 6) prefill_rope_kernel(const PrefillParams p) {
  __shared__ float4 cs[kHeadDim / 2];  // (cos_hi, sin_hi, cos_lo, sin_lo) of pair i
  __shared__ __align__(8) uint64_t rows_bar;
  extern __shared__ __align__(16) uint8_t rope_rows[];  // [H_q + 2 H_kv][128] bf16: q, k, v rows
  griddep_launch_dependents();
  const int b = blockIdx.x / p.T, i = blockIdx.x - b * p.T;
  const int s = p.q_start[b];
  const bool ok = chunk_ok(p, s);
  const long long tok = static_cast<long long>(b) * p.T + i;
  const uint32_t qbytes = static_cast<uint32_t>(p.Hq) * kHeadDim * 2, kvbytes = static_cast<uint32_t>(p.Hkv) * kHeadDim * 2;
  const uint32_t bar = smem_addr(&rows_bar);
  if (threadIdx.x == 0 && ok) {
    mbar_init(bar, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(bar, qbytes + 2 * kvbytes);
    bulk_load(smem_addr(rope_rows), p.q_new + tok * p.Hq * kHeadDim, qbytes, bar);
    bulk_load(smem_addr(rope_rows) + qbytes, p.k_new + tok * p.Hkv * kHeadDim, kvbytes, bar);
    bulk_load(smem_addr(rope_rows) + qbytes + kvbytes, p.v_new + tok * p.Hkv * kHeadDim, kvbytes, bar);
  }
  const int pos = s + i;
  if (ok && threadIdx.x < kHeadDim / 2) {
    double sv, cv;
    sincos(static_cast<double>(pos) * p.inv_freq[threadIdx.x], &sv, &cv);
    const float ch = static_cast<float>(cv), sh = static_cast<float>(sv);
    cs[threadIdx.x] = make_float4(ch, sh, static_cast<float>(cv - ch), static_cast<float>(sv - sh));
  }
  griddep_wait();  // `out` and the cache rows are written below
  if (!ok) {
    // a chunk outside [0, max_seq_len): flagged, nothing appended, zeros for its output
    // (the attention kernel gives it no work)
    if (i == 0 && threadIdx.x == 0) atomicOr(p.err, s < 0 ? GQA_DEVERR_POSITION : GQA_DEVERR_SEQLEN);
    uint4 *dst = reinterpret_cast<uint4 *>(p.out + tok * p.Hq * kHeadDim);
    for (int c = threadIdx.x; c < p.Hq * kHeadDim / 8; c += blockDim.x) dst[c] = make_uint4(0, 0, 0, 0);
    return;
  }
  __syncthreads();  // cos/sin (and the barrier's initialisation) visible
  const bool landed = mbar_wait(bar, 0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (!__all_sync(0xffffffffu, landed)) {  // the row copies never arrived: flag, write nothing
    if (lane == 0) atomicOr(p.err, GQA_DEVERR_TIMEOUT);
    return;
  }
  const long long crow = cache_row_of(p, b, pos);
  if (crow < 0 && threadIdx.x == 0) atomicOr(p.err, GQA_DEVERR_PAGE);
  // Lane l holds dims 2l, 2l + 1 and their RoPE partners 2l + 64, 2l + 65 of a row (one
  // 32-bit word each half), so that a row is read and written in two 32-bit accesses a lane
  // and both pairs stay in the lane.
  const float4 c0 = cs[2 * lane], c1 = cs[2 * lane + 1];
  const uint32_t *rw = reinterpret_cast<const uint32_t *>(rope_rows);  // [row][64] bf16 pairs
  uint32_t qw0 = 0u, qw1 = 0u, kw0 = 0u, kw1 = 0u;  // the norm weights of the lane's dims
  if (p.q_norm_w) {
    qw0 = reinterpret_cast<const uint32_t *>(p.q_norm_w)[lane];
    qw1 = reinterpret_cast<const uint32_t *>(p.q_norm_w)[32 + lane];
  }
  if (p.k_norm_w) {
    kw0 = reinterpret_cast<const uint32_t *>(p.k_norm_w)[lane];
    kw1 = reinterpret_cast<const uint32_t *>(p.k_norm_w)[32 + lane];
  }
  for (int r = warp; r < p.Hq + p.Hkv; r += 8) {
    if (r < p.Hq) {
      // query row: binary32, one bf16 rounding (it is not stored in the cache)
      const uint32_t a = rw[r * 64 + lane], c = rw[r * 64 + 32 + lane];
      const float x[4] = {bf16_lo_to_float(a), bf16_hi_to_float(a), bf16_lo_to_float(c), bf16_hi_to_float(c)};
      float ss = 0.f;
#pragma unroll
      for (int t = 0; t < 4; ++t) ss = fmaf(x[t], x[t], ss);
      float y[4];
      if (p.q_norm_w) {
        y[0] = x[0] * bf16_lo_to_float(qw0), y[1] = x[1] * bf16_hi_to_float(qw0);
        y[2] = x[2] * bf16_lo_to_float(qw1), y[3] = x[3] * bf16_hi_to_float(qw1);
      } else {
#pragma unroll
        for (int t = 0; t < 4; ++t) y[t] = x[t];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float rn = p.q_norm_w ? 1.0f / sqrtf(ss * (1.0f / 128.0f) + p.eps) : 1.0f;
      const float z0 = rn * fmaf(y[0], c0.x, -y[2] * c0.y), z2 = rn * fmaf(y[2], c0.x, y[0] * c0.y);
      const float z1 = rn * fmaf(y[1], c1.x, -y[3] * c1.y), z3 = rn * fmaf(y[3], c1.x, y[1] * c1.y);
      uint32_t *dst = reinterpret_cast<uint32_t *>(p.out + (tok * p.Hq + r) * kHeadDim);
      dst[lane] = pack_bf16(z0, z1);
      dst[32 + lane] = pack_bf16(z2, z3);
    } else if (crow >= 0) {
      const int kv = r - p.Hq;
      const uint32_t a = rw[(p.Hq + kv) * 64 + lane], c = rw[(p.Hq + kv) * 64 + 32 + lane];
      const uint16_t x[4] = {static_cast<uint16_t>(a & 0xffffu), static_cast<uint16_t>(a >> 16),
                             static_cast<uint16_t>(c & 0xffffu), static_cast<uint16_t>(c >> 16)};
      const uint16_t w[4] = {static_cast<uint16_t>(kw0 & 0xffffu), static_cast<uint16_t>(kw0 >> 16),
                             static_cast<uint16_t>(kw1 & 0xffffu), static_cast<uint16_t>(kw1 >> 16)};
      uint16_t kz[4];
      rotate_row_k(x, w, p.k_norm_w != nullptr, p.eps, c0, c1, kz);
      uint32_t *kd = reinterpret_cast<uint32_t *>(p.k_cache + (crow * p.Hkv + kv) * kHeadDim);
      uint32_t *vd = reinterpret_cast<uint32_t *>(p.v_cache + (crow * p.Hkv + kv) * kHeadDim);
      kd[lane] = static_cast<uint32_t>(kz[0]) | (static_cast<uint32_t>(kz[1]) << 16);
      kd[32 + lane] = static_cast<uint32_t>(kz[2]) | (static_cast<uint32_t>(kz[3]) << 16);
      vd[lane] = rw[(p.Hq + p.Hkv + kv) * 64 + lane];
      vd[32 + lane] = rw[(p.Hq + p.Hkv + kv) * 64 + 32 + lane];
    }
  }
}

// ----------------------------------------------------------------------------- attention
__global__ void __launch_bounds__(kPfThreads, kPfCtasPerSm)
    prefill_attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_addr(smem_raw) & 1023u) != 0u) {  // a launch assumption broken: no work at all
    if (threadIdx.x == 0) atomicOr(p.err, GQA_DEVERR_LAUNCH);
    return;
  }
  uint8_t *smem = smem_raw;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
  uint64_t *q_full = bars;
  uint64_t *k_full = bars + 1;
  uint64_t *k_empty = k_full + kPfKStages;
  uint64_t *v_full = k_empty + kPfKStages;
  uint64_t *v_empty = v_full + kPfVStages;
  uint64_t *s_full = v_empty + kPfVStages;
  uint64_t *p_full = s_full + 2;
  uint64_t *o_done = p_full + 2;
  uint64_t *drain = o_done + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBars);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Work item: query tiles in decreasing order of their key count (query blocks from the
  // last to the first), so that the longest start first.  The first ndp items are whole
  // tiles; the rest are the KV parts of the last ntail tiles -- the final partial round of
  // CTA slots -- which fill the slots that free up first.
  const int x = static_cast<int>(blockIdx.x);
  int tile = x, part = 0;
  if (x >= p.ndp) {
    tile = p.ndp + (x - p.ndp) / p.ksplit;
    part = (x - p.ndp) % p.ksplit;
  }
  const bool split = x >= p.ndp;
  const int bk = p.B * p.Hkv;
  const int qb = p.nqb - 1 - tile / bk;
  const int rem = tile % bk;
  const int b = rem / p.Hkv, kv = rem - b * p.Hkv;
  const int t0 = qb * p.Tt;                       // first chunk token of the block
  const int t_end = min(t0 + p.Tt, p.T);          // one past its last

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i)  // p_full collects one arrival per softmax warp
      mbar_init(smem_addr(&bars[i]), (&bars[i] == &p_full[0] || &bars[i] == &p_full[1]) ? kPfSoftmaxWarps : 1);
    fence_barrier_init();
  }
  if (warp == kPfProducerWarp && lane == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  if (warp == kPfMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), kPfTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Everything below reads what the prologue kernel wrote (the rotated queries in `out`,
  // the appended cache rows).
  griddep_wait();
  const int s0 = p.q_start[b];
  const bool seq_ok = chunk_ok(p, s0);
  // KV tiles the block needs: up to the one holding its last query's position; the
  // tiles after it are wholly in the future of every query and are never loaded.
  const int kmax = s0 + t_end - 1;
  const int n = seq_ok ? kmax / kTile + 1 : 0;  // 0: the prologue kernel wrote its zeros
  // this item's KV tiles [j0, j1) of the n (a part of a cut tile may be empty)
  const int j0 = split ? n * part / p.ksplit : 0, j1 = split ? n * (part + 1) / p.ksplit : n;
  const int nt = j1 - j0;
  uint8_t *const qs = smem + kOffQ;
  auto k_ptr = [&](int s) { return smem + kOffK + s * kKvTileBytes; };
  auto v_ptr = [&](int s) { return smem + kOffV + s * kKvTileBytes; };

  if (warp == kPfProducerWarp) {
    // ------------------------------------------------------------------ TMA producer
    // Order: K_0, V_0, K_1, V_1, ... -- each V tile goes out with its K tile, so that it has
    // landed by the time its P is ready (the V ring is one stage deeper than the K ring,
    // since a V tile is held until P V).
    if (lane == 0 && nt > 0) {
      const uint32_t qb_bytes = 2u * 64u * 2u * static_cast<uint32_t>(p.G * p.Tt);
      mbar_arrive_expect_tx(smem_addr(q_full), qb_bytes);
      tma_load_4d(smem_addr(qs), &tmQ, smem_addr(q_full), 0, kv * p.G, t0, b);
      tma_load_4d(smem_addr(qs + kPfRows * kHalfRowBytes), &tmQ, smem_addr(q_full), 64, kv * p.G, t0, b);
      auto row_of = [&](int j) {
        if (!p.paged) return b * p.max_seq + j * kTile;
        const int pg = p.page_table[static_cast<long long>(b) * p.max_blocks + j];
        if (pg < 0 || pg >= p.num_blocks) {
          atomicOr(p.err, GQA_DEVERR_PAGE);
          return -kTile;  // the whole box out of bounds: TMA fills zeros
        }
        return pg * kTile;
      };
      int kissued = 0, vissued = 0;
      bool ok = true;
      // i counts the item's KV tiles (stages and phases), j = j0 + i is the tile
      auto load_k = [&](int i) -> bool {
        const int s = i % kPfKStages;
        if (i >= kPfKStages && !mbar_wait(smem_addr(&k_empty[s]), static_cast<uint32_t>((i / kPfKStages - 1) & 1)))
          return false;
        const int row = row_of(j0 + i);
        const uint32_t fb = smem_addr(&k_full[s]), base = smem_addr(k_ptr(s));
        mbar_arrive_expect_tx(fb, 2 * kHalfTileBytes);
        tma_load_3d(base, &tmK, fb, 0, kv, row);
        tma_load_3d(base + kHalfTileBytes, &tmK, fb, 64, kv, row);
        kissued = i + 1;
        return true;
      };
      auto load_v = [&](int i) -> bool {
        const int s = i % kPfVStages;
        if (i >= kPfVStages && !mbar_wait(smem_addr(&v_empty[s]), static_cast<uint32_t>((i / kPfVStages - 1) & 1)))
          return false;
        const int row = row_of(j0 + i);
        const uint32_t fb = smem_addr(&v_full[s]), base = smem_addr(v_ptr(s));
        mbar_arrive_expect_tx(fb, 2 * kHalfTileBytes);
        tma_load_3d(base, &tmV, fb, 0, kv, row);
        tma_load_3d(base + kHalfTileBytes, &tmV, fb, 64, kv, row);
        vissued = i + 1;
        return true;
      };
      for (int i = 0; i < nt && ok; ++i) {
        ok = load_k(i);
        if (ok) ok = load_v(i);
      }
      if (!ok) {
        atomicOr(p.err, GQA_DEVERR_TIMEOUT);
        // Do not leave while copies into this CTA's shared memory may still be in flight.
        (void)mbar_wait(smem_addr(q_full), 0);
        for (int j = (kissued > kPfKStages ? kissued - kPfKStages : 0); j < kissued; ++j)
          (void)mbar_wait(smem_addr(&k_full[j % kPfKStages]), static_cast<uint32_t>((j / kPfKStages) & 1));
        for (int j = (vissued > kPfVStages ? vissued - kPfVStages : 0); j < vissued; ++j)
          (void)mbar_wait(smem_addr(&v_full[j % kPfVStages]), static_cast<uint32_t>((j / kPfVStages) & 1));
      }
    }
  } else if (warp == kPfMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    // Issue order: S_0, S_1, PV_0, S_2, PV_1, ...  S_j overwrites the buffer that held
    // P_{j-2}; P_{j-2} V was issued before it and the tensor pipe runs them in order.
    if (lane == 0 && nt > 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(kPfRows, kTile, false, false);
      constexpr uint32_t kIdO = idesc_bf16_f32(kPfRows, kHeadDim, false, true);
      const uint32_t qa = smem_addr(qs);
      bool ok = mbar_wait(smem_addr(q_full), 0);
      // O += P_t V_t (hi then lo part of P, read from tensor memory), then release V_t
      // and mark O current.
      auto issue_pv = [&](int t) -> bool {
        const int pb = t & 1, s = t % kPfVStages;
        if (!mbar_wait(smem_addr(&v_full[s]), static_cast<uint32_t>((t / kPfVStages) & 1))) return false;
        if (!mbar_wait(smem_addr(&p_full[pb]), static_cast<uint32_t>((t >> 1) & 1))) return false;
        tc_fence_after();
        const uint32_t va = smem_addr(v_ptr(s));
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k)
          umma_bf16_ts(tmem + kTmemO, tmem + 64 * pb + 8 * k, sdesc_sw128(va + 2048 * k, kHalfTileBytes, 1024), kIdO,
                       (t > 0 || k > 0) ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k)
          umma_bf16_ts(tmem + kTmemO, tmem + 64 * pb + 32 + 8 * k, sdesc_sw128(va + 2048 * k, kHalfTileBytes, 1024),
                       kIdO, 1u);
        umma_commit(smem_addr(&v_empty[s]));
        umma_commit(smem_addr(o_done));
        return true;
      };
      for (int j = 0; j < nt && ok; ++j) {  // j counts the item's KV tiles
        const int s = j % kPfKStages, sb = j & 1;
        ok = mbar_wait(smem_addr(&k_full[s]), static_cast<uint32_t>((j / kPfKStages) & 1));
        if (!ok) break;
        tc_fence_after();
        const uint32_t ka = smem_addr(k_ptr(s));
#pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k)
          umma_bf16(tmem + 64 * sb, sdesc_sw128(qa + (k >> 2) * (kPfRows * kHalfRowBytes) + 32 * (k & 3), 16, 1024),
                    sdesc_sw128(ka + (k >> 2) * kHalfTileBytes + 32 * (k & 3), 16, 1024), kIdS, k > 0 ? 1u : 0u);
        umma_commit(smem_addr(&k_empty[s]));
        umma_commit(smem_addr(&s_full[sb]));
        if (j >= 1) ok = issue_pv(j - 1);
      }
      if (ok) ok = issue_pv(nt - 1);
      if (!ok) atomicOr(p.err, GQA_DEVERR_TIMEOUT);
      umma_commit(smem_addr(drain));  // lets the teardown wait for every MMA issued
    }
  } else {
    // ------------------------------------------------------------------ softmax warps
    const int row = warp * 32 + lane;
    const int tl = row / p.G, g = row - tl * p.G;
    const int t = t0 + tl;
    const bool in_block = tl < p.Tt && t < t_end;
    const bool valid = in_block && seq_ok;
    const int qpos = valid ? s0 + t : -1;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float m_run = valid ? -INFINITY : 0.f;  // invalid rows: every score masked, P = 0
    float l_run = 0.f;
    bool ok = true;
    for (int i = 0; i < nt; ++i) {  // i counts the item's KV tiles, j is the tile
      const int j = j0 + i, sb = i & 1;
      ok = mbar_wait(smem_addr(&s_full[sb]), static_cast<uint32_t>((i >> 1) & 1));
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[64];
      {
        float a[32], c[32];
        tmem_ld32(tmem + lane_base + 64 * sb, a);
        tmem_ld32(tmem + lane_base + 64 * sb + 32, c);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          sv[e] = a[e];
          sv[32 + e] = c[e];
        }
      }

      // The causal mask -- key j*64 + c is visible iff <= qpos -- only on tiles that some
      // row of the warp does not see whole (the partial tiles of the page's tile classes).
      const int klim = qpos - j * kTile;  // last visible column (may be >= 64 or < 0)
      if (!__all_sync(0xffffffffu, klim >= kTile - 1)) {
#pragma unroll
        for (int c = 0; c < 64; ++c) sv[c] = c <= klim ? sv[c] : -INFINITY;
      }
      float m8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) m8[e] = fmaxf(sv[e], sv[e + 8]);
#pragma unroll
      for (int c = 16; c < 64; c += 8)
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = fmaxf(m8[e], sv[c + e]);
      const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      // scores in log2 units: s * scale_log2 (a positive scale keeps the maximum's place)
      const float m_new = fmaxf(m_run, mx * p.scale_log2);
      float corr = 1.f;
      bool resc = false;
      if (m_new > m_run + kRescaleLog2) {
        corr = fast_exp2(m_run - m_new);  // m_run = -inf before the row's first visible key: 0
        m_run = m_new;
        l_run *= corr;
        resc = i > 0;
      }
      if (__any_sync(0xffffffffu, resc)) {
        // O must hold P_0..P_{j-1} V before it is scaled: wait for the last P V.  (S_j was
        // issued after P_{j-2} V, so o_done has completed that phase: the parity wait
        // below is never more than one phase ahead of the barrier.)
        ok = mbar_wait(smem_addr(o_done), static_cast<uint32_t>((i - 1) & 1));
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          float o[32];
          tmem_ld32(tmem + lane_base + kTmemO + 32 * c4, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= corr;
          tmem_st32(tmem + lane_base + kTmemO + 32 * c4, o);
        }
      }

      // P = 2^(s - m) as bf16 hi + lo pairs into the S buffer's columns
      uint32_t ph[32], pl[32];
      float rs8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      // (a row that has seen no visible key yet -- in a part that starts past its position --
      // keeps m = -inf and gets P = 0)
      const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float v0 = fast_exp2(fmaf(sv[2 * c], p.scale_log2, neg_m));
        const float v1 = fast_exp2(fmaf(sv[2 * c + 1], p.scale_log2, neg_m));
        rs8[c & 7] += v0 + v1;
        ph[c] = pack_bf16(v0, v1);
        pl[c] = pack_bf16(v0 - bf16_lo_to_float(ph[c]), v1 - bf16_hi_to_float(ph[c]));
      }
      tmem_st32(tmem + lane_base + 64 * sb, ph);
      tmem_st32(tmem + lane_base + 64 * sb + 32, pl);
      l_run += ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));

      // The last tile may hold cache rows past the block's last query, which nothing
      // has written: zero those V rows so that P = 0 never meets a non-finite value.
      if (j == n - 1) {
        const int vz = kmax - j * kTile + 1;  // first row to clear
        if (vz < kTile) {
          const int s = i % kPfVStages;
          (void)mbar_wait(smem_addr(&v_full[s]), static_cast<uint32_t>((i / kPfVStages) & 1));
          uint4 *v0 = reinterpret_cast<uint4 *>(v_ptr(s));
          uint4 *v1 = reinterpret_cast<uint4 *>(v_ptr(s) + kHalfTileBytes);
          for (int c = vz * 8 + row; c < kTile * 8; c += kPfRows) {
            v0[c] = make_uint4(0, 0, 0, 0);
            v1[c] = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&p_full[sb]));
    }
    if (!ok && lane == 0) atomicOr(p.err, GQA_DEVERR_TIMEOUT);

    // epilogue: O / l as bf16 into this row's output, or, for a part of a cut tile, its
    // partial and the merge
    griddep_launch_dependents();
    // The final O is complete when the MMA thread's last commit (`drain`, one phase) fires.
    // (o_done cannot say it: when the last S has been read, the P V before the last one may
    // still be running, so o_done can be two phases behind, where a parity wait is
    // ambiguous.)
    bool have_o = false;
    if (ok && nt > 0) {
      const bool done = mbar_wait(smem_addr(drain), 0);
      have_o = __all_sync(0xffffffffu, done);
      if (!have_o && lane == 0) atomicOr(p.err, GQA_DEVERR_TIMEOUT);
    }
    if (have_o) tc_fence_after();
    uint16_t *dst = p.out + ((static_cast<long long>(b) * p.T + t) * p.Hq + kv * p.G + g) * kHeadDim;
    if (nt > 0 && !split) {
      const float inv = (valid && l_run > 0.f) ? 1.f / l_run : 0.f;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float o[32];
        if (have_o) {
          tmem_ld32(tmem + lane_base + kTmemO + 32 * c4, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0.f;
        }
        if (in_block) {
          uint4 *d4 = reinterpret_cast<uint4 *>(dst + 32 * c4);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            d4[q] = make_uint4(pack_bf16(o[8 * q] * inv, o[8 * q + 1] * inv),
                               pack_bf16(o[8 * q + 2] * inv, o[8 * q + 3] * inv),
                               pack_bf16(o[8 * q + 4] * inv, o[8 * q + 5] * inv),
                               pack_bf16(o[8 * q + 6] * inv, o[8 * q + 7] * inv));
        }
      }
    } else if (nt > 0) {
      // A part of a cut tile: leave (O, m, l) in its slot for prefill_merge_kernel.
      float *mine = p.part + (static_cast<long long>(tile - p.ndp) * p.ksplit + part) * kPartFloats;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float o[32];
        if (have_o) {
          tmem_ld32(tmem + lane_base + kTmemO + 32 * c4, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) mine[(32 * c4 + e) * kPfRows + row] = o[e];
      }
      mine[kHeadDim * kPfRows + row] = m_run;
      mine[(kHeadDim + 1) * kPfRows + row] = have_o ? l_run : 0.f;
    }
  }

  // ------------------------------------------------------------------ teardown
  __syncwarp();  // the producer and MMA warps ran their loops on lane 0 alone
  tc_fence_before();
  __syncthreads();
  if (warp == kPfMmaWarp) {
    tc_fence_after();
    if (nt > 0) (void)mbar_wait(smem_addr(drain), 0);
    __syncwarp();
    tmem_dealloc(tmem, kPfTmemCols);
  }
}

// ------------------------------------------------------------------------------ merge
// One CTA per (cut query tile r, 16 dims); a thread takes four consecutive rows of the
// tile's 128-row M tile (row = token-in-block * G + head, as in the attention kernel) and
// four dims, so that every partial it reads is a 16-byte vector of the column-major
// partials (a warp reads 512 contiguous bytes).  It waits for the attention kernel, weighs
// the non-empty parts of each row -- w_k = 2^(m_k - M) / L with M = max m_k,
// L = sum 2^(m_k - M) l_k -- and writes its dims of the rows in bf16.  All of a thread's
// loads are issued before the sums.
constexpr int kPfMergeDims = 16;                                      // dims a merge CTA covers
constexpr int kPfMergeThreads = (kPfRows / 4) * (kPfMergeDims / 4);  // 128
__device__ __forceinline__ float f4_at(const float4 &v, int k) {
  return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}
__global__ void __launch_bounds__(kPfMergeThreads) prefill_merge_kernel(const PrefillParams p) {
  griddep_wait();  // the attention kernel's partials
  const int r = static_cast<int>(blockIdx.x);
  const int r0 = 4 * (static_cast<int>(threadIdx.x) % (kPfRows / 4));  // rows r0 .. r0 + 3
  const int d0 = kPfMergeDims * static_cast<int>(blockIdx.y) + 4 * (static_cast<int>(threadIdx.x) / (kPfRows / 4));
  const int tile = p.ndp + r;
  const int bk = p.B * p.Hkv;
  const int qb = p.nqb - 1 - tile / bk;
  const int rem = tile % bk;
  const int b = rem / p.Hkv, kv = rem - b * p.Hkv;
  const int t0 = qb * p.Tt, t_end = min(t0 + p.Tt, p.T);
  const int s0 = p.q_start[b];
  if (!chunk_ok(p, s0)) return;  // the prologue wrote this chunk's zeros
  const int n = (s0 + t_end - 1) / kTile + 1;  // the tile's KV tiles, cut into ksplit parts
  auto slot = [&](int pt) { return p.part + (static_cast<long long>(r) * p.ksplit + pt) * kPartFloats; };
  float4 mv[kPfMaxSplit], lv[kPfMaxSplit], x[kPfMaxSplit][4];
  const float4 none_m = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY), zero = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int pt = 0; pt < kPfMaxSplit; ++pt) {  // every load first: (m, l) and the four dims, four rows each
    const bool has = pt < p.ksplit && n * pt / p.ksplit < n * (pt + 1) / p.ksplit;
    const float *sp = slot(pt < p.ksplit ? pt : 0);
    mv[pt] = has ? __ldcg(reinterpret_cast<const float4 *>(sp + kHeadDim * kPfRows + r0)) : none_m;
    lv[pt] = has ? __ldcg(reinterpret_cast<const float4 *>(sp + (kHeadDim + 1) * kPfRows + r0)) : zero;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      x[pt][e] = has ? __ldcg(reinterpret_cast<const float4 *>(sp + (d0 + e) * kPfRows + r0)) : zero;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {  // row r0 + k
    const int row = r0 + k;
    const int tl = row / p.G, g = row - tl * p.G, t = t0 + tl;
    float M = -INFINITY;
#pragma unroll
    for (int pt = 0; pt < kPfMaxSplit; ++pt)  // a part that saw none of the row's keys has l = 0
      if (f4_at(lv[pt], k) > 0.f) M = fmaxf(M, f4_at(mv[pt], k));
    float L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int pt = 0; pt < kPfMaxSplit; ++pt) {
      const float l = f4_at(lv[pt], k);
      const float f = l > 0.f ? fast_exp2(f4_at(mv[pt], k) - M) : 0.f;
      L += f * l;
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[e] = fmaf(f, f4_at(x[pt][e], k), acc[e]);
    }
    if (tl < p.Tt && t < t_end) {
      const float inv = L > 0.f ? 1.f / L : 0.f;
      uint16_t *dst = p.out + ((static_cast<long long>(b) * p.T + t) * p.Hq + kv * p.G + g) * kHeadDim + d0;
      *reinterpret_cast<uint2 *>(dst) =
          make_uint2(pack_bf16(acc[0] * inv, acc[1] * inv), pack_bf16(acc[2] * inv, acc[3] * inv));
    }
  }
}

// --------------------------------------------------------------------------- host side

namespace {

std::mutex g_pf_mu;
struct PfDevice {
  bool configured = false;
  int sms = 0;
  float *part = nullptr;
};
PfDevice g_pf_dev[64];

gqa_status_t check_desc(const gqa_prefill_desc_t &d) {
  if (d.head_dim != kHeadDim) return GQA_ERR_UNSUPPORTED;
  if (d.batch < 1 || d.batch > GQA_MAX_BATCH || d.num_q_heads < 1 || d.num_kv_heads < 1 || d.chunk_len < 1 ||
      d.max_seq_len < 1 || d.chunk_len > d.max_seq_len)
    return GQA_ERR_INVALID_ARG;
  if (d.num_q_heads % d.num_kv_heads != 0) return GQA_ERR_UNSUPPORTED;
  if (d.num_q_heads / d.num_kv_heads > GQA_MAX_GROUP) return GQA_ERR_UNSUPPORTED;
  if (d.block_size != 0 && d.block_size != GQA_BLOCK_SIZE) return GQA_ERR_UNSUPPORTED;
  if (d.block_size > 0 && d.num_cache_blocks < 1) return GQA_ERR_INVALID_ARG;
  const long long rows = d.block_size > 0 ? static_cast<long long>(d.num_cache_blocks) * kTile
                                          : static_cast<long long>(d.batch) * d.max_seq_len;
  if (rows > 0x7fffffffLL) return GQA_ERR_UNSUPPORTED;  // TMA row coordinates are int32
  if (static_cast<long long>(d.num_q_heads + 2 * d.num_kv_heads) * kHeadDim * 2 > kRopeMaxSmem)
    return GQA_ERR_UNSUPPORTED;  // a token's rows must fit the prologue's shared memory
  return GQA_OK;
}

bool aligned_to(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

// A per-call error word when the caller passes none (nothing reads it).
static __device__ uint32_t g_prefill_err_sink;
// Partials of the query tiles cut into KV parts.
static __device__ __align__(16) float g_pf_part[kPfMaxSlots * kPartFloats];

}  // namespace gqa

using namespace gqa;

extern "C" gqa_status_t gqa_prefill_attn(const gqa_prefill_desc_t *desc, const void *q_new, const void *k_new,
                                         const void *v_new, void *k_cache, void *v_cache, const int32_t *page_table,
                                         const int32_t *q_start, const void *q_norm_w, const void *k_norm_w,
                                         float rope_theta, float eps, void *out, uint32_t *device_errors,
                                         void *stream) {
  if (!desc) return GQA_ERR_INVALID_ARG;
  const gqa_prefill_desc_t d = *desc;
  gqa_status_t st = check_desc(d);
  if (st != GQA_OK) return st;
  if (!q_new || !k_new || !v_new || !k_cache || !v_cache || !q_start || !out) return GQA_ERR_INVALID_ARG;
  const bool paged = d.block_size > 0;
  if (paged != (page_table != nullptr)) return GQA_ERR_INVALID_ARG;
  if (!(isfinite(rope_theta) && rope_theta > 0.f) || !isfinite(eps) || eps < 0.f) return GQA_ERR_INVALID_ARG;
  if (!aligned_to(q_new, 16) || !aligned_to(k_new, 16) || !aligned_to(v_new, 16) || !aligned_to(k_cache, 16) ||
      !aligned_to(v_cache, 16) || !aligned_to(out, 16) || !aligned_to(q_norm_w, 16) || !aligned_to(k_norm_w, 16) ||
      !aligned_to(page_table, 4) || !aligned_to(q_start, 4))
    return GQA_ERR_INVALID_ARG;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) return GQA_ERR_CUDA;
  if (d.device < 0 || d.device >= ndev) return GQA_ERR_INVALID_ARG;
  if (d.device >= 64) return GQA_ERR_UNSUPPORTED;
  DeviceGuard guard(d.device);
  if (!guard.ok) return GQA_ERR_CUDA;
  PfDevice dev;
  {
    // first call on the device: shared-memory limits, SM count, the split-tile scratch
    std::lock_guard<std::mutex> lk(g_pf_mu);
    PfDevice &pd = g_pf_dev[d.device];
    if (!pd.configured) {
      void *part = nullptr;
      if (cudaFuncSetAttribute(prefill_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
              cudaSuccess ||
          cudaFuncSetAttribute(prefill_rope_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRopeMaxSmem) !=
              cudaSuccess ||
          cudaFuncSetAttribute(prefill_attn_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
          cudaDeviceGetAttribute(&pd.sms, cudaDevAttrMultiProcessorCount, d.device) != cudaSuccess ||
          cudaGetSymbolAddress(&part, g_pf_part) != cudaSuccess) {
        cudaGetLastError();
        return GQA_ERR_CUDA;
      }
      pd.part = static_cast<float *>(part);
      pd.configured = true;
    }
    dev = pd;
  }
  uint32_t *err = device_errors;
  if (!err) {
    void *sink = nullptr;
    if (cudaGetSymbolAddress(&sink, g_prefill_err_sink) != cudaSuccess) {
      cudaGetLastError();
      return GQA_ERR_CUDA;
    }
    err = static_cast<uint32_t *>(sink);
  }

  PrefillParams p;
  memset(&p, 0, sizeof p);
  p.q_new = static_cast<const uint16_t *>(q_new);
  p.k_new = static_cast<const uint16_t *>(k_new);
  p.v_new = static_cast<const uint16_t *>(v_new);
  p.k_cache = static_cast<uint16_t *>(k_cache);
  p.v_cache = static_cast<uint16_t *>(v_cache);
  p.page_table = page_table;
  p.q_start = q_start;
  p.q_norm_w = static_cast<const uint16_t *>(q_norm_w);
  p.k_norm_w = static_cast<const uint16_t *>(k_norm_w);
  p.out = static_cast<uint16_t *>(out);
  p.err = err;
  p.part = dev.part;
  p.B = d.batch;
  p.T = d.chunk_len;
  p.Hq = d.num_q_heads;
  p.Hkv = d.num_kv_heads;
  p.G = d.num_q_heads / d.num_kv_heads;
  p.Tt = kPfRows / p.G;
  p.nqb = (p.T + p.Tt - 1) / p.Tt;
  // Work items: whole query tiles fill complete rounds of the CTA slots (two per SM); the
  // tiles of the last, partial round are cut into up to kPfMaxSplit KV parts each, so that
  // their parts fill the slots the whole tiles leave free (the cut tiles' partials must fit
  // the static scratch: ntail * ksplit <= kPfMaxSlots).
  {
    const long long tiles = static_cast<long long>(p.nqb) * p.B * p.Hkv;
    const long long slots = std::min<long long>(static_cast<long long>(dev.sms) * kPfCtasPerSm, kPfMaxSlots);
    const long long tail = tiles % slots;
    const long long k = tail > 0 ? std::min<long long>(kPfMaxSplit, slots / tail) : 1;
    if (k > 1) {
      p.ndp = static_cast<int>(tiles - tail);
      p.ntail = static_cast<int>(tail);
      p.ksplit = static_cast<int>(k);
    } else {
      p.ndp = static_cast<int>(tiles);
      p.ntail = 0;
      p.ksplit = 1;
    }
  }
  p.paged = paged ? 1 : 0;
  p.max_seq = d.max_seq_len;
  p.max_blocks = (d.max_seq_len + kTile - 1) / kTile;
  p.num_blocks = paged ? d.num_cache_blocks : 0;
  p.eps = eps;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(kHeadDim)));
  for (int i = 0; i < kHeadDim / 2; ++i)
    p.inv_freq[i] = pow(static_cast<double>(rope_theta), -2.0 * i / static_cast<double>(kHeadDim));

  const long long rows = paged ? static_cast<long long>(d.num_cache_blocks) * kTile
                               : static_cast<long long>(d.batch) * d.max_seq_len;
  CUtensorMap tq, tk, tv;
  // queries (in `out`) viewed as [B][T][H_q][128]; box = 64 dims x G heads x Tt tokens x 1
  const cuuint64_t qdims[4] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(p.Hq),
                               static_cast<cuuint64_t>(p.T), static_cast<cuuint64_t>(p.B)};
  const cuuint64_t qstrides[3] = {static_cast<cuuint64_t>(kHeadDim) * 2, static_cast<cuuint64_t>(p.Hq) * kHeadDim * 2,
                                  static_cast<cuuint64_t>(p.T) * p.Hq * kHeadDim * 2};
  const cuuint32_t qbox[4] = {64, static_cast<cuuint32_t>(p.G), static_cast<cuuint32_t>(p.Tt), 1};
  if (!encode_bf16_map(&tq, 4, out, qdims, qstrides, qbox) || !make_cache_map(&tk, k_cache, p.Hkv, rows) ||
      !make_cache_map(&tv, v_cache, p.Hkv, rows))
    return GQA_ERR_CUDA;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t rope_smem = static_cast<size_t>(p.Hq + 2 * p.Hkv) * kHeadDim * 2;
  if (launch_pdl(prefill_rope_kernel, dim3(static_cast<unsigned>(p.B * p.T)), dim3(256), rope_smem, s, p) !=
      cudaSuccess)
    return GQA_ERR_CUDA;
  const unsigned grid = static_cast<unsigned>(p.ndp + p.ntail * p.ksplit);
  if (launch_pdl(prefill_attn_kernel, dim3(grid), dim3(kPfThreads), static_cast<size_t>(kSmemBytes), s, tq, tk, tv,
                 p) != cudaSuccess)
    return GQA_ERR_CUDA;
  if (p.ntail > 0 && launch_pdl(prefill_merge_kernel, dim3(static_cast<unsigned>(p.ntail), kHeadDim / kPfMergeDims),
                                dim3(kPfMergeThreads), 0, s, p) != cudaSuccess)
    return GQA_ERR_CUDA;
  return GQA_OK;
}
