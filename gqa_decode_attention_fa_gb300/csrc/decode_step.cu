// The fused GQA decode step on sm_103a: QK-norm + RoPE, KV-cache append, split-KV
// attention and the log-sum-exp combine, in one kernel launch.
//
// What it computes, for every sequence b and query head h (KV head kv = h / G):
//   q = bf16(RoPE_p(RMSNorm(q_new))), k_row = bf16(RoPE_p(RMSNorm(k_new))) appended with
//   v_new at position p = positions[b], then out = softmax(q K^T / sqrt(d)) V over the
//   L_b cached tokens ("Qwen3-14B Optimization", section 2.1 Shape 4 and #796: QK-norm and
//   RoPE folded into the fused attention; section 3.3: the lo/hi RoPE halves;
//   "ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)", section 0.5.1: K cached
//   post-RoPE, V raw).  The attention is the FlashAttention per-tile recurrence of
//   ADR-0060 section 3 -- S = scale q K_j^T (masked past L_b), m' = max(m, rowmax S),
//   P = exp(S - m'), c = exp(m - m'), l = l c + rowsum P, O = O c + P V_j, seeded
//   m = -inf, l = 0, O = 0 with no peeled first iteration ("Qwen3-14B Optimization",
//   section 2.1 Shape 3) -- over split-KV pieces merged with the associative log-sum-exp
//   merge of ADR-0060 section 4 and normalised once (FlashDecoding).
//
// GB300 design:
//  * The G query heads sharing KV head kv are folded into one operand (ADR-0060 section
//    5.2, M-fold): one K/V tile serves all G heads.  Decode is KV-bandwidth bound, so the
//    fold is laid out token-major: S^T[64 tokens x 8*NT heads] = K_j[64 x 128] Q^T and
//    O^T[128 x 8*NT] += V_j^T P^T on legacy mma.sync m16n8k16 (bf16 in, fp32 accumulate):
//    G <= 8 pads to 8 columns, G <= 16 to 16.
//  * P enters the P.V product as bf16 hi + bf16 lo (two mma), so rounding P costs no
//    accuracy; the bf16 output rounding is the only sizeable error.
//  * One CTA per SM.  A producer warp streams 64-token K/V tiles (4 x 8 KiB boxes) with
//    3-D TMA loads (128-byte swizzle, no multicast) into a 6-stage mbarrier ring; six
//    consumer warps each own one stage and take every sixth tile.  A consumer rotates the
//    group's queries itself (binary32) whenever it enters a new (b, kv) segment, and the
//    consumer that owns the tile holding a sequence's new token appends the k row
//    (binary64, one bf16 rounding) and the v row to the cache and patches both into its
//    shared-memory tile (the TMA read the slot before the append).
//  * Workers own equal contiguous ranges of the batch's tiles (ADR-0060 section 2.1
//    placement applied to the whole batch), so ragged batches stay balanced.  At the end
//    each CTA merges its warps' partials per segment: a segment it holds entirely is
//    normalised and written out directly; a segment shared with neighbouring CTAs gets a
//    CTA partial and an arrival ticket, and the CTA that draws the last ticket merges the
//    segment's CTA partials (the reduce-to-root of ADR-0060 section 4 within one GPU).
//    Nothing waits on another CTA.
#include "launch.h"
#include "rowmath.cuh"

namespace gqa {

namespace {

// Largest b with pre[b] <= x; pre[] is non-decreasing with pre[B] > x.  The sequence
// found always has at least one tile.
__device__ __forceinline__ void locate(const uint32_t *pre, const int32_t *Ls, int B, int Hkv, long long x,
                                       int &b, int &kv, int &j) {
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<long long>(pre[mid]) <= x) lo = mid;
    else hi = mid;
  }
  b = lo;
  const int nt = (Ls[lo] + kTile - 1) / kTile;
  const int within = static_cast<int>(x - static_cast<long long>(pre[lo]));
  kv = within / nt;
  j = within - kv * nt;
}

template <int NT>
struct Cfg {
  static constexpr int kNpad = 8 * NT;
  static constexpr int kQBytes = kNpad * 256;              // one rotated-q tile (one ring slot)
  static constexpr int kRing = NT == 1 ? 2 * kStages : kStages;  // q ring slots (as many as fit)
  static constexpr int kStageBytes = 4 * kHalfTileBytes;   // K lo, K hi, V lo, V hi
  static constexpr int kQOffset = kStages * kStageBytes;
  static constexpr int kBarOffset = kQOffset + kRing * kQBytes;
  static_assert(kStageBytes % 1024 == 0 && kQOffset % 1024 == 0, "1024-byte alignment for the 128B swizzle");
};

__device__ __forceinline__ void consumer_barrier() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// Appends sequence b's new token for KV head kv: k = RoPE_pos(RMSNorm(k_new)) in binary64
// rounded once to bf16, v = v_new, written to the cache row of position pos (skipped when
// the page id is out of range; the producer flags that) and returned per lane (dims
// lane + 32 t) for the shared-memory patch.
__device__ __forceinline__ void append_new_row(const StepParams &p, int b, int kv, int pos, int lane,
                                               uint16_t (&kz)[4], uint16_t (&vz)[4]) {
  const long long nrow = (static_cast<long long>(b) * p.Hkv + kv) * kHeadDim;
  const double2 cs0 = p.rope_tab[static_cast<long long>(pos) * 64 + lane];
  const double2 cs1 = p.rope_tab[static_cast<long long>(pos) * 64 + lane + 32];
#pragma unroll
  for (int t = 0; t < 4; ++t) vz[t] = p.v_new[nrow + lane + 32 * t];
  rotate_row_fp64(p.k_new + nrow, p.k_norm_w, p.eps, cs0, cs1, lane, kz);
  long long grow = -1;
  if (p.paged) {
    const int pg = p.page_table[static_cast<long long>(b) * p.max_blocks + pos / kTile];
    if (pg >= 0 && pg < p.num_blocks) grow = static_cast<long long>(pg) * kTile + (pos & (kTile - 1));
  } else {
    grow = static_cast<long long>(b) * p.max_seq + pos;
  }
  if (grow >= 0) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      p.k_cache[(grow * p.Hkv + kv) * kHeadDim + lane + 32 * t] = kz[t];
      p.v_cache[(grow * p.Hkv + kv) * kHeadDim + lane + 32 * t] = vz[t];
    }
  }
}

// Rotated query row (segment sg = b * H_kv + kv, head g of the group) into q slot `slot`
// of the CTA's ring -- each slot a swizzled tile [half][npad rows][128 B] whose rows >= G
// stay zero -- and, with `publish`, into the diagnostic copy q_rot [B, Hq, d].
template <int NT>
__device__ __forceinline__ void store_q_row(const StepParams &p, uint8_t *qslots, int slot, int b, int kv, int g,
                                            const uint16_t (&z)[4], int lane, bool publish) {
  uint8_t *qbuf = qslots + slot * Cfg<NT>::kQBytes;
  const long long h = static_cast<long long>(b) * p.Hq + kv * p.G + g;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int e = lane + 32 * t;
    const uint32_t off = (e >> 6) * (Cfg<NT>::kNpad * 128) + swz128(g, (e & 63) >> 3) + (e & 7) * 2;
    *reinterpret_cast<uint16_t *>(qbuf + off) = z[t];
    if (publish) p.q_rot[h * kHeadDim + e] = z[t];
  }
}

// Rotates rows first, first + stride, ... (< nrows) of the segment run starting at
// seg_first (row r = segment seg_first + r / G, head r % G) into their ring slots.  BATCH
// rows' inputs are loaded before any is used, so the loads overlap.  A segment's rows are
// published when this CTA holds the segment's first tile.
template <int NT, int BATCH>
__device__ __forceinline__ void rotate_q_rows(const StepParams &p, const uint32_t *pre, const int32_t *Ls,
                                              int seg_first, int first, int stride, int nrows, long long xs,
                                              uint8_t *qslots, int lane) {
  for (int r0 = first; r0 < nrows; r0 += BATCH * stride) {
    uint16_t x[BATCH][4];
    float2 c0[BATCH], c1[BATCH];
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int r = r0 + u * stride;
      if (r < nrows) {
        const int sg = seg_first + r / p.G, g = r % p.G;
        const int b = sg / p.Hkv, kv = sg - b * p.Hkv;
        const int pos = Ls[b] > 0 ? p.positions[b] : 0;
        const uint16_t *src = p.q_new + ((static_cast<long long>(b) * p.Hq) + kv * p.G + g) * kHeadDim;
#pragma unroll
        for (int t = 0; t < 4; ++t) x[u][t] = src[lane + 32 * t];
        const double2 d0 = p.rope_tab[static_cast<long long>(pos) * 64 + lane];
        const double2 d1 = p.rope_tab[static_cast<long long>(pos) * 64 + lane + 32];
        c0[u] = make_float2(static_cast<float>(d0.x), static_cast<float>(d0.y));
        c1[u] = make_float2(static_cast<float>(d1.x), static_cast<float>(d1.y));
      }
    }
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int r = r0 + u * stride;
      if (r < nrows) {
        const int sg = seg_first + r / p.G, g = r % p.G;
        const int b = sg / p.Hkv, kv = sg - b * p.Hkv;
        if (Ls[b] <= 0) continue;  // a skipped sequence inside the run
        uint16_t z[4];
        rotate_row_fp32_regs(x[u], p.q_norm_w, static_cast<float>(p.eps), c0[u], c1[u], lane, z);
        const int nt = (Ls[b] + kTile - 1) / kTile;
        const long long beg = static_cast<long long>(pre[b]) + static_cast<long long>(kv) * nt;
        store_q_row<NT>(p, qslots, (sg - seg_first) % Cfg<NT>::kRing, b, kv, g, z, lane, beg >= xs);
      }
    }
  }
}

// Folds partial (m2, l2, o2) into the running (m, l, o) with the log-sum-exp merge
// (m in log2 units).
__device__ __forceinline__ void merge_into(float &m, float &l, float4 &o, float m2, float l2, float4 o2) {
  const float mn = fmaxf(m, m2);
  const float sa = exp2f(m - mn), sb = exp2f(m2 - mn);
  l = l * sa + l2 * sb;
  o.x = o.x * sa + o2.x * sb;
  o.y = o.y * sa + o2.y * sb;
  o.z = o.z * sa + o2.z * sb;
  o.w = o.w * sa + o2.w * sb;
  m = mn;
}

__device__ __forceinline__ void store_out4(uint16_t *dst, float4 o, float l) {
  const float inv = 1.0f / l;
  uint2 v;
  v.x = pack_bf16(o.x * inv, o.y * inv);
  v.y = pack_bf16(o.z * inv, o.w * inv);
  *reinterpret_cast<uint2 *>(dst) = v;
}

}  // namespace

template <int NT>
__global__ void __launch_bounds__(kThreadsAttn, 1)
    decode_step_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const StepParams p) {
  using C = Cfg<NT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + C::kBarOffset);
  uint64_t *empty_bar = full_bar + kStages;
  uint32_t *pre = reinterpret_cast<uint32_t *>(empty_bar + kStages);  // [B + 1]
  int32_t *Ls = reinterpret_cast<int32_t *>(pre + p.B + 1);           // [B], 0 = sequence skipped
  __shared__ int s_abort;
  __shared__ int s_last[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), 1);
    }
    fence_barrier_init();
    s_abort = 0;
  }
  if (warp == kConsumerWarps && lane == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  // Inputs may come from the previous kernel on the stream: read nothing before this.
  griddep_wait();
  if (warp == 0) {  // tile prefix over the batch; a sequence with a bad length or position is skipped
    uint32_t run = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int b = b0 + lane;
      uint32_t v = 0;
      if (b < p.B) {
        const int L = p.seq_lens[b], pos = p.positions[b];
        int nt = tiles_of(L, p.max_seq);
        uint32_t bad = 0;
        if (nt == 0) bad = GQA_DEVERR_SEQLEN;
        else if (pos < 0 || pos >= L) bad = GQA_DEVERR_POSITION;
        if (bad) {
          nt = 0;
          if (blockIdx.x == 0) atomicOr(p.err, bad);
        }
        Ls[b] = nt ? L : 0;
        v = static_cast<uint32_t>(nt) * static_cast<uint32_t>(p.Hkv);
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
      }
      if (b < p.B) pre[b + 1] = run + v;
      run += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) pre[0] = 0;
  }
  __syncthreads();
  griddep_launch_dependents();  // the next kernel may launch; it waits for this grid to finish

  // Skipped sequences get a zero output row.
  for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
    if (Ls[b] != 0) continue;
    uint16_t *o = p.out + static_cast<long long>(b) * p.Hq * kHeadDim;
    for (int i = tid; i < p.Hq * kHeadDim; i += blockDim.x) o[i] = 0;
  }

  const long long T = pre[p.B];
  const int W = gridDim.x, w = blockIdx.x;
  const long long xs = worker_begin(T, W, w), xe = worker_begin(T, W, w + 1);
  const long long n = xe - xs;
  if (n <= 0) return;

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------------- producer warp
    bool fail = false;
    long long issued = 0;
    for (long long i0 = 0; i0 < n && !fail; i0 += 32) {
      const long long i = i0 + lane;
      int row = 0, kv = 0;
      if (i < n) {
        int b, j;
        locate(pre, Ls, p.B, p.Hkv, xs + i, b, kv, j);
        if (p.paged) {
          const int pg = p.page_table[static_cast<long long>(b) * p.max_blocks + j];
          if (pg < 0 || pg >= p.num_blocks) {
            atomicOr(p.err, GQA_DEVERR_PAGE);
            row = -kTile;  // whole box out of bounds: TMA fills zeros
          } else {
            row = pg * kTile;
          }
        } else {
          row = b * p.max_seq + j * kTile;
        }
      }
      const int cnt = static_cast<int>(n - i0 < 32 ? n - i0 : 32);
      for (int k = 0; k < cnt; ++k) {
        const int r_row = __shfl_sync(0xffffffffu, row, k);
        const int r_kv = __shfl_sync(0xffffffffu, kv, k);
        const long long ii = i0 + k;
        const int s = static_cast<int>(ii % kStages);
        int ok = 1;
        if (lane == 0) {
          if (ii >= kStages)
            ok = mbar_wait(smem_addr(&empty_bar[s]), static_cast<uint32_t>(((ii / kStages) - 1) & 1));
          if (ok) {
            const uint32_t fb = smem_addr(&full_bar[s]);
            const uint32_t base = smem_addr(smem + s * C::kStageBytes);
            mbar_arrive_expect_tx(fb, C::kStageBytes);
            tma_load_3d(base, &tmK, fb, 0, r_kv, r_row);
            tma_load_3d(base + kHalfTileBytes, &tmK, fb, 64, r_kv, r_row);
            tma_load_3d(base + 2 * kHalfTileBytes, &tmV, fb, 0, r_kv, r_row);
            tma_load_3d(base + 3 * kHalfTileBytes, &tmV, fb, 64, r_kv, r_row);
            issued = ii + 1;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          fail = true;
          break;
        }
      }
    }
    if (fail && lane == 0) {
      atomicOr(p.err, GQA_DEVERR_TIMEOUT);
      s_abort = 1;
      // Do not leave while copies into this CTA's shared memory may still be in flight.
      for (long long ii = (issued > kStages ? issued - kStages : 0); ii < issued; ++ii)
        (void)mbar_wait(smem_addr(&full_bar[ii % kStages]), static_cast<uint32_t>((ii / kStages) & 1));
    }
    return;
  }

  // ------------------------------------------------------------------ consumer warps
  const int cw = warp;
  // The q ring: slot (seg - seg_first) % kRing holds the rotated queries of segment seg.
  // The first kRing segments are rotated up front by all consumer warps; a warp entering a
  // later segment rotates it into its slot only once it holds the segment's tile.  While a
  // warp holds tile i, no warp holds a tile outside [i - 5, i + 5] (the producer refills a
  // stage only after its owner releases it), and segments sharing a slot are at least
  // kRing - 1 >= 5 whole segments (>= 5 tiles) apart, so a slot is never rewritten while
  // another warp still reads it for an older segment.
  uint8_t *qslots = smem + C::kQOffset;
  int seg_first, seg_last;
  {
    int b0, kv0, j0, b1, kv1, j1;
    locate(pre, Ls, p.B, p.Hkv, xs, b0, kv0, j0);
    locate(pre, Ls, p.B, p.Hkv, xe - 1, b1, kv1, j1);
    seg_first = b0 * p.Hkv + kv0;
    seg_last = b1 * p.Hkv + kv1;
  }
  for (int i = tid; i < C::kRing * C::kQBytes / 16; i += kConsumerWarps * 32)
    reinterpret_cast<uint4 *>(qslots)[i] = make_uint4(0, 0, 0, 0);
  consumer_barrier();
  // The first kRing segments' queries are rotated by all consumer warps together while the
  // first tiles load.
  const int nseg_ring = min(seg_last - seg_first + 1, C::kRing);
  rotate_q_rows<NT, 8>(p, pre, Ls, seg_first, cw, kConsumerWarps, nseg_ring * p.G, xs, qslots, lane);

  // The new-token k/v rows this warp appends: the first two are computed now, while the
  // first tiles are still in flight, written to the cache and kept packed in registers for
  // the shared-memory patch; any further ones are computed when their tile arrives.
  long long ex0 = -1, ex1 = -1;
  uint32_t ek0[2] = {0, 0}, ev0[2] = {0, 0}, ek1[2] = {0, 0}, ev1[2] = {0, 0};
  {
    for (int sg = seg_first; sg <= seg_last && ex1 < 0; ++sg) {
      const int b = sg / p.Hkv, kv = sg - b * p.Hkv;
      const int L = Ls[b];
      if (L <= 0) continue;
      const int pos = p.positions[b];
      const int nt = (L + kTile - 1) / kTile;
      const long long x_new = static_cast<long long>(pre[b]) + static_cast<long long>(kv) * nt + pos / kTile;
      if (x_new < xs || x_new >= xe || (x_new - xs) % kConsumerWarps != cw) continue;
      uint16_t kz[4], vz[4];
      append_new_row(p, b, kv, pos, lane, kz, vz);
      uint32_t *ek = ex0 < 0 ? ek0 : ek1, *ev = ex0 < 0 ? ev0 : ev1;
      ek[0] = kz[0] | (uint32_t(kz[1]) << 16), ek[1] = kz[2] | (uint32_t(kz[3]) << 16);
      ev[0] = vz[0] | (uint32_t(vz[1]) << 16), ev[1] = vz[2] | (uint32_t(vz[3]) << 16);
      if (ex0 < 0) ex0 = x_new;
      else ex1 = x_new;
    }
  }
  consumer_barrier();  // the ring's first segments are rotated

  float o[8][NT][4];
  float m_run[NT][2], l_run[NT][2];
#pragma unroll
  for (int md = 0; md < 8; ++md)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[md][nt][e] = 0.f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      m_run[nt][jj] = -INFINITY;
      l_run[nt][jj] = 0.f;
    }

  // Writes this warp's (m, l, O) partial of segment seg and resets the running state.
  auto flush = [&](int seg) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        float l = l_run[nt][jj];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        l_run[nt][jj] = l;
      }
    const long long base_row = (static_cast<long long>(seg + w) * kConsumerWarps + cw) * p.G;
#pragma unroll
    for (int md = 0; md < 8; ++md)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int g = 8 * nt + 2 * (lane & 3) + (e & 1);
          const int d = 16 * md + (lane >> 2) + ((e >> 1) << 3);
          if (g < p.G) p.part_o[(base_row + g) * kHeadDim + d] = o[md][nt][e];
          o[md][nt][e] = 0.f;
        }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int g = 8 * nt + 2 * lane + jj;
        if (lane < 4 && g < p.G) {
          p.part_ml[(base_row + g) * 2 + 0] = m_run[nt][jj];
          p.part_ml[(base_row + g) * 2 + 1] = l_run[nt][jj];
        }
        m_run[nt][jj] = -INFINITY;
        l_run[nt][jj] = 0.f;
      }
  };

  int cur_seg = -1;
  for (long long i = cw; i < n; i += kConsumerWarps) {
    int b, kv, j;
    locate(pre, Ls, p.B, p.Hkv, xs + i, b, kv, j);
    const int seg = b * p.Hkv + kv;
    const int pos_b = p.positions[b];
    const bool entering = seg != cur_seg;
    if (entering) {
      if (cur_seg >= 0) flush(cur_seg);
      cur_seg = seg;
    }
    const int qslot = (seg - seg_first) % C::kRing;
    const int s = static_cast<int>(i % kStages);
    const bool ready = mbar_wait(smem_addr(&full_bar[s]), static_cast<uint32_t>((i / kStages) & 1));
    __syncwarp();  // reconverge before the warp-collective ldmatrix / mma below
    if (!__all_sync(0xffffffffu, ready)) {
      if (lane == 0) {
        atomicOr(p.err, GQA_DEVERR_TIMEOUT);
        s_abort = 1;
      }
      break;
    }
    if (entering && seg - seg_first >= C::kRing) {  // beyond the pre-rotated segments
      rotate_q_rows<NT, 2>(p, pre, Ls, seg, 0, 1, p.G, xs + i - j, qslots + qslot * C::kQBytes, lane);
      __syncwarp();
    }
    const int valid = min(kTile, Ls[b] - j * kTile);
    uint8_t *stage = smem + s * C::kStageBytes;
    const uint32_t kLo = smem_addr(stage), kHi = kLo + kHalfTileBytes;
    const uint32_t vLo = kLo + 2 * kHalfTileBytes, vHi = kLo + 3 * kHalfTileBytes;
    const uint32_t qS = smem_addr(qslots + qslot * C::kQBytes);

    if (valid < kTile) {
      // Rows past L_b hold whatever the cache holds there; zero the V rows so that
      // P = 0 never meets a non-finite value.  Whole 128-byte rows, so the swizzle
      // does not matter.
      uint4 *v0 = reinterpret_cast<uint4 *>(stage + 2 * kHalfTileBytes);
      uint4 *v1 = reinterpret_cast<uint4 *>(stage + 3 * kHalfTileBytes);
      const int nchunks = (kTile - valid) * 8;
      for (int c = lane; c < nchunks; c += 32) {
        v0[valid * 8 + c] = make_uint4(0, 0, 0, 0);
        v1[valid * 8 + c] = make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }
    // The tile holding sequence b's new token: the TMA may have read the slot before the
    // append, so patch the appended k and v rows into it.
    const bool holds_new = (pos_b >> 6) == j;
    if (holds_new) {
      uint16_t kz[4], vz[4];
      const long long x = xs + i;
      if (x == ex0 || x == ex1) {
        const uint32_t *k2 = x == ex0 ? ek0 : ek1, *v2 = x == ex0 ? ev0 : ev1;
        kz[0] = k2[0] & 0xffff, kz[1] = k2[0] >> 16, kz[2] = k2[1] & 0xffff, kz[3] = k2[1] >> 16;
        vz[0] = v2[0] & 0xffff, vz[1] = v2[0] >> 16, vz[2] = v2[1] & 0xffff, vz[3] = v2[1] >> 16;
      } else {
        append_new_row(p, b, kv, pos_b, lane, kz, vz);
      }
      const int r = pos_b & (kTile - 1);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int e = lane + 32 * t;
        const uint32_t off = (e >> 6) * kHalfTileBytes + swz128(r, (e & 63) >> 3) + (e & 7) * 2;
        *reinterpret_cast<uint16_t *>(stage + off) = kz[t];
        *reinterpret_cast<uint16_t *>(stage + 2 * kHalfTileBytes + off) = vz[t];
      }
      __syncwarp();
    }

    // q^T as the B operand: 8 k-steps (16 dims) x NT column tiles of 8 heads.
    uint32_t qf[8][NT][2];
#pragma unroll
    for (int ks2 = 0; ks2 < 4; ++ks2)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int chunk = 4 * ks2 + (lane >> 3);
        const int g = 8 * nt + (lane & 7);
        const uint32_t addr = qS + (chunk >> 3) * (C::kNpad * 128) + swz128(g, chunk & 7);
        ldsm_x4(addr, qf[2 * ks2][nt][0], qf[2 * ks2][nt][1], qf[2 * ks2 + 1][nt][0], qf[2 * ks2 + 1][nt][1]);
      }

    // S^T = K_j q^T : 4 token blocks of 16 x NT head blocks of 8.
    float sacc[4][NT][4];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[mt][nt][e] = 0.f;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int qd = lane >> 3;
        const int tok = 16 * mt + (lane & 7) + ((qd & 1) << 3);
        const int chunk = 2 * ks + (qd >> 1);
        const uint32_t addr = ((chunk >> 3) ? kHi : kLo) + swz128(tok, chunk & 7);
        uint32_t a0, a1, a2, a3;
        ldsm_x4(addr, a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16(sacc[mt][nt], a0, a1, a2, a3, qf[ks][nt][0], qf[ks][nt][1]);
      }

    // scale (log2 domain) and mask tokens >= valid
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = 16 * mt + (lane >> 2) + ((e >> 1) << 3);
          sacc[mt][nt][e] = tok < valid ? sacc[mt][nt][e] * p.scale_log2 : -INFINITY;
        }

    // online-softmax update per head column
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        float mx = -INFINITY;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) mx = fmaxf(mx, fmaxf(sacc[mt][nt][jj], sacc[mt][nt][jj + 2]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float m_new = fmaxf(m_run[nt][jj], mx);
        const float corr = fast_exp2(m_run[nt][jj] - m_new);  // 0 on the first tile
        m_run[nt][jj] = m_new;
        l_run[nt][jj] *= corr;
#pragma unroll
        for (int md = 0; md < 8; ++md) {
          o[md][nt][jj] *= corr;
          o[md][nt][jj + 2] *= corr;
        }
      }

    // P = 2^(s - m), split into bf16 hi + lo, transposed into B fragments of P^T
    uint32_t ph[4][NT][2], pl[4][NT][2];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          pv[e] = fast_exp2(sacc[mt][nt][e] - m_run[nt][e & 1]);
          l_run[nt][e & 1] += pv[e];
        }
        const uint32_t h01 = pack_bf16(pv[0], pv[1]), h23 = pack_bf16(pv[2], pv[3]);
        const uint32_t l01 = pack_bf16(pv[0] - bf16_lo_to_float(h01), pv[1] - bf16_hi_to_float(h01));
        const uint32_t l23 = pack_bf16(pv[2] - bf16_lo_to_float(h23), pv[3] - bf16_hi_to_float(h23));
        ph[mt][nt][0] = movmatrix_t(h01);
        ph[mt][nt][1] = movmatrix_t(h23);
        pl[mt][nt][0] = movmatrix_t(l01);
        pl[mt][nt][1] = movmatrix_t(l23);
      }

    // O^T += V_j^T P^T : 8 dim blocks of 16 x 4 token k-steps
#pragma unroll
    for (int md = 0; md < 8; ++md)
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        const int qd = lane >> 3;
        const int tok = 16 * mt + (lane & 7) + ((qd >> 1) << 3);
        const int chunk = 2 * md + (qd & 1);
        const uint32_t addr = ((chunk >> 3) ? vHi : vLo) + swz128(tok, chunk & 7);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(addr, a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_bf16(o[md][nt], a0, a1, a2, a3, ph[mt][nt][0], ph[mt][nt][1]);
          mma_bf16(o[md][nt], a0, a1, a2, a3, pl[mt][nt][0], pl[mt][nt][1]);
        }
      }

    if (valid < kTile || holds_new) fence_proxy_async_smem();  // generic writes precede the next TMA here
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty_bar[s]));
  }
  if (cur_seg >= 0) flush(cur_seg);

  // ------------------------------------------------------------------ merge
  consumer_barrier();
  if (s_abort) return;
  auto seg_range = [&](int sg, long long &beg, long long &end) {
    const int b = sg / p.Hkv, kv = sg - b * p.Hkv;
    const int nt = (Ls[b] + kTile - 1) / kTile;
    beg = static_cast<long long>(pre[b]) + static_cast<long long>(kv) * nt;
    end = beg + nt;
  };
  // Phase A: this CTA's warp partials per (segment, head).  A segment held entirely by
  // this CTA is normalised and written out; a shared one leaves a CTA partial.
  const int nseg = seg_last - seg_first + 1;
  for (int pr = cw; pr < nseg * p.G; pr += kConsumerWarps) {
    const int sg = seg_first + pr / p.G, g = pr % p.G;
    long long beg, end;
    seg_range(sg, beg, end);
    if (end <= beg) continue;  // a skipped sequence inside the range
    const long long a = beg > xs ? beg : xs, e = end < xe ? end : xe;
    float m = -INFINITY, l = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float2 ml[kConsumerWarps];
    float4 ov[kConsumerWarps];
#pragma unroll
    for (int c = 0; c < kConsumerWarps; ++c) {
      ml[c] = make_float2(-INFINITY, 0.f);
      if (warp_has_tile(a - xs, e - xs, c)) {
        const long long r = (static_cast<long long>(sg + w) * kConsumerWarps + c) * p.G + g;
        ml[c] = *reinterpret_cast<const float2 *>(p.part_ml + r * 2);
        ov[c] = *reinterpret_cast<const float4 *>(p.part_o + r * kHeadDim + 4 * lane);
      }
    }
#pragma unroll
    for (int c = 0; c < kConsumerWarps; ++c)
      if (ml[c].y > 0.f) merge_into(m, l, acc, ml[c].x, ml[c].y, ov[c]);
    const int b = sg / p.Hkv, kv = sg - b * p.Hkv;
    if (beg >= xs && end <= xe) {
      store_out4(p.out + (static_cast<long long>(b) * p.Hq + kv * p.G + g) * kHeadDim + 4 * lane, acc, l);
    } else {
      const long long r = static_cast<long long>(sg + w) * p.G + g;
      *reinterpret_cast<float4 *>(p.cpart_o + r * kHeadDim + 4 * lane) = acc;
      if (lane == 0) *reinterpret_cast<float2 *>(p.cpart_ml + r * 2) = make_float2(m, l);
      __threadfence();  // publish the CTA partial before the ticket below
    }
  }
  consumer_barrier();
  // Phase B: an arrival ticket for each shared segment (only the first and the last
  // segment of a CTA's range can be shared); the CTA drawing the last ticket merges it.
  if (tid == 0) {
    for (int k = 0; k < 2; ++k) {
      s_last[k] = -1;
      const int sg = k == 0 ? seg_first : seg_last;
      if (k == 1 && seg_last == seg_first) break;
      long long beg, end;
      seg_range(sg, beg, end);
      if (end <= beg || (beg >= xs && end <= xe)) continue;
      const int pieces = workers_of_segment(T, W, beg, end);
      __threadfence();
      const unsigned prev = atomicAdd(&p.seg_count[sg], 1u);
      if (prev == static_cast<unsigned>(pieces - 1)) {
        s_last[k] = sg;
        p.seg_count[sg] = 0;  // ready for the next call
        __threadfence();
      }
    }
  }
  consumer_barrier();
  // Phase C: merge every CTA partial of the segments this CTA closed.
  for (int k = 0; k < 2; ++k) {
    const int sg = s_last[k];
    if (sg < 0) continue;
    long long beg, end;
    seg_range(sg, beg, end);
    const int wa = worker_of(T, W, beg), wb = worker_of(T, W, end - 1);
    const int b = sg / p.Hkv, kv = sg - b * p.Hkv;
    for (int g = cw; g < p.G; g += kConsumerWarps) {
      float m = -INFINITY, l = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int w0 = wa; w0 <= wb; w0 += 8) {
        float2 ml[8];
        float4 ov[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          ml[u] = make_float2(-INFINITY, 0.f);
          if (w0 + u <= wb && worker_nonempty(T, W, w0 + u)) {
            const long long r = static_cast<long long>(sg + w0 + u) * p.G + g;
            ml[u] = __ldcg(reinterpret_cast<const float2 *>(p.cpart_ml + r * 2));
            ov[u] = __ldcg(reinterpret_cast<const float4 *>(p.cpart_o + r * kHeadDim + 4 * lane));
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (ml[u].y > 0.f) merge_into(m, l, acc, ml[u].x, ml[u].y, ov[u]);
      }
      store_out4(p.out + (static_cast<long long>(b) * p.Hq + kv * p.G + g) * kHeadDim + 4 * lane, acc, l);
    }
  }
}

size_t step_smem_bytes(int npad, int batch) {
  const size_t ring = npad == 8 ? Cfg<1>::kRing * Cfg<1>::kQBytes : Cfg<2>::kRing * Cfg<2>::kQBytes;
  return 1024 + static_cast<size_t>(kStages) * 4 * kHalfTileBytes + ring + 16 * kStages + 4 * (batch + 1) +
         4 * batch;
}

cudaError_t step_configure(int npad, int batch) {
  const int bytes = static_cast<int>(step_smem_bytes(npad, batch));
  if (npad == 8) return cudaFuncSetAttribute(decode_step_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  return cudaFuncSetAttribute(decode_step_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t launch_step(const CUtensorMap &tmK, const CUtensorMap &tmV, const StepParams &p, int npad,
                        int num_workers, cudaStream_t stream) {
  const size_t bytes = step_smem_bytes(npad, p.B);
  if (npad == 8)
    return launch_pdl(decode_step_kernel<1>, dim3(num_workers), dim3(kThreadsAttn), bytes, stream, tmK, tmV, p);
  return launch_pdl(decode_step_kernel<2>, dim3(num_workers), dim3(kThreadsAttn), bytes, stream, tmK, tmV, p);
}

}  // namespace gqa
