// Split-KV decode attention over a bf16 KV cache (sm_103a).
//
// What it computes -- for each query head h of sequence b, over its KV tiles -- is the
// FlashAttention per-tile recurrence of "ADR-0060: AHBM GQA Fused Attention Kernel
// (Llama3-70B)", section 3:  S = scale * q K_j^T (masked past L_b), m' = max(m, rowmax S),
// P = exp(S - m'), c = exp(m - m'), l = l*c + rowsum P, O = O*c + P V_j, seeded
// m = -inf, l = 0, O = 0 ("Qwen3-14B Optimization", section 2.1 Shape 3: the running
// state lives on-chip across the block loop with no peeled first iteration).  Each worker
// leaves unnormalised (m, l, O) partials for the log-sum-exp combine (ADR-0060 section 4;
// FlashDecoding split-KV).
//
// GB300 design:
//  * The G query heads sharing KV head kv are folded into one operand (ADR-0060 section
//    5.2, M-fold): one K/V tile serves all G heads.  Because decode is KV-bandwidth bound,
//    the fold is laid out token-major: S^T[64 tokens x 8*NT heads] = K_j[64 x 128] *
//    Q^T[128 x 8*NT], and O^T[128 x 8*NT] += V_j^T * P^T, with legacy mma.sync m16n8k16
//    (bf16 in, fp32 accumulate).  G <= 8 pads to 8 columns (G = 5 wastes 3), not 16 rows.
//  * P enters the P.V product as bf16 hi + bf16 lo (two mma), so rounding P costs no
//    accuracy (the bf16 output rounding is then the only sizeable error).
//  * One CTA per SM: a producer warp streams 64-token K/V tiles (2 x 16 KiB) with 3-D
//    TMA loads (128-byte swizzle, no multicast) into a 6-stage mbarrier ring; six
//    consumer warps each own one stage, take every sixth tile, run the recurrence in
//    registers and release the stage.
//  * The decode prologue is folded in ("Qwen3-14B Optimization", section 2.1 Shape 4 and
//    "Then: buy it" (#796): QK-norm and RoPE inside the attention kernel).  Each consumer
//    warp builds the rotated queries of the segment it works on straight into its mma B
//    fragments (binary32, one bf16 rounding), and the warp owning the tile that holds a
//    sequence's new token computes the rotated key (double-word arithmetic, rounded as the
//    exact value rounds), appends k and v to the cache and patches them into its tile.  Their inputs are loaded before
//    the KV stream starts, and both happen before the kernel waits on the preceding
//    kernel, overlapping the first KV loads.
//  * Workers own contiguous, equal ranges of the batch's tiles (see gqa_common.cuh), so
//    ragged batches stay balanced.
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

// Inputs of one new-token k/v row, loaded ahead of their use (lane l holds dims l + 32 t).
struct KvRowIn {
  uint16_t x[4], v[4], w[4];  // bf16 bits of k_new, v_new and k_norm_w (w unused without a norm)
  float4 cs0, cs1;            // double-word (cos, sin) of pairs l and l + 32
  long long grow;             // cache row of the new token; -1 when its page is out of range
};

__device__ __forceinline__ void load_kv_row(const AttnParams &p, int b, int kv, int pos, int lane, KvRowIn &in) {
  const long long nrow = (static_cast<long long>(b) * p.Hkv + kv) * kHeadDim;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    in.x[t] = p.k_new[nrow + lane + 32 * t];
    in.v[t] = p.v_new[nrow + lane + 32 * t];
    in.w[t] = p.k_norm_w ? p.k_norm_w[lane + 32 * t] : uint16_t(0);
  }
  in.cs0 = p.rope_dw[static_cast<long long>(pos) * 64 + lane];
  in.cs1 = p.rope_dw[static_cast<long long>(pos) * 64 + lane + 32];
  in.grow = -1;
  if (p.paged) {
    const int pg = p.page_table[static_cast<long long>(b) * p.max_blocks + pos / kTile];
    if (pg >= 0 && pg < p.num_blocks) in.grow = static_cast<long long>(pg) * kTile + (pos & (kTile - 1));
  } else {
    in.grow = static_cast<long long>(b) * p.max_seq + pos;
  }
}

// Appends one new token for KV head kv: k = RoPE_pos(RMSNorm(k_new)) rounded once to bf16
// as its exact value rounds (rotate_row_k), v = v_new, written to the token's cache row
// (skipped when its page id is out of range; the producer flags that) and returned per
// lane for the shared-memory patch.
__device__ __forceinline__ void append_kv_row(const AttnParams &p, int kv, int lane, const KvRowIn &in,
                                              uint16_t (&kz)[4], uint16_t (&vz)[4]) {
  rotate_row_k(in.x, in.w, p.k_norm_w != nullptr, static_cast<float>(p.eps), in.cs0, in.cs1, kz);
#pragma unroll
  for (int t = 0; t < 4; ++t) vz[t] = in.v[t];
  if (in.grow >= 0) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      p.k_cache[(in.grow * p.Hkv + kv) * kHeadDim + lane + 32 * t] = kz[t];
      p.v_cache[(in.grow * p.Hkv + kv) * kHeadDim + lane + 32 * t] = vz[t];
    }
  }
}

// The rotated queries of segment (b, kv) -- RoPE_pos(RMSNorm(q_new)) for the G heads
// kv*G .. kv*G+G-1, in binary32, rounded once to bf16 -- go straight into the B operand of
// S^T = K_j q^T: lane l holds head 8 nt + l/4 (zero past G) at dims
// 16 ks + 8 hf + 2 (l mod 4) + {0, 1} in qf[ks][nt][hf].  The RoPE partner of dim i is
// i + 64, i.e. ks + 4 in the same lane; the norm's sum of squares is completed over the
// four lanes that share a head.  QIn holds the inputs, loaded ahead of their use.
template <int NT>
struct QIn {
  uint32_t x[NT][8][2];  // q_new bf16 pairs
  uint32_t w[8][2];      // q_norm_w bf16 pairs at the same dims
  float4 cs[4][2];       // (cos, sin) of pairs i and i + 1, i = 16 ks + 8 hf + 2 (l mod 4), ks < 4
};

template <int NT>
__device__ __forceinline__ void load_q_inputs(const AttnParams &p, int b, int kv, int pos, int lane, QIn<NT> &in) {
  const int c2 = 2 * (lane & 3);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int g = 8 * nt + (lane >> 2);
    const long long row = (static_cast<long long>(b) * p.Hq + kv * p.G + g) * kHeadDim;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
        in.x[nt][ks][hf] = g < p.G ? *reinterpret_cast<const uint32_t *>(p.q_new + row + 16 * ks + 8 * hf + c2) : 0u;
  }
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
      in.w[ks][hf] = p.q_norm_w ? *reinterpret_cast<const uint32_t *>(p.q_norm_w + 16 * ks + 8 * hf + c2) : 0u;
  const float2 *cs = p.rope_tab32 + static_cast<long long>(pos) * 64;
#pragma unroll
  for (int ks = 0; ks < 4; ++ks)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) in.cs[ks][hf] = *reinterpret_cast<const float4 *>(cs + 16 * ks + 8 * hf + c2);
}

// `publish`: also store the rows, as plain [B, H_q, d] rows, to the workspace copy of the
// rotated queries.
template <int NT>
__device__ __forceinline__ void rotate_q(const AttnParams &p, int b, int kv, int lane, bool publish,
                                         const QIn<NT> &in, uint32_t (&qf)[8][NT][2]) {
  const int c2 = 2 * (lane & 3);
  const float eps = static_cast<float>(p.eps);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int g = 8 * nt + (lane >> 2);
    const bool real = g < p.G;
    const long long row = (static_cast<long long>(b) * p.Hq + kv * p.G + g) * kHeadDim;
    float ss = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const float a = bf16_lo_to_float(in.x[nt][ks][hf]), c = bf16_hi_to_float(in.x[nt][ks][hf]);
        ss = fmaf(a, a, ss);
        ss = fmaf(c, c, ss);
      }
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    const float r = p.q_norm_w ? 1.0f / sqrtf(ss * (1.0f / 128.0f) + eps) : 1.0f;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int i = 16 * ks + 8 * hf + c2;  // pairs i, i + 1 (< 64)
        float y0 = bf16_lo_to_float(in.x[nt][ks][hf]), y1 = bf16_hi_to_float(in.x[nt][ks][hf]);
        float p0 = bf16_lo_to_float(in.x[nt][ks + 4][hf]), p1 = bf16_hi_to_float(in.x[nt][ks + 4][hf]);
        if (p.q_norm_w) {
          y0 *= bf16_lo_to_float(in.w[ks][hf]), y1 *= bf16_hi_to_float(in.w[ks][hf]);
          p0 *= bf16_lo_to_float(in.w[ks + 4][hf]), p1 *= bf16_hi_to_float(in.w[ks + 4][hf]);
        }
        const float4 cs = in.cs[ks][hf];  // (cos_i, sin_i, cos_i+1, sin_i+1)
        uint32_t lo = pack_bf16(r * fmaf(y0, cs.x, -p0 * cs.y), r * fmaf(y1, cs.z, -p1 * cs.w));
        uint32_t hi = pack_bf16(r * fmaf(p0, cs.x, y0 * cs.y), r * fmaf(p1, cs.z, y1 * cs.w));
        if (!real) lo = hi = 0u;
        qf[ks][nt][hf] = lo;
        qf[ks + 4][nt][hf] = hi;
        if (publish && real) {
          *reinterpret_cast<uint32_t *>(p.q_rot + row + i) = lo;
          *reinterpret_cast<uint32_t *>(p.q_rot + row + i + 64) = hi;
        }
      }
  }
}

template <int NT>
struct Cfg {
  static constexpr int kStageBytes = 4 * kHalfTileBytes;
  static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment for the 128B swizzle");
};

}  // namespace

template <int NT>
__global__ void __launch_bounds__(kThreadsAttn, 1)
    attn_splitkv_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const AttnParams p) {
  using C = Cfg<NT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align_smem_1024(smem_raw);
  uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + kStages * C::kStageBytes);
  uint64_t *empty_bar = full_bar + kStages;
  uint32_t *pre = reinterpret_cast<uint32_t *>(empty_bar + kStages);  // [B + 1]
  int32_t *Ls = reinterpret_cast<int32_t *>(pre + p.B + 1);           // [B], 0 if invalid
  int32_t *Ps = Ls + p.B;                                              // [B], -1 if invalid

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), 1);
    }
    fence_barrier_init();
  }
  if (warp == kConsumerWarps && lane == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  if (warp == kConsumerWarps && lane < 3 && !p.inputs_in_host_memory) {
    // Every CTA pulls its share of the new-token rows into L2 while the batch prefix (which
    // says whose rows it needs) is still being worked out.
    const uint16_t *src = lane == 0 ? p.q_new : lane == 1 ? p.k_new : p.v_new;
    const long long bytes = static_cast<long long>(p.B) * (lane == 0 ? p.Hq : p.Hkv) * kHeadDim * 2;
    const long long chunk = ((bytes + gridDim.x - 1) / gridDim.x + 15) & ~15LL;
    const long long off = chunk * blockIdx.x;
    if (off < bytes) {
      const long long len = bytes - off < chunk ? bytes - off : chunk;
      prefetch_l2(reinterpret_cast<const char *>(src) + off, static_cast<uint32_t>(len));
    }
  }
  if (warp == kConsumerWarps && p.spec && lane < kStages) {
    // The first tiles this worker streamed at the previous launch: unless the lengths
    // changed the tile partition (in decode, once every 64 steps of a sequence), they are
    // its first tiles again, so they are pulled into L2 now, a DRAM round trip before the
    // partition is known.  A wrong guess costs only the prefetched bytes.  (The host
    // passes spec for contiguous caches only: with a page table the producer needs one
    // more small dependent read before its first load, and measured, a stream of
    // prefetches ahead of it cost more than it saved.)
    const int2 t = p.spec[blockIdx.x * kStages + lane];
    if (t.x >= 0) {
      tma_prefetch_3d(&tmK, 0, t.y, t.x);
      tma_prefetch_3d(&tmK, 64, t.y, t.x);
      tma_prefetch_3d(&tmV, 0, t.y, t.x);
      tma_prefetch_3d(&tmV, 64, t.y, t.x);
    }
  }
  if (warp == 0) {  // tile prefix over the batch; lengths and positions checked once
    uint32_t run = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int b = b0 + lane;
      uint32_t v = 0;
      if (b < p.B) {
        int L = p.seq_lens[b], pos = p.positions[b];
        const int nt = tiles_of(L, p.max_seq);
        if (nt == 0) {
          if (blockIdx.x == 0) atomicOr(p.err, GQA_DEVERR_SEQLEN);
          L = 0;
          pos = -1;
        } else if (pos < 0 || pos >= L) {
          if (blockIdx.x == 0) atomicOr(p.err, GQA_DEVERR_POSITION);
          pos = -1;
        }
        Ls[b] = L;
        Ps[b] = pos;
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

  const long long T = pre[p.B];
  const int W = gridDim.x, w = blockIdx.x;
  const long long xs = worker_begin(T, W, w), xe = worker_begin(T, W, w + 1);
  const long long n = xe - xs;
  const bool producer = warp == kConsumerWarps;
  const int cw = warp;

  // Where tile xs + i lives: its (b, kv) segment and the cache row of its first token (the
  // TMA z coordinate).
  auto describe = [&](long long i, int &row, int &kv, int &seg) {
    int b, j;
    locate(pre, Ls, p.B, p.Hkv, xs + i, b, kv, j);
    seg = b * p.Hkv + kv;
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
  };

  // ---------------------------------------------------------------- early loads
  // The producer resolves its first tiles' cache rows; each consumer warp loads what the
  // rotated queries of its first segment and the first new-token row it appends need.
  // These small reads go out before the KV stream starts; the new-token rows among them
  // were prefetched into L2 above, so they do not wait behind the stream.
  const int npre = static_cast<int>(n < kStages ? n : kStages);
  int row = 0, kv = 0, seg = 0;                 // producer: lane k < npre describes tile k
  QIn<NT> qin;
  KvRowIn kin;
  int q_b = -1, q_kv = 0, q_j = 0;              // consumer: first tile's segment
  long long ex0 = -1, ex1 = -1;                 // consumer: tiles holding new tokens it appends
  int ex0_b = 0, ex0_kv = 0, ex1_b = 0, ex1_kv = 0;
  if (producer) {
    if (lane < npre) describe(lane, row, kv, seg);
    if (p.spec && lane < kStages)
      p.spec[blockIdx.x * kStages + lane] = lane < npre ? make_int2(row, kv) : make_int2(-1, 0);
  } else if (n > 0) {
    if (cw < n) {
      locate(pre, Ls, p.B, p.Hkv, xs + cw, q_b, q_kv, q_j);
      if (Ps[q_b] >= 0) load_q_inputs<NT>(p, q_b, q_kv, Ps[q_b], lane, qin);
    }
    int b0, kv0, j0, b1, kv1, j1;
    locate(pre, Ls, p.B, p.Hkv, xs, b0, kv0, j0);
    locate(pre, Ls, p.B, p.Hkv, xe - 1, b1, kv1, j1);
    const int seg_first = b0 * p.Hkv + kv0, seg_last = b1 * p.Hkv + kv1;
    for (int sg = seg_first; sg <= seg_last && ex1 < 0; ++sg) {
      const int b = sg / p.Hkv, k = sg - b * p.Hkv;
      const int pos = Ps[b];
      if (pos < 0) continue;
      const int nt = (Ls[b] + kTile - 1) / kTile;
      const long long x_new = static_cast<long long>(pre[b]) + static_cast<long long>(k) * nt + pos / kTile;
      if (x_new < xs || x_new >= xe || (x_new - xs) % kConsumerWarps != cw) continue;
      if (ex0 < 0) {
        ex0 = x_new, ex0_b = b, ex0_kv = k;
      } else {
        ex1 = x_new, ex1_b = b, ex1_kv = k;
      }
    }
    if (ex0 >= 0) load_kv_row(p, ex0_b, ex0_kv, Ps[ex0_b], lane, kin);
  }
  __syncthreads();

  if (producer) {
    // ---------------------------------------------------------------- producer warp
    // The producer reads only the cache and the page table.  The preceding step has
    // finished by the time this kernel starts (the combine between the two launches it
    // only after waiting for that step's attention kernel), and this step's new rows are
    // patched into the shared-memory tiles by their consumers, so it streams from the
    // start and never waits on the preceding kernel.
    if (n <= 0) return;
    for (int k = 0; k < npre; ++k) {
      const int r_row = __shfl_sync(0xffffffffu, row, k), r_kv = __shfl_sync(0xffffffffu, kv, k);
      if (lane == 0) {
        const uint32_t fb = smem_addr(&full_bar[k]);
        const uint32_t base = smem_addr(smem + k * C::kStageBytes);
        mbar_arrive_expect_tx(fb, C::kStageBytes);
        tma_load_3d(base, &tmK, fb, 0, r_kv, r_row);
        tma_load_3d(base + kHalfTileBytes, &tmK, fb, 64, r_kv, r_row);
        tma_load_3d(base + 2 * kHalfTileBytes, &tmV, fb, 0, r_kv, r_row);
        tma_load_3d(base + 3 * kHalfTileBytes, &tmV, fb, 64, r_kv, r_row);
      }
    }
    bool fail = false;
    long long issued = npre;
    for (long long i0 = npre; i0 < n && !fail; i0 += 32) {
      const long long i = i0 + lane;
      row = 0, kv = 0, seg = 0;
      if (i < n) describe(i, row, kv, seg);
      const int cnt = static_cast<int>(n - i0 < 32 ? n - i0 : 32);
      for (int k = 0; k < cnt; ++k) {
        const int r_row = __shfl_sync(0xffffffffu, row, k);
        const int r_kv = __shfl_sync(0xffffffffu, kv, k);
        const long long ii = i0 + k;
        const int s = static_cast<int>(ii % kStages);
        int ok = 1;
        if (lane == 0) {
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
      // Do not leave while copies into this CTA's shared memory may still be in flight.
      for (long long ii = (issued > kStages ? issued - kStages : 0); ii < issued; ++ii)
        (void)mbar_wait(smem_addr(&full_bar[ii % kStages]), static_cast<uint32_t>((ii / kStages) & 1));
    }
    return;
  }

  // ------------------------------------------------------------------ consumer warps
  // Until griddep_wait() returns, the preceding kernel in the stream (the previous step's
  // combine) may still be reading the partials, so those are written only after it;
  // everything before it reads only the caller's inputs and the RoPE table and writes only
  // the new cache rows, which that kernel does not touch.
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

  auto flush = [&](int sg) {
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
    const long long base_row = (static_cast<long long>(sg + w) * kConsumerWarps + cw) * p.G;
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

  // The rotated queries of the segment in hand, as mma B fragments (rebuilt whenever the
  // warp moves to another segment; the warp holding a segment's first tile also publishes
  // them to the workspace).  A sequence whose position is out of range gets zeros.
  uint32_t qf[8][NT][2];
  auto zero_q = [&]() {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) qf[ks][nt][0] = qf[ks][nt][1] = 0u;
  };
  int cur_seg = -1;
  if (q_b >= 0) {
    if (Ps[q_b] >= 0) rotate_q<NT>(p, q_b, q_kv, lane, q_j == 0, qin, qf);
    else zero_q();
    cur_seg = q_b * p.Hkv + q_kv;
  }

  // The new-token k/v rows this warp appends: the first two are computed now, while the
  // first tiles are still in flight, written to the cache and kept packed in registers for
  // the shared-memory patch; any further ones are computed when their tile arrives.
  uint32_t ek0[2] = {0, 0}, ev0[2] = {0, 0}, ek1[2] = {0, 0}, ev1[2] = {0, 0};
  if (ex0 >= 0) {
    uint16_t kz[4], vz[4];
    append_kv_row(p, ex0_kv, lane, kin, kz, vz);
    ek0[0] = kz[0] | (uint32_t(kz[1]) << 16), ek0[1] = kz[2] | (uint32_t(kz[3]) << 16);
    ev0[0] = vz[0] | (uint32_t(vz[1]) << 16), ev0[1] = vz[2] | (uint32_t(vz[3]) << 16);
  }
  if (ex1 >= 0) {
    uint16_t kz[4], vz[4];
    load_kv_row(p, ex1_b, ex1_kv, Ps[ex1_b], lane, kin);
    append_kv_row(p, ex1_kv, lane, kin, kz, vz);
    ek1[0] = kz[0] | (uint32_t(kz[1]) << 16), ek1[1] = kz[2] | (uint32_t(kz[3]) << 16);
    ev1[0] = vz[0] | (uint32_t(vz[1]) << 16), ev1[1] = vz[2] | (uint32_t(vz[3]) << 16);
  }

  griddep_wait();
  griddep_launch_dependents();

  for (long long i = cw; i < n; i += kConsumerWarps) {
    int b, kv, j;
    locate(pre, Ls, p.B, p.Hkv, xs + i, b, kv, j);
    const int sg = b * p.Hkv + kv;
    const int pos_b = Ps[b];
    if (sg != cur_seg) {
      flush(cur_seg);
      cur_seg = sg;
      if (pos_b >= 0) {
        load_q_inputs<NT>(p, b, kv, pos_b, lane, qin);
        rotate_q<NT>(p, b, kv, lane, j == 0, qin, qf);
      } else {
        zero_q();
      }
    }
    const int s = static_cast<int>(i % kStages);
    const bool ready = mbar_wait(smem_addr(&full_bar[s]), static_cast<uint32_t>((i / kStages) & 1));
    __syncwarp();  // reconverge before the warp-collective ldmatrix / mma below
    if (!__all_sync(0xffffffffu, ready)) {
      if (lane == 0) atomicOr(p.err, GQA_DEVERR_TIMEOUT);
      return;
    }
    const int valid = min(kTile, Ls[b] - j * kTile);
    uint8_t *stage = smem + s * C::kStageBytes;
    const uint32_t kLo = smem_addr(stage), kHi = kLo + kHalfTileBytes;
    const uint32_t vLo = kLo + 2 * kHalfTileBytes, vHi = kLo + 3 * kHalfTileBytes;

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
    // The tile holding sequence b's new token: the TMA filled this stage from the cache
    // before the row was appended, so patch the appended k and v rows into it.
    const bool holds_new = pos_b >= 0 && (pos_b >> 6) == j;
    if (holds_new) {
      uint16_t kz[4], vz[4];
      const long long x = xs + i;
      if (x == ex0 || x == ex1) {
        const uint32_t *k2 = x == ex0 ? ek0 : ek1, *v2 = x == ex0 ? ev0 : ev1;
        kz[0] = k2[0] & 0xffff, kz[1] = k2[0] >> 16, kz[2] = k2[1] & 0xffff, kz[3] = k2[1] >> 16;
        vz[0] = v2[0] & 0xffff, vz[1] = v2[0] >> 16, vz[2] = v2[1] & 0xffff, vz[3] = v2[1] >> 16;
      } else {
        load_kv_row(p, b, kv, pos_b, lane, kin);
        append_kv_row(p, kv, lane, kin, kz, vz);
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
}

size_t attn_smem_bytes(int npad, int batch) {
  (void)npad;  // the rotated queries live in registers: the stage size does not depend on G
  const int stage = 4 * kHalfTileBytes;
  return 1024 + static_cast<size_t>(kStages) * stage + 16 * kStages + 4 * (batch + 1) + 8 * batch;
}

cudaError_t attn_configure(int npad) {
  const int bytes = static_cast<int>(attn_smem_bytes(npad, GQA_MAX_BATCH));
  if (npad == 8) return cudaFuncSetAttribute(attn_splitkv_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  return cudaFuncSetAttribute(attn_splitkv_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t launch_attention(const CUtensorMap &tmK, const CUtensorMap &tmV, const AttnParams &p, int npad,
                             int num_workers, bool pdl, cudaStream_t stream) {
  const size_t bytes = attn_smem_bytes(npad, p.B);
  if (npad == 8)
    return launch_ex(pdl, attn_splitkv_kernel<1>, dim3(num_workers), dim3(kThreadsAttn), bytes, stream, tmK, tmV, p);
  return launch_ex(pdl, attn_splitkv_kernel<2>, dim3(num_workers), dim3(kThreadsAttn), bytes, stream, tmK, tmV, p);
}

}  // namespace gqa
