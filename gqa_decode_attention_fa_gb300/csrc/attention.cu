// Decode attention over a bf16 KV cache (sm_103a): the split-KV kernel (a worker
// partition of the batch's tiles, partials merged by the combine kernel) and, further
// down, the single-launch kernel (a thread-block cluster per segment, merged on chip),
// which share the producer / consumer ring and the per-tile recurrence.
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

// The inputs of the new row that do not depend on its position (k_new, v_new, k_norm_w) ...
__device__ __forceinline__ void load_kv_inputs(const AttnParams &p, int b, int kv, int lane, KvRowIn &in) {
  const long long nrow = (static_cast<long long>(b) * p.Hkv + kv) * kHeadDim;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    in.x[t] = p.k_new[nrow + lane + 32 * t];
    in.v[t] = p.v_new[nrow + lane + 32 * t];
    in.w[t] = p.k_norm_w ? p.k_norm_w[lane + 32 * t] : uint16_t(0);
  }
}
// ... and those that do (the RoPE table row, the cache row).
__device__ __forceinline__ void load_kv_place(const AttnParams &p, int b, int pos, int lane, KvRowIn &in) {
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
__device__ __forceinline__ void load_kv_row(const AttnParams &p, int b, int kv, int pos, int lane, KvRowIn &in) {
  load_kv_inputs(p, b, kv, lane, in);
  load_kv_place(p, b, pos, lane, in);
}

// Appends one new token for KV head kv: k = RoPE_pos(RMSNorm(k_new)) rounded once to bf16
// as its exact value rounds (rotate_row_k), v = v_new, written to the token's cache row
// (skipped when its page id is out of range; the producer flags that) and returned per
// lane for the shared-memory patch.
__device__ __forceinline__ void rotated_kv_row(const AttnParams &p, const KvRowIn &in, uint16_t (&kz)[4],
                                               uint16_t (&vz)[4]) {
  rotate_row_k(in.x, in.w, p.k_norm_w != nullptr, static_cast<float>(p.eps), in.cs0, in.cs1, kz);
#pragma unroll
  for (int t = 0; t < 4; ++t) vz[t] = in.v[t];
}
__device__ __forceinline__ void store_kv_row(const AttnParams &p, int kv, int lane, const KvRowIn &in,
                                             const uint16_t (&kz)[4], const uint16_t (&vz)[4]) {
  if (in.grow >= 0) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      p.k_cache[(in.grow * p.Hkv + kv) * kHeadDim + lane + 32 * t] = kz[t];
      p.v_cache[(in.grow * p.Hkv + kv) * kHeadDim + lane + 32 * t] = vz[t];
    }
  }
}
__device__ __forceinline__ void append_kv_row(const AttnParams &p, int kv, int lane, const KvRowIn &in,
                                              uint16_t (&kz)[4], uint16_t (&vz)[4]) {
  rotated_kv_row(p, in, kz, vz);
  store_kv_row(p, kv, lane, in, kz, vz);
}
// The same store from the packed form (two bf16 a register: dims l + 32 t, t = 0..3).
__device__ __forceinline__ void store_packed_row(const AttnParams &p, int kv, int lane, long long grow,
                                                 const uint32_t (&k2)[2], const uint32_t (&v2)[2]) {
  if (grow < 0) return;
  uint16_t *kr = p.k_cache + (grow * p.Hkv + kv) * kHeadDim + lane;
  uint16_t *vr = p.v_cache + (grow * p.Hkv + kv) * kHeadDim + lane;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    kr[32 * t] = static_cast<uint16_t>(k2[t >> 1] >> (16 * (t & 1)));
    vr[32 * t] = static_cast<uint16_t>(v2[t >> 1] >> (16 * (t & 1)));
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

// The query rows and q_norm_w (independent of the position) ...
template <int NT>
__device__ __forceinline__ void load_q_rows(const AttnParams &p, int b, int kv, int lane, QIn<NT> &in) {
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
}
// ... and the RoPE table row of the position.
template <int NT>
__device__ __forceinline__ void load_q_rope(const AttnParams &p, int pos, int lane, QIn<NT> &in) {
  const int c2 = 2 * (lane & 3);
  const float2 *cs = p.rope_tab32 + static_cast<long long>(pos) * 64;
#pragma unroll
  for (int ks = 0; ks < 4; ++ks)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) in.cs[ks][hf] = *reinterpret_cast<const float4 *>(cs + 16 * ks + 8 * hf + c2);
}
template <int NT>
__device__ __forceinline__ void load_q_inputs(const AttnParams &p, int b, int kv, int pos, int lane, QIn<NT> &in) {
  load_q_rows<NT>(p, b, kv, lane, in);
  load_q_rope<NT>(p, pos, lane, in);
}

template <int NT>
__device__ __forceinline__ void rotate_q(const AttnParams &p, int lane, const QIn<NT> &in, uint32_t (&qf)[8][NT][2]) {
  const float eps = static_cast<float>(p.eps);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int g = 8 * nt + (lane >> 2);
    const bool real = g < p.G;
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
      for (int hf = 0; hf < 2; ++hf) {  // pairs i, i + 1 (< 64), i = 16 ks + 8 hf + 2 (l mod 4)
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
      }
  }
}

// Stores the rotated queries held in qf, as plain [B, H_q, d] rows, to the workspace copy
// of the rotated queries (for tests and debugging; the kernel itself keeps q in registers).
template <int NT>
__device__ __forceinline__ void publish_q(const AttnParams &p, int b, int kv, int lane,
                                          const uint32_t (&qf)[8][NT][2]) {
  const int c2 = 2 * (lane & 3);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int g = 8 * nt + (lane >> 2);
    if (g >= p.G) continue;
    const long long row = (static_cast<long long>(b) * p.Hq + kv * p.G + g) * kHeadDim;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int i = 16 * ks + 8 * hf + c2;
        *reinterpret_cast<uint32_t *>(p.q_rot + row + i) = qf[ks][nt][hf];
        *reinterpret_cast<uint32_t *>(p.q_rot + row + i + 64) = qf[ks + 4][nt][hf];
      }
  }
}

// Rows past L_b hold whatever the cache holds there; zero the V rows from `valid` on so
// that P = 0 never meets a non-finite value.  Whole 128-byte rows, so the swizzle does not
// matter.
__device__ __forceinline__ void zero_v_tail(uint8_t *stage, int valid, int lane) {
  uint4 *v0 = reinterpret_cast<uint4 *>(stage + 2 * kHalfTileBytes);
  uint4 *v1 = reinterpret_cast<uint4 *>(stage + 3 * kHalfTileBytes);
  const int nchunks = (kTile - valid) * 8;
  for (int c = lane; c < nchunks; c += 32) {
    v0[valid * 8 + c] = make_uint4(0, 0, 0, 0);
    v1[valid * 8 + c] = make_uint4(0, 0, 0, 0);
  }
  __syncwarp();
}

// Writes an appended k/v row (lane l holds dims l + 32 t) into row r of a ring stage: the
// TMA filled the stage from the cache before the row was appended.
__device__ __forceinline__ void patch_row(uint8_t *stage, int r, const uint16_t (&kz)[4], const uint16_t (&vz)[4],
                                          int lane) {
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int e = lane + 32 * t;
    const uint32_t off = (e >> 6) * kHalfTileBytes + swz128(r, (e & 63) >> 3) + (e & 7) * 2;
    *reinterpret_cast<uint16_t *>(stage + off) = kz[t];
    *reinterpret_cast<uint16_t *>(stage + 2 * kHalfTileBytes + off) = vz[t];
  }
  __syncwarp();
}


// One 64-token tile of the recurrence for a warp's G heads, on a ring stage holding the
// tile's K and V halves (128-byte swizzled): S^T = K_j q^T scaled to the log2 domain with
// tokens >= valid masked to -inf, the online-softmax update of (m, l, O), and
// O^T += V_j^T P^T with P split into bf16 hi + lo.
template <int NT>
__device__ __forceinline__ void tile_update(const uint8_t *stage, int valid, float scale_log2, int lane,
                                            const uint32_t (&qf)[8][NT][2], float (&o)[8][NT][4],
                                            float (&m_run)[NT][2], float (&l_run)[NT][2]) {
  const uint32_t kLo = smem_addr(stage), kHi = kLo + kHalfTileBytes;
  const uint32_t vLo = kLo + 2 * kHalfTileBytes, vHi = kLo + 3 * kHalfTileBytes;
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
        sacc[mt][nt][e] = tok < valid ? sacc[mt][nt][e] * scale_log2 : -INFINITY;
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
  // combine) may still be reading the partials, so nothing is written before it: the work
  // before the wait only reads (the caller's inputs, the RoPE table, the cache) and
  // computes the first new rows.  The new cache rows, the workspace copy of the rotated
  // queries and the partials are all written after it -- a workspace laid out per call
  // (the static-scratch entry point) can put this call's copy where the previous call's
  // partials were, and the preceding step may still read a row this one rewrites.
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
    if (Ps[q_b] >= 0) rotate_q<NT>(p, lane, qin, qf);
    else zero_q();
    cur_seg = q_b * p.Hkv + q_kv;
  }

  // The new-token k/v rows this warp appends: the first two are computed now, while the
  // first tiles are still in flight, kept packed in registers for the shared-memory patch
  // and written to the cache right after the wait below (a preceding single-launch step
  // may still be reading the rows a repeated position rewrites); any further ones are
  // computed and written when their tile arrives.
  uint32_t ek0[2] = {0, 0}, ev0[2] = {0, 0}, ek1[2] = {0, 0}, ev1[2] = {0, 0};
  long long grow0 = -1, grow1 = -1;
  if (ex0 >= 0) {
    uint16_t kz[4], vz[4];
    rotated_kv_row(p, kin, kz, vz);
    grow0 = kin.grow;
    ek0[0] = kz[0] | (uint32_t(kz[1]) << 16), ek0[1] = kz[2] | (uint32_t(kz[3]) << 16);
    ev0[0] = vz[0] | (uint32_t(vz[1]) << 16), ev0[1] = vz[2] | (uint32_t(vz[3]) << 16);
  }
  if (ex1 >= 0) {
    uint16_t kz[4], vz[4];
    load_kv_row(p, ex1_b, ex1_kv, Ps[ex1_b], lane, kin);
    rotated_kv_row(p, kin, kz, vz);
    grow1 = kin.grow;
    ek1[0] = kz[0] | (uint32_t(kz[1]) << 16), ek1[1] = kz[2] | (uint32_t(kz[3]) << 16);
    ev1[0] = vz[0] | (uint32_t(vz[1]) << 16), ev1[1] = vz[2] | (uint32_t(vz[3]) << 16);
  }

  griddep_wait();
  griddep_launch_dependents();
  if (ex0 >= 0) store_packed_row(p, ex0_kv, lane, grow0, ek0, ev0);
  if (ex1 >= 0) store_packed_row(p, ex1_kv, lane, grow1, ek1, ev1);
  if (q_b >= 0 && q_j == 0 && Ps[q_b] >= 0) publish_q<NT>(p, q_b, q_kv, lane, qf);

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
        rotate_q<NT>(p, lane, qin, qf);
        if (j == 0) publish_q<NT>(p, b, kv, lane, qf);
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
    if (valid < kTile) zero_v_tail(stage, valid, lane);
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
      patch_row(stage, pos_b & (kTile - 1), kz, vz, lane);
    }

    tile_update<NT>(stage, valid, p.scale_log2, lane, qf, o, m_run, l_run);

    if (valid < kTile || holds_new) fence_proxy_async_smem();  // generic writes precede the next TMA here
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty_bar[s]));
  }
  if (cur_seg >= 0) flush(cur_seg);
}

// ------------------------------------------------------------------ single-launch form
// The whole decode step in one launch: one thread-block cluster of C = p.csize CTAs per
// (sequence, KV head) segment -- several CTAs per segment for a few long sequences, C = 1
// for batches with more segments than SMs (then, when the clusters come in more than one
// wave and the plan gives an order, the segments start longest first).  CTA rank r of the cluster
// streams the segment's tiles r, r + C, r + 2C, ... through the same producer / consumer
// ring as the split-KV kernel and runs the same per-tile recurrence; the partials never
// leave the chip.  Each CTA merges its six consumer warps' (m, l, O) in shared memory and
// pushes the merged state to the cluster: CTA q owns dims [q 128/C, (q+1) 128/C) of the
// segment's G heads, and every CTA stores its (m, l) and its O values for those dims into
// CTA q's receive area with remote asynchronous stores that count their bytes on CTA q's
// mbarrier.  CTA q waits for the C contributions, merges them in a fixed order (ADR-0060
// section 4's merge) and writes its dims normalised in bf16.  No partials in HBM, no
// second kernel and no grid-wide wait inside the step.
//
// Ordering with the neighbouring kernels in the stream (programmatic dependent launch):
// the whole computation -- streaming the cache, the tiles, the merges -- runs without
// waiting on the preceding kernel; only the writes to global memory wait for it: the
// cache append (the preceding step may still read the row this one rewrites), the
// rotated-query copy and `out` (it may write the same buffers).  The producer warp waits
// first, appends the new row when this CTA holds it, fences it and lets the next kernel
// launch, since the next step streams the cache before its own wait.  So the next step's
// CTAs start as soon as this one's rows are in place and compute on the SMs this one
// leaves free while it finishes; a step's time is about half its latency.
//
// Cluster protocol: every thread arrives on the cluster barrier once its CTA's mbarriers
// are initialised and waits on it before the first remote store (so no store reaches an
// uninitialised barrier), and arrives again once its CTA has received everything and waits
// before leaving (so no CTA leaves while stores to or from it are in flight).  No thread
// leaves early and every mbarrier wait is bounded, so a pipeline timeout cannot hang the
// cluster.
namespace {
constexpr int kPartStride = 132;          // floats per (warp, head) partial row in shared memory
// Receive area of the single-launch kernel, after the ring's barriers: (m, l) of every
// sender and head, then O for the owned dims, [sender][head][128 / C].
constexpr int kRecvMlFloats = GQA_MAX_GROUP * GQA_MAX_GROUP * 2;
constexpr int kRecvOFloats = GQA_MAX_GROUP * kHeadDim;
constexpr int kRecvOffset = kStages * 4 * kHalfTileBytes + 1024;   // from the aligned base
constexpr int kKvRowOffset = kRecvOffset + 4 * (kRecvMlFloats + kRecvOFloats);  // the appended k/v row
constexpr size_t kClusterSmemBytes = 1024 + kKvRowOffset + 2 * kHeadDim * 2;

// Barrier 1 hands the appended k/v row from the ordering warp to the consumer warp whose
// tile holds it (the ordering warp arrives, that consumer waits).
__device__ __forceinline__ void kvrow_arrive() { asm volatile("bar.arrive 1, 64;" ::: "memory"); }
__device__ __forceinline__ void kvrow_sync() { asm volatile("bar.sync 1, 64;" ::: "memory"); }
// Barrier 2: the producer warp arrives once the ring's barriers are initialised; the
// consumer warps wait for it before their first wait on a ring stage.
constexpr int kRingReadyThreads = 32 * (kConsumerWarps + 1);
__device__ __forceinline__ void ring_ready_arrive() {
  asm volatile("bar.arrive 2, %0;" ::"n"(kRingReadyThreads) : "memory");
}
__device__ __forceinline__ void ring_ready_sync() { asm volatile("bar.sync 2, %0;" ::"n"(kRingReadyThreads) : "memory"); }
// Warps: the consumers, the producer, and an ordering warp that waits on the preceding
// kernel, appends the new row (in the CTA whose tile holds it) and lets the next launch.
constexpr int kOrderWarp = kConsumerWarps + 1;
constexpr int kThreadsCluster = 32 * (kConsumerWarps + 2);
}  // namespace

// L2 prefetch of local tiles [first, n) of a single-launch CTA (rank `rank` of C in the
// cluster of segment (b, kv)), lane t taking tile first + t; kept out of line so that the
// producer's start-up code stays short for the launches that do not use it.
__device__ __noinline__ void spec_prefetch_l2(const CUtensorMap *tmK, const CUtensorMap *tmV,
                                              const int32_t *page_table, int max_blocks, int num_blocks,
                                              int max_seq, int b, int kv, int rank, int C, int first, int n,
                                              int lane) {
  const int i = first + lane;
  if (i < n) {
    const int j = rank + C * i;
    int row = -kTile;  // a page id outside the pool prefetches nothing
    if (page_table == nullptr) {
      row = b * max_seq + j * kTile;
    } else if (j < max_blocks) {
      const int pg = page_table[static_cast<long long>(b) * max_blocks + j];
      if (pg >= 0 && pg < num_blocks) row = pg * kTile;
    }
    tma_prefetch_3d(tmK, 0, kv, row);
    tma_prefetch_3d(tmK, 64, kv, row);
    tma_prefetch_3d(tmV, 0, kv, row);
    tma_prefetch_3d(tmV, 64, kv, row);
  }
}

// kOrder: the launch order of the segments comes from p.seg_order (a separate instance, so
// that the launches without it keep their start-up path unchanged).
template <int NT, bool kOrder>
__global__ void __launch_bounds__(kThreadsCluster, 1)
    attn_cluster_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const AttnParams p) {
  using Cf = Cfg<NT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align_smem_1024(smem_raw);
  uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + kStages * Cf::kStageBytes);
  uint64_t *empty_bar = full_bar + kStages;
  uint64_t *recv_bar = empty_bar + kStages;
  float *recv_ml = reinterpret_cast<float *>(smem + kRecvOffset);   // [C][G][2]
  float *recv_o = recv_ml + kRecvMlFloats;                          // [C][G][128 / C]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = p.csize;
  const int rank = static_cast<int>(cluster_ctarank());
  // CTA q owns dims [q * 128 / C, (q + 1) * 128 / C) of the segment's heads
  const int d0 = rank * kHeadDim / C, nd = (rank + 1) * kHeadDim / C - d0;
  // the cluster's segment: launch order longest first when the plan gives one (a batch of
  // more clusters than the device holds at once then ends with its short segments)
  const int seg = kOrder ? p.seg_order[blockIdx.x / C] : static_cast<int>(blockIdx.x) / C;
  const int b = seg / p.Hkv, kv = seg - b * p.Hkv;
  const bool producer = warp == kConsumerWarps;
  uint16_t *kvrow = reinterpret_cast<uint16_t *>(smem + kKvRowOffset);  // [2][128]: k, v

  // Cache row of local tile i's first token (the TMA z coordinate); a page id outside the
  // pool reads as a box wholly out of bounds (zeros) and is flagged when `flag`.
  auto tile_row = [&](int i, bool flag) -> int {
    const int j = rank + C * i;
    if (p.paged) {
      const int pg = p.page_table[static_cast<long long>(b) * p.max_blocks + j];
      if (pg < 0 || pg >= p.num_blocks) {
        if (flag) atomicOr(p.err, GQA_DEVERR_PAGE);
        return -kTile;
      }
      return pg * kTile;
    }
    return b * p.max_seq + j * kTile;
  };
  auto issue = [&](int s, int r_row) {  // one tile into stage s (lane 0 of the producer)
    const uint32_t fb = smem_addr(&full_bar[s]);
    const uint32_t base = smem_addr(smem + s * Cf::kStageBytes);
    mbar_arrive_expect_tx(fb, Cf::kStageBytes);
    tma_load_3d(base, &tmK, fb, 0, kv, r_row);
    tma_load_3d(base + kHalfTileBytes, &tmK, fb, 64, kv, r_row);
    tma_load_3d(base + 2 * kHalfTileBytes, &tmV, fb, 0, kv, r_row);
    tma_load_3d(base + 3 * kHalfTileBytes, &tmV, fb, 64, kv, r_row);
  };

  // The plan's expectation of the segment's tiles (the longest segment of the lengths it
  // was made with) and of this CTA's share.
  const int st_all = p.spec_tiles < p.max_blocks ? p.spec_tiles : p.max_blocks;
  const int st_cta = st_all > rank ? (st_all - rank + C - 1) / C : 0;
  // The producer initialises the barriers and, before the segment's length is known, loads
  // the first tiles the plan expects this CTA to stream (a tile's cache row does not depend
  // on the length); tiles that turn out to lie past the length are waited for and dropped.
  int nspec = 0, spec_row = 0;
  if (producer) {
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) {
        mbar_init(smem_addr(&full_bar[s]), 1);
        mbar_init(smem_addr(&empty_bar[s]), 1);
      }
      mbar_init(smem_addr(recv_bar), 1);
      fence_barrier_init();
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
    }
    nspec = st_cta < kStages ? st_cta : kStages;
    if (lane < nspec) spec_row = tile_row(lane, false);
    __syncwarp();
    for (int k = 0; k < nspec; ++k) {
      const int r_row = __shfl_sync(0xffffffffu, spec_row, k);
      if (lane == 0) issue(k, r_row);
    }
    // A CTA expected to stream more than one ring but at most two (a short, latency-bound
    // step) also prefetches the tiles past the ring into L2, which then arrive from L2 as
    // stages free instead of starting a DRAM round trip then.  (Measured on a 4k step: 5.87
    // -> 5.46 us; prefetching one ring ahead all along slowed the bandwidth-bound steps.)
    if (st_cta > kStages && st_cta <= 2 * kStages)
      spec_prefetch_l2(&tmK, &tmV, p.paged ? p.page_table : nullptr, p.max_blocks, p.num_blocks, p.max_seq, b, kv,
                       rank, C, kStages, st_cta, lane);
    ring_ready_arrive();
  }
  // The cluster barrier's first phase: every CTA's barriers are initialised (the producer's
  // lane 0 arrives after its initialisation; it is waited for before the first remote store).
  cluster_arrive();
  // The segment's length and new-token position (one broadcast load per warp), then the
  // inputs that do not depend on the position -- the queries (consumer warps), the new k
  // and v rows (ordering warp) -- requested before the position arrives, so that the
  // latencies overlap (a layer's inputs are usually not in L2 when its kernel starts).
  int L = p.seq_lens[b], pos = p.positions[b];
  QIn<NT> qin;
  KvRowIn kin;
  if (warp < kConsumerWarps) load_q_rows<NT>(p, b, kv, lane, qin);
  else if (warp == kOrderWarp) load_kv_inputs(p, b, kv, lane, kin);
  const int nt = tiles_of(L, p.max_seq);
  if (nt == 0) {
    if (tid == 0 && rank == 0 && kv == 0) atomicOr(p.err, GQA_DEVERR_SEQLEN);
    L = 0;
    pos = -1;
  } else if (pos < 0 || pos >= L) {
    if (tid == 0 && rank == 0 && kv == 0) atomicOr(p.err, GQA_DEVERR_POSITION);
    pos = -1;
  }
  const int n = nt > rank ? (nt - rank + C - 1) / C : 0;  // local tile i is segment tile rank + C i
  // The warp (of this CTA) whose tile holds the new token, or -1.
  int owner = -1;
  if (pos >= 0 && (pos >> 6) % C == rank) owner = ((pos >> 6) / C) % kConsumerWarps;

  float o[8][NT][4];
  float m_run[NT][2], l_run[NT][2];
#pragma unroll
  for (int md = 0; md < 8; ++md)
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[md][t][e] = 0.f;
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      m_run[t][jj] = -INFINITY;
      l_run[t][jj] = 0.f;
    }

  uint32_t qkeep[8][NT][2];  // warp 0 of rank 0: the rotated queries to publish
  bool qpub = false;
  if (warp == kOrderWarp) {
    // ------------------------------------------------------------------ ordering warp
    // Computes the new row (when this CTA's tiles hold it) while the preceding kernel
    // drains, appends it once that kernel has completed, fences it and lets the next
    // kernel launch.
    uint16_t kz[4], vz[4];
    if (owner >= 0) {
      load_kv_place(p, b, pos, lane, kin);
      rotated_kv_row(p, kin, kz, vz);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        kvrow[lane + 32 * t] = kz[t];
        kvrow[kHeadDim + lane + 32 * t] = vz[t];
      }
      kvrow_arrive();  // the owning consumer warp patches its tile with these
    }
    griddep_wait();
    if (owner >= 0) {
      store_kv_row(p, kv, lane, kin, kz, vz);
      __threadfence();
    }
    __syncwarp();
    if (lane == 0) griddep_launch_dependents();
  } else if (producer) {
    // ---------------------------------------------------------------- producer warp
    // The producer streams from the start and never waits on the preceding kernel: that
    // kernel let this grid launch only after its own cache rows were appended and fenced
    // (the single-launch kernel) or after the attention kernel it waits on had completed
    // (the combine), and this step's own new row is patched into its tile by the consumer
    // that owns it.
    const int npre = n < kStages ? n : kStages;
    if (lane < nspec && lane < n && spec_row < 0) atomicOr(p.err, GQA_DEVERR_PAGE);  // now known to be read
    int row = 0;
    if (lane >= nspec && lane < npre) row = tile_row(lane, true);
    for (int k = nspec; k < npre; ++k) {
      const int r_row = __shfl_sync(0xffffffffu, row, k);
      if (lane == 0) issue(k, r_row);
    }
    bool fail = false;
    int issued = npre > nspec ? npre : nspec;
    for (int i0 = npre; i0 < n && !fail; i0 += 32) {
      row = i0 + lane < n ? tile_row(i0 + lane, true) : 0;
      const int cnt = n - i0 < 32 ? n - i0 : 32;
      for (int k = 0; k < cnt; ++k) {
        const int r_row = __shfl_sync(0xffffffffu, row, k);
        const int ii = i0 + k, s = ii % kStages;
        int ok = 1;
        if (lane == 0) {
          ok = mbar_wait(smem_addr(&empty_bar[s]), static_cast<uint32_t>(((ii / kStages) - 1) & 1));
          if (ok) {
            issue(s, r_row);
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
    if (lane == 0) {
      if (fail) atomicOr(p.err, GQA_DEVERR_TIMEOUT);
      // No copy may still be landing in this CTA's shared memory when it is reused below:
      // after a failure, the last ring's worth; else the speculative tiles past the length,
      // which no consumer waits for.
      const int from = fail ? (issued > kStages ? issued - kStages : 0) : n;
      for (int ii = from; ii < issued; ++ii)
        (void)mbar_wait(smem_addr(&full_bar[ii % kStages]), static_cast<uint32_t>((ii / kStages) & 1));
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ consumer warps
    const int cw = warp;
    const bool has_tiles = cw < n;
    const int i_new = cw == owner ? (pos >> 6) / C : -1;  // local index of the new token's tile
    if (has_tiles && pos >= 0) load_q_rope<NT>(p, pos, lane, qin);
    uint32_t qf[8][NT][2];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
#pragma unroll
      for (int t = 0; t < NT; ++t) qf[ks][t][0] = qf[ks][t][1] = 0u;
    if (has_tiles && pos >= 0) rotate_q<NT>(p, lane, qin, qf);
    ring_ready_sync();  // the ring's barriers are initialised
    if (rank == 0 && cw == 0) {  // the rotated queries, published after the wait below
      qpub = has_tiles && pos >= 0;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
#pragma unroll
        for (int t = 0; t < NT; ++t) qkeep[ks][t][0] = qf[ks][t][0], qkeep[ks][t][1] = qf[ks][t][1];
    }

    for (int i = cw; i < n; i += kConsumerWarps) {
      const int s = i % kStages;
      const bool ready = mbar_wait(smem_addr(&full_bar[s]), static_cast<uint32_t>((i / kStages) & 1));
      __syncwarp();
      if (!__all_sync(0xffffffffu, ready)) {
        if (lane == 0) atomicOr(p.err, GQA_DEVERR_TIMEOUT);
        break;
      }
      const int valid = min(kTile, L - (rank + C * i) * kTile);
      uint8_t *stage = smem + s * Cf::kStageBytes;
      if (valid < kTile) zero_v_tail(stage, valid, lane);
      if (i == i_new) {  // the appended row, from the ordering warp
        kvrow_sync();
        uint16_t kz[4], vz[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) kz[t] = kvrow[lane + 32 * t], vz[t] = kvrow[kHeadDim + lane + 32 * t];
        patch_row(stage, pos & (kTile - 1), kz, vz, lane);
      }
      tile_update<NT>(stage, valid, p.scale_log2, lane, qf, o, m_run, l_run);
      if (valid < kTile || i == i_new) fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty_bar[s]));
    }
  }

  // ------------------------------------------------------------------ merge
  // Each consumer warp's (m, l) per head go to shared memory; once all are there, every
  // warp rescales its own O (in registers) and l to the CTA's maximum m and stores them,
  // so that the CTA's partial of an element is a plain sum over the six warps.
  float *wpart = reinterpret_cast<float *>(smem);                          // [6][16][kPartStride]
  float *wml = wpart + kConsumerWarps * GQA_MAX_GROUP * kPartStride;       // [6][16][2]
  float *wm = wml + kConsumerWarps * GQA_MAX_GROUP * 2;                    // [6][16]
  __syncthreads();  // every issued tile has been consumed: the ring is free
  if (!producer && warp != kOrderWarp) {
    const int cw = warp;
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int g = 8 * t + 2 * lane + jj;
        if (lane < 4 && g < p.G) wm[cw * GQA_MAX_GROUP + g] = m_run[t][jj];
      }
  }
  __syncthreads();
  if (!producer && warp != kOrderWarp) {
    const int cw = warp;
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int g = 8 * t + 2 * (lane & 3) + jj;  // the head column this lane holds
        float M = -INFINITY;
#pragma unroll
        for (int c = 0; c < kConsumerWarps; ++c) M = fmaxf(M, wm[c * GQA_MAX_GROUP + (g < p.G ? g : 0)]);
        const float f = m_run[t][jj] == -INFINITY ? 0.f : exp2f(m_run[t][jj] - M);
        float l = l_run[t][jj] * f;
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        if (lane < 4 && g < p.G) {
          wml[(cw * GQA_MAX_GROUP + g) * 2 + 0] = M;
          wml[(cw * GQA_MAX_GROUP + g) * 2 + 1] = l;
        }
#pragma unroll
        for (int md = 0; md < 8; ++md) {
          o[md][t][jj] *= f;
          o[md][t][jj + 2] *= f;
        }
      }
#pragma unroll
    for (int md = 0; md < 8; ++md)
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int g = 8 * t + 2 * (lane & 3) + (e & 1);
          const int d = 16 * md + (lane >> 2) + ((e >> 1) << 3);
          if (g < p.G) wpart[(cw * GQA_MAX_GROUP + g) * kPartStride + d] = o[md][t][e];
        }
  }
  __syncthreads();
  // This CTA's partial per element -- (M, sum of the warps' rescaled l, sum of their
  // rescaled O) -- pushed straight to the CTA that owns the element's dims.
  const int E = p.G * kHeadDim;
  const uint32_t bar_local = smem_addr(recv_bar);
  if (tid == 0)  // this CTA's own receive phase: C senders x (G (m, l) pairs + G x nd floats)
    mbar_arrive_expect_tx(bar_local, static_cast<uint32_t>(C * p.G * (8 + 4 * nd)));
  cluster_wait();  // every CTA of the cluster has initialised its barriers
  for (int e = tid; e < E; e += kThreadsCluster) {
    const int g = e >> 7, d = e & (kHeadDim - 1);
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < kConsumerWarps; ++c) acc += wpart[(c * GQA_MAX_GROUP + g) * kPartStride + d];
    const int q = ((d + 1) * C - 1) / kHeadDim;  // the owner of dim d
    const int dq = q * kHeadDim / C, ndq = (q + 1) * kHeadDim / C - dq, dd = d - dq;
    const uint32_t bar_q = mapa_shared(bar_local, q);
    st_async_f32(mapa_shared(smem_addr(recv_o + (rank * p.G + g) * ndq + dd), q), acc, bar_q);
    if (dd == 0) {
      float den = 0.f;
#pragma unroll
      for (int c = 0; c < kConsumerWarps; ++c) den += wml[(c * GQA_MAX_GROUP + g) * 2 + 1];
      st_async_v2f32(mapa_shared(smem_addr(recv_ml + (rank * p.G + g) * 2), q), wml[g * 2], den, bar_q);
    }
  }
  // The owned dims: merge the C contributions and write them (global writes: after the
  // preceding kernel has completed).
  const bool got = mbar_wait(bar_local, 0);
  if (!got && (tid & 31) == 0) atomicOr(p.err, GQA_DEVERR_TIMEOUT);
  cluster_arrive_relaxed();  // this CTA has received everything (or given up)
  griddep_wait();
  if (qpub) publish_q<NT>(p, b, kv, lane, qkeep);
  // (Code that runs once per launch is kept compact: on a latency-bound step its
  // instruction fetches, not its arithmetic, set the time.)
  for (int e = tid; e < p.G * nd; e += kThreadsCluster) {
    const int g = e / nd, dd = e - g * nd;
    float M = -INFINITY;
#pragma unroll 1
    for (int r = 0; r < C; ++r) M = fmaxf(M, recv_ml[(r * p.G + g) * 2]);
    float acc = 0.f, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll 1
      for (int r = 0; r < C; ++r) {
        const float f = exp2f(recv_ml[(r * p.G + g) * 2] - M);
        acc = fmaf(f, recv_o[(r * p.G + g) * nd + dd], acc);
        den = fmaf(f, recv_ml[(r * p.G + g) * 2 + 1], den);
      }
    }
    const float v = den > 0.f ? acc / den : 0.f;  // zeros for an invalid length (flagged above)
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    p.out[(static_cast<long long>(b) * p.Hq + kv * p.G + g) * kHeadDim + d0 + dd] =
        *reinterpret_cast<const uint16_t *>(&h);
  }
  cluster_wait();  // every CTA has received everything: no store to or from this CTA is in flight
}

size_t attn_smem_bytes(int npad, int batch) {
  (void)npad;  // the rotated queries live in registers: the stage size does not depend on G
  const int stage = 4 * kHalfTileBytes;
  return 1024 + static_cast<size_t>(kStages) * stage + 16 * kStages + 4 * (batch + 1) + 8 * batch;
}

size_t attn_cluster_smem_bytes() { return kClusterSmemBytes; }

namespace {
using ClusterKernel = void (*)(CUtensorMap, CUtensorMap, AttnParams);
ClusterKernel cluster_kernel(int npad, bool order) {
  if (npad == 8) return order ? attn_cluster_kernel<1, true> : attn_cluster_kernel<1, false>;
  return order ? attn_cluster_kernel<2, true> : attn_cluster_kernel<2, false>;
}
}  // namespace

cudaError_t attn_configure(int npad) {
  const int bytes = static_cast<int>(attn_smem_bytes(npad, GQA_MAX_BATCH));
  const int cbytes = static_cast<int>(attn_cluster_smem_bytes());
  void (*split)(CUtensorMap, CUtensorMap, AttnParams) = npad == 8 ? attn_splitkv_kernel<1> : attn_splitkv_kernel<2>;
  cudaError_t e = cudaFuncSetAttribute(split, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  for (bool order : {false, true}) {
    const ClusterKernel single = cluster_kernel(npad, order);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(single, cudaFuncAttributeMaxDynamicSharedMemorySize, cbytes);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(single, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  }
  return e;
}

int attn_cluster_capacity(int npad, int csize) {
  const ClusterKernel single = cluster_kernel(npad, false);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(csize));
  cfg.blockDim = dim3(kThreadsCluster);
  cfg.dynamicSmemBytes = attn_cluster_smem_bytes();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(csize);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, single, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_attention_cluster(const CUtensorMap &tmK, const CUtensorMap &tmV, const AttnParams &p, int npad,
                                     bool pdl, cudaStream_t stream) {
  const ClusterKernel single = cluster_kernel(npad, p.seg_order != nullptr);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.B * p.Hkv * p.csize));
  cfg.blockDim = dim3(kThreadsCluster);
  cfg.dynamicSmemBytes = attn_cluster_smem_bytes();
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.csize);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, single, tmK, tmV, p);
}

cudaError_t launch_attention(const CUtensorMap &tmK, const CUtensorMap &tmV, const AttnParams &p, int npad,
                             int num_workers, bool pdl, cudaStream_t stream) {
  const size_t bytes = attn_smem_bytes(npad, p.B);
  if (npad == 8)
    return launch_ex(pdl, attn_splitkv_kernel<1>, dim3(num_workers), dim3(kThreadsAttn), bytes, stream, tmK, tmV, p);
  return launch_ex(pdl, attn_splitkv_kernel<2>, dim3(num_workers), dim3(kThreadsAttn), bytes, stream, tmK, tmV, p);
}

}  // namespace gqa
