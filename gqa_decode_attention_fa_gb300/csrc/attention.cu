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
//  * One CTA per SM: a producer warp streams 64-token K/V tiles (2 x 8 KiB each) with
//    3-D TMA loads (128-byte swizzle, no multicast) into a 6-stage mbarrier ring, plus
//    the group's rotated q (2-4 KiB bulk copy); six consumer warps each own one stage,
//    take every sixth tile, run the recurrence in registers and release the stage.
//  * Workers own contiguous, equal ranges of the batch's tiles (see gqa_common.cuh), so
//    ragged batches stay balanced; CTA 0 publishes the batch prefix for the combine.
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

// Appends sequence b's new token for KV head kv: k = RoPE_pos(RMSNorm(k_new)) in binary64
// rounded once to bf16, v = v_new, written to the cache row of position pos (skipped when
// the page id is out of range; the producer flags that) and returned per lane (dims
// lane + 32 t) for the shared-memory patch.
__device__ __forceinline__ void append_new_row(const AttnParams &p, int b, int kv, int pos, int lane,
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

template <int NT>
struct Cfg {
  static constexpr int kNpad = 8 * NT;
  static constexpr int kQBytes = kNpad * 256;
  static constexpr int kStageBytes = 4 * kHalfTileBytes + kQBytes;
  static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment for the 128B swizzle");
};

}  // namespace

template <int NT>
__global__ void __launch_bounds__(kThreadsAttn, 1)
    attn_splitkv_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const AttnParams p) {
  using C = Cfg<NT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + kStages * C::kStageBytes);
  uint64_t *empty_bar = full_bar + kStages;
  uint32_t *pre = reinterpret_cast<uint32_t *>(empty_bar + kStages);  // [B + 1]
  int32_t *Ls = reinterpret_cast<int32_t *>(pre + p.B + 1);           // [B], 0 if invalid

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
  if (warp == 0) {  // tile prefix over the batch
    uint32_t run = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int b = b0 + lane;
      uint32_t v = 0;
      if (b < p.B) {
        int L = p.seq_lens[b];
        const int nt = tiles_of(L, p.max_seq);
        if (nt == 0) {
          if (blockIdx.x == 0) atomicOr(p.err, GQA_DEVERR_SEQLEN);
          L = 0;
        }
        Ls[b] = L;
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

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------------- producer warp
    // The first kStages tiles' K/V loads go out before waiting on the prologue: they read
    // only the caller's cache (the prologue writes none of it; a tile holding a new
    // token's row is patched in shared memory by its consumer).  The rotated q follows
    // once the prologue has finished.
    if (n <= 0) {
      griddep_wait();
      griddep_launch_dependents();
      return;
    }
    const int npre = static_cast<int>(n < kStages ? n : kStages);
    int row = 0, kv = 0, seg = 0;
    if (lane < npre) describe(lane, row, kv, seg);
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
    griddep_wait();
    griddep_launch_dependents();
    for (int k = 0; k < npre; ++k) {
      const int r_seg = __shfl_sync(0xffffffffu, seg, k);
      if (lane == 0) {
        const uint32_t fb = smem_addr(&full_bar[k]);
        const uint32_t base = smem_addr(smem + k * C::kStageBytes);
        bulk_load(base + 4 * kHalfTileBytes, p.q_rot + static_cast<long long>(r_seg) * C::kNpad * kHeadDim,
                  C::kQBytes, fb);
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
        const int r_seg = __shfl_sync(0xffffffffu, seg, k);
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
            bulk_load(base + 4 * kHalfTileBytes, p.q_rot + static_cast<long long>(r_seg) * C::kNpad * kHeadDim,
                      C::kQBytes, fb);
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

  // The rotated q, the appended cache rows and the workspace belong to earlier kernels
  // until this returns.
  griddep_wait();
  griddep_launch_dependents();
  if (blockIdx.x == 0) {
    for (int i = tid; i <= p.B; i += kConsumerWarps * 32) p.prefix[i] = pre[i];
  }
  if (n <= 0) return;

  // ------------------------------------------------------------------ consumer warps
  const int cw = warp;
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

  // The new-token k/v rows this warp appends: the first two are computed now, while the
  // first tiles are still in flight, written to the cache and kept packed in registers for
  // the shared-memory patch; any further ones are computed when their tile arrives.
  long long ex0 = -1, ex1 = -1;
  uint32_t ek0[2] = {0, 0}, ev0[2] = {0, 0}, ek1[2] = {0, 0}, ev1[2] = {0, 0};
  {
    int b0, kv0, j0, b1, kv1, j1;
    locate(pre, Ls, p.B, p.Hkv, xs, b0, kv0, j0);
    locate(pre, Ls, p.B, p.Hkv, xe - 1, b1, kv1, j1);
    const int seg_first = b0 * p.Hkv + kv0, seg_last = b1 * p.Hkv + kv1;
    for (int sg = seg_first; sg <= seg_last && ex1 < 0; ++sg) {
      const int b = sg / p.Hkv, kv = sg - b * p.Hkv;
      const int L = Ls[b], pos = p.positions[b];
      if (L <= 0 || pos < 0 || pos >= L) continue;
      const int nt = (L + kTile - 1) / kTile;
      const long long x_new = static_cast<long long>(pre[b]) + static_cast<long long>(kv) * nt + pos / kTile;
      if (x_new < xs || x_new >= xe || (x_new - xs) % kConsumerWarps != cw) continue;
      uint16_t kz[4], vz[4];
      append_new_row(p, b, kv, pos, lane, kz, vz);
      if (ex0 < 0) {
        ex0 = x_new;
        ek0[0] = kz[0] | (uint32_t(kz[1]) << 16), ek0[1] = kz[2] | (uint32_t(kz[3]) << 16);
        ev0[0] = vz[0] | (uint32_t(vz[1]) << 16), ev0[1] = vz[2] | (uint32_t(vz[3]) << 16);
      } else {
        ex1 = x_new;
        ek1[0] = kz[0] | (uint32_t(kz[1]) << 16), ek1[1] = kz[2] | (uint32_t(kz[3]) << 16);
        ev1[0] = vz[0] | (uint32_t(vz[1]) << 16), ev1[1] = vz[2] | (uint32_t(vz[3]) << 16);
      }
    }
  }

  int cur_seg = -1;
  for (long long i = cw; i < n; i += kConsumerWarps) {
    int b, kv, j;
    locate(pre, Ls, p.B, p.Hkv, xs + i, b, kv, j);
    const int seg = b * p.Hkv + kv;
    const int pos_b = p.positions[b];
    if (seg != cur_seg) {
      if (cur_seg >= 0) flush(cur_seg);
      cur_seg = seg;
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
    const uint32_t qS = kLo + 4 * kHalfTileBytes;

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
    const bool holds_new = pos_b >= 0 && pos_b < Ls[b] && (pos_b >> 6) == j;
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
}

size_t attn_smem_bytes(int npad, int batch) {
  const int stage = 4 * kHalfTileBytes + npad * 256;
  return 1024 + static_cast<size_t>(kStages) * stage + 16 * kStages + 4 * (batch + 1) + 4 * batch;
}

cudaError_t attn_configure(int npad) {
  const int bytes = static_cast<int>(attn_smem_bytes(npad, GQA_MAX_BATCH));
  if (npad == 8) return cudaFuncSetAttribute(attn_splitkv_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  return cudaFuncSetAttribute(attn_splitkv_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t launch_attention(const CUtensorMap &tmK, const CUtensorMap &tmV, const AttnParams &p, int npad,
                             int num_workers, cudaStream_t stream) {
  const size_t bytes = attn_smem_bytes(npad, p.B);
  if (npad == 8)
    return launch_pdl(attn_splitkv_kernel<1>, dim3(num_workers), dim3(kThreadsAttn), bytes, stream, tmK, tmV, p);
  return launch_pdl(attn_splitkv_kernel<2>, dim3(num_workers), dim3(kThreadsAttn), bytes, stream, tmK, tmV, p);
}

}  // namespace gqa
