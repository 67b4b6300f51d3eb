// The decode step over a 4-bit KV cache (sm_103a).
//
// The cache format of "Qwen3-14B Optimization", section 2.3 (TurboQuant): every cache row
// (token, KV head) is 128 Lloyd-Max codebook indices, two per byte -- byte c holds
// idx[c + 64] * 16 + idx[c] -- dequantized by gather -> renormalize -> scale -> unrotate.
// Readings where the page is silent: the codebook is the caller's 16 bf16 levels; the
// rotation is R = H D / sqrt(d) (Sylvester Walsh-Hadamard H, caller's +-1 signs D); a row
// keeps one fp32 scale sigma = ||x|| / ||c[idx]||, so it dequantizes to
// x^ = sigma R^T c[idx].
//
// R is orthogonal, so the step never unrotates a cache row: with q~ = R q,
//   q . x^_t = sigma_t (q~ . c[idx_t])   and   sum_t p_t x^_t = R^T sum_t p_t sigma_t c[idx_t],
// i.e. the scores and the value sum run on the raw codewords in the rotated domain, and
// the merged output row is rotated back once.  Two forms, as for the bf16 cache: the
// single-launch form (q4_cluster_kernel, at the end of this file: the whole step in one
// launch, the merge on chip) and the split-KV form's three kernels:
//  * q4_prologue_kernel (one warp per row): q~ = R RoPE(RMSNorm(q_new)) in binary32,
//    kept as bf16 hi + lo (so that rounding q~ costs no accuracy); the new token's k row
//    RoPE(RMSNorm(k_new)) and v row quantized and appended (R by a fast Walsh-Hadamard
//    transform across the warp, the nearest level by the midpoint thresholds).
//  * q4_attn_kernel: the split-KV attention of attention.cu -- the same worker partition
//    and partial slots -- on 4 KB index tiles, through a 12-stage TMA ring whose stages
//    also carry the tile's per-token scales (cp.async) and its (sequence, head, length).
//    The consumer warp that owns a stage builds its mma fragments directly from a
//    256-entry table of codeword pairs (no expanded tile in shared memory), runs
//    S = K~ q~^T (hi and lo), scales each token's scores by its sigma_K, runs the online
//    softmax, folds sigma_V into P and accumulates O~ += C_V^T (P sigma_V)^T.
//  * q4_combine_kernel (combine.cu): the log-sum-exp merge, then R^T.
#include "launch.h"

namespace gqa {

namespace {

constexpr int kQ4TileBytes = kTile * 64;                 // 64 tokens x 64 bytes of indices
constexpr int kQ4StageBytes = 2 * kQ4TileBytes;          // K and V index tiles
constexpr int kQ4Stages = 2 * kConsumerWarps;          // ring depth: two stages per consumer warp
static_assert(kQ4Stages % kConsumerWarps == 0, "each stage must belong to exactly one consumer warp");
constexpr float kInvSqrtD = 0.08838834764831845f;        // 1 / sqrt(128)

// Smem: [12 stages][pair table, one copy per lane][per-stage scales][per-stage tile info]
// [barriers][prefix]
constexpr int kQ4OffStage = 0;
constexpr int kQ4OffPair = kQ4OffStage + kQ4Stages * kQ4StageBytes;
constexpr int kQ4PairBytes = 256 * 32 * 4;
constexpr int kQ4OffScale = kQ4OffPair + kQ4PairBytes;               // [stage][K, V][64] fp32
constexpr int kQ4OffInfo = kQ4OffScale + kQ4Stages * 2 * kTile * 4;  // [stage] int4
constexpr int kQ4OffBar = kQ4OffInfo + kQ4Stages * 16;

// Fast Walsh-Hadamard transform (Sylvester order) of a 128-vector held by a warp, lane l
// holding dims 4 l .. 4 l + 3: bits 0-1 of the dim within the lane, bits 2-6 across lanes.
__device__ __forceinline__ void fwht128(float (&v)[4], int lane) {
  float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
  v[0] = a0 + a2;
  v[1] = a1 + a3;
  v[2] = a0 - a2;
  v[3] = a1 - a3;
#pragma unroll
  for (int hb = 1; hb < 32; hb <<= 1) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float o = __shfl_xor_sync(0xffffffffu, v[u], hb);
      v[u] = (lane & hb) ? o - v[u] : v[u] + o;
    }
  }
}

// 4-byte asynchronous global -> shared copy, and the arrive-on that fires on the barrier
// once this thread's earlier copies have landed (no pending-count increment: the barrier's
// expected count includes these arrivals)
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void unpack4(uint2 w, float (&f)[4]) {
  f[0] = __uint_as_float(w.x << 16);
  f[1] = __uint_as_float(w.x & 0xffff0000u);
  f[2] = __uint_as_float(w.y << 16);
  f[3] = __uint_as_float(w.y & 0xffff0000u);
}

// Per-warp constants of the 4-bit row arithmetic, lane l holding dims 4 l .. 4 l + 3: the
// RoPE (cos, sin) of those dims' pairs at a position, the rotation's signs, the codebook
// and the midpoints between consecutive levels (exact in binary32).
struct Q4RowConsts {
  float cs_c[4], cs_s[4], sg[4], cb[16], thr[15];
};
__device__ __forceinline__ void q4_row_consts(const float2 *rope_tab32, int pos, const int8_t *signs,
                                              const uint16_t *codebook, int lane, Q4RowConsts &k) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    k.cs_c[u] = 1.f;
    k.cs_s[u] = 0.f;
  }
  if (pos >= 0) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float2 t = rope_tab32[static_cast<long long>(pos) * 64 + 4 * (lane & 15) + u];
      k.cs_c[u] = t.x;
      k.cs_s[u] = t.y;
    }
  }
  const char4 s4 = reinterpret_cast<const char4 *>(signs)[lane];
  k.sg[0] = s4.x;
  k.sg[1] = s4.y;
  k.sg[2] = s4.z;
  k.sg[3] = s4.w;
#pragma unroll
  for (int j = 0; j < 16; ++j) k.cb[j] = __uint_as_float(static_cast<uint32_t>(codebook[j]) << 16);
#pragma unroll
  for (int j = 0; j < 15; ++j) k.thr[j] = 0.5f * (k.cb[j] + k.cb[j + 1]);
}

// RMSNorm (optional weight) and RoPE of a bf16 row whose dims 4 l .. 4 l + 3 lane l holds
// (`bits`), binary32; the RoPE partner of dim e (e +- 64) is in lane l ^ 16.
__device__ __forceinline__ void q4_norm_rope(uint2 bits, const uint16_t *w, float eps, const Q4RowConsts &k, int lane,
                                             float (&z)[4]) {
  float x[4], y[4], ss = 0.f;
  unpack4(bits, x);
  float wv[4] = {1.f, 1.f, 1.f, 1.f};
  if (w) unpack4(reinterpret_cast<const uint2 *>(w)[lane], wv);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    ss = fmaf(x[u], x[u], ss);
    y[u] = x[u] * wv[u];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float rn = w ? 1.0f / sqrtf(ss * (1.0f / 128.0f) + eps) : 1.0f;
  const bool first_half = lane < 16;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float yp = __shfl_xor_sync(0xffffffffu, y[u], 16);
    z[u] = rn * (first_half ? fmaf(y[u], k.cs_c[u], -yp * k.cs_s[u]) : fmaf(y[u], k.cs_c[u], yp * k.cs_s[u]));
  }
}
__device__ __forceinline__ void q4_norm_rope(const uint16_t *src, const uint16_t *w, float eps, const Q4RowConsts &k,
                                             int lane, float (&z)[4]) {
  q4_norm_rope(reinterpret_cast<const uint2 *>(src)[lane], w, eps, k, lane, z);
}

// Quantizes a row z: t = sqrt(d) R z / ||z||, idx = the nearest level (the lower one on a
// tie); the indices packed into bytes 4 l .. 4 l + 3 (lanes < 16) and sigma.
__device__ __forceinline__ void q4_quantize(const float (&z)[4], const Q4RowConsts &k, int lane, uint32_t &packed,
                                            float &sigma) {
  float ss = 0.f, y[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    ss = fmaf(z[u], z[u], ss);
    y[u] = k.sg[u] * z[u];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float s = sqrtf(ss);
  fwht128(y, lane);  // H D z = sqrt(d) R z
  int idx[4];
  float cn = 0.f;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float t = s > 0.f ? y[u] / s : 0.f;  // sqrt(d) (R z)_i / ||z||
    int j = 0;
    float cj = k.cb[0];  // the chosen level, selected in registers (no indexed local array)
#pragma unroll
    for (int q = 0; q < 15; ++q) {
      const bool above = k.thr[q] < t;
      j += above ? 1 : 0;
      cj = above ? k.cb[q + 1] : cj;
    }
    idx[u] = j;
    cn = fmaf(cj, cj, cn);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cn += __shfl_xor_sync(0xffffffffu, cn, o);
  sigma = s > 0.f ? s / sqrtf(cn) : 0.f;
  const uint32_t mine = idx[0] | (idx[1] << 8) | (idx[2] << 16) | (idx[3] << 24);
  const uint32_t hi = __shfl_xor_sync(0xffffffffu, mine, 16);  // dims + 64 from lane l + 16
  packed = mine | (hi << 4);
}

// q~ = R bf16(z) = H D bf16(z) / sqrt(d) (q is a bf16 activation), in place.
__device__ __forceinline__ void q4_rotate_query(float (&z)[4], const Q4RowConsts &k, int lane) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const __nv_bfloat16 zq = __float2bfloat16_rn(z[u]);
    z[u] = k.sg[u] * __bfloat162float(zq);
  }
  fwht128(z, lane);
#pragma unroll
  for (int u = 0; u < 4; ++u) z[u] *= kInvSqrtD;
}

}  // namespace

// ----------------------------------------------------------------------------- prologue
// One warp per row: CTA (b, y) of 8 warps handles rows 8 y .. 8 y + 7 of sequence b's H_q
// query rows, then its H_kv key rows, then its H_kv value rows.  Lane l holds dims 4 l .. 4 l + 3; the
// RoPE partner of dim e (e +- 64) is in lane l ^ 16.
// The kernel waits on the preceding kernel in the stream only at its end.  That kernel is
// the previous step's combine (which lets this one start once the previous attention
// kernel has finished, so the rotated-query buffer and the cache are free) or a kernel of
// the caller (which has then finished); a RoPE table rebuild is ordered before it by a
// plain launch.  The wait at the end keeps this grid from completing before the previous
// combine has read its partials, which the next attention kernel overwrites.
__global__ void __launch_bounds__(256) q4_prologue_kernel(const Q4PrologueParams p) {
  griddep_launch_dependents();
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.y * 8 + warp;  // this warp's row
  if (r >= p.Hq + 2 * p.Hkv) {
    griddep_wait();
    return;
  }
  const int L = p.seq_lens[b], pos = p.positions[b];
  const bool len_ok = L >= 1 && L <= p.max_seq;
  const bool pos_ok = len_ok && pos >= 0 && pos < L;
  if (threadIdx.x == 0 && blockIdx.y == 0) {
    if (!len_ok) atomicOr(p.err, GQA_DEVERR_SEQLEN);
    else if (!pos_ok) atomicOr(p.err, GQA_DEVERR_POSITION);
  }
  long long crow = -1;
  if (pos_ok) {
    if (p.paged) {
      const int pg = p.page_table[static_cast<long long>(b) * p.max_blocks + pos / kTile];
      if (pg >= 0 && pg < p.num_blocks) crow = static_cast<long long>(pg) * kTile + (pos & (kTile - 1));
      else if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(p.err, GQA_DEVERR_PAGE);
    } else {
      crow = static_cast<long long>(b) * p.max_seq + pos;
    }
  }
  Q4RowConsts kc;
  q4_row_consts(p.rope_tab32, pos_ok ? pos : -1, p.signs, p.codebook, lane, kc);

  {
    if (r < p.Hq) {
      const long long row = static_cast<long long>(b) * p.Hq + r;
      float z[4] = {0.f, 0.f, 0.f, 0.f};
      if (pos_ok) {
        q4_norm_rope(p.q_new + row * kHeadDim, p.q_norm_w, p.eps, kc, lane, z);
        q4_rotate_query(z, kc, lane);
      }
      uint32_t h[2], l[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        h[u] = pack_bf16(z[2 * u], z[2 * u + 1]);
        l[u] = pack_bf16(z[2 * u] - bf16_lo_to_float(h[u]), z[2 * u + 1] - bf16_hi_to_float(h[u]));
      }
      reinterpret_cast<uint2 *>(p.q_hi + row * kHeadDim)[lane] = make_uint2(h[0], h[1]);
      reinterpret_cast<uint2 *>(p.q_lo + row * kHeadDim)[lane] = make_uint2(l[0], l[1]);
    } else if (crow >= 0) {
      const bool is_k = r < p.Hq + p.Hkv;
      const int kv = is_k ? r - p.Hq : r - p.Hq - p.Hkv;
      const long long nrow = static_cast<long long>(b) * p.Hkv + kv;
      float z[4];
      if (is_k) {
        q4_norm_rope(p.k_new + nrow * kHeadDim, p.k_norm_w, p.eps, kc, lane, z);
      } else {
        unpack4(reinterpret_cast<const uint2 *>(p.v_new + nrow * kHeadDim)[lane], z);
      }
      uint32_t packed;
      float sigma;
      q4_quantize(z, kc, lane, packed, sigma);
      const long long crow_kv = crow * p.Hkv + kv;
      uint8_t *dst = (is_k ? p.k_idx : p.v_idx) + crow_kv * 64;
      if (lane < 16) reinterpret_cast<uint32_t *>(dst)[lane] = packed;
      if (lane == 0) (is_k ? p.k_scale : p.v_scale)[crow_kv] = sigma;
    }
  }
  griddep_wait();
}

// ----------------------------------------------------------------------------- attention
namespace {

__device__ __forceinline__ void q4_locate(const uint32_t *pre, const int32_t *Ls, int B, long long x, int &b,
                                          int &kv, int &j) {
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

}  // namespace

// One 64-token index tile of the 4-bit recurrence for a warp's G heads: kt holds the K and
// V index tiles ([64 tokens][64 bytes] each), sk / sv the tokens' sigma_K * scale (log2
// domain) and sigma_V for this lane's 8 tokens (16 mt + lane / 4 + 8 h), 0 past the
// length.  S = C_K q~^T with q~ as bf16 hi + lo, the online-softmax update of (m, l, O~)
// and O~^T += C_V^T (P sigma_V)^T, with the mma fragments built from pair-table lookups
// (the dim orders are described at the consumer loop of q4_attn_kernel).
//
// The pair table holds one copy of its 256 entries per lane.  kWide = false: entry e of
// lane l at tbl + 128 e (tbl = the table's shared address + 4 l), so a lookup is a byte
// permute, a shift-add and the load.  kWide = true: the table starts on a 64 KiB boundary T
// of the shared window with entries 256 bytes apart, tbl = T + 4 l, and one byte permute
// that puts the index byte into bits 8-15 of tbl gives the address (T has zero low 16 bits
// and lies below 2^18), so a lookup is two instructions.
template <int NT, bool kWide>
__device__ __forceinline__ void q4_tile_update(const uint8_t *kt, int valid, const float (&sk)[4][2],
                                               const float (&sv)[4][2], uint32_t tbl, int lane,
                                               const uint32_t (&qh)[8][NT][2], const uint32_t (&ql)[8][NT][2],
                                               float (&o)[8][NT][4], float (&m_run)[NT][2], float (&l_run)[NT][2]) {
  const int r8 = lane >> 2, c4 = lane & 3;
  auto pair_entry = [&](uint32_t w, int k) {
    uint32_t a;
    if constexpr (kWide) {
      a = __byte_perm(w, tbl, 0x7604u | (static_cast<uint32_t>(k) << 4));  // bytes: tbl.0, w.k, tbl.2, tbl.3
    } else {
      a = tbl + (__byte_perm(w, 0u, 0x4440u | static_cast<uint32_t>(k)) << 7);
    }
    uint32_t v;
    asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
  };
  const uint8_t *vt = kt + kQ4TileBytes;

  // S^T = C_K q~^T (hi and lo parts of q~; with one head block in two accumulators, so
  // that the two mma chains interleave): 4 token blocks of 16 x NT head blocks of 8
  float sacc[4][NT][4], sacl[4][NT][4];
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[mt][nt][e] = sacl[mt][nt][e] = 0.f;
  // tokens 16 mt + r (A rows 0-7) and + 8 (rows 8-15), index bytes 16 c .. 16 c + 15; the
  // token blocks innermost, so that consecutive mma feed different accumulators
  uint32_t xk[4][2][4];
#pragma unroll
  for (int mt = 0; mt < 4; ++mt) {
    const uint4 w0 = *reinterpret_cast<const uint4 *>(kt + (16 * mt + r8) * 64 + 16 * c4);
    const uint4 w1 = *reinterpret_cast<const uint4 *>(kt + (16 * mt + r8 + 8) * 64 + 16 * c4);
    xk[mt][0][0] = w0.x, xk[mt][0][1] = w0.y, xk[mt][0][2] = w0.z, xk[mt][0][3] = w0.w;
    xk[mt][1][0] = w1.x, xk[mt][1][1] = w1.y, xk[mt][1][2] = w1.z, xk[mt][1][3] = w1.w;
  }
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const int wd = ks >> 1, k0 = 2 * (ks & 1);  // bytes 2 ks and 2 ks + 1
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const uint32_t a0 = pair_entry(xk[mt][0][wd], k0), a2 = pair_entry(xk[mt][0][wd], k0 + 1);
      const uint32_t a1 = pair_entry(xk[mt][1][wd], k0), a3 = pair_entry(xk[mt][1][wd], k0 + 1);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma_bf16(sacc[mt][nt], a0, a1, a2, a3, qh[ks][nt][0], qh[ks][nt][1]);
        mma_bf16(NT == 1 ? sacl[mt][nt] : sacc[mt][nt], a0, a1, a2, a3, ql[ks][nt][0], ql[ks][nt][1]);
      }
    }
  }
  if constexpr (NT == 1) {
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[mt][0][e] += sacl[mt][0][e];
  }

  // sigma_K * scale (log2 domain) per token, and the mask past the length
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = 16 * mt + (lane >> 2) + ((e >> 1) << 3);
        sacc[mt][nt][e] = tok < valid ? sacc[mt][nt][e] * sk[mt][e >> 1] : -INFINITY;
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
  // P = 2^(s - m) (l sums P), then P sigma_V split into bf16 hi + lo, transposed into B
  // fragments of (P sigma_V)^T
  uint32_t ph[4][NT][2], pl[4][NT][2];
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float pv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float pe = fast_exp2(sacc[mt][nt][e] - m_run[nt][e & 1]);
        l_run[nt][e & 1] += pe;
        pv[e] = pe * sv[mt][e >> 1];
      }
      const uint32_t h01 = pack_bf16(pv[0], pv[1]), h23 = pack_bf16(pv[2], pv[3]);
      const uint32_t l01 = pack_bf16(pv[0] - bf16_lo_to_float(h01), pv[1] - bf16_hi_to_float(h01));
      const uint32_t l23 = pack_bf16(pv[2] - bf16_lo_to_float(h23), pv[3] - bf16_hi_to_float(h23));
      // lanes with odd c hold their two k-slots (tokens) swapped, as their V index rows are
      // loaded below (both mma operands of a k-slot pair come from lanes of the same c)
      const uint32_t sw = (c4 & 1) ? 0x1032u : 0x3210u;
      ph[mt][nt][0] = __byte_perm(movmatrix_t(h01), 0u, sw);
      ph[mt][nt][1] = __byte_perm(movmatrix_t(h23), 0u, sw);
      pl[mt][nt][0] = __byte_perm(movmatrix_t(l01), 0u, sw);
      pl[mt][nt][1] = __byte_perm(movmatrix_t(l23), 0u, sw);
    }
  // O~^T += C_V^T (P sigma_V)^T: 4 token k-steps x 8 dim blocks of 16 (rows 8 r + md and
  // 64 + 8 r + md); tokens t0, t0 + 1 (k-slots 2 c, +1) and t0 + 8, t0 + 9 (slots + 8).
  // Lanes with odd c take the rows of a token pair in the other order (t0 + 1 first), so
  // that each 8-byte load touches two even and two odd 64-byte rows, i.e. all 32 banks;
  // their P fragments were swapped to match.
  const int tswap = c4 & 1;
#pragma unroll
  for (int mt = 0; mt < 4; ++mt) {
    const int t0 = 16 * mt + 2 * c4;
    const uint8_t *vr = vt + t0 * 64 + 8 * r8;
    const uint2 y0 = *reinterpret_cast<const uint2 *>(vr + tswap * 64);
    const uint2 y1 = *reinterpret_cast<const uint2 *>(vr + (1 - tswap) * 64);
    const uint2 y2 = *reinterpret_cast<const uint2 *>(vr + (8 + tswap) * 64);
    const uint2 y3 = *reinterpret_cast<const uint2 *>(vr + (9 - tswap) * 64);
#pragma unroll
    for (int hw = 0; hw < 2; ++hw) {
      const uint32_t u0 = hw ? y0.y : y0.x, u1 = hw ? y1.y : y1.x, u2 = hw ? y2.y : y2.x, u3 = hw ? y3.y : y3.x;
      // byte m of each: entry (nibble of token t) | (same nibble of token t + 1) << 4
      const uint32_t lo01 = (u0 & 0x0f0f0f0fu) | ((u1 << 4) & 0xf0f0f0f0u);
      const uint32_t hi01 = ((u0 >> 4) & 0x0f0f0f0fu) | (u1 & 0xf0f0f0f0u);
      const uint32_t lo23 = (u2 & 0x0f0f0f0fu) | ((u3 << 4) & 0xf0f0f0f0u);
      const uint32_t hi23 = ((u2 >> 4) & 0x0f0f0f0fu) | (u3 & 0xf0f0f0f0u);
      // the four dim blocks' hi products, then their lo products (no accumulator is
      // used by two consecutive mma)
      uint32_t av[4][4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        av[m][0] = pair_entry(lo01, m), av[m][1] = pair_entry(hi01, m);
        av[m][2] = pair_entry(lo23, m), av[m][3] = pair_entry(hi23, m);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int m = 0; m < 4; ++m)
          mma_bf16(o[4 * hw + m][nt], av[m][0], av[m][1], av[m][2], av[m][3], ph[mt][nt][0], ph[mt][nt][1]);
#pragma unroll
        for (int m = 0; m < 4; ++m)
          mma_bf16(o[4 * hw + m][nt], av[m][0], av[m][1], av[m][2], av[m][3], pl[mt][nt][0], pl[mt][nt][1]);
      }
    }
  }
}

template <int NT>
__global__ void __launch_bounds__(kThreadsAttn, 1)
    q4_attn_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const Q4AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align_smem_1024(smem_raw);
  uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + kQ4OffBar);
  uint64_t *empty_bar = full_bar + kQ4Stages;
  // pair table: entry (a | b << 4) = bf16 c[a] | bf16 c[b] << 16, the codewords of two
  // adjacent dims from their two nibbles; 32 copies interleaved word by word, lane l
  // reading copy l (word 32 e + l, always bank l), so random entries never conflict
  uint32_t *cpair = reinterpret_cast<uint32_t *>(smem + kQ4OffPair);  // [256][32]
  float *scl = reinterpret_cast<float *>(smem + kQ4OffScale);        // [stage][2][64]
  int4 *info = reinterpret_cast<int4 *>(smem + kQ4OffInfo);           // [stage]
  uint32_t *pre = reinterpret_cast<uint32_t *>(empty_bar + kQ4Stages);  // [B + 1]
  int32_t *Ls = reinterpret_cast<int32_t *>(pre + p.B + 1);            // [B]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kQ4Stages; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1 + 32);  // the TMA issue + one arrive per producer lane
      mbar_init(smem_addr(&empty_bar[s]), 1);
    }
    fence_barrier_init();
  }
  if (warp == kConsumerWarps && lane == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  for (int e = tid; e < 256 * 32; e += blockDim.x) {
    const int v = e >> 5;
    cpair[e] = static_cast<uint32_t>(p.codebook[v & 15]) | (static_cast<uint32_t>(p.codebook[v >> 4]) << 16);
  }
  griddep_wait();  // the prologue kernel appended the new rows and wrote q~
  if (warp == 0) {  // tile prefix over the batch
    uint32_t run = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int b = b0 + lane;
      uint32_t v = 0;
      if (b < p.B) {
        const int L = p.seq_lens[b];
        const int nt = tiles_of(L, p.max_seq);
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

  const long long T = pre[p.B];
  const int W = gridDim.x, w = blockIdx.x;
  const long long xs = worker_begin(T, W, w), xe = worker_begin(T, W, w + 1);
  const long long n = xe - xs;
  auto tile_row = [&](int b, int j) {
    if (!p.paged) return b * p.max_seq + j * kTile;
    const int pg = p.page_table[static_cast<long long>(b) * p.max_blocks + j];
    if (pg < 0 || pg >= p.num_blocks) {
      atomicOr(p.err, GQA_DEVERR_PAGE);
      return -kTile;  // the whole box out of bounds: TMA fills zeros
    }
    return pg * kTile;
  };

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------------- producer warp
    // Lane l looks up tile i0 + l of the next 32 (sequence, head, page, length), so that
    // one page-table round trip serves 32 tiles; then per tile lane 0 stores the tile's
    // info and issues the two index-tile TMAs, and every lane copies the scales of tokens
    // l and l + 32 (the ones inside the sequence) with cp.async, whose arrivals complete
    // the stage with the TMA bytes.
    long long issued = 0;
    bool ok = true;
    for (long long i0 = 0; i0 < n && ok; i0 += 32) {
      int mb = 0, mkv = 0, mrow = -kTile, mvalid = 0;
      if (i0 + lane < n) {
        int mj;
        q4_locate(pre, Ls, p.B, xs + i0 + lane, mb, mkv, mj);
        mrow = tile_row(mb, mj);
        mvalid = min(kTile, Ls[mb] - mj * kTile);
      }
      const int cnt = static_cast<int>(min(32LL, n - i0));
      for (int u = 0; u < cnt; ++u) {
        const long long i = i0 + u;
        const int b = __shfl_sync(0xffffffffu, mb, u), kv = __shfl_sync(0xffffffffu, mkv, u);
        const int row = __shfl_sync(0xffffffffu, mrow, u), valid = __shfl_sync(0xffffffffu, mvalid, u);
        const int s = static_cast<int>(i % kQ4Stages);
        if (i >= kQ4Stages) ok = mbar_wait(smem_addr(&empty_bar[s]), static_cast<uint32_t>(((i / kQ4Stages) - 1) & 1));
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const uint32_t fb = smem_addr(&full_bar[s]);
        if (lane == 0) {
          info[s] = make_int4(b, kv, valid, row >= 0 ? 1 : 0);
          const uint32_t base = smem_addr(smem + kQ4OffStage + s * kQ4StageBytes);
          mbar_arrive_expect_tx(fb, kQ4StageBytes);
          tma_load_3d(base, &tmK, fb, 0, kv, row);
          tma_load_3d(base + kQ4TileBytes, &tmV, fb, 0, kv, row);
        }
        const uint32_t sdst = smem_addr(scl + s * 2 * kTile);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int tok = lane + 32 * hh;
          if (tok < valid && row >= 0) {
            const long long r = (static_cast<long long>(row) + tok) * p.Hkv + kv;
            cp_async4(sdst + 4 * tok, p.k_scale + r);
            cp_async4(sdst + 4 * (kTile + tok), p.v_scale + r);
          }
        }
        cp_async_arrive_noinc(fb);
        issued = i + 1;
      }
    }
    if (!ok) {
      if (lane == 0) {
        atomicOr(p.err, GQA_DEVERR_TIMEOUT);
        for (long long ii = (issued > kQ4Stages ? issued - kQ4Stages : 0); ii < issued; ++ii)
          (void)mbar_wait(smem_addr(&full_bar[ii % kQ4Stages]), static_cast<uint32_t>((ii / kQ4Stages) & 1));
      }
    }
    cp_async_wait_all();
    return;
  }

  // ------------------------------------------------------------------ consumer warps
  // The mma fragments of the codeword tiles come straight from pair-table lookups, with no
  // expanded tile in shared memory: each A register is two bf16 codewords, i.e. one
  // lookup, once the dims are ordered so that the two nibbles of a lookup are
  //  * for S = C_K q~^T (contraction over dims): the two nibbles of one index byte --
  //    k-slot pair (2 c, 2 c + 1) of k-step ks for lane group c holds dims (j, j + 64) with
  //    j = 16 c + 2 ks (and j + 1 for slots 8 + 2 c, +1), so a lane reads its token's 16
  //    index bytes 16 c .. 16 c + 15 in one load and each byte is a table entry; q~ is
  //    loaded in the same order;
  //  * for O~^T = C_V^T (P sigma_V)^T (contraction over tokens): the same nibble of two
  //    consecutive tokens -- row r of dim block md is dim 8 r + md (rows 8..15: 64 + 8 r
  //    + md), so a lane reads 8 index bytes per token row and forms four entries per
  //    word with two logic operations; the accumulator rows are written back in natural
  //    dim order by the flush.
  const int cw = warp;
  // Entry of byte k of w in this lane's copy of the table: the byte moved down by a byte
  // permute, then one shift-add onto the lane's 32-bit shared address.  The table is
  // constant after the start-up barrier, so the load is a plain (reorderable) asm.
  const uint32_t tbl_lane = smem_addr(cpair) + 4u * lane;
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
          const int d = ((e >> 1) << 6) + 8 * (lane >> 2) + md;
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

  const int r8 = lane >> 2, c4 = lane & 3;
  uint32_t qh[8][NT][2], ql[8][NT][2];
  int cur_seg = -1;
  for (long long i = cw; i < n; i += kConsumerWarps) {
    const int s = static_cast<int>(i % kQ4Stages);
    const bool ready = mbar_wait(smem_addr(&full_bar[s]), static_cast<uint32_t>((i / kQ4Stages) & 1));
    __syncwarp();
    if (!__all_sync(0xffffffffu, ready)) {
      if (lane == 0) atomicOr(p.err, GQA_DEVERR_TIMEOUT);
      return;
    }
    const int4 ti = info[s];
    const int b = ti.x, kv = ti.y, valid = ti.z;
    const bool page_ok = ti.w != 0;
    const int sg = b * p.Hkv + kv;
    if (sg != cur_seg) {
      if (cur_seg >= 0) flush(cur_seg);
      cur_seg = sg;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int g = 8 * nt + r8;
        const long long row = (static_cast<long long>(b) * p.Hq + kv * p.G + g) * kHeadDim;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int j = 16 * c4 + 2 * ks + hf;  // dims j (low half) and j + 64 (high half)
            uint32_t vh = 0u, vl = 0u;
            if (g < p.G) {
              vh = static_cast<uint32_t>(p.q_hi[row + j]) | (static_cast<uint32_t>(p.q_hi[row + j + 64]) << 16);
              vl = static_cast<uint32_t>(p.q_lo[row + j]) | (static_cast<uint32_t>(p.q_lo[row + j + 64]) << 16);
            }
            qh[ks][nt][hf] = vh;
            ql[ks][nt][hf] = vl;
          }
      }
    }
    // per-token scales of this lane's 8 tokens (16 mt + lane / 4 + 8 h), staged with the
    // tile; 0 past the length and on a page outside the pool (its tiles read as zeros)
    float sk[4][2], sv[4][2];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int tok = 16 * mt + r8 + 8 * hh;
        const bool in = tok < valid && page_ok;
        sk[mt][hh] = in ? scl[s * 2 * kTile + tok] * p.scale_log2 : 0.f;
        sv[mt][hh] = in ? scl[s * 2 * kTile + kTile + tok] : 0.f;
      }
    q4_tile_update<NT, false>(smem + kQ4OffStage + s * kQ4StageBytes, valid, sk, sv, tbl_lane, lane, qh, ql, o, m_run,
                       l_run);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty_bar[s]));  // the stage's index tiles are consumed
  }
  if (cur_seg >= 0) flush(cur_seg);
}

// ------------------------------------------------------------------ single-launch form
// The whole 4-bit step in one launch, as the bf16 step's single-launch form (attention.cu):
// one thread-block cluster of C CTAs per (sequence, KV head), CTA rank r streaming the
// segment's index tiles r, r + C, ...  The prologue is folded in: the consumer warps
// compute the segment's rotated queries q~ into shared memory, and an ordering warp
// quantizes the new k and v rows, hands them to the consumer whose tile holds them, waits
// on the preceding kernel, appends them, fences them and lets the next kernel launch.  The
// merge is partitioned by query head (CTA q owns the heads g with g mod C = q): every CTA
// pushes its partial of a head to the head's owner with remote st.async stores counted on
// the owner's mbarrier, and the owner merges the C contributions, rotates the row back
// (R^T: a Walsh-Hadamard transform across a warp) and writes it in bf16.  The ordering and
// cluster protocol are the bf16 kernel's: only the global writes (the append and `out`)
// wait on the preceding kernel, no thread leaves early, every mbarrier wait is bounded.
namespace {
constexpr int kQ4CPartStride = 132;                                       // floats per (warp, head) row
constexpr int kQ4CTableBytes = 65536;
constexpr int kQ4CRecvRows = 2 * GQA_MAX_GROUP;                           // C x ceil(G / C) <= G + C - 1
// Warps and shared memory of q4_cluster_kernel<NT>: six consumer warps, a producer warp
// and an ordering warp; a ring of two stages per consumer warp (a stage is always consumed
// by the same warp, so that a warp never waits on a stage barrier two phases ahead).
// (Eight consumer warps with sixteen stages measured slower: 70.8 against 65.0 us on the
// ragged 4-bit batch.)
//
// Layout.  The pair table (the wide form of q4_tile_update: 256 entries x 256 bytes) starts
// at T, the first 64 KiB boundary of the shared window at or after the 1024-aligned base A.
// The ring's stages fill [A, T) as far as whole stages fit (n1 of them, n1 <= 7 because
// T - A < 64 KiB) and continue after the table; the rest follows them:
//   [stages 0 .. n1-1][unused < 8 KiB][table, 64 KiB][stages n1 .. 11][misc]
// with misc = [scales][tile info][q~][new rows][receive area][barriers].  The whole layout
// takes at most 64 KiB + 12 stages + 7 KiB + misc from A.  After the tile loop the table's
// space holds the merge's warp partials.
template <int NT>
struct Q4C {
  static constexpr int kWarps = kConsumerWarps;
  static constexpr int kStages = 2 * kWarps;
  static constexpr int kOrderWarp = kWarps + 1;
  static constexpr int kThreads = 32 * (kWarps + 2);
  static constexpr int kMiscScale = 0;                                           // [stage][K, V][64] fp32
  static constexpr int kMiscInfo = kMiscScale + kStages * 2 * kTile * 4;         // [stage] page inside the pool
  static constexpr int kMiscQ = kMiscInfo + 4 * kStages;                         // [hi, lo][16][128] bf16 q~
  static constexpr int kMiscNew = kMiscQ + 2 * GQA_MAX_GROUP * kHeadDim * 2;     // new K, V index rows, sigmas
  static constexpr int kMiscRecv = kMiscNew + 256;                               // [C x owned][2], [..][128]
  static constexpr int kMiscBar = kMiscRecv + kQ4CRecvRows * (2 + kHeadDim) * 4;
  static constexpr int kMiscBytes = kMiscBar + 8 * (2 * kStages + 1);
  static constexpr size_t kSmemBytes =
      1024 + kQ4CTableBytes + kStages * kQ4StageBytes + (kQ4StageBytes - 1024) + kMiscBytes;
  // the merge's partials: [W][16][132] O, [W][16][2] (m, l), [W][16] m
  static constexpr int kPartBytes = kWarps * GQA_MAX_GROUP * (kQ4CPartStride + 2 + 1) * 4;
  static_assert(kMiscQ % 16 == 0 && kMiscRecv % 16 == 0 && kMiscBar % 8 == 0, "misc alignment");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert(kPartBytes <= kQ4CTableBytes, "the partials fit in the table's space");
};

// Barrier 1: the ordering warp hands the new rows to the consumer whose tile holds them;
// barrier 2: the consumer warps' rotated queries are in shared memory.
__device__ __forceinline__ void q4c_newrow_arrive() { asm volatile("bar.arrive 1, 64;" ::: "memory"); }
__device__ __forceinline__ void q4c_newrow_sync() { asm volatile("bar.sync 1, 64;" ::: "memory"); }
template <int W>
__device__ __forceinline__ void q4c_consumers_sync() {
  asm volatile("bar.sync 2, %0;" ::"n"(32 * W) : "memory");
}
// Heads of a segment owned by cluster rank q: g = q, q + C, ...
__device__ __forceinline__ int q4c_owned(int G, int C, int q) { return q < G ? (G - q + C - 1) / C : 0; }
}  // namespace

// kOrder: the launch order of the segments comes from p.seg_order.
template <int NT, bool kOrder>
__global__ void __launch_bounds__(Q4C<NT>::kThreads, 1)
    q4_cluster_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const Q4ClusterParams p) {
  using K = Q4C<NT>;
  constexpr int kW = K::kWarps, kS = K::kStages, kThreads = K::kThreads;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align_smem_1024(smem_raw);
  // the layout described above (the same in every CTA of the launch)
  const uint32_t base_a = smem_addr(smem);
  const uint32_t region1 = ((base_a + 0xFFFFu) & ~0xFFFFu) - base_a;   // T - A
  const int n1 = static_cast<int>(region1 / kQ4StageBytes);            // stages before the table (< 8)
  uint8_t *table = smem + region1;
  uint8_t *region2 = table + kQ4CTableBytes;
  uint8_t *misc = region2 + (kS - n1) * kQ4StageBytes;
  auto stage_ptr = [&](int s) -> uint8_t * {
    return s < n1 ? smem + s * kQ4StageBytes : region2 + (s - n1) * kQ4StageBytes;
  };
  uint64_t *full_bar = reinterpret_cast<uint64_t *>(misc + K::kMiscBar);
  uint64_t *empty_bar = full_bar + kS;
  uint64_t *recv_bar = empty_bar + kS;
  uint32_t *cpair = reinterpret_cast<uint32_t *>(table);              // [256][64]: lane copies in [0, 32)
  float *scl = reinterpret_cast<float *>(misc + K::kMiscScale);       // [stage][2][64]
  int *pinfo = reinterpret_cast<int *>(misc + K::kMiscInfo);          // [stage]
  uint16_t *qbuf = reinterpret_cast<uint16_t *>(misc + K::kMiscQ);     // [2][16][128]
  uint32_t *newrow = reinterpret_cast<uint32_t *>(misc + K::kMiscNew); // K words [16], V words [16], sigmas
  float *recv_ml = reinterpret_cast<float *>(misc + K::kMiscRecv);    // [C x owned][2]
  float *recv_o = recv_ml + 2 * kQ4CRecvRows;                         // [C x owned][128]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = p.csize;
  const int rank = static_cast<int>(cluster_ctarank());
  const int seg = kOrder ? p.seg_order[blockIdx.x / C] : static_cast<int>(blockIdx.x) / C;
  const int b = seg / p.Hkv, kv = seg - b * p.Hkv;
  const bool producer = warp == kW;

  if (producer && lane == 0) {
    for (int s = 0; s < kS; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1 + 32);  // the TMA issue + one arrive per producer lane
      mbar_init(smem_addr(&empty_bar[s]), 1);
    }
    mbar_init(smem_addr(recv_bar), 1);
    fence_barrier_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  // The segment's length and new-token position, then the rows that do not depend on the
  // position -- a consumer warp's first query head, the ordering warp's new k and v rows --
  // requested before the pair table is built, so that their latencies overlap it.
  int L = p.seq_lens[b], pos = p.positions[b];
  uint2 xraw = make_uint2(0u, 0u), vraw = make_uint2(0u, 0u);
  {
    const long long krow = (static_cast<long long>(b) * p.Hkv + kv) * kHeadDim;
    if (warp < kW && warp < p.G) {
      xraw = reinterpret_cast<const uint2 *>(p.q_new + (static_cast<long long>(b) * p.Hq + kv * p.G + warp) *
                                                           kHeadDim)[lane];
    } else if (warp == K::kOrderWarp) {
      xraw = reinterpret_cast<const uint2 *>(p.k_new + krow)[lane];
      vraw = reinterpret_cast<const uint2 *>(p.v_new + krow)[lane];
    }
  }
  {
    // the pair table: entry v = (c[v & 15], c[v >> 4]) in each lane's copy, four copies
    // (16 bytes) a store; thread t writes entries v = t / 8 + 32 k (k < 8), copies
    // 4 (t mod 8) .. + 3, so its low codeword c[(t / 8) mod 16] is the same for all eight
    static_assert(kThreads == 256, "pair-table build layout");
    const int c0 = 4 * (tid & 7);
    const uint32_t lo = p.codebook[(tid >> 3) & 15];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int v = (tid >> 3) + 32 * k;
      const uint32_t e = lo | (static_cast<uint32_t>(p.codebook[v >> 4]) << 16);
      *reinterpret_cast<uint4 *>(&cpair[v * 64 + c0]) = make_uint4(e, e, e, e);
    }
  }
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
  int owner = -1;  // the consumer warp whose tile holds the new token
  if (pos >= 0 && (pos >> 6) % C == rank) owner = ((pos >> 6) / C) % kW;
  __syncthreads();   // barriers and the pair table ready in the CTA
  cluster_arrive();  // ... and the receive barrier for the cluster

  const uint32_t tbl_lane = smem_addr(cpair) + 4u * lane;  // T + 4 lane: the wide table
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

  if (warp == K::kOrderWarp) {
    // ------------------------------------------------------------------ ordering warp
    Q4RowConsts kc;
    uint32_t pk = 0, pv = 0;
    float sgk = 0.f, sgv = 0.f;
    long long crow = -1;
    if (owner >= 0) {
      q4_row_consts(p.rope_tab32, pos, p.signs, p.codebook, lane, kc);
      float z[4];
      q4_norm_rope(xraw, p.k_norm_w, p.eps, kc, lane, z);
      q4_quantize(z, kc, lane, pk, sgk);
      unpack4(vraw, z);
      q4_quantize(z, kc, lane, pv, sgv);
      if (lane < 16) {
        newrow[lane] = pk;
        newrow[16 + lane] = pv;
      }
      if (lane == 0) {
        newrow[32] = __float_as_uint(sgk);
        newrow[33] = __float_as_uint(sgv);
      }
      if (p.paged) {
        const int pg = p.page_table[static_cast<long long>(b) * p.max_blocks + (pos >> 6)];
        if (pg >= 0 && pg < p.num_blocks) crow = static_cast<long long>(pg) * kTile + (pos & (kTile - 1));
      } else {
        crow = static_cast<long long>(b) * p.max_seq + pos;
      }
      q4c_newrow_arrive();
    }
    griddep_wait();
    if (crow >= 0) {
      const long long r = crow * p.Hkv + kv;
      if (lane < 16) {
        reinterpret_cast<uint32_t *>(p.k_idx + r * 64)[lane] = pk;
        reinterpret_cast<uint32_t *>(p.v_idx + r * 64)[lane] = pv;
      }
      if (lane == 0) {
        p.k_scale[r] = sgk;
        p.v_scale[r] = sgv;
      }
      __threadfence();
    }
    __syncwarp();
    if (lane == 0) griddep_launch_dependents();
  } else if (producer) {
    // ---------------------------------------------------------------- producer warp
    // Index tiles by TMA; each lane copies the scales of tokens l and l + 32 (inside the
    // sequence) with cp.async, whose arrivals complete the stage with the TMA bytes.
    bool ok = true;
    int issued = 0;
    for (int i0 = 0; i0 < n && ok; i0 += 32) {
      int mrow = -kTile, mok = 0;
      if (i0 + lane < n) {
        const int j = rank + C * (i0 + lane);
        if (p.paged) {
          const int pg = p.page_table[static_cast<long long>(b) * p.max_blocks + j];
          if (pg >= 0 && pg < p.num_blocks) mrow = pg * kTile, mok = 1;
          else atomicOr(p.err, GQA_DEVERR_PAGE);
        } else {
          mrow = b * p.max_seq + j * kTile;
          mok = 1;
        }
      }
      const int cnt = n - i0 < 32 ? n - i0 : 32;
      for (int u = 0; u < cnt; ++u) {
        const int i = i0 + u;
        const int row = __shfl_sync(0xffffffffu, mrow, u), pok = __shfl_sync(0xffffffffu, mok, u);
        const int valid = min(kTile, L - (rank + C * i) * kTile);
        const int s = i % kS;
        if (i >= kS) ok = mbar_wait(smem_addr(&empty_bar[s]), static_cast<uint32_t>(((i / kS) - 1) & 1));
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const uint32_t fb = smem_addr(&full_bar[s]);
        if (lane == 0) {
          pinfo[s] = pok;
          const uint32_t base = smem_addr(stage_ptr(s));
          mbar_arrive_expect_tx(fb, kQ4StageBytes);
          tma_load_3d(base, &tmK, fb, 0, kv, row);
          tma_load_3d(base + kQ4TileBytes, &tmV, fb, 0, kv, row);
        }
        const uint32_t sdst = smem_addr(scl + s * 2 * kTile);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int tok = lane + 32 * hh;
          if (tok < valid && pok) {
            const long long r = (static_cast<long long>(row) + tok) * p.Hkv + kv;
            cp_async4(sdst + 4 * tok, p.k_scale + r);
            cp_async4(sdst + 4 * (kTile + tok), p.v_scale + r);
          }
        }
        cp_async_arrive_noinc(fb);
        issued = i + 1;
      }
    }
    if (lane == 0 && !ok) {
      atomicOr(p.err, GQA_DEVERR_TIMEOUT);
      for (int ii = (issued > kS ? issued - kS : 0); ii < issued; ++ii)
        (void)mbar_wait(smem_addr(&full_bar[ii % kS]), static_cast<uint32_t>((ii / kS) & 1));
    }
    cp_async_wait_all();
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ consumer warps
    const int cw = warp, r8 = lane >> 2, c4 = lane & 3;
    // the segment's rotated queries q~ (hi + lo), one head a warp at a time
    {
      Q4RowConsts kc;
      q4_row_consts(p.rope_tab32, pos, p.signs, p.codebook, lane, kc);
      for (int g = cw; g < p.G; g += kW) {
        float z[4] = {0.f, 0.f, 0.f, 0.f};
        if (pos >= 0) {
          const uint2 bits = g == cw ? xraw
                                     : reinterpret_cast<const uint2 *>(
                                           p.q_new + (static_cast<long long>(b) * p.Hq + kv * p.G + g) * kHeadDim)[lane];
          q4_norm_rope(bits, p.q_norm_w, p.eps, kc, lane, z);
          q4_rotate_query(z, kc, lane);
        }
        uint32_t h[2], l[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          h[u] = pack_bf16(z[2 * u], z[2 * u + 1]);
          l[u] = pack_bf16(z[2 * u] - bf16_lo_to_float(h[u]), z[2 * u + 1] - bf16_hi_to_float(h[u]));
        }
        reinterpret_cast<uint2 *>(qbuf + g * kHeadDim)[lane] = make_uint2(h[0], h[1]);
        reinterpret_cast<uint2 *>(qbuf + (GQA_MAX_GROUP + g) * kHeadDim)[lane] = make_uint2(l[0], l[1]);
      }
    }
    q4c_consumers_sync<kW>();
    uint32_t qh[8][NT][2], ql[8][NT][2];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int g = 8 * t + r8;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int j = 16 * c4 + 2 * ks + hf;  // dims j (low half) and j + 64 (high half)
          uint32_t vh = 0u, vl = 0u;
          if (g < p.G) {
            vh = static_cast<uint32_t>(qbuf[g * kHeadDim + j]) | (static_cast<uint32_t>(qbuf[g * kHeadDim + j + 64]) << 16);
            vl = static_cast<uint32_t>(qbuf[(GQA_MAX_GROUP + g) * kHeadDim + j]) |
                 (static_cast<uint32_t>(qbuf[(GQA_MAX_GROUP + g) * kHeadDim + j + 64]) << 16);
          }
          qh[ks][t][hf] = vh;
          ql[ks][t][hf] = vl;
        }
    }
    const int i_new = cw == owner ? (pos >> 6) / C : -1;
    for (int i = cw; i < n; i += kW) {
      const int s = i % kS;
      const bool ready = mbar_wait(smem_addr(&full_bar[s]), static_cast<uint32_t>((i / kS) & 1));
      __syncwarp();
      if (!__all_sync(0xffffffffu, ready)) {
        if (lane == 0) atomicOr(p.err, GQA_DEVERR_TIMEOUT);
        break;
      }
      const int valid = min(kTile, L - (rank + C * i) * kTile);
      const bool page_ok = pinfo[s] != 0;
      uint8_t *kt = stage_ptr(s);
      if (i == i_new) {  // the new row, from the ordering warp, into its place in the stage
        q4c_newrow_sync();
        const int r = pos & (kTile - 1);
        if (lane < 16) {
          reinterpret_cast<uint32_t *>(kt + r * 64)[lane] = newrow[lane];
          reinterpret_cast<uint32_t *>(kt + kQ4TileBytes + r * 64)[lane] = newrow[16 + lane];
        }
        if (lane == 0) {
          scl[s * 2 * kTile + r] = __uint_as_float(newrow[32]);
          scl[s * 2 * kTile + kTile + r] = __uint_as_float(newrow[33]);
        }
        __syncwarp();
      }
      float sk[4][2], sv[4][2];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int tok = 16 * mt + r8 + 8 * hh;
          const bool in = tok < valid && page_ok;
          sk[mt][hh] = in ? scl[s * 2 * kTile + tok] * p.scale_log2 : 0.f;
          sv[mt][hh] = in ? scl[s * 2 * kTile + kTile + tok] : 0.f;
        }
      q4_tile_update<NT, true>(kt, valid, sk, sv, tbl_lane, lane, qh, ql, o, m_run, l_run);
      if (i == i_new) fence_proxy_async_smem();  // generic writes precede the next TMA into the stage
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty_bar[s]));
    }
  }

  // ------------------------------------------------------------------ merge
  float *wpart = reinterpret_cast<float *>(table);  // [W][16][132], over the table
  float *wml = wpart + kW * GQA_MAX_GROUP * kQ4CPartStride;  // [W][16][2]
  float *wm = wml + kW * GQA_MAX_GROUP * 2;                  // [W][16]
  __syncthreads();  // every issued tile has been consumed: the table is no longer read
  const bool consumer = !producer && warp != K::kOrderWarp;
  if (consumer) {
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int g = 8 * t + 2 * lane + jj;
        if (lane < 4 && g < p.G) wm[warp * GQA_MAX_GROUP + g] = m_run[t][jj];
      }
  }
  __syncthreads();
  if (consumer) {
    const int cw = warp;
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int g = 8 * t + 2 * (lane & 3) + jj;
        float M = -INFINITY;
#pragma unroll
        for (int c = 0; c < kW; ++c) M = fmaxf(M, wm[c * GQA_MAX_GROUP + (g < p.G ? g : 0)]);
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
          const int d = ((e >> 1) << 6) + 8 * (lane >> 2) + md;  // natural dim order
          if (g < p.G) wpart[(cw * GQA_MAX_GROUP + g) * kQ4CPartStride + d] = o[md][t][e];
        }
  }
  __syncthreads();
  const int own = q4c_owned(p.G, C, rank);
  const uint32_t bar_local = smem_addr(recv_bar);
  if (tid == 0) mbar_arrive_expect_tx(bar_local, static_cast<uint32_t>(C * own * (8 + 4 * kHeadDim)));
  cluster_wait();  // every CTA of the cluster has initialised its barriers
  for (int e = tid; e < p.G * kHeadDim; e += kThreads) {
    const int g = e >> 7, d = e & (kHeadDim - 1);
    const int q = g % C, slot = g / C, own_q = q4c_owned(p.G, C, q);
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < kW; ++c) acc += wpart[(c * GQA_MAX_GROUP + g) * kQ4CPartStride + d];
    const uint32_t bar_q = mapa_shared(bar_local, q);
    const int rrow = rank * own_q + slot;
    st_async_f32(mapa_shared(smem_addr(recv_o + rrow * kHeadDim + d), q), acc, bar_q);
    if (d == 0) {
      float den = 0.f;
#pragma unroll
      for (int c = 0; c < kW; ++c) den += wml[(c * GQA_MAX_GROUP + g) * 2 + 1];
      st_async_v2f32(mapa_shared(smem_addr(recv_ml + rrow * 2), q), wml[g * 2], den, bar_q);
    }
  }
  const bool got = mbar_wait(bar_local, 0);
  if (!got && lane == 0) atomicOr(p.err, GQA_DEVERR_TIMEOUT);
  cluster_arrive_relaxed();  // this CTA has received everything (or given up)
  griddep_wait();
  // the owned heads: merge, rotate back (R^T o = D H o / sqrt(d)) and write; a warp a head
  for (int slot = warp; slot < own; slot += kThreads / 32) {
    const int g = rank + C * slot;
    float M = -INFINITY;
#pragma unroll 1
    for (int r = 0; r < C; ++r) M = fmaxf(M, recv_ml[(r * own + slot) * 2]);
    float v[4] = {0.f, 0.f, 0.f, 0.f}, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll 1
      for (int r = 0; r < C; ++r) {
        const int rr = r * own + slot;
        const float f = exp2f(recv_ml[rr * 2] - M);
        const float4 x = reinterpret_cast<const float4 *>(recv_o + rr * kHeadDim)[lane];
        v[0] = fmaf(f, x.x, v[0]);
        v[1] = fmaf(f, x.y, v[1]);
        v[2] = fmaf(f, x.z, v[2]);
        v[3] = fmaf(f, x.w, v[3]);
        den = fmaf(f, recv_ml[rr * 2 + 1], den);
      }
    }
    const float inv = den > 0.f ? 1.0f / den : 0.f;  // zeros for an invalid length (flagged above)
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] *= inv;
    fwht128(v, lane);
    const char4 s4 = reinterpret_cast<const char4 *>(p.signs)[lane];
    const float sg[4] = {static_cast<float>(s4.x), static_cast<float>(s4.y), static_cast<float>(s4.z),
                         static_cast<float>(s4.w)};
    uint32_t w2[2];
#pragma unroll
    for (int u = 0; u < 2; ++u)
      w2[u] = pack_bf16(sg[2 * u] * v[2 * u] * kInvSqrtD, sg[2 * u + 1] * v[2 * u + 1] * kInvSqrtD);
    reinterpret_cast<uint2 *>(p.out + (static_cast<long long>(b) * p.Hq + kv * p.G + g) * kHeadDim)[lane] =
        make_uint2(w2[0], w2[1]);
  }
  cluster_wait();  // every CTA has received everything: no store to or from this CTA is in flight
}

size_t q4_attn_smem_bytes(int batch) {
  return 1024 + static_cast<size_t>(kQ4OffBar) + 16 * kQ4Stages + 4 * (batch + 1) + 4 * batch;
}

cudaError_t q4_configure() {
  const int bytes = static_cast<int>(q4_attn_smem_bytes(GQA_MAX_BATCH));
  cudaError_t e = cudaFuncSetAttribute(q4_attn_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(q4_attn_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  void (*ck[4])(CUtensorMap, CUtensorMap, Q4ClusterParams) = {q4_cluster_kernel<1, false>, q4_cluster_kernel<2, false>,
                                                              q4_cluster_kernel<1, true>, q4_cluster_kernel<2, true>};
  const int cbytes[4] = {static_cast<int>(Q4C<1>::kSmemBytes), static_cast<int>(Q4C<2>::kSmemBytes),
                         static_cast<int>(Q4C<1>::kSmemBytes), static_cast<int>(Q4C<2>::kSmemBytes)};
  for (int i = 0; i < 4; ++i) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ck[i], cudaFuncAttributeMaxDynamicSharedMemorySize, cbytes[i]);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ck[i], cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  }
  return e;
}

cudaError_t launch_q4_cluster(const CUtensorMap &tmK, const CUtensorMap &tmV, const Q4ClusterParams &p, int npad,
                              bool pdl, cudaStream_t stream) {
  const bool one = npad == 8;
  const bool order = p.seg_order != nullptr;
  void (*k)(CUtensorMap, CUtensorMap, Q4ClusterParams) =
      one ? (order ? q4_cluster_kernel<1, true> : q4_cluster_kernel<1, false>)
          : (order ? q4_cluster_kernel<2, true> : q4_cluster_kernel<2, false>);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.B * p.Hkv * p.csize));
  cfg.blockDim = dim3(one ? Q4C<1>::kThreads : Q4C<2>::kThreads);
  cfg.dynamicSmemBytes = one ? Q4C<1>::kSmemBytes : Q4C<2>::kSmemBytes;
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
  return cudaLaunchKernelEx(&cfg, k, tmK, tmV, p);
}

cudaError_t launch_q4_prologue(const Q4PrologueParams &p, bool pdl, cudaStream_t stream) {
  return launch_ex(pdl, q4_prologue_kernel, dim3(static_cast<unsigned>(p.B), static_cast<unsigned>((p.Hq + 2 * p.Hkv + 7) / 8)),
                    dim3(256), 0, stream, p);
}

cudaError_t launch_q4_attention(const CUtensorMap &tmK, const CUtensorMap &tmV, const Q4AttnParams &p, int npad,
                                int num_workers, cudaStream_t stream) {
  const size_t bytes = q4_attn_smem_bytes(p.B);
  if (npad == 8)
    return launch_pdl(q4_attn_kernel<1>, dim3(num_workers), dim3(kThreadsAttn), bytes, stream, tmK, tmV, p);
  return launch_pdl(q4_attn_kernel<2>, dim3(num_workers), dim3(kThreadsAttn), bytes, stream, tmK, tmV, p);
}

}  // namespace gqa
