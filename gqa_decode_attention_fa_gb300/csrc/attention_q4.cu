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
// the merged output row is rotated back once, by the combine.  Three kernels:
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
  const bool first_half = lane < 16;
  float cs_c[4] = {1.f, 1.f, 1.f, 1.f}, cs_s[4] = {0.f, 0.f, 0.f, 0.f};
  if (pos_ok) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float2 t = p.rope_tab32[static_cast<long long>(pos) * 64 + 4 * (lane & 15) + u];
      cs_c[u] = t.x;
      cs_s[u] = t.y;
    }
  }
  float sg[4];
  {
    const char4 s4 = reinterpret_cast<const char4 *>(p.signs)[lane];
    sg[0] = s4.x;
    sg[1] = s4.y;
    sg[2] = s4.z;
    sg[3] = s4.w;
  }
  // codebook and the midpoints between consecutive levels (exact in binary32)
  float cb[16], thr[15];
#pragma unroll
  for (int j = 0; j < 16; ++j) cb[j] = __uint_as_float(static_cast<uint32_t>(p.codebook[j]) << 16);
#pragma unroll
  for (int j = 0; j < 15; ++j) thr[j] = 0.5f * (cb[j] + cb[j + 1]);

  // RMSNorm (optional weight) and RoPE of a row, binary32
  auto norm_rope = [&](const uint16_t *src, const uint16_t *w, float (&z)[4]) {
    float x[4], y[4], ss = 0.f;
    unpack4(reinterpret_cast<const uint2 *>(src)[lane], x);
    float wv[4] = {1.f, 1.f, 1.f, 1.f};
    if (w) unpack4(reinterpret_cast<const uint2 *>(w)[lane], wv);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      ss = fmaf(x[u], x[u], ss);
      y[u] = x[u] * wv[u];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rn = w ? 1.0f / sqrtf(ss * (1.0f / 128.0f) + p.eps) : 1.0f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float yp = __shfl_xor_sync(0xffffffffu, y[u], 16);
      z[u] = rn * (first_half ? fmaf(y[u], cs_c[u], -yp * cs_s[u]) : fmaf(y[u], cs_c[u], yp * cs_s[u]));
    }
  };
  // quantize a row z: indices packed into bytes 4 l .. 4 l + 3 (lanes < 16) and sigma
  auto quantize = [&](const float (&z)[4], uint32_t &packed, float &sigma) {
    float ss = 0.f, y[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      ss = fmaf(z[u], z[u], ss);
      y[u] = sg[u] * z[u];
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
      int k = 0;
#pragma unroll
      for (int j = 0; j < 15; ++j) k += thr[j] < t ? 1 : 0;
      idx[u] = k;
      cn = fmaf(cb[k], cb[k], cn);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cn += __shfl_xor_sync(0xffffffffu, cn, o);
    sigma = s > 0.f ? s / sqrtf(cn) : 0.f;
    uint32_t mine = idx[0] | (idx[1] << 8) | (idx[2] << 16) | (idx[3] << 24);
    const uint32_t hi = __shfl_xor_sync(0xffffffffu, mine, 16);  // dims + 64 from lane l + 16
    packed = mine | (hi << 4);
  };

  {
    if (r < p.Hq) {
      const long long row = static_cast<long long>(b) * p.Hq + r;
      float z[4] = {0.f, 0.f, 0.f, 0.f};
      if (pos_ok) {
        norm_rope(p.q_new + row * kHeadDim, p.q_norm_w, z);
#pragma unroll
        for (int u = 0; u < 4; ++u) {  // q~ = R z = H D z / sqrt(d)
          const __nv_bfloat16 zq = __float2bfloat16_rn(z[u]);  // q is a bf16 activation
          z[u] = sg[u] * __bfloat162float(zq);
        }
        fwht128(z, lane);
#pragma unroll
        for (int u = 0; u < 4; ++u) z[u] *= kInvSqrtD;
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
        norm_rope(p.k_new + nrow * kHeadDim, p.k_norm_w, z);
      } else {
        unpack4(reinterpret_cast<const uint2 *>(p.v_new + nrow * kHeadDim)[lane], z);
      }
      uint32_t packed;
      float sigma;
      quantize(z, packed, sigma);
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
  auto pair_entry = [&](uint32_t w, int k) {
    const uint32_t e = __byte_perm(w, 0u, 0x4440u | static_cast<uint32_t>(k));
    uint32_t v;
    asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(tbl_lane + (e << 7)));
    return v;
  };
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
    const uint8_t *kt = smem + kQ4OffStage + s * kQ4StageBytes;  // [64 tokens][64 index bytes]
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
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      // tokens 16 mt + r (A rows 0-7) and + 8 (rows 8-15), index bytes 16 c .. 16 c + 15
      const uint4 w0 = *reinterpret_cast<const uint4 *>(kt + (16 * mt + r8) * 64 + 16 * c4);
      const uint4 w1 = *reinterpret_cast<const uint4 *>(kt + (16 * mt + r8 + 8) * 64 + 16 * c4);
      const uint32_t x0[4] = {w0.x, w0.y, w0.z, w0.w}, x1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int wd = ks >> 1, k0 = 2 * (ks & 1);  // bytes 2 ks and 2 ks + 1
        const uint32_t a0 = pair_entry(x0[wd], k0), a2 = pair_entry(x0[wd], k0 + 1);
        const uint32_t a1 = pair_entry(x1[wd], k0), a3 = pair_entry(x1[wd], k0 + 1);
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
        ph[mt][nt][0] = movmatrix_t(h01);
        ph[mt][nt][1] = movmatrix_t(h23);
        pl[mt][nt][0] = movmatrix_t(l01);
        pl[mt][nt][1] = movmatrix_t(l23);
      }
    // O~^T += C_V^T (P sigma_V)^T: 4 token k-steps x 8 dim blocks of 16 (rows 8 r + md and
    // 64 + 8 r + md); tokens t0, t0 + 1 (k-slots 2 c, +1) and t0 + 8, t0 + 9 (slots + 8)
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const int t0 = 16 * mt + 2 * c4;
      const uint8_t *vr = vt + t0 * 64 + 8 * r8;
      const uint2 y0 = *reinterpret_cast<const uint2 *>(vr), y1 = *reinterpret_cast<const uint2 *>(vr + 64);
      const uint2 y2 = *reinterpret_cast<const uint2 *>(vr + 8 * 64), y3 = *reinterpret_cast<const uint2 *>(vr + 9 * 64);
#pragma unroll
      for (int hw = 0; hw < 2; ++hw) {
        const uint32_t u0 = hw ? y0.y : y0.x, u1 = hw ? y1.y : y1.x, u2 = hw ? y2.y : y2.x, u3 = hw ? y3.y : y3.x;
        // byte m of each: entry (nibble of token t) | (same nibble of token t + 1) << 4
        const uint32_t lo01 = (u0 & 0x0f0f0f0fu) | ((u1 << 4) & 0xf0f0f0f0u);
        const uint32_t hi01 = ((u0 >> 4) & 0x0f0f0f0fu) | (u1 & 0xf0f0f0f0u);
        const uint32_t lo23 = (u2 & 0x0f0f0f0fu) | ((u3 << 4) & 0xf0f0f0f0u);
        const uint32_t hi23 = ((u2 >> 4) & 0x0f0f0f0fu) | (u3 & 0xf0f0f0f0u);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int md = 4 * hw + m;
          const uint32_t a0 = pair_entry(lo01, m), a1 = pair_entry(hi01, m);
          const uint32_t a2 = pair_entry(lo23, m), a3 = pair_entry(hi23, m);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma_bf16(o[md][nt], a0, a1, a2, a3, ph[mt][nt][0], ph[mt][nt][1]);
            mma_bf16(o[md][nt], a0, a1, a2, a3, pl[mt][nt][0], pl[mt][nt][1]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty_bar[s]));  // the stage's index tiles are consumed
  }
  if (cur_seg >= 0) flush(cur_seg);
}

size_t q4_attn_smem_bytes(int batch) {
  return 1024 + static_cast<size_t>(kQ4OffBar) + 16 * kQ4Stages + 4 * (batch + 1) + 4 * batch;
}

cudaError_t q4_configure() {
  const int bytes = static_cast<int>(q4_attn_smem_bytes(GQA_MAX_BATCH));
  cudaError_t e = cudaFuncSetAttribute(q4_attn_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(q4_attn_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  return e;
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
