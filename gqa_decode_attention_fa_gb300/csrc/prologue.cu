// Prologue of the decode step: per-head QK RMSNorm + RoPE of the new token, k/v append.
//
// "Qwen3-14B Optimization", section 2.1 (Shape 4, and #796 in "Then: buy it") folds
// QK-norm and RoPE into the attention path; section 3.3 batches the G query heads of a
// (batch, KV head) pair into one tile and notes that the RMSNorm reciprocal commutes with
// RoPE.  "ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)", section 0.5.1 fixes
// what must hold before attention reads the cache: K stored post-RoPE (P2), V raw (P4),
// the new row appended at its position first (P3).
//
// One CTA per (b, kv): it writes the G rotated query rows of the group into the
// workspace -- already in the 128-byte-swizzled shared-memory image the attention
// kernel's ldmatrix reads, padded to npad rows with zeros -- and the post-RoPE k row and
// the raw v row into cache slot (b, positions[b]).
//
// Precision: the k row is computed in binary64 and rounded once to bf16 (round to
// nearest even), so the appended cache row equals the exact-arithmetic result rounded
// once, except where that value lies within ~1e-15 (relative) of a bf16 rounding
// midpoint.  Binary64 runs at ~1/64 of the binary32 rate on this GPU, so the G query
// rows, which are not stored in the cache, are computed in binary32 (x*w is exact,
// one rounding for the norm scalar, fused multiply-add for the rotation) and rounded to
// bf16 once.
#include "gqa_common.cuh"
#include "launch.h"

namespace gqa {

// Round a binary64 value to bf16 bits, nearest with ties to even, in one step.
// bf16 keeps 8 significant bits; the unit in the last place of a normal bf16 at
// exponent e is 2^(e-7); subnormal bf16 values are multiples of 2^-133.
__device__ __forceinline__ uint16_t round_bf16_rne(double z) {
  const unsigned long long u = static_cast<unsigned long long>(__double_as_longlong(z));
  const uint16_t sign = static_cast<uint16_t>((u >> 48) & 0x8000u);
  const unsigned long long a = u & 0x7fffffffffffffffULL;
  if (a > 0x7ff0000000000000ULL) return 0x7fc0;                       // NaN
  const int e = static_cast<int>(a >> 52) - 1023;                      // unbiased exponent
  if (e >= 128) return static_cast<uint16_t>(sign | 0x7f80);           // inf or overflow
  if (e < -134) return sign;                                           // below half of 2^-133
  const unsigned long long M = (a & ((1ULL << 52) - 1)) | (1ULL << 52);  // 53-bit significand
  if (e >= -126) {                                                     // normal bf16 range
    unsigned long long q = M >> 45;                                    // 8 bits: 1.xxxxxxx
    const unsigned long long rem = M & ((1ULL << 45) - 1), half = 1ULL << 44;
    if (rem > half || (rem == half && (q & 1))) ++q;
    int ee = e;
    if (q == 256) { q = 128; ++ee; }
    if (ee >= 128) return static_cast<uint16_t>(sign | 0x7f80);
    return static_cast<uint16_t>(sign | ((ee + 127) << 7) | (q & 127));
  }
  // subnormal bf16: value / 2^-133 = M * 2^(e + 81); shift right by -(e + 81) in [46, 53]
  const int shift = -81 - e;
  unsigned long long q = M >> shift;
  const unsigned long long rem = M & ((1ULL << shift) - 1), half = 1ULL << (shift - 1);
  if (rem > half || (rem == half && (q & 1))) ++q;
  return static_cast<uint16_t>(sign | q);                              // q == 128 is 2^-126
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t v) { return __uint_as_float(uint32_t(v) << 16); }

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Offset (in bf16 elements) of element (row g, dim e) in one group's swizzled q tile:
// [half = e / 64][npad rows][128 B], 16-byte chunk index XOR (g mod 8).
__device__ __forceinline__ int qtile_offset(int g, int e, int npad) {
  const int half = e >> 6, chunk = (e & 63) >> 3, within = e & 7;
  return (half * npad * 128 + static_cast<int>(swz128(g, chunk))) / 2 + within;
}

__global__ void __launch_bounds__(128) prologue_kernel(const PrologueParams p) {
  const int seg = blockIdx.x;
  const int b = seg / p.Hkv, kv = seg - b * p.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ double s_cos[64], s_sin[64];
  __shared__ long long s_row;
  __shared__ int s_ok;
  uint16_t *qtile = p.q_rot + static_cast<long long>(seg) * p.npad * kHeadDim;

  if (tid == 0) {
    const int L = p.seq_lens[b], pos = p.positions[b];
    uint32_t bad = 0;
    long long row = -1;
    if (L < 1 || L > p.max_seq) bad |= GQA_DEVERR_SEQLEN;
    else if (pos < 0 || pos >= L) bad |= GQA_DEVERR_POSITION;
    else if (p.paged) {
      const int pg = p.page_table[static_cast<long long>(b) * p.max_blocks + pos / kTile];
      if (pg < 0 || pg >= p.num_blocks) bad |= GQA_DEVERR_PAGE;
      else row = static_cast<long long>(pg) * kTile + pos % kTile;
    } else {
      row = static_cast<long long>(b) * p.max_seq + pos;
    }
    if (bad && kv == 0) atomicOr(p.err, bad);
    s_ok = bad == 0;
    s_row = row;
  }
  __syncthreads();
  if (!s_ok) {  // leave a zero q tile: the attention kernel skips this sequence anyway
    for (int i = tid; i < p.npad * kHeadDim; i += blockDim.x) qtile[i] = 0;
    return;
  }
  const int pos = p.positions[b];
  if (tid < 64) {
    double sv, cv;
    sincos(static_cast<double>(pos) * p.inv_freq[tid], &sv, &cv);
    s_cos[tid] = cv;
    s_sin[tid] = sv;
  }
  __syncthreads();

  // Lane owns dims {lane, lane+32, lane+64, lane+96}: the RoPE pairs (lane, lane+64) and
  // (lane+32, lane+96) stay inside the lane.
  const double c0 = s_cos[lane], sn0 = s_sin[lane], c1 = s_cos[lane + 32], sn1 = s_sin[lane + 32];
  const long long row = s_row;

  for (int v = warp; v <= p.G; v += 4) {
    if (v == 0) {
      // k row: binary64 throughout, one rounding to bf16.
      const uint16_t *src = p.k_new + (static_cast<long long>(b) * p.Hkv + kv) * kHeadDim;
      double y[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) y[t] = static_cast<double>(bf16_bits_to_float(src[lane + 32 * t]));
      if (p.k_norm_w) {
        double ss = 0.0;
#pragma unroll
        for (int t = 0; t < 4; ++t) ss += y[t] * y[t];
        ss = warp_sum(ss);
        const double r = 1.0 / sqrt(ss / 128.0 + p.eps);
#pragma unroll
        for (int t = 0; t < 4; ++t) y[t] = y[t] * r * static_cast<double>(bf16_bits_to_float(p.k_norm_w[lane + 32 * t]));
      }
      const double z0 = y[0] * c0 - y[2] * sn0, z2 = y[2] * c0 + y[0] * sn0;
      const double z1 = y[1] * c1 - y[3] * sn1, z3 = y[3] * c1 + y[1] * sn1;
      uint16_t *dst = p.k_cache + (row * p.Hkv + kv) * kHeadDim;
      dst[lane] = round_bf16_rne(z0);
      dst[lane + 32] = round_bf16_rne(z1);
      dst[lane + 64] = round_bf16_rne(z2);
      dst[lane + 96] = round_bf16_rne(z3);
    } else {
      // query row g = v - 1 of the group: binary32, one rounding to bf16.
      const int g = v - 1, h = kv * p.G + g;
      const uint16_t *src = p.q_new + (static_cast<long long>(b) * p.Hq + h) * kHeadDim;
      float y[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) y[t] = bf16_bits_to_float(src[lane + 32 * t]);
      float r = 1.0f;
      if (p.q_norm_w) {
        float ss = 0.f;
#pragma unroll
        for (int t = 0; t < 4; ++t) ss = fmaf(y[t], y[t], ss);
        ss = warp_sum(ss);
        r = 1.0f / sqrtf(ss * (1.0f / 128.0f) + static_cast<float>(p.eps));
#pragma unroll
        for (int t = 0; t < 4; ++t) y[t] *= bf16_bits_to_float(p.q_norm_w[lane + 32 * t]);  // exact
      }
      const float fc0 = static_cast<float>(c0), fs0 = static_cast<float>(sn0);
      const float fc1 = static_cast<float>(c1), fs1 = static_cast<float>(sn1);
      const float z0 = r * fmaf(y[0], fc0, -y[2] * fs0), z2 = r * fmaf(y[2], fc0, y[0] * fs0);
      const float z1 = r * fmaf(y[1], fc1, -y[3] * fs1), z3 = r * fmaf(y[3], fc1, y[1] * fs1);
      const float zz[4] = {z0, z1, z2, z3};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        __nv_bfloat16 hb = __float2bfloat16_rn(zz[t]);
        qtile[qtile_offset(g, lane + 32 * t, p.npad)] = *reinterpret_cast<uint16_t *>(&hb);
      }
    }
  }
  // v row: raw copy, 16 B per lane of the last warp.
  if (warp == 3 && lane < 16) {
    const uint4 *src = reinterpret_cast<const uint4 *>(p.v_new + (static_cast<long long>(b) * p.Hkv + kv) * kHeadDim);
    uint4 *dst = reinterpret_cast<uint4 *>(p.v_cache + (row * p.Hkv + kv) * kHeadDim);
    dst[lane] = src[lane];
  }
  // zero padding rows G..npad-1 of the q tile (both halves)
  const int pad_rows = p.npad - p.G;
  for (int i = tid; i < pad_rows * kHeadDim; i += blockDim.x) {
    const int g = p.G + i / kHeadDim, e = i % kHeadDim;
    qtile[qtile_offset(g, e, p.npad)] = 0;
  }
}

cudaError_t launch_prologue(const PrologueParams &p, cudaStream_t stream) {
  prologue_kernel<<<p.B * p.Hkv, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gqa
