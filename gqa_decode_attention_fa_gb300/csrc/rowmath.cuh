// Per-row arithmetic of the decode prologue shared by the kernels: bf16 rounding of
// binary64 values and the QK-norm + RoPE of one 128-dim head row held by one warp.
//
// "Qwen3-14B Optimization", section 2.1 (Shape 4) and section 3.3: per-head RMSNorm of q
// and k folded into RoPE, the RoPE halves (i, i + d/2) rotated together, the norm
// reciprocal a per-row scalar that commutes with the rotation.
#pragma once

#include "gqa_common.cuh"

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

// One warp computes RoPE_pos(RMSNorm(x, w)) of a 128-dim bf16 row x in binary64 and
// rounds each element once to bf16.  Lane l handles dims {l, l+32, l+64, l+96}, so the
// RoPE pairs (l, l+64) and (l+32, l+96) stay in the lane; out[t] is dim l + 32 t.
// cs0/cs1 are (cos, sin) of the pair angles for pairs l and l+32; w may be null.
__device__ __forceinline__ void rotate_row_fp64(const uint16_t *x, const uint16_t *w, double eps, double2 cs0,
                                                double2 cs1, int lane, uint16_t (&out)[4]) {
  double y[4];
  if (w) {
    float xf[4];
    double ss = 0.0;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      xf[t] = bf16_bits_to_float(x[lane + 32 * t]);
      const double xd = static_cast<double>(xf[t]);
      ss = fma(xd, xd, ss);
    }
    ss = warp_sum(ss);
    const double r = rsqrt(ss * (1.0 / 128.0) + eps);
#pragma unroll
    for (int t = 0; t < 4; ++t)  // x * w is exact in binary32 (two 8-bit significands)
      y[t] = static_cast<double>(xf[t] * bf16_bits_to_float(w[lane + 32 * t])) * r;
  } else {
#pragma unroll
    for (int t = 0; t < 4; ++t) y[t] = static_cast<double>(bf16_bits_to_float(x[lane + 32 * t]));
  }
  out[0] = round_bf16_rne(fma(y[0], cs0.x, -y[2] * cs0.y));
  out[2] = round_bf16_rne(fma(y[2], cs0.x, y[0] * cs0.y));
  out[1] = round_bf16_rne(fma(y[1], cs1.x, -y[3] * cs1.y));
  out[3] = round_bf16_rne(fma(y[3], cs1.x, y[1] * cs1.y));
}

// The same in binary32 (for query rows, which are not stored): x*w is exact, one rounding
// for the norm scalar, one fused multiply-add per rotated element, one rounding to bf16.
__device__ __forceinline__ void rotate_row_fp32(const uint16_t *x, const uint16_t *w, float eps, float2 cs0,
                                                float2 cs1, int lane, uint16_t (&out)[4]) {
  float y[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) y[t] = bf16_bits_to_float(x[lane + 32 * t]);
  float r = 1.0f;
  if (w) {
    float ss = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) ss = fmaf(y[t], y[t], ss);
    ss = warp_sum(ss);
    r = 1.0f / sqrtf(ss * (1.0f / 128.0f) + eps);
#pragma unroll
    for (int t = 0; t < 4; ++t) y[t] *= bf16_bits_to_float(w[lane + 32 * t]);
  }
  const float z[4] = {r * fmaf(y[0], cs0.x, -y[2] * cs0.y), r * fmaf(y[1], cs1.x, -y[3] * cs1.y),
                      r * fmaf(y[2], cs0.x, y[0] * cs0.y), r * fmaf(y[3], cs1.x, y[1] * cs1.y)};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const __nv_bfloat16 hb = __float2bfloat16_rn(z[t]);
    out[t] = *reinterpret_cast<const uint16_t *>(&hb);
  }
}

}  // namespace gqa
