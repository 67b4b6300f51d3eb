// Per-row arithmetic of the new key row: the QK-norm + RoPE of one 128-dim head row held by
// one warp, rounded once to bf16 as the exact value rounds.
//
// "Qwen3-14B Optimization", section 2.1 (Shape 4) and section 3.3: per-head RMSNorm of q
// and k folded into RoPE, the RoPE halves (i, i + d/2) rotated together, the norm
// reciprocal a per-row scalar that commutes with the rotation.
//
// The stored key must round like the definition's exact value, so the row is computed in
// double-word (float-float) arithmetic -- about 44 significant bits from binary32
// operations: GB300's binary64 units are too slow for this to stay off the critical path.
// The building blocks are the classical error-free transformations (Knuth's TwoSum,
// Dekker's Fast2Sum, the FMA-based product TwoProd) and the double-word sum and product of
// Joldes, Muller and Popescu, "Tight and rigorous error bounds for basic building blocks
// of double-word arithmetic" (ACM TOMS 44(2), 2017): relative errors below 3u^2 and 5u^2,
// u = 2^-24.  The intrinsics (__fadd_rn, ...) keep the compiler from contracting or
// reassociating them.
#pragma once

#include "gqa_common.cuh"

namespace gqa {

__device__ __forceinline__ float bf16_bits_to_float(uint16_t v) { return __uint_as_float(uint32_t(v) << 16); }

// A double-word number hi + lo with |lo| <= ulp(hi) / 2.
struct dw {
  float hi, lo;
};

__device__ __forceinline__ dw two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
// Requires |a| >= |b| (or a == 0).
__device__ __forceinline__ dw fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ dw two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return {p, __fmaf_rn(a, b, -p)};
}
__device__ __forceinline__ dw dw_add(dw a, dw b) {
  const dw s = two_sum(a.hi, b.hi), t = two_sum(a.lo, b.lo);
  const dw v = fast_two_sum(s.hi, __fadd_rn(s.lo, t.hi));
  return fast_two_sum(v.hi, __fadd_rn(v.lo, t.lo));
}
__device__ __forceinline__ dw dw_mul(dw a, dw b) {
  const dw p = two_prod(a.hi, b.hi);
  const float t = __fmaf_rn(a.hi, b.lo, __fmul_rn(a.lo, b.hi));
  return fast_two_sum(p.hi, __fadd_rn(p.lo, t));
}
__device__ __forceinline__ dw dw_mul_f(dw a, float b) {
  const dw p = two_prod(a.hi, b);
  return fast_two_sum(p.hi, __fmaf_rn(a.lo, b, p.lo));
}
__device__ __forceinline__ dw dw_neg(dw a) { return {-a.hi, -a.lo}; }

// bf16 bits of the value hi + lo, rounded to nearest with ties to even.  Only when hi is
// itself a bf16 rounding midpoint can lo change the result (|lo| is below half a binary32
// ulp of hi, while any other hi is at least one ulp away from the nearest midpoint).
__device__ __forceinline__ uint16_t round_dw_bf16(dw z) {
  const uint32_t b = __float_as_uint(z.hi);
  if ((b & 0xffffu) == 0x8000u && z.lo != 0.f && (b & 0x7f800000u) != 0x7f800000u) {
    const bool away = (z.lo > 0.f) == (z.hi > 0.f);  // the value lies beyond the midpoint
    return static_cast<uint16_t>((b >> 16) + (away ? 1u : 0u));
  }
  const __nv_bfloat16 h = __float2bfloat16_rn(z.hi);
  return *reinterpret_cast<const uint16_t *>(&h);
}

// One warp computes RoPE_pos(RMSNorm(x, w)) of a 128-dim bf16 row x and rounds each element
// once to bf16.  Each lane holds four dims of x (and of w, when has_w) as two RoPE pairs:
// x[0] with its partner x[2], x[1] with x[3] (the decode step: dims l, l+32, l+64, l+96; the
// prefill prologue: 2l, 2l+1, 2l+64, 2l+65); out[t] is the dim of x[t].  cs0/cs1 are the
// double-word (cos_hi, sin_hi, cos_lo, sin_lo) of the angles of the pairs of x[0] and x[1].
//   ss = sum x^2: the squares are exact in binary32 (8-bit significands) and are summed in
//     double-word, in the lane and over the shuffle tree (every lane gets the same sum);
//   r = 1/sqrt(ss/128 + eps): a correctly rounded binary32 seed and one Newton step in
//     double-word (relative error about 2^-45);
//   y = x w is exact in binary32;  z_i = r (y_i cos - y_p sin), z_p = r (y_p cos + y_i sin)
//     in double-word.
// The result differs from the definition's exact value by about 2^-44 r (|y_i| + |y_p|), so
// its bf16 rounding differs only if that value lies closer than this to a rounding
// midpoint.
__device__ __forceinline__ void rotate_row_k(const uint16_t (&x)[4], const uint16_t (&w)[4], bool has_w, float eps,
                                             float4 cs0, float4 cs1, uint16_t (&out)[4]) {
  float y[4];
  dw r = {1.f, 0.f};
  if (has_w) {
    dw ss = {0.f, 0.f};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float xf = bf16_bits_to_float(x[t]);
      ss = dw_add(ss, dw{__fmul_rn(xf, xf), 0.f});
      y[t] = __fmul_rn(xf, bf16_bits_to_float(w[t]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const dw other = {__shfl_xor_sync(0xffffffffu, ss.hi, o), __shfl_xor_sync(0xffffffffu, ss.lo, o)};
      ss = dw_add(ss, other);
    }
    const dw t = dw_add(dw{__fmul_rn(ss.hi, 1.0f / 128.0f), __fmul_rn(ss.lo, 1.0f / 128.0f)}, dw{eps, 0.f});
    const float r0 = __frcp_rn(__fsqrt_rn(t.hi));
    const dw e = dw_add(dw{1.f, 0.f}, dw_neg(dw_mul(t, two_prod(r0, r0))));  // 1 - t r0^2
    r = fast_two_sum(r0, __fmul_rn(__fmul_rn(0.5f, r0), e.hi));
  } else {
#pragma unroll
    for (int t = 0; t < 4; ++t) y[t] = bf16_bits_to_float(x[t]);
  }
  const dw c0 = {cs0.x, cs0.z}, s0 = {cs0.y, cs0.w}, c1 = {cs1.x, cs1.z}, s1 = {cs1.y, cs1.w};
  dw z[4];
  z[0] = dw_add(dw_mul_f(c0, y[0]), dw_neg(dw_mul_f(s0, y[2])));
  z[2] = dw_add(dw_mul_f(c0, y[2]), dw_mul_f(s0, y[0]));
  z[1] = dw_add(dw_mul_f(c1, y[1]), dw_neg(dw_mul_f(s1, y[3])));
  z[3] = dw_add(dw_mul_f(c1, y[3]), dw_mul_f(s1, y[1]));
#pragma unroll
  for (int t = 0; t < 4; ++t) out[t] = round_dw_bf16(has_w ? dw_mul(z[t], r) : z[t]);
}

}  // namespace gqa
