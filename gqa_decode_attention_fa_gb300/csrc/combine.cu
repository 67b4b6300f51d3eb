// Log-sum-exp combine of the split-KV partials (sm_103a).
//
// "ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)", section 4: partials
// (m_i, l_i, O_i) merge associatively and commutatively --
//   m = max(m_a, m_b),  l = l_a e^(m_a - m) + l_b e^(m_b - m),  O = O_a e^(m_a - m) + O_b e^(m_b - m)
// -- and are normalised once, out = O / l.  On one GPU the reduce-to-root of that
// section becomes this kernel: one CTA per (b, h), 128 threads (one per dim), reading
// the fp32 partials (L2-resident) of every (worker, warp) piece that touched the
// sequence's KV head, first for the maximum m, then for the weighted sums.  The m values
// are in log2 units (the attention kernel works with exp2), so the weights are 2^(m - M).
#include "gqa_common.cuh"
#include "launch.h"

namespace gqa {

__global__ void __launch_bounds__(128) combine_kernel(const CombineParams p) {
  const int bh = blockIdx.x;
  const int b = bh / p.Hq, h = bh - b * p.Hq;
  const int kv = h / p.G, g = h - kv * p.G;
  const int d = threadIdx.x;
  uint16_t *out = p.out + static_cast<long long>(bh) * kHeadDim;
  const int nt = tiles_of(p.seq_lens[b], p.max_seq);
  if (nt == 0) {  // invalid length: the attention kernel skipped it and flagged the error
    out[d] = 0;
    return;
  }
  const long long T = p.prefix[p.B];
  const long long seg_begin = static_cast<long long>(p.prefix[b]) + static_cast<long long>(kv) * nt;
  const long long seg_end = seg_begin + nt;
  const int seg = b * p.Hkv + kv;
  const int w0 = worker_of(T, p.W, seg_begin), w1 = worker_of(T, p.W, seg_end - 1);

  float M = -INFINITY;
  for (int w = w0; w <= w1; ++w) {
    const long long wb = worker_begin(T, p.W, w), we = worker_begin(T, p.W, w + 1);
    const long long a = seg_begin > wb ? seg_begin : wb, e = seg_end < we ? seg_end : we;
    for (int c = 0; c < kConsumerWarps; ++c) {
      if (!warp_has_tile(a - wb, e - wb, c)) continue;
      const long long r = (static_cast<long long>(seg + w) * kConsumerWarps + c) * p.G + g;
      M = fmaxf(M, p.part_ml[r * 2]);
    }
  }
  float num = 0.f, den = 0.f;
  for (int w = w0; w <= w1; ++w) {
    const long long wb = worker_begin(T, p.W, w), we = worker_begin(T, p.W, w + 1);
    const long long a = seg_begin > wb ? seg_begin : wb, e = seg_end < we ? seg_end : we;
    for (int c = 0; c < kConsumerWarps; ++c) {
      if (!warp_has_tile(a - wb, e - wb, c)) continue;
      const long long r = (static_cast<long long>(seg + w) * kConsumerWarps + c) * p.G + g;
      const float f = exp2f(p.part_ml[r * 2] - M);
      num = fmaf(f, p.part_o[r * kHeadDim + d], num);
      den = fmaf(f, p.part_ml[r * 2 + 1], den);
    }
  }
  const __nv_bfloat16 v = __float2bfloat16_rn(num / den);
  out[d] = *reinterpret_cast<const uint16_t *>(&v);
}

cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream) {
  combine_kernel<<<p.B * p.Hq, kHeadDim, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gqa
