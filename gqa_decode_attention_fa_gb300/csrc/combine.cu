// Log-sum-exp combine of the split-KV partials (sm_103a).
//
// "ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)", section 4: partials
// (m_i, l_i, O_i) merge associatively and commutatively --
//   m = max(m_a, m_b),  l = l_a e^(m_a - m) + l_b e^(m_b - m),  O = O_a e^(m_a - m) + O_b e^(m_b - m)
// -- and are normalised once, out = O / l.  On one GPU the reduce-to-root of that
// section becomes this kernel: one CTA per (b, h) merges the fp32 partials (L2-resident)
// of every (worker, consumer warp) piece that touched the sequence's KV head.  Each of
// the eight warps folds an eighth of the pieces with the merge above (a lane holds four
// of the 128 dims, so one 16-byte load per lane fetches a whole partial row; eight
// pieces' loads are in flight per warp), and the warp results are merged once more
// through shared memory.  The m values are in log2 units (the attention kernel works
// with exp2).
#include "gqa_common.cuh"
#include "launch.h"

namespace gqa {

namespace {

constexpr int kCombineWarps = 8;
constexpr int kCombineThreads = 32 * kCombineWarps;
constexpr int kUnroll = 8;         // pieces whose loads a warp keeps in flight at once
constexpr int kWorkerChunk = 128;  // worker range starts cached in shared memory per pass

}  // namespace

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineParams p) {
  __shared__ __align__(16) float s_o[kCombineWarps][kHeadDim];  // float4 stores below
  __shared__ long long s_wb[kWorkerChunk + 1];
  __shared__ float s_ml[kCombineWarps][2];
  griddep_wait();               // the partials come from the attention kernel
  griddep_launch_dependents();
  const int bh = blockIdx.x;
  const int b = bh / p.Hq, h = bh - b * p.Hq;
  const int kv = h / p.G, g = h - kv * p.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint16_t *out = p.out + static_cast<long long>(bh) * kHeadDim;
  const int nt = tiles_of(p.seq_lens[b], p.max_seq);
  if (nt == 0) {  // invalid length: the attention kernel skipped it and flagged the error
    if (tid < kHeadDim) out[tid] = 0;
    return;
  }
  const long long T = p.prefix[p.B];
  const long long seg_begin = static_cast<long long>(p.prefix[b]) + static_cast<long long>(kv) * nt;
  const long long seg_end = seg_begin + nt;
  const int seg = b * p.Hkv + kv;
  const int w0 = worker_of(T, p.W, seg_begin), w1 = worker_of(T, p.W, seg_end - 1);

  float m_run = -INFINITY, l_run = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int wc = w0; wc <= w1; wc += kWorkerChunk) {
    const int nw = min(kWorkerChunk, w1 - wc + 1);
    for (int k = tid; k <= nw; k += kCombineThreads) s_wb[k] = worker_begin(T, p.W, wc + k);
    __syncthreads();
    const int ncand = nw * kConsumerWarps;
    // kUnroll pieces per round: all their loads are issued before any is used
    for (int cand0 = warp; cand0 < ncand; cand0 += kCombineWarps * kUnroll) {
      long long r[kUnroll];
      float2 ml[kUnroll];
      float4 o[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int cand = cand0 + u * kCombineWarps;
        r[u] = -1;
        if (cand < ncand) {
          const int wi = cand / kConsumerWarps, c = cand - wi * kConsumerWarps;
          const long long wb = s_wb[wi], we = s_wb[wi + 1];
          const long long a = seg_begin > wb ? seg_begin : wb, e = seg_end < we ? seg_end : we;
          if (warp_has_tile(a - wb, e - wb, c))
            r[u] = (static_cast<long long>(seg + wc + wi) * kConsumerWarps + c) * p.G + g;
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (r[u] >= 0) {
          ml[u] = *reinterpret_cast<const float2 *>(p.part_ml + r[u] * 2);
          o[u] = *reinterpret_cast<const float4 *>(p.part_o + r[u] * kHeadDim + 4 * lane);
        } else {
          ml[u] = make_float2(-INFINITY, 0.f);
          o[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (r[u] < 0) continue;
        const float m_new = fmaxf(m_run, ml[u].x);
        const float sa = exp2f(m_run - m_new), sb = exp2f(ml[u].x - m_new);
        l_run = l_run * sa + ml[u].y * sb;
        acc.x = acc.x * sa + o[u].x * sb;
        acc.y = acc.y * sa + o[u].y * sb;
        acc.z = acc.z * sa + o[u].z * sb;
        acc.w = acc.w * sa + o[u].w * sb;
        m_run = m_new;
      }
    }
    __syncthreads();
  }
  // merge the warps' partials
  *reinterpret_cast<float4 *>(&s_o[warp][4 * lane]) = acc;
  if (lane == 0) {
    s_ml[warp][0] = m_run;
    s_ml[warp][1] = l_run;
  }
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < kCombineWarps; ++i) M = fmaxf(M, s_ml[i][0]);
  if (tid >= kHeadDim) return;
  float num = 0.f, den = 0.f;
#pragma unroll
  for (int i = 0; i < kCombineWarps; ++i) {
    if (s_ml[i][1] == 0.f) continue;  // a warp that merged no piece
    const float f = exp2f(s_ml[i][0] - M);
    num = fmaf(f, s_o[i][tid], num);
    den = fmaf(f, s_ml[i][1], den);
  }
  const __nv_bfloat16 v = __float2bfloat16_rn(num / den);
  out[tid] = *reinterpret_cast<const uint16_t *>(&v);
}

cudaError_t configure_combine() {
  return cudaFuncSetAttribute(combine_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared);
}

cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream) {
  return launch_pdl(combine_kernel, dim3(p.B * p.Hq), dim3(kCombineThreads), 0, stream, p);
}

}  // namespace gqa
