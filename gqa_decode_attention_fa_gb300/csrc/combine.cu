// Log-sum-exp combine of the split-KV partials (sm_103a).
//
// "ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)", section 4: partials
// (m_i, l_i, O_i) merge associatively and commutatively --
//   m = max(m_a, m_b),  l = l_a e^(m_a - m) + l_b e^(m_b - m),  O = O_a e^(m_a - m) + O_b e^(m_b - m)
// -- and are normalised once, out = O / l.  On one GPU the reduce-to-root of that
// section becomes this kernel: the fp32 partials (L2-resident) of every (worker, consumer
// warp) piece that touched a sequence's KV head are merged per query head.  The m values
// are in log2 units (the attention kernel works with exp2).
//
// The step is latency-bound, so the kernels are shaped around dependent round trips:
//  * Everything that does not depend on the attention kernel's output -- the tile prefix
//    of the batch (from seq_lens), the workers that touched the segment and the list of
//    pieces to merge -- is worked out before the kernel waits on the attention kernel
//    (programmatic dependent launch), i.e. while the attention kernel is still running.
//  * After the wait, the piece loads go out side by side, a 16-byte load per lane.
// Two shapes, chosen by the host:
//  * combine_head_kernel<NSPLIT>: a CTA merges 128 / NSPLIT dims of one query head; a
//    group of 32 / NSPLIT lanes loads one piece's dims and the groups merge disjoint
//    subsets of the pieces before a last merge across groups in shared memory.  For few
//    sequences with many pieces each (long contexts split over many workers).
//  * combine_seg_kernel: a CTA per (sequence, KV head) segment with one warp per query
//    head of the group, which merges all the pieces of its head alone.  For many
//    segments with few pieces each (batched decode): a fifth of the CTAs, each planned
//    once for the whole group.
// The merge order is fixed, so results are deterministic.
#include "gqa_common.cuh"
#include "launch.h"

namespace gqa {

namespace {

constexpr int kHeadThreads = 128;                   // combine_head_kernel CTA size
constexpr int kMaxWarps = GQA_MAX_GROUP;            // combine_seg_kernel: one warp per head
constexpr int kMaxPieces = 1024;                    // pieces listed per planning pass
constexpr int kUnroll = 4;                          // piece loads in flight: head kernel
constexpr int kUnrollSeg = 4;                       // the same in the segment kernel

// Sum over the CTA (nwarps full warps) of two 64-bit counts; every thread gets the sums.
__device__ __forceinline__ void block_sum2(long long &a, long long &b, long long (*red)[2], int nwarps) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  if (lane == 0) {
    red[warp][0] = a;
    red[warp][1] = b;
  }
  __syncthreads();
  a = b = 0;
  for (int i = 0; i < nwarps; ++i) {
    a += red[i][0];
    b += red[i][1];
  }
}

// Where segment (b, kv)'s tiles sit in the batch's tile order (from the lengths, as the
// attention kernel numbers them) and which workers hold them.
struct SegSpan {
  long long T, begin, end;  // all tiles; the segment's [begin, end)
  int nt, w0, w1;           // its tile count (0: invalid length) and first / last worker
};

__device__ __forceinline__ SegSpan seg_span(const CombineParams &p, int b, int kv, long long (*red)[2],
                                            int nwarps) {
  const int nthreads = nwarps * 32;
  long long before = 0, total = 0;
  for (int i = threadIdx.x; i < p.B; i += nthreads) {
    const long long t = tiles_of(p.seq_lens[i], p.max_seq);
    total += t;
    if (i < b) before += t;
  }
  block_sum2(before, total, red, nwarps);
  SegSpan s;
  s.nt = tiles_of(p.seq_lens[b], p.max_seq);
  s.T = total * p.Hkv;
  s.begin = before * p.Hkv + static_cast<long long>(kv) * s.nt;
  s.end = s.begin + s.nt;
  s.w0 = s.nt > 0 ? worker_of(s.T, p.W, s.begin) : 0;
  s.w1 = s.nt > 0 ? worker_of(s.T, p.W, s.end - 1) : -1;
  return s;
}

// Lists, in (worker, consumer warp) order, the pieces among candidates
// [base, base + kMaxPieces) of the segment's (worker, warp) pairs that hold tiles of it:
// s_piece[k] = slot * 6 + warp for the partial rows of that piece.  Each warp compacts
// its candidates with a ballot.  Returns the count (the same in every thread).
__device__ __forceinline__ int plan_pieces(const CombineParams &p, const SegSpan &s, int seg, long long base,
                                           int *s_piece, int *s_wcount, int nwarps) {
  const int nthreads = nwarps * 32, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long npairs = static_cast<long long>(s.w1 - s.w0 + 1) * kConsumerWarps;
  const long long lim = npairs - base < kMaxPieces ? npairs - base : kMaxPieces;
  int count = 0;
  for (long long r0 = 0; r0 < lim; r0 += nthreads) {
    const long long k = base + r0 + threadIdx.x;
    bool has = false;
    int piece = 0;
    if (r0 + threadIdx.x < lim) {
      const int wi = s.w0 + static_cast<int>(k / kConsumerWarps), c = static_cast<int>(k % kConsumerWarps);
      const long long wb = worker_begin(s.T, p.W, wi), we = worker_begin(s.T, p.W, wi + 1);
      const long long a = s.begin > wb ? s.begin : wb, e = s.end < we ? s.end : we;
      has = warp_has_tile(a - wb, e - wb, c);
      piece = (seg + wi) * kConsumerWarps + c;
    }
    const unsigned m = __ballot_sync(0xffffffffu, has);
    if (lane == 0) s_wcount[warp] = __popc(m);
    __syncthreads();
    int off = count;
    for (int i = 0; i < warp; ++i) off += s_wcount[i];
    for (int i = 0; i < nwarps; ++i) count += s_wcount[i];
    if (has) s_piece[off + __popc(m & ((1u << lane) - 1u))] = piece;
    __syncthreads();
  }
  return count;
}

// Folds pieces first, first + step, ... (< count) of head g, dims [d0, d0 + 4) into the
// running (m, l, acc), U loads in flight.
template <int kUnroll>
__device__ __forceinline__ void merge_pieces(const CombineParams &p, const int *s_piece, int count, int first,
                                             int step, int g, int d0, float &m_run, float &l_run, float4 &acc) {
  for (int k0 = first; k0 < count; k0 += step * kUnroll) {
    float2 ml[kUnroll];
    float4 o[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int k = k0 + u * step;
      if (k < count) {
        const long long row = static_cast<long long>(s_piece[k]) * p.G + g;
        ml[u] = *reinterpret_cast<const float2 *>(p.part_ml + row * 2);
        o[u] = *reinterpret_cast<const float4 *>(p.part_o + row * kHeadDim + d0);
      } else {
        ml[u] = make_float2(-INFINITY, 0.f);
        o[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (k0 + u * step >= count) continue;
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
}

__device__ __forceinline__ uint32_t pack2_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}

}  // namespace

// At most 64 registers a thread: a combine CTA (four warps) launched early (programmatic
// dependent launch) then fits on an SM beside a running attention CTA -- two of them do,
// within each SM sub-partition's register file -- and so does the next step's attention
// CTA beside combine CTAs still running.
template <int NSPLIT>
__global__ void __launch_bounds__(kHeadThreads, 8) combine_head_kernel(const CombineParams p) {
  constexpr int kWarps = kHeadThreads / 32;
  constexpr int kDims = kHeadDim / NSPLIT;             // dims merged by this CTA
  constexpr int kLanes = kDims / 4;                    // lanes per piece (4 dims each)
  constexpr int kGroups = kHeadThreads / kLanes;       // pieces loaded side by side
  __shared__ int s_piece[kMaxPieces];
  __shared__ int s_wcount[kWarps];
  __shared__ long long s_red[kWarps][2];
  __shared__ __align__(16) float s_o[kGroups][kDims];  // float4 stores below
  __shared__ float s_m[kGroups], s_l[kGroups];

  const int tid = threadIdx.x;
  const int bh = blockIdx.x / NSPLIT, part = blockIdx.x - bh * NSPLIT;
  const int b = bh / p.Hq, h = bh - b * p.Hq;
  const int kv = h / p.G, g = h - kv * p.G;
  const int grp = tid / kLanes, sub = tid - grp * kLanes;
  uint16_t *out = p.out + static_cast<long long>(bh) * kHeadDim + part * kDims;

  const SegSpan s = seg_span(p, b, kv, s_red, kWarps);
  const long long npairs = static_cast<long long>(s.w1 - s.w0 + 1) * kConsumerWarps;
  float m_run = -INFINITY, l_run = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  bool waited = false;
  for (long long base = 0; base < npairs; base += kMaxPieces) {
    const int count = plan_pieces(p, s, b * p.Hkv + kv, base, s_piece, s_wcount, kWarps);
    if (!waited) {
      griddep_wait();  // the partials come from the attention kernel
      griddep_launch_dependents();
      waited = true;
    }
    merge_pieces<kUnroll>(p, s_piece, count, grp, kGroups, g, part * kDims + 4 * sub, m_run, l_run, acc);
    __syncthreads();  // the list is rebuilt by the next pass
  }
  if (!waited) {
    griddep_wait();
    griddep_launch_dependents();
  }
  if (s.nt == 0) {  // invalid length: the attention kernel skipped it and flagged the error
    if (tid < kDims) out[tid] = 0;
    return;
  }

  // merge the groups' partials
  *reinterpret_cast<float4 *>(&s_o[grp][4 * sub]) = acc;
  if (sub == 0) {
    s_m[grp] = m_run;
    s_l[grp] = l_run;
  }
  __syncthreads();
  if (tid >= kDims) return;
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < kGroups; ++i) M = fmaxf(M, s_m[i]);
  float num = 0.f, den = 0.f;
#pragma unroll
  for (int i = 0; i < kGroups; ++i) {
    if (s_l[i] == 0.f) continue;  // a group that merged no piece
    const float f = exp2f(s_m[i] - M);
    num = fmaf(f, s_o[i][tid], num);
    den = fmaf(f, s_l[i], den);
  }
  const __nv_bfloat16 v = __float2bfloat16_rn(num / den);
  out[tid] = *reinterpret_cast<const uint16_t *>(&v);
}

// One CTA of 32 * G threads per segment; warp g merges query head kv * G + g.
__global__ void __launch_bounds__(32 * kMaxWarps, 2) combine_seg_kernel(const CombineParams p) {
  __shared__ int s_piece[kMaxPieces];
  __shared__ int s_wcount[kMaxWarps];
  __shared__ long long s_red[kMaxWarps][2];
  const int nwarps = p.G, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = blockIdx.x, b = seg / p.Hkv, kv = seg - b * p.Hkv;
  uint16_t *out = p.out + (static_cast<long long>(b) * p.Hq + kv * p.G + warp) * kHeadDim + 4 * lane;

  const SegSpan s = seg_span(p, b, kv, s_red, nwarps);
  const long long npairs = static_cast<long long>(s.w1 - s.w0 + 1) * kConsumerWarps;
  float m_run = -INFINITY, l_run = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  bool waited = false;
  for (long long base = 0; base < npairs; base += kMaxPieces) {
    const int count = plan_pieces(p, s, seg, base, s_piece, s_wcount, nwarps);
    if (!waited) {
      griddep_wait();  // the partials come from the attention kernel
      griddep_launch_dependents();
      waited = true;
    }
    merge_pieces<kUnrollSeg>(p, s_piece, count, 0, 1, warp, 4 * lane, m_run, l_run, acc);
    __syncthreads();  // the list is rebuilt by the next pass
  }
  if (!waited) {
    griddep_wait();
    griddep_launch_dependents();
  }
  uint2 v = make_uint2(0u, 0u);  // zeros for an invalid length (flagged by the attention kernel)
  if (s.nt > 0) {
    const float inv = 1.0f / l_run;
    v = make_uint2(pack2_bf16(acc.x * inv, acc.y * inv), pack2_bf16(acc.z * inv, acc.w * inv));
  }
  *reinterpret_cast<uint2 *>(out) = v;
}

// The combine of the 4-bit-cache step: the same log-sum-exp merge over the same pieces (one
// CTA per query head, all 128 dims, four groups of 32 lanes), then the merged row -- still
// in the rotated domain of the cache's codewords -- is rotated back before the bf16
// rounding: out = R^T o = D H o / sqrt(d), H the Sylvester Hadamard matrix applied as a
// fast Walsh-Hadamard transform across the 128 threads (thread = dim).
__global__ void __launch_bounds__(kHeadThreads, 8) q4_combine_kernel(const CombineParams p, const int8_t *signs) {
  constexpr int kWarps = kHeadThreads / 32;
  constexpr int kGroups = kHeadThreads / 32;
  __shared__ int s_piece[kMaxPieces];
  __shared__ int s_wcount[kWarps];
  __shared__ long long s_red[kWarps][2];
  __shared__ __align__(16) float s_o[kGroups][kHeadDim];
  __shared__ float s_m[kGroups], s_l[kGroups];
  __shared__ float s_x[kHeadDim];

  const int tid = threadIdx.x;
  const int bh = blockIdx.x, b = bh / p.Hq, h = bh - b * p.Hq;
  const int kv = h / p.G, g = h - kv * p.G;
  const int grp = tid / 32, sub = tid - grp * 32;
  uint16_t *out = p.out + static_cast<long long>(bh) * kHeadDim;

  const SegSpan s = seg_span(p, b, kv, s_red, kWarps);
  const long long npairs = static_cast<long long>(s.w1 - s.w0 + 1) * kConsumerWarps;
  float m_run = -INFINITY, l_run = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  bool waited = false;
  for (long long base = 0; base < npairs; base += kMaxPieces) {
    const int count = plan_pieces(p, s, b * p.Hkv + kv, base, s_piece, s_wcount, kWarps);
    if (!waited) {
      griddep_wait();  // the partials come from the attention kernel
      griddep_launch_dependents();
      waited = true;
    }
    merge_pieces<kUnroll>(p, s_piece, count, grp, kGroups, g, 4 * sub, m_run, l_run, acc);
    __syncthreads();  // the list is rebuilt by the next pass
  }
  if (!waited) {
    griddep_wait();
    griddep_launch_dependents();
  }
  if (s.nt == 0) {  // invalid length: the attention kernel skipped it and flagged the error
    out[tid] = 0;
    return;
  }
  *reinterpret_cast<float4 *>(&s_o[grp][4 * sub]) = acc;
  if (sub == 0) {
    s_m[grp] = m_run;
    s_l[grp] = l_run;
  }
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < kGroups; ++i) M = fmaxf(M, s_m[i]);
  float num = 0.f, den = 0.f;
#pragma unroll
  for (int i = 0; i < kGroups; ++i) {
    if (s_l[i] == 0.f) continue;  // a group that merged no piece
    const float f = exp2f(s_m[i] - M);
    num = fmaf(f, s_o[i][tid], num);
    den = fmaf(f, s_l[i], den);
  }
  float v = num / den;
  // H v: butterflies over dim bits 0..4 within the warp, bits 5 and 6 through shared memory
#pragma unroll
  for (int hb = 1; hb < 32; hb <<= 1) {
    const float u = __shfl_xor_sync(0xffffffffu, v, hb);
    v = (tid & hb) ? u - v : v + u;
  }
#pragma unroll
  for (int hb = 32; hb < kHeadDim; hb <<= 1) {
    s_x[tid] = v;
    __syncthreads();
    const float u = s_x[tid ^ hb];
    __syncthreads();
    v = (tid & hb) ? u - v : v + u;
  }
  const __nv_bfloat16 r = __float2bfloat16_rn(static_cast<float>(signs[tid]) * v * 0.08838834764831845f);
  out[tid] = *reinterpret_cast<const uint16_t *>(&r);
}

cudaError_t launch_q4_combine(const CombineParams &p, const int8_t *signs, cudaStream_t stream) {
  return launch_pdl(q4_combine_kernel, dim3(static_cast<unsigned>(p.B * p.Hq)), dim3(kHeadThreads), 0, stream, p,
                    signs);
}

cudaError_t configure_combine() {
  const void *fns[5] = {reinterpret_cast<const void *>(combine_head_kernel<1>),
                        reinterpret_cast<const void *>(combine_head_kernel<2>),
                        reinterpret_cast<const void *>(combine_head_kernel<4>),
                        reinterpret_cast<const void *>(combine_seg_kernel),
                        reinterpret_cast<const void *>(q4_combine_kernel)};
  for (const void *f : fns) {
    const cudaError_t e =
        cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int combine_split(int batch, int num_q_heads, int num_kv_heads, int num_workers, int num_sms) {
  const long long segs = static_cast<long long>(batch) * num_kv_heads;
  // expected pieces per query head: consumer warps x workers a segment spans
  const long long pieces = kConsumerWarps * ((num_workers + segs - 1) / segs + 1);
  if (2 * segs >= num_sms && pieces <= 4 * kUnroll * kConsumerWarps / 2) return 0;
  const long long heads = static_cast<long long>(batch) * num_q_heads;
  if (heads * 4 <= 2 * num_sms) return 4;
  if (heads * 2 <= 2 * num_sms) return 2;
  return 1;
}

cudaError_t launch_combine(const CombineParams &p, int split, cudaStream_t stream) {
  if (split == 0)
    return launch_pdl(combine_seg_kernel, dim3(static_cast<unsigned>(p.B * p.Hkv)), dim3(32 * p.G), 0, stream, p);
  const dim3 grid(static_cast<unsigned>(p.B * p.Hq * split));
  if (split == 4) return launch_pdl(combine_head_kernel<4>, grid, dim3(kHeadThreads), 0, stream, p);
  if (split == 2) return launch_pdl(combine_head_kernel<2>, grid, dim3(kHeadThreads), 0, stream, p);
  return launch_pdl(combine_head_kernel<1>, grid, dim3(kHeadThreads), 0, stream, p);
}

}  // namespace gqa
