// Prologue of the decode step: per-head QK RMSNorm + RoPE of the new token's queries.
//
// "Qwen3-14B Optimization", section 2.1 (Shape 4, and #796 in "Then: buy it") folds
// QK-norm and RoPE into the attention path; section 3.3 batches the G query heads of a
// (batch, KV head) pair into one tile.  The new token's key and value are appended by the
// split-KV attention kernel itself (the warp that owns the tile holding the new token
// computes the rotated key, patches it into its shared-memory tile and writes it to the
// cache), so this kernel only produces the rotated queries.
//
// One CTA per (b, kv): it writes the G rotated query rows of the group into the
// workspace -- already in the 128-byte-swizzled shared-memory image the attention
// kernel's ldmatrix reads, padded to npad rows with zeros.  Query rows are not stored,
// so they are computed in binary32 and rounded to bf16 once (rotate_row_fp32); the
// rotation factors cos/sin(pos * theta^(-2i/d)) come from the plan's binary64 table,
// built once per theta by rope_table_kernel.
#include "launch.h"
#include "rowmath.cuh"

namespace gqa {

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
  uint16_t *qtile = p.q_rot + static_cast<long long>(seg) * p.npad * kHeadDim;
  griddep_wait();               // inputs and the workspace are free once earlier kernels finish
  griddep_launch_dependents();  // the attention kernel may now launch; it waits for us itself

  const int L = p.seq_lens[b], pos = p.positions[b];
  uint32_t bad = 0;
  if (L < 1 || L > p.max_seq) bad = GQA_DEVERR_SEQLEN;
  else if (pos < 0 || pos >= L) bad = GQA_DEVERR_POSITION;
  if (bad) {  // leave a zero q tile: the attention kernel skips or zero-fills this sequence
    if (tid == 0 && kv == 0) atomicOr(p.err, bad);
    for (int i = tid; i < p.npad * kHeadDim; i += blockDim.x) qtile[i] = 0;
    return;
  }
  const double2 d0 = p.rope_tab[static_cast<long long>(pos) * 64 + lane];
  const double2 d1 = p.rope_tab[static_cast<long long>(pos) * 64 + lane + 32];
  const float2 cs0 = make_float2(static_cast<float>(d0.x), static_cast<float>(d0.y));
  const float2 cs1 = make_float2(static_cast<float>(d1.x), static_cast<float>(d1.y));
  for (int g = warp; g < p.G; g += 4) {
    const int h = kv * p.G + g;
    uint16_t z[4];
    rotate_row_fp32(p.q_new + (static_cast<long long>(b) * p.Hq + h) * kHeadDim, p.q_norm_w,
                    static_cast<float>(p.eps), cs0, cs1, lane, z);
#pragma unroll
    for (int t = 0; t < 4; ++t) qtile[qtile_offset(g, lane + 32 * t, p.npad)] = z[t];
  }
  // zero padding rows G..npad-1 of the q tile (both halves)
  const int pad_rows = p.npad - p.G;
  for (int i = tid; i < pad_rows * kHeadDim; i += blockDim.x) {
    const int g = p.G + i / kHeadDim, e = i % kHeadDim;
    qtile[qtile_offset(g, e, p.npad)] = 0;
  }
}

// cos and sin of pos * theta^(-2i/d) for every position below max_seq and pair i < 64,
// in binary64 (CUDA's sincos), rebuilt only when the call's theta changes.
__global__ void __launch_bounds__(256) rope_table_kernel(const RopeTableParams p) {
  griddep_wait();
  griddep_launch_dependents();
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(p.max_seq) * 64) return;
  const int pos = static_cast<int>(idx >> 6), i = static_cast<int>(idx & 63);
  double sv, cv;
  sincos(static_cast<double>(pos) * p.inv_freq[i], &sv, &cv);
  p.rope_tab[idx] = make_double2(cv, sv);
}

cudaError_t launch_rope_table(const RopeTableParams &p, cudaStream_t stream) {
  const long long n = static_cast<long long>(p.max_seq) * 64;
  return launch_pdl(rope_table_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0, stream, p);
}

cudaError_t configure_combine();

cudaError_t configure_small_kernels() {
  cudaError_t e = cudaFuncSetAttribute(prologue_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(rope_table_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) e = configure_combine();
  return e;
}

cudaError_t launch_prologue(const PrologueParams &p, cudaStream_t stream) {
  return launch_pdl(prologue_kernel, dim3(p.B * p.Hkv), dim3(128), 0, stream, p);
}

}  // namespace gqa
