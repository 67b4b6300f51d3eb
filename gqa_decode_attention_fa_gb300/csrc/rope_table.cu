// The RoPE tables of a plan: cos and sin of pos * theta^(-2i/d) for every position below
// max_seq and pair i < 64 ("Qwen3-14B Optimization", section 3.3: the lo/hi halves of a
// 128-dim head rotate as pairs (i, i + 64)).  The attention kernel rotates the new token's
// query (binary32) and key (double-word) with them.
#include "launch.h"

namespace gqa {

// cos and sin of pos * theta^(-2i/d) for every position below max_seq and pair i < 64,
// computed in binary64 (CUDA's sincos) and stored as double-word pairs (hi = the binary32
// rounding, lo = the binary32 rounding of the rest: 48 significant bits) for the key row,
// and as binary32 for the query rotation; rebuilt only when the call's theta changes.
__global__ void __launch_bounds__(256) rope_table_kernel(const RopeTableParams p) {
  griddep_wait();
  griddep_launch_dependents();
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(p.max_seq) * 64) return;
  const int pos = static_cast<int>(idx >> 6), i = static_cast<int>(idx & 63);
  double sv, cv;
  sincos(static_cast<double>(pos) * p.inv_freq[i], &sv, &cv);
  const float ch = static_cast<float>(cv), sh = static_cast<float>(sv);
  p.rope_dw[idx] = make_float4(ch, sh, static_cast<float>(cv - ch), static_cast<float>(sv - sh));
  p.rope_tab32[idx] = make_float2(ch, sh);
}

cudaError_t launch_rope_table(const RopeTableParams &p, cudaStream_t stream) {
  const long long n = static_cast<long long>(p.max_seq) * 64;
  return launch_pdl(rope_table_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0, stream, p);
}

cudaError_t configure_combine();

cudaError_t configure_small_kernels() {
  cudaError_t e = cudaFuncSetAttribute(rope_table_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) e = configure_combine();
  return e;
}

}  // namespace gqa
