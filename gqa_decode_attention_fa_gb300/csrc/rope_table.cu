// The plan's RoPE table: cos and sin of pos * theta^(-2i/d) for every position below
// max_seq and every pair i < 64, in binary64 (CUDA's sincos).  It is rebuilt only when a
// call's theta differs from the table's, so a decode step evaluates no transcendental
// function ("Qwen3-14B Optimization", section 3.3: the rotation of the half-split pairs
// (i, i + d/2) at the token's position).
#include "launch.h"

namespace gqa {

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

cudaError_t rope_table_configure() {
  // same carveout as the step kernel, so the two never make an SM switch configuration
  return cudaFuncSetAttribute(rope_table_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared);
}

cudaError_t launch_rope_table(const RopeTableParams &p, cudaStream_t stream) {
  const long long n = static_cast<long long>(p.max_seq) * 64;
  return launch_pdl(rope_table_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0, stream, p);
}

}  // namespace gqa
