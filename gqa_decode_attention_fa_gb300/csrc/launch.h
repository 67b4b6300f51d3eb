// Internal launchers shared by the kernel files and the C-ABI layer (not part of the ABI).
#pragma once

#include <utility>

#include "gqa_common.cuh"

namespace gqa {

cudaError_t launch_prologue(const PrologueParams &p, cudaStream_t stream);
cudaError_t launch_rope_table(const RopeTableParams &p, cudaStream_t stream);

// Launches `kernel` with programmatic stream serialization (it may begin while the
// previous kernel in the stream finishes; the kernels order themselves with
// griddepcontrol.wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Dynamic shared memory the split-KV kernel needs for a group padded to npad rows.
size_t attn_smem_bytes(int npad, int batch);
// Raises the kernel's dynamic shared-memory limit on the current device to what a launch
// of the largest supported batch needs.  The limit is per function, not per plan, so it
// never depends on one plan's batch: a plan made later for a smaller batch must not lower
// it under an earlier plan's launches.
cudaError_t attn_configure(int npad);
cudaError_t launch_attention(const CUtensorMap &tmK, const CUtensorMap &tmV, const AttnParams &p, int npad,
                             int num_workers, cudaStream_t stream);

cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream);

// Gives the prologue, combine and table kernels the attention kernel's shared-memory
// carveout, so that consecutive kernels of a step never make an SM switch configuration.
cudaError_t configure_small_kernels();

}  // namespace gqa
