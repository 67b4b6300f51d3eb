// Internal launchers shared by the kernel files and the C-ABI layer (not part of the ABI).
#pragma once

#include <utility>

#include "gqa_common.cuh"

namespace gqa {

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

// The fused decode step (decode_step.cu).
size_t step_smem_bytes(int npad, int batch);
cudaError_t step_configure(int npad, int batch);  // dynamic shared-memory limit on the current device
cudaError_t launch_step(const CUtensorMap &tmK, const CUtensorMap &tmV, const StepParams &p, int npad,
                        int num_workers, cudaStream_t stream);

// The binary64 RoPE table (rope_table.cu).
cudaError_t launch_rope_table(const RopeTableParams &p, cudaStream_t stream);
cudaError_t rope_table_configure();

}  // namespace gqa
