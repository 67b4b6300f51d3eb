// Internal launchers shared by the kernel files and the C-ABI layer (not part of the ABI).
#pragma once

#include "gqa_common.cuh"

namespace gqa {

cudaError_t launch_prologue(const PrologueParams &p, cudaStream_t stream);

// Dynamic shared memory the split-KV kernel needs for a group padded to npad rows.
size_t attn_smem_bytes(int npad, int batch);
// Raises the kernel's dynamic shared-memory limit on the current device.
cudaError_t attn_configure(int npad, int batch);
cudaError_t launch_attention(const CUtensorMap &tmK, const CUtensorMap &tmV, const AttnParams &p, int npad,
                             int num_workers, cudaStream_t stream);

cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream);

}  // namespace gqa
