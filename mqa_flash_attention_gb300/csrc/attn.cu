// Translation unit of the fused attention kernel.
#include "attn_kernel.cuh"
#include "internal.h"

namespace ds4a {

cudaError_t prepare_attn_kernel() {
  return cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
}

cudaError_t launch_attn(const AttnParams &p, int grid, cudaStream_t s) {
  attn_fwd_kernel<<<grid, kThreads, kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace ds4a
