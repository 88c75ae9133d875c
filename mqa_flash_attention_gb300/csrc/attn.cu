// Translation unit of the fused attention kernel.
#include "attn_kernel.cuh"
#include "internal.h"

namespace ds4a {

cudaError_t prepare_attn_kernel() {
  return cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
}

// Launched with programmatic stream serialization: the kernel's prologue may
// overlap the previous kernel in the stream; it waits (griddepcontrol.wait)
// before touching global memory.
cudaError_t launch_attn(const AttnParams &p, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_fwd_kernel, p);
}

}  // namespace ds4a
