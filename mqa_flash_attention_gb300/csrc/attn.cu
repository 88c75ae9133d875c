// Translation unit of the fused attention kernel.
#include "attn_kernel.cuh"
#include "internal.h"

namespace ds4a {

cudaError_t prepare_attn_kernel() {
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(attn_fwd_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
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
  return p.comp_fp8 ? cudaLaunchKernelEx(&cfg, attn_fwd_kernel<true>, p) : cudaLaunchKernelEx(&cfg, attn_fwd_kernel<false>, p);
}

}  // namespace ds4a
