// Translation unit of the fused attention kernel.
#include "attn_kernel.cuh"
#include "internal.h"

namespace ds4a {

cudaError_t prepare_attn_kernel() {
  const void *k[4] = {(const void *)attn_fwd_kernel<false, false>, (const void *)attn_fwd_kernel<false, true>,
                      (const void *)attn_fwd_kernel<true, false>, (const void *)attn_fwd_kernel<true, true>};
  for (const void *f : k) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
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
  const bool la = look_ahead_suits(p);
  if (p.comp_fp8)
    return la ? cudaLaunchKernelEx(&cfg, attn_fwd_kernel<true, true>, p)
              : cudaLaunchKernelEx(&cfg, attn_fwd_kernel<true, false>, p);
  return la ? cudaLaunchKernelEx(&cfg, attn_fwd_kernel<false, true>, p)
            : cudaLaunchKernelEx(&cfg, attn_fwd_kernel<false, false>, p);
}

}  // namespace ds4a
