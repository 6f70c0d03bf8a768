// Kernel launches with programmatic dependent launch (PDL).
//
// Every kernel of the library is launched with programmatic stream serialization
// allowed. Each kernel calls pdl_trigger() at entry, so the next kernel on the stream
// may be scheduled as soon as all of this kernel's CTAs are resident, and calls
// pdl_wait() before its first access to global memory that a previous kernel may write
// or that a previous kernel may still read, which returns only once the previous kernel
// on the stream has completed and its writes are visible. Before that wait a kernel does
// only work that neither reads what an earlier kernel writes nor writes anything:
// shared-memory setup, TMEM allocation, tensor-map prefetch, and (the narrow grouped-GEMM
// launch) L2 prefetches of expert weight tiles, which are inputs of the whole forward
// that no kernel of the library writes. Stream order is therefore preserved by
// construction. Without a preceding kernel both calls are no-ops.
#pragma once

#include <utility>

#include <cuda_runtime.h>

namespace moe {

__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
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

}  // namespace moe
