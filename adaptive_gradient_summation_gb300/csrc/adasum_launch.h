// adasum_launch.h -- host-side launch helper shared by the launcher translation units.
#pragma once

#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <utility>

namespace adasum {

// Dependent launch is on.  A test build (-DADASUM_TEST_HOOKS) switches it off with
// ADASUM_PDL=0, for comparisons; the product library reads no environment.
inline bool pdl_enabled() {
#ifdef ADASUM_TEST_HOOKS
  static const bool on = [] {
    const char* v = std::getenv("ADASUM_PDL");
    return v == nullptr || std::strcmp(v, "0") != 0;
  }();
  return on;
#else
  return true;
#endif
}

// Launches `kernel` on `stream` with programmatic stream serialization: the kernel may be
// scheduled while the previous kernel of the stream finishes (every kernel of the chain
// starts with pdl_enter(), which waits for that kernel before touching memory).
// Returns the cudaError_t as int.
template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                      Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return static_cast<int>(cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...));
}

}  // namespace adasum
