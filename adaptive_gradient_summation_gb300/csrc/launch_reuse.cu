// launch_reuse.cu -- launcher of the persistent reuse kernel (adasum_reuse.cuh).
#include "adasum_reuse.cuh"

namespace adasum {

namespace {
template <int KG>
int max_grid() {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reuse_kernel<KG>, kReuseThreads, 0) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return per_sm >= 1 ? sms : 0;  // one CTA per SM
}
}  // namespace

int reuse_max_grid(int KG) {
  static int cached[2] = {-1, -1};
  const int i = KG == 16 ? 1 : 0;
  if (cached[i] < 0) cached[i] = KG == 16 ? max_grid<16>() : max_grid<8>();
  return cached[i];
}

// Cooperative launch: every CTA must be resident, since C steps wait (bounded) on
// coefficients that other CTAs' finisher warps publish.
int launch_reuse(const ReuseArgs& a, int KG, int grid, void* stream, const char** name) {
  void* args[] = {const_cast<ReuseArgs*>(&a)};
  const void* fn = KG == 16 ? reinterpret_cast<const void*>(reuse_kernel<16>)
                            : reinterpret_cast<const void*>(reuse_kernel<8>);
  *name = KG == 16 ? "reuse<bf16,16>" : "reuse<bf16,8>";
  if (KG != 8 && KG != 16) return static_cast<int>(cudaErrorInvalidValue);
  return static_cast<int>(cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kReuseThreads), args, 0,
                                                      static_cast<cudaStream_t>(stream)));
}

}  // namespace adasum
