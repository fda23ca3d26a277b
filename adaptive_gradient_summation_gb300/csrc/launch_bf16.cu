// launch_bf16.cu -- launchers for bf16 gradients (tensor-core Gram for 8 and 16
// workers, CUDA-core Gram for 2 and 4).
#include "adasum_kernels.cuh"
#include "adasum_launch.h"

namespace adasum {

namespace {
template <typename Kernel>
int launch(Kernel k, dim3 grid, dim3 block, const StageArgs& a, void* stream) {
  return launch_pdl(k, grid, block, 0, static_cast<cudaStream_t>(stream), a);
}
// The CTA Gram launch goes out without the dependent-launch attribute: launched early,
// its large grid fills the SMs with CTAs waiting on the previous kernel, and behind a
// latency-bound kernel (the small-segment ones) that wait slowed the predecessor's tail
// (K=64 set: 1.94 -> 1.74 ms per call without the attribute here).
template <typename Kernel>
int launch_serial(Kernel k, dim3 grid, dim3 block, const StageArgs& a, void* stream) {
  k<<<grid, block, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return static_cast<int>(cudaGetLastError());
}
}  // namespace

int launch_gram_bf16(const StageArgs& a, void* stream, const char** name) {
  const dim3 grid(a.tile_list ? a.ntile_list : a.ntiles, a.G), block(kThreads);
  switch (a.Kg) {
    case 2: *name = "gram_simt<bf16,2>"; return launch_serial(gram_simt_kernel<BF16Tag, 2>, grid, block, a, stream);
    case 4: *name = "gram_simt<bf16,4>"; return launch_serial(gram_simt_kernel<BF16Tag, 4>, grid, block, a, stream);
    case 8: *name = "gram_mma<bf16,8>"; return launch_serial(gram_mma_bf16_kernel<8>, grid, block, a, stream);
    case 16: *name = "gram_mma<bf16,16>"; return launch_serial(gram_mma_bf16_kernel<16>, grid, block, a, stream);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

template <typename OutTag, bool MOM>
static int combine_bf16_k(const StageArgs& a, int warp, void* stream, const char** name) {
  if (warp) {  // short tiles, one warp each
    const dim3 grid(warp_tile_grid(a.nsmall, a.num_sms), a.G), block(kCombineWarpThreads);
    switch (a.Kg) {
      case 1: *name = "combine_warp<bf16,1>"; return launch(combine_warp_kernel<BF16Tag, OutTag, 1, MOM>, grid, block, a, stream);
      case 2: *name = "combine_warp<bf16,2>"; return launch(combine_warp_kernel<BF16Tag, OutTag, 2, MOM>, grid, block, a, stream);
      case 4: *name = "combine_warp<bf16,4>"; return launch(combine_warp_kernel<BF16Tag, OutTag, 4, MOM>, grid, block, a, stream);
      case 8: *name = "combine_warp<bf16,8>"; return launch(combine_warp_kernel<BF16Tag, OutTag, 8, MOM>, grid, block, a, stream);
      case 16: *name = "combine_warp<bf16,16>"; return launch(combine_warp_kernel<BF16Tag, OutTag, 16, MOM>, grid, block, a, stream);
      default: return static_cast<int>(cudaErrorInvalidValue);
    }
  }
  const int n = a.tile_list ? a.ntile_list : a.ntiles;
  const dim3 grid((n + a.combine_tiles - 1) / a.combine_tiles, a.G), block(kThreads);
  switch (a.Kg) {
    case 1: *name = "combine<bf16,1>"; return launch(combine_kernel<BF16Tag, OutTag, 1, MOM>, grid, block, a, stream);
    case 2: *name = "combine<bf16,2>"; return launch(combine_kernel<BF16Tag, OutTag, 2, MOM>, grid, block, a, stream);
    case 4: *name = "combine<bf16,4>"; return launch(combine_kernel<BF16Tag, OutTag, 4, MOM>, grid, block, a, stream);
    case 8: *name = "combine<bf16,8>"; return launch(combine_kernel<BF16Tag, OutTag, 8, MOM>, grid, block, a, stream);
    case 16: *name = "combine<bf16,16>"; return launch(combine_kernel<BF16Tag, OutTag, 16, MOM>, grid, block, a, stream);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

int launch_combine_bf16in(const StageArgs& a, int out_dtype, int momentum, int warp, void* stream,
                          const char** name) {
  if (out_dtype == kF32)
    return momentum ? combine_bf16_k<F32Tag, true>(a, warp, stream, name)
                    : combine_bf16_k<F32Tag, false>(a, warp, stream, name);
  return momentum ? combine_bf16_k<BF16Tag, true>(a, warp, stream, name)
                  : combine_bf16_k<BF16Tag, false>(a, warp, stream, name);
}

}  // namespace adasum
