// launch_f32.cu -- launchers for fp32 inputs (user fp32 gradients and the fp32
// intermediates of multi-stage trees) and for the per-segment coefficient kernel.
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

int launch_gram_f32(const StageArgs& a, void* stream, const char** name) {
  const dim3 grid(a.tile_list ? a.ntile_list : a.ntiles, a.G), block(kThreads);
  switch (a.Kg) {
    case 2: *name = "gram_simt<f32,2>"; return launch_serial(gram_simt_kernel<F32Tag, 2>, grid, block, a, stream);
    case 4: *name = "gram_simt<f32,4>"; return launch_serial(gram_simt_kernel<F32Tag, 4>, grid, block, a, stream);
    case 8: *name = "gram_simt<f32,8>"; return launch_serial(gram_simt_kernel<F32Tag, 8>, grid, block, a, stream);
    case 16:  // the tensor cores on an exact three-part bf16 split
      *name = "gram_mma<f32,16>";
      return launch_serial(gram_mma_f32_kernel<16>, grid, block, a, stream);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

int launch_gram_warp(const StageArgs& a, int in_dtype, void* stream, const char** name) {
  constexpr int wpb = kGramWarpThreads / 32;
  const dim3 grid((a.nsmall + wpb - 1) / wpb, a.G), block(kGramWarpThreads);
  if (in_dtype == kF32) {
    switch (a.Kg) {
      case 2: *name = "gram_warp<f32,2>"; return launch(gram_warp_kernel<F32Tag, 2>, grid, block, a, stream);
      case 4: *name = "gram_warp<f32,4>"; return launch(gram_warp_kernel<F32Tag, 4>, grid, block, a, stream);
      case 8: *name = "gram_warp<f32,8>"; return launch(gram_warp_kernel<F32Tag, 8>, grid, block, a, stream);
      case 16: {
        *name = "gram_warp_mma<f32,16>";
        if (!a.aligned) return launch(gram_warp_mma_f32_kernel<16>, grid, block, a, stream);
        // aligned rows: the staged kernel, with its warps' copy rings in dynamic shared memory
        static const int attr = static_cast<int>(cudaFuncSetAttribute(
            gram_warp_staged_f32_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
            static_cast<int>(kGramWarpRingBytes)));
        if (attr != 0) return attr;
        return launch_pdl(gram_warp_staged_f32_kernel<16>, grid, block, kGramWarpRingBytes,
                          static_cast<cudaStream_t>(stream), a);
      }
      default: return static_cast<int>(cudaErrorInvalidValue);
    }
  }
  switch (a.Kg) {
    case 2: *name = "gram_warp<bf16,2>"; return launch(gram_warp_kernel<BF16Tag, 2>, grid, block, a, stream);
    case 4: *name = "gram_warp<bf16,4>"; return launch(gram_warp_kernel<BF16Tag, 4>, grid, block, a, stream);
    case 8: *name = "gram_warp<bf16,8>"; return launch(gram_warp_kernel<BF16Tag, 8>, grid, block, a, stream);
    case 16:  // the tensor cores, as in the CTA Gram
      *name = "gram_warp_mma<bf16,16>";
      return launch(gram_warp_mma_bf16_kernel<16>, grid, block, a, stream);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

int launch_reduce_chunks(const StageArgs& a, void* stream, const char** name) {
  const int per = a.nmulti >= 16 * a.num_sms ? kChunksPerCta : 1;
  const dim3 grid((a.nmulti + per - 1) / per, a.G), block(kThreads);
  switch (a.Kg) {
    case 2: *name = "reduce_chunks<2>"; return launch(reduce_chunks_kernel<2>, grid, block, a, stream);
    case 4: *name = "reduce_chunks<4>"; return launch(reduce_chunks_kernel<4>, grid, block, a, stream);
    case 8: *name = "reduce_chunks<8>"; return launch(reduce_chunks_kernel<8>, grid, block, a, stream);
    case 16: *name = "reduce_chunks<16>"; return launch(reduce_chunks_kernel<16>, grid, block, a, stream);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

int launch_coef(const StageArgs& a, void* stream, const char** name) {
  // several trees per CTA only when there are many more items than SMs
  const int items = (a.seg_list ? a.nseg_list : a.nsegs) * a.G;
  if (items >= 8 * a.num_sms) {
    const dim3 grid((items + kCoefWarps - 1) / kCoefWarps), block(32 * kCoefWarps);
    switch (a.Kg) {
      case 2: *name = "coef<2>"; return launch(coef_warp_kernel<2>, grid, block, a, stream);
      case 4: *name = "coef<4>"; return launch(coef_warp_kernel<4>, grid, block, a, stream);
      case 8: *name = "coef<8>"; return launch(coef_warp_kernel<8>, grid, block, a, stream);
      case 16: *name = "coef<16>"; return launch(coef_warp_kernel<16>, grid, block, a, stream);
      default: return static_cast<int>(cudaErrorInvalidValue);
    }
  }
  const dim3 grid(items), block(32 * kCoefWarps);
  switch (a.Kg) {
    case 2: *name = "coef<2>"; return launch(coef_kernel<2>, grid, block, a, stream);
    case 4: *name = "coef<4>"; return launch(coef_kernel<4>, grid, block, a, stream);
    case 8: *name = "coef<8>"; return launch(coef_kernel<8>, grid, block, a, stream);
    case 16: *name = "coef<16>"; return launch(coef_kernel<16>, grid, block, a, stream);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

template <typename OutTag, bool MOM>
static int combine_f32_k(const StageArgs& a, int warp, void* stream, const char** name) {
  if (warp) {  // short tiles, one warp each
    const dim3 grid(warp_tile_grid(a.nsmall, a.num_sms), a.G), block(kCombineWarpThreads);
    switch (a.Kg) {
      case 1: *name = "combine_warp<f32,1>"; return launch(combine_warp_kernel<F32Tag, OutTag, 1, MOM>, grid, block, a, stream);
      case 2: *name = "combine_warp<f32,2>"; return launch(combine_warp_kernel<F32Tag, OutTag, 2, MOM>, grid, block, a, stream);
      case 4: *name = "combine_warp<f32,4>"; return launch(combine_warp_kernel<F32Tag, OutTag, 4, MOM>, grid, block, a, stream);
      case 8: *name = "combine_warp<f32,8>"; return launch(combine_warp_kernel<F32Tag, OutTag, 8, MOM>, grid, block, a, stream);
      case 16: *name = "combine_warp<f32,16>"; return launch(combine_warp_kernel<F32Tag, OutTag, 16, MOM>, grid, block, a, stream);
      default: return static_cast<int>(cudaErrorInvalidValue);
    }
  }
  const int n = a.tile_list ? a.ntile_list : a.ntiles;
  const dim3 grid((n + a.combine_tiles - 1) / a.combine_tiles, a.G), block(kThreads);
  switch (a.Kg) {
    case 1: *name = "combine<f32,1>"; return launch(combine_kernel<F32Tag, OutTag, 1, MOM>, grid, block, a, stream);
    case 2: *name = "combine<f32,2>"; return launch(combine_kernel<F32Tag, OutTag, 2, MOM>, grid, block, a, stream);
    case 4: *name = "combine<f32,4>"; return launch(combine_kernel<F32Tag, OutTag, 4, MOM>, grid, block, a, stream);
    case 8: *name = "combine<f32,8>"; return launch(combine_kernel<F32Tag, OutTag, 8, MOM>, grid, block, a, stream);
    case 16: *name = "combine<f32,16>"; return launch(combine_kernel<F32Tag, OutTag, 16, MOM>, grid, block, a, stream);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

int launch_combine_f32in(const StageArgs& a, int out_dtype, int momentum, int warp, void* stream,
                         const char** name) {
  if (out_dtype == kF32)
    return momentum ? combine_f32_k<F32Tag, true>(a, warp, stream, name)
                    : combine_f32_k<F32Tag, false>(a, warp, stream, name);
  return momentum ? combine_f32_k<BF16Tag, true>(a, warp, stream, name)
                  : combine_f32_k<BF16Tag, false>(a, warp, stream, name);
}

}  // namespace adasum
