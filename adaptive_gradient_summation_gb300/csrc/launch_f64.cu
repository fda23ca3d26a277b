// launch_f64.cu -- launchers of the fp64 recompute path (flagged segments only) and of
// the list-building kernel.
#include <algorithm>

#include "adasum_kernels.cuh"
#include "adasum_launch.h"

namespace adasum {

namespace {
template <typename Kernel>
int launch(Kernel k, dim3 grid, dim3 block, const StageArgs& a, void* stream) {
  return launch_pdl(k, grid, block, 0, static_cast<cudaStream_t>(stream), a);
}

int kind_of(int dtype, int is_f64) { return is_f64 ? kKindF64 : (dtype == kBF16 ? kKindBF16 : kKindF32); }

template <int IN>
int gram64_k(const StageArgs& a, dim3 grid, void* stream, const char** name) {
  switch (a.Kg) {
    case 2: *name = "gram64<2>"; return launch(gram64_kernel<IN, 2>, grid, dim3(kThreads), a, stream);
    case 4: *name = "gram64<4>"; return launch(gram64_kernel<IN, 4>, grid, dim3(kThreads), a, stream);
    case 8: *name = "gram64<8>"; return launch(gram64_kernel<IN, 8>, grid, dim3(kThreads), a, stream);
    case 16: *name = "gram64<16>"; return launch(gram64_kernel<IN, 16>, grid, dim3(kThreads), a, stream);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

template <int IN, int OUT, bool MOM>
int combine64_k(const StageArgs& a, dim3 grid, void* stream, const char** name) {
  *name = "combine64";
  switch (a.Kg) {
    case 1: return launch(combine64_kernel<IN, OUT, 1, MOM>, grid, dim3(kThreads), a, stream);
    case 2: return launch(combine64_kernel<IN, OUT, 2, MOM>, grid, dim3(kThreads), a, stream);
    case 4: return launch(combine64_kernel<IN, OUT, 4, MOM>, grid, dim3(kThreads), a, stream);
    case 8: return launch(combine64_kernel<IN, OUT, 8, MOM>, grid, dim3(kThreads), a, stream);
    case 16: return launch(combine64_kernel<IN, OUT, 16, MOM>, grid, dim3(kThreads), a, stream);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}
}  // namespace

int launch_local_momentum(const void* g, int dtype, float* v, int64_t n, float mu, int aligned,
                          int num_sms, void* stream, const char** name) {
  *name = "local_momentum";
  const int64_t vw = dtype == kBF16 ? 8 : 4;
  const int64_t blocks = std::min<int64_t>((n / vw + kThreads) / kThreads, 8LL * num_sms);
  const dim3 grid(static_cast<unsigned>(std::max<int64_t>(1, blocks)));
  if (dtype == kBF16)
    return launch_pdl(local_momentum_kernel<BF16Tag>, grid, dim3(kThreads), 0, static_cast<cudaStream_t>(stream), g,
                      v, n, mu, aligned);
  return launch_pdl(local_momentum_kernel<F32Tag>, grid, dim3(kThreads), 0, static_cast<cudaStream_t>(stream), g, v,
                    n, mu, aligned);
}

int launch_orthogonality(const double* outnorm2, const double* diag_sum, int groups, int nsegs,
                         float* ortho, void* stream, const char** name) {
  *name = "orthogonality";
  const int grid = (nsegs + kThreads - 1) / kThreads;
  return launch_pdl(orthogonality_kernel, dim3(grid), dim3(kThreads), 0, static_cast<cudaStream_t>(stream),
                    outnorm2, diag_sum, groups, nsegs, ortho);
}

int launch_collect(const StageArgs& a, int grid, void* stream, const char** name) {
  *name = "collect";
  return launch(collect_kernel, dim3(grid), dim3(kThreads), a, stream);
}

int launch_tiny64(const StageArgs& a, int in_dtype, int out_dtype, int momentum, int grid,
                  void* stream, const char** name) {
  *name = "tiny64";
  const dim3 g(grid), b(kThreads);
  const bool bf = in_dtype == kBF16;
  if (out_dtype != in_dtype) return static_cast<int>(cudaErrorInvalidValue);
  if (momentum)
    return bf ? launch(tiny64_kernel<kKindBF16, kKindBF16, true>, g, b, a, stream)
              : launch(tiny64_kernel<kKindF32, kKindF32, true>, g, b, a, stream);
  return bf ? launch(tiny64_kernel<kKindBF16, kKindBF16, false>, g, b, a, stream)
            : launch(tiny64_kernel<kKindF32, kKindF32, false>, g, b, a, stream);
}

int launch_segmax(const StageArgs& a, int in_dtype, int grid, void* stream, const char** name) {
  *name = "segmax";
  switch (kind_of(in_dtype, 0)) {
    case kKindF32: return launch(segmax_kernel<kKindF32>, dim3(grid), dim3(kThreads), a, stream);
    default: return launch(segmax_kernel<kKindBF16>, dim3(grid), dim3(kThreads), a, stream);
  }
}

int launch_gram64(const StageArgs& a, int in_dtype, int grid, void* stream, const char** name) {
  const dim3 g(grid, a.G);
  switch (kind_of(in_dtype, a.in_f64)) {
    case kKindF32: return gram64_k<kKindF32>(a, g, stream, name);
    case kKindBF16: return gram64_k<kKindBF16>(a, g, stream, name);
    default: return gram64_k<kKindF64>(a, g, stream, name);
  }
}

int launch_coef64(const StageArgs& a, int grid, void* stream, const char** name) {
  const dim3 g(grid, a.G), b(128);
  switch (a.Kg) {
    case 2: *name = "coef64<2>"; return launch(coef64_kernel<2>, g, b, a, stream);
    case 4: *name = "coef64<4>"; return launch(coef64_kernel<4>, g, b, a, stream);
    case 8: *name = "coef64<8>"; return launch(coef64_kernel<8>, g, b, a, stream);
    case 16: *name = "coef64<16>"; return launch(coef64_kernel<16>, g, b, a, stream);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

int launch_combine64(const StageArgs& a, int in_dtype, int out_dtype, int momentum, int grid,
                     void* stream, const char** name) {
  const dim3 g(grid, a.G);
  const int in = kind_of(in_dtype, a.in_f64);
  const int out = kind_of(out_dtype, a.out_f64);
  if (momentum) {  // final stage only
    if (in == kKindF32 && out == kKindF32) return combine64_k<kKindF32, kKindF32, true>(a, g, stream, name);
    if (in == kKindBF16 && out == kKindBF16) return combine64_k<kKindBF16, kKindBF16, true>(a, g, stream, name);
    if (in == kKindF64 && out == kKindF32) return combine64_k<kKindF64, kKindF32, true>(a, g, stream, name);
    if (in == kKindF64 && out == kKindBF16) return combine64_k<kKindF64, kKindBF16, true>(a, g, stream, name);
    return static_cast<int>(cudaErrorInvalidValue);
  }
  if (in == kKindF32 && out == kKindF64) return combine64_k<kKindF32, kKindF64, false>(a, g, stream, name);
  if (in == kKindF32 && out == kKindF32) return combine64_k<kKindF32, kKindF32, false>(a, g, stream, name);
  if (in == kKindBF16 && out == kKindF64) return combine64_k<kKindBF16, kKindF64, false>(a, g, stream, name);
  if (in == kKindBF16 && out == kKindBF16) return combine64_k<kKindBF16, kKindBF16, false>(a, g, stream, name);
  if (in == kKindF64 && out == kKindF64) return combine64_k<kKindF64, kKindF64, false>(a, g, stream, name);
  if (in == kKindF64 && out == kKindF32) return combine64_k<kKindF64, kKindF32, false>(a, g, stream, name);
  if (in == kKindF64 && out == kKindBF16) return combine64_k<kKindF64, kKindBF16, false>(a, g, stream, name);
  return static_cast<int>(cudaErrorInvalidValue);
}

}  // namespace adasum
