// launch_pipe.cu -- launchers of the fused single-stage kernel (one instantiation per
// input type, output type, group size and momentum flag).
#include "adasum_kernels.cuh"

namespace adasum {

namespace {

template <typename In, typename Out, int KG, bool MOM>
int launch_k(const StageArgs& a, const PipeArgs& p, int grid, void* stream) {
  pipeline_kernel<In, Out, KG, MOM><<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(a, p);
  return static_cast<int>(cudaGetLastError());
}

template <typename In, typename Out, int KG, bool MOM>
int occupancy_k() {
  int blocks = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, pipeline_kernel<In, Out, KG, MOM>,
                                                kThreads, 0);
  return blocks > 0 ? blocks : 1;
}

// Calls F<In, Out, KG, MOM>() for the runtime combination (in, out, Kg, momentum).
template <template <typename, typename, int, bool> class F, typename... Args>
int dispatch(int in_dtype, int out_dtype, int Kg, int momentum, Args&&... args) {
#define ADASUM_DISPATCH_KG(IN, OUT, MOM)                                      \
  switch (Kg) {                                                             \
    case 1: return F<IN, OUT, 1, MOM>::run(args...);                        \
    case 2: return F<IN, OUT, 2, MOM>::run(args...);                        \
    case 4: return F<IN, OUT, 4, MOM>::run(args...);                        \
    case 8: return F<IN, OUT, 8, MOM>::run(args...);                        \
    case 16: return F<IN, OUT, 16, MOM>::run(args...);                      \
    default: return -1;                                                     \
  }
  if (in_dtype != out_dtype) return -1;  // single stage: output type = input type
  if (in_dtype == kBF16) {
    if (momentum) { ADASUM_DISPATCH_KG(BF16Tag, BF16Tag, true) }
    ADASUM_DISPATCH_KG(BF16Tag, BF16Tag, false)
  }
  if (momentum) { ADASUM_DISPATCH_KG(F32Tag, F32Tag, true) }
  ADASUM_DISPATCH_KG(F32Tag, F32Tag, false)
#undef ADASUM_DISPATCH_KG
}

template <typename In, typename Out, int KG, bool MOM>
struct Launch {
  static int run(const StageArgs& a, const PipeArgs& p, int grid, void* stream) {
    return launch_k<In, Out, KG, MOM>(a, p, grid, stream);
  }
};

template <typename In, typename Out, int KG, bool MOM>
struct Occupancy {
  static int run() { return occupancy_k<In, Out, KG, MOM>(); }
};

}  // namespace

int pipeline_grid(int in_dtype, int out_dtype, int Kg, int momentum, int num_sms) {
  const int per_sm = dispatch<Occupancy>(in_dtype, out_dtype, Kg, momentum);
  return per_sm > 0 ? per_sm * num_sms : num_sms;
}

int launch_pipeline(const StageArgs& a, const PipeArgs& p, int in_dtype, int out_dtype,
                    int momentum, int grid, void* stream, const char** name) {
  *name = "pipeline";
  const int rc = dispatch<Launch>(in_dtype, out_dtype, a.Kg, momentum, a, p, grid, stream);
  return rc < 0 ? static_cast<int>(cudaErrorInvalidValue) : rc;
}

}  // namespace adasum
