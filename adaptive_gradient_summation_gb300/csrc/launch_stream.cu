// launch_stream.cu -- cooperative launch of the streaming single-stage kernel.
#include "adasum_stream.cuh"

namespace adasum {

namespace {

template <typename In, int KG, bool MOM>
int launch_k(const StageArgs& a, const StreamArgs& s, int grid, size_t smem, void* stream) {
  auto fn = stream_kernel<In, KG, MOM>;
  static bool configured = false;  // per instantiation; calls are serialised by the library
  if (!configured) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return static_cast<int>(cudaGetLastError());
    configured = true;
  } else {
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  }
  StageArgs a_copy = a;
  StreamArgs s_copy = s;
  void* args[] = {&a_copy, &s_copy};
  const cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(fn), dim3(grid),
                                                    dim3(kStreamThreads), args, smem,
                                                    static_cast<cudaStream_t>(stream));
  return static_cast<int>(e != cudaSuccess ? e : cudaGetLastError());
}

template <typename In, bool MOM>
int by_kg(const StageArgs& a, const StreamArgs& s, int grid, size_t smem, void* stream) {
  switch (a.Kg) {
    case 2: return launch_k<In, 2, MOM>(a, s, grid, smem, stream);
    case 4: return launch_k<In, 4, MOM>(a, s, grid, smem, stream);
    case 8: return launch_k<In, 8, MOM>(a, s, grid, smem, stream);
    case 16:
      if constexpr (ElemTraits<In>::kVW == 8) return launch_k<In, 16, MOM>(a, s, grid, smem, stream);
      return static_cast<int>(cudaErrorInvalidValue);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

}  // namespace

bool stream_supported(int dtype, int Kg) {
  if (Kg < 2 || Kg > 16) return false;
  return dtype == kBF16 || Kg <= 8;
}

int stream_smem_bytes(int dtype, int Kg, int stage_pos) {
  const int es = dtype == kBF16 ? 2 : 4;
  return kStages * Kg * (stage_pos * es + kRowPad);
}

int launch_stream(const StageArgs& a, const StreamArgs& s, int dtype, int momentum, int grid,
                  void* stream, const char** name) {
  *name = "stream";
  const size_t smem = static_cast<size_t>(stream_smem_bytes(dtype, a.Kg, s.stage_pos));
  if (dtype == kBF16)
    return momentum ? by_kg<BF16Tag, true>(a, s, grid, smem, stream)
                    : by_kg<BF16Tag, false>(a, s, grid, smem, stream);
  return momentum ? by_kg<F32Tag, true>(a, s, grid, smem, stream)
                  : by_kg<F32Tag, false>(a, s, grid, smem, stream);
}

}  // namespace adasum
