// launch_onchip.cu -- launchers of the small-segment kernels (adasum_onchip.cuh): the
// on-chip kernel, one launch per cluster size (1..16 CTAs, set at launch time), and the
// one-warp-per-segment kernel for tiny segments.
#include <mutex>
#include <string>

#include "adasum_launch.h"
#include "adasum_onchip.cuh"
#include "adasum_pair.cuh"

namespace adasum {

namespace {

template <typename Tag, int KG1, int NG>
cudaError_t configure(int C) {
  auto kern = onchip_kernel<Tag, KG1, NG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       onchip_dynamic_smem(KG1 * NG));
  if (e == cudaSuccess && C > 8) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

template <typename Tag, int KG1, int NG>
cudaLaunchConfig_t make_config(int count, int C, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(count) * static_cast<unsigned>(C));
  cfg.blockDim = dim3(kOnchipThreads);
  cfg.dynamicSmemBytes = onchip_dynamic_smem(KG1 * NG);
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <typename Tag, int KG1, int NG>
int launch_k(const OnchipArgs& a, int count, int C, void* stream) {
  cudaError_t e = configure<Tag, KG1, NG>(C);
  if (e != cudaSuccess) return static_cast<int>(e);
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = make_config<Tag, KG1, NG>(count, C, static_cast<cudaStream_t>(stream), attr);
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_enter()
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  return static_cast<int>(cudaLaunchKernelEx(&cfg, onchip_kernel<Tag, KG1, NG>, a));
}

// Clusters of C CTAs that fit on the device at once (0: this cluster size cannot run).
template <typename Tag, int KG1, int NG>
int active_clusters(int C) {
  if (configure<Tag, KG1, NG>(C) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_config<Tag, KG1, NG>(C, C, nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, onchip_kernel<Tag, KG1, NG>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

// Profiler names: onchip<dtype,K,cC> (K as groups of 16 when above 16).
const char* kernel_name(bool f32, int K, int C) {
  static std::string names[2][7][5];
  int ki = 0, ci = 0;
  for (int k = 2; k < K; k *= 2) ++ki;
  for (int c = 1; c < C; c *= 2) ++ci;
  std::string& n = names[f32 ? 0 : 1][ki][ci];
  if (n.empty()) {
    const std::string ks = K > 16 ? "16x" + std::to_string(K / 16) : std::to_string(K);
    n = std::string("onchip<") + (f32 ? "f32," : "bf16,") + ks + ",c" + std::to_string(C) + ">";
  }
  return n.c_str();
}

template <typename Tag>
int dispatch(const OnchipArgs& a, int K, int count, int C, void* stream, const char** name) {
  constexpr bool f32 = sizeof(typename ElemTraits<Tag>::Storage) == 4;
  *name = kernel_name(f32, K, C);
  switch (K) {
    case 2: return launch_k<Tag, 2, 1>(a, count, C, stream);
    case 4: return launch_k<Tag, 4, 1>(a, count, C, stream);
    case 8: return launch_k<Tag, 8, 1>(a, count, C, stream);
    case 16: return launch_k<Tag, 16, 1>(a, count, C, stream);
    case 32: return launch_k<Tag, 16, 2>(a, count, C, stream);
    case 64: return launch_k<Tag, 16, 4>(a, count, C, stream);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

template <typename Tag>
int clusters_for(int K, int C) {
  switch (K) {
    case 2: return active_clusters<Tag, 2, 1>(C);
    case 4: return active_clusters<Tag, 4, 1>(C);
    case 8: return active_clusters<Tag, 8, 1>(C);
    case 16: return active_clusters<Tag, 16, 1>(C);
    case 32: return active_clusters<Tag, 16, 2>(C);
    case 64: return active_clusters<Tag, 16, 4>(C);
    default: return 0;
  }
}

}  // namespace

// Clusters of C CTAs of the kernel for (dtype, K) that fit on the current device at
// once, cached per (device, dtype, K, C): the answer depends only on the kernel and the
// device.  -1 for an unsupported dtype or K or a device query that failed.
int onchip_resident_clusters(int dtype, int K, int C) {
  static std::mutex mu;
  static int cache[64][2][7][5];
  static bool init = false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return -1;
  }
  int kidx = 0, cidx = 0;
  for (int k = 2; k < K; k *= 2) ++kidx;
  for (int c = 1; c < C; c *= 2) ++cidx;
  if (kidx > 5 || cidx > 4 || (dtype != kF32 && dtype != kBF16)) return -1;
  std::lock_guard<std::mutex> lock(mu);
  if (!init) {
    for (auto& d : cache)
      for (auto& t : d)
        for (auto& k : t)
          for (int& v : k) v = -1;
    init = true;
  }
  int& slot = cache[dev][dtype][kidx][cidx];
  if (slot < 0) slot = dtype == kF32 ? clusters_for<F32Tag>(K, 1 << cidx) : clusters_for<BF16Tag>(K, 1 << cidx);
  return slot;
}

int onchip_max_cluster(int dtype, int K) {
  int kidx = 0;
  for (int k = 2; k < K; k *= 2) ++kidx;
  if (kidx > 5 || (dtype != kF32 && dtype != kBF16)) return 0;
  for (int C = kOnchipMaxCluster; C >= 2; C /= 2)
    if (onchip_resident_clusters(dtype, K, C) > 0) return C;
  return 1;
}

int launch_onchip(const OnchipArgs& a, int dtype, int K, int count, int C, void* stream,
                  const char** name) {
  if (count <= 0) return 0;
  return dtype == kF32 ? dispatch<F32Tag>(a, K, count, C, stream, name)
                       : dispatch<BF16Tag>(a, K, count, C, stream, name);
}

namespace {
template <typename Tag>
int launch_tiny_tag(const TinyArgs& a, dim3 grid, dim3 block, cudaStream_t s) {
  switch (a.K) {
    case 2: return launch_pdl(tiny_reg_kernel<Tag, 2>, grid, block, 0, s, a);
    case 4: return launch_pdl(tiny_reg_kernel<Tag, 4>, grid, block, 0, s, a);
    case 8: return launch_pdl(tiny_reg_kernel<Tag, 8>, grid, block, 0, s, a);
    case 16: return launch_pdl(tiny_reg_kernel<Tag, 16>, grid, block, 0, s, a);
    case 32: return launch_pdl(tiny_reg_kernel<Tag, 32>, grid, block, 0, s, a);
    case 64: return launch_pdl(tiny_reg_kernel<Tag, 64>, grid, block, 0, s, a);
    default: return launch_pdl(tiny_df_kernel<Tag>, grid, block, 0, s, a);
  }
}
}  // namespace

int launch_tiny_df(const TinyArgs& a, int dtype, void* stream, const char** name) {
  if (a.count <= 0) return 0;
  const bool reg = a.K <= 64;
  // warps: the register kernel packs short segments (see tiny_reg_kernel)
  const int warps = reg ? (a.count8 + 3) / 4 + (a.count16 + 1) / 2 + (a.count - a.count8 - a.count16) : a.count;
  const dim3 grid((warps + kOnchipWarps - 1) / kOnchipWarps), block(kOnchipThreads);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == kF32) {
    *name = reg ? "tiny_reg<f32>" : "tiny_df<f32>";
    return launch_tiny_tag<F32Tag>(a, grid, block, s);
  }
  *name = reg ? "tiny_reg<bf16>" : "tiny_df<bf16>";
  return launch_tiny_tag<BF16Tag>(a, grid, block, s);
}

int pair_fused_max_grid(int dtype) {
  static std::mutex mu;
  static int cache[64][2];
  static bool init = false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || (dtype != kF32 && dtype != kBF16)) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!init) {
    for (auto& d : cache) d[0] = d[1] = -1;
    init = true;
  }
  int& slot = cache[dev][dtype];
  if (slot < 0) {
    int per_sm = 0, sms = 0;
    const cudaError_t e1 =
        dtype == kF32 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pair_fused_kernel<F32Tag>, kPairThreads, 0)
                      : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pair_fused_kernel<BF16Tag>, kPairThreads, 0);
    const cudaError_t e2 = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e1 != cudaSuccess || e2 != cudaSuccess) {
      cudaGetLastError();
      slot = 0;
    } else {
      slot = per_sm * sms;
    }
  }
  return slot;
}

int launch_pair_fused(const PairArgs& a, int dtype, int grid, void* stream, const char** name) {
  PairArgs copy = a;
  void* args[] = {&copy};
  const void* fn = dtype == kF32 ? reinterpret_cast<const void*>(pair_fused_kernel<F32Tag>)
                                 : reinterpret_cast<const void*>(pair_fused_kernel<BF16Tag>);
  *name = dtype == kF32 ? "pair_fused<f32>" : "pair_fused<bf16>";
  const cudaError_t e = cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kPairThreads), args, 0,
                                                    static_cast<cudaStream_t>(stream));
  return static_cast<int>(e);
}

}  // namespace adasum
