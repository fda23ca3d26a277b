// adasum_noalloc.cu -- adasum_pair_noalloc: the two-worker Adasum of adasum_pair for
// callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they need the reduction: a
// framework's caching allocator may already own nearly all of the GPU's memory (a fresh
// cudaMalloc then fails, or forces the framework to release and re-fragment its pool),
// cudaMalloc and cudaFree synchronise the device and so stall a latency-sensitive loop,
// and some serving processes fix their memory footprint at start-up and forbid any
// allocation afterwards.  The regular entry points grow a library workspace with
// cudaMalloc on first use; this one never allocates.  Its scratch memory is a fixed
// file-scope __device__ array (64 KiB plus a few bytes), which every GPU that loads the
// library holds until the process exits.
//
// What it computes: Adasum(a, b) = (1 - a.b/(2|a|^2)) a + (1 - a.b/(2|b|^2)) b over one
// segment of n elements, by the same three steps as the regular path (per-tile partial
// dot products, fp64 coefficients from their compensated sum, a symmetric combine).  It
// runs only the fp32 pass: it does not estimate the conditioning or recompute
// ill-conditioned inputs in fp64 as adasum_pair does.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/adasum.h"
#include "adasum_kernels.cuh"

namespace adasum {
namespace noalloc {

constexpr int kTile = 8192;                   // positions per tile
constexpr int kMaxTiles = 4096;               // tiles per call
constexpr int64_t kMaxN = int64_t(kTile) * kMaxTiles;
static_assert(kMaxN == ADASUM_NOALLOC_MAX_N, "header and implementation disagree");
constexpr int kCoefOffset = 4 * kMaxTiles;    // floats: per-tile partials come first
constexpr int kScratchFloats = kCoefOffset + 64;

// The scratch: per-tile partial sums (a.b, |a|^2, |b|^2, unused) followed by the two
// coefficients.  Every call writes each slot it later reads (tiles [0, ntiles) and the
// two coefficients) before reading it, so nothing has to start at zero and nothing is
// carried from one call to the next.  Calls that overlap on the GPU share these slots
// and race.
static __device__ __align__(256) float g_scratch[kScratchFloats];

template <typename Tag>
__global__ void __launch_bounds__(kThreads) pair_gram_kernel(const void* a, const void* b,
                                                             int64_t n, int aligned,
                                                             float* scratch) {
  using S = typename ElemTraits<Tag>::Storage;
  constexpr int VW = ElemTraits<Tag>::kVW;
  const int tile = blockIdx.x;
  const int64_t lo = static_cast<int64_t>(tile) * kTile;
  const int64_t hi = lo + kTile < n ? lo + kTile : n;
  const S* x = static_cast<const S*>(a);
  const S* y = static_cast<const S*>(b);
  float acc[3] = {0.f, 0.f, 0.f};
  for (int64_t v = lo / VW + threadIdx.x; v < (hi + VW - 1) / VW; v += kThreads) {
    const uint4 ra = load_vec_raw<Tag, kLoadKeep>(x, v, lo, hi, aligned != 0);
    const uint4 rb = load_vec_raw<Tag, kLoadKeep>(y, v, lo, hi, aligned != 0);
#pragma unroll
    for (int e = 0; e < VW; ++e) {
      const float xa = vec_elem<Tag>(ra, e), xb = vec_elem<Tag>(rb, e);
      acc[0] = __fmaf_rn(xa, xb, acc[0]);
      acc[1] = __fmaf_rn(xa, xa, acc[1]);
      acc[2] = __fmaf_rn(xb, xb, acc[2]);
    }
  }
  block_reduce_store<3>(acc, scratch + 4 * tile);
}

// One CTA of three warps, warp w summing quantity w (a.b, |a|^2, |b|^2) of the tile
// partials: lane l takes tiles l, l + 32, ... (compensated fp32, in tile order), then
// the lanes' sums are added in fp64 by a fixed butterfly, so the result is the same bits
// on every run.  Then the coefficients in fp64 (a zero-norm operand gets coefficient 1).
constexpr int kCoefThreads = 96;
__global__ void __launch_bounds__(kCoefThreads) pair_coef_kernel(int ntiles, float* scratch) {
  __shared__ double sums[3];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float s = 0.f, comp = 0.f;
  for (int t = lane; t < ntiles; t += 32) kahan_add(s, comp, scratch[4 * t + w]);
  double v = static_cast<double>(s) - static_cast<double>(comp);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
  if (lane == 0) sums[w] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    const double d = sums[0], p = sums[1], q = sums[2];
    const double alpha = 1.0 - (p == 0.0 ? 0.0 : d / (2.0 * p));
    const double beta = 1.0 - (q == 0.0 ? 0.0 : d / (2.0 * q));
    scratch[kCoefOffset] = static_cast<float>(alpha);
    scratch[kCoefOffset + 1] = static_cast<float>(beta);
  }
}

// out = alpha a + beta b, both products rounded before the sum, so swapping a and b
// gives the same bits.
template <typename Tag>
__global__ void __launch_bounds__(kThreads) pair_combine_kernel(const void* a, const void* b,
                                                                void* out, int64_t n,
                                                                int aligned,
                                                                const float* scratch) {
  using S = typename ElemTraits<Tag>::Storage;
  constexpr int VW = ElemTraits<Tag>::kVW;
  const int tile = blockIdx.x;
  const int64_t lo = static_cast<int64_t>(tile) * kTile;
  const int64_t hi = lo + kTile < n ? lo + kTile : n;
  const float alpha = scratch[kCoefOffset], beta = scratch[kCoefOffset + 1];
  const S* x = static_cast<const S*>(a);
  const S* y = static_cast<const S*>(b);
  S* o = static_cast<S*>(out);
  for (int64_t v = lo / VW + threadIdx.x; v < (hi + VW - 1) / VW; v += kThreads) {
    const uint4 ra = load_vec_raw<Tag, kLoadStream>(x, v, lo, hi, aligned != 0);
    const uint4 rb = load_vec_raw<Tag, kLoadStream>(y, v, lo, hi, aligned != 0);
    float val[VW];
#pragma unroll
    for (int e = 0; e < VW; ++e)
      val[e] = __fadd_rn(__fmul_rn(alpha, vec_elem<Tag>(ra, e)), __fmul_rn(beta, vec_elem<Tag>(rb, e)));
    store_vec<Tag, VW>(o, v * VW, lo, hi, aligned != 0, val);
  }
}

// Device address of g_scratch, looked up once per device with that device current.
constexpr int kMaxDevices = 128;
std::mutex g_setup_mu;
float* g_scratch_ptr[kMaxDevices] = {};

adasum_status_t scratch_for_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ADASUM_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return ADASUM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return ADASUM_ERR_CUDA;
    }
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
  return ADASUM_OK;
}

// One launch through cudaLaunchKernelEx, whose return value is that launch's own error.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), int grid, int block, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

bool overlap(const void* p, const void* q, size_t bytes) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(p), y = reinterpret_cast<uintptr_t>(q);
  return x < y + bytes && y < x + bytes;
}

}  // namespace noalloc
}  // namespace adasum

extern "C" adasum_status_t adasum_pair_noalloc(const void* a, const void* b, int64_t n,
                                               adasum_dtype_t dtype, void* out,
                                               adasum_stream_t stream) {
  using namespace adasum;
  using namespace adasum::noalloc;
  if (dtype != ADASUM_F32 && dtype != ADASUM_BF16) return ADASUM_ERR_INVALID_ARG;
  if (n < 0) return ADASUM_ERR_INVALID_ARG;
  if (n > kMaxN) return ADASUM_ERR_UNSUPPORTED;
  if (n == 0) return ADASUM_OK;
  if (a == nullptr || b == nullptr || out == nullptr) return ADASUM_ERR_INVALID_ARG;
  const size_t bytes = static_cast<size_t>(n) * (dtype == ADASUM_BF16 ? 2 : 4);
  if ((out != a && overlap(out, a, bytes)) || (out != b && overlap(out, b, bytes)))
    return ADASUM_ERR_ALIAS;
  float* scratch = nullptr;
  if (adasum_status_t st = scratch_for_current_device(&scratch)) return st;
  const int aligned = ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) |
                        reinterpret_cast<uintptr_t>(out)) & 15u) == 0;
  const int ntiles = static_cast<int>((n + kTile - 1) / kTile);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // Each launch's own return code decides the status (an error left pending by other
  // code on this thread is neither reported as this call's nor cleared).
  const bool bf16 = dtype == ADASUM_BF16;
  if (launch(bf16 ? pair_gram_kernel<BF16Tag> : pair_gram_kernel<F32Tag>, ntiles, kThreads, s,
             a, b, n, aligned, scratch) != cudaSuccess ||
      launch(pair_coef_kernel, 1, kCoefThreads, s, ntiles, scratch) != cudaSuccess ||
      launch(bf16 ? pair_combine_kernel<BF16Tag> : pair_combine_kernel<F32Tag>, ntiles, kThreads, s,
             a, b, out, n, aligned, static_cast<const float*>(scratch)) != cudaSuccess)
    return ADASUM_ERR_CUDA;
  return ADASUM_OK;
}
