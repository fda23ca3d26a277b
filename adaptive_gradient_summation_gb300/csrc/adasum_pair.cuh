// adasum_pair.cuh -- Adasum(a, b) of two workers over one segment in a single cooperative
// kernel (Scaling Distributed Training with Adaptive Summation, Section 3, the operator
// for two gradients).
//
// For two workers the Gram matrix has three entries, so the coefficient step is a few
// divisions; what costs time in the tiled route is its chain of launches.  Here one
// kernel does all of it, with one grid-wide barrier:
//   1. every thread sums a.b, |a|^2 and |b|^2 over its elements in double-float
//      arithmetic (products exact by TwoProduct), the values first scaled by a power of
//      two from the thread's own largest |value| so that squares stay inside fp32's
//      range; the sums are brought to the CTA's largest exponent (exact power-of-two
//      scaling) and added in a fixed order; each CTA publishes its three sums;
//   2. grid barrier;
//   3. every CTA adds the partials of all CTAs in a fixed order (the same result in every
//      CTA), forms alpha = 1 - a.b / (2|a|^2) and beta = 1 - a.b / (2|b|^2) in
//      double-float (a zero-norm operand gets 1), and combines its own elements as
//      alpha a + beta b in double-float, rounded once to the output type.
// Every thread holds its elements (at most kPairVecs 16-byte vectors of each input) in
// registers from step 1 to step 3, so the inputs are read once and the output written
// once; the host sends only segments that fit the co-resident CTAs that way.  The Gram
// sums carry
// about 2^-48 relative error and the combine rounds once, so there is no conditioning
// check and no recompute.  Exchanging a and b leaves every value bitwise unchanged.
#pragma once

#include "adasum_kernels.cuh"

namespace adasum {

constexpr int kNoExponent = -1000;  // exponent of a thread or CTA that saw no data

// Grid barrier for a cooperative launch: arrivals are counted in bar[0]; the CTA that
// arrives last resets the count and advances the generation in bar[1], which the others
// wait for (clock-bounded: bit 8 of the error word when the budget runs out).  The count
// is back at zero after every barrier, so the state carries over from call to call, and
// from one replay of a captured graph to the next.  no_arrival (the timeout test): the
// CTA waits without arriving, so every wait runs out and the state stays as it was.
__device__ __forceinline__ void pair_grid_barrier(unsigned* bar, unsigned nctas, bool no_arrival,
                                                  long long budget, int* error) {
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile unsigned* gen = bar + 1;
    const unsigned g = *gen;
    __threadfence();  // this CTA's partials before its arrival
    if (!no_arrival && atomicAdd(bar, 1u) == nctas - 1) {
      bar[0] = 0u;
      __threadfence();
      atomicAdd(bar + 1, 1u);
    } else {
      const long long t0 = clock64();
      while (*gen == g) {
        if (clock64() - t0 > budget) {
          atomicOr(error, 8);
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
  }
  __syncthreads();
}

// Largest value over the CTA (every thread gets it).
__device__ __forceinline__ int pair_block_max(int e, int* sh) {
  for (int off = 16; off > 0; off >>= 1) e = max(e, __shfl_xor_sync(0xFFFFFFFFu, e, off));
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = e;
  __syncthreads();
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) e = max(e, sh[w]);
  __syncthreads();
  return e;
}

// Double-float sums over the CTA of three values, every term brought to exponent E
// first: x * 2^(2(e - E)).  A fixed order -- a butterfly within each warp, then one over
// the warps' sums on the first lanes of warp 0 -- so every CTA that adds the same values
// gets the same bits.  Thread 0 gets the results in v.
__device__ __forceinline__ void pair_block_sum3(df32 (&v)[3], int e, int E, df32 (*sh)[kPairThreads / 32]) {
  constexpr int kW = kPairThreads / 32;
  const float f = ldexpf(1.f, 2 * (e - E));
#pragma unroll
  for (int i = 0; i < 3; ++i) v[i] = {v[i].hi * f, v[i].lo * f};
  for (int off = 16; off > 0; off >>= 1)
#pragma unroll
    for (int i = 0; i < 3; ++i) v[i] = df_add(v[i], df_shfl_xor(v[i], off));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0)
#pragma unroll
    for (int i = 0; i < 3; ++i) sh[i][warp] = v[i];
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int i = 0; i < 3; ++i) v[i] = lane < kW ? sh[i][lane] : df32{0.f, 0.f};
    for (int off = kW / 2; off > 0; off >>= 1)
#pragma unroll
      for (int i = 0; i < 3; ++i) v[i] = df_add(v[i], df_shfl_xor(v[i], off));
  }
  __syncthreads();
}

__device__ __forceinline__ df32 pair_coefficient(df32 d, df32 p) {
  if (p.hi == 0.f) return {1.f, 0.f};  // a zero operand: the pair is a plain sum
  return df_add(df32{1.f, 0.f}, df_neg(df_div(d, df32{2.f * p.hi, 2.f * p.lo})));
}

template <typename Tag>
__global__ void __launch_bounds__(kPairThreads) pair_fused_kernel(const PairArgs a) {
  using S = typename ElemTraits<Tag>::Storage;
  constexpr int VW = ElemTraits<Tag>::kVW;
  constexpr int kWarpsPair = kPairThreads / 32;
  __shared__ df32 sh[3][kWarpsPair];
  __shared__ int sh_e[kWarpsPair];
  __shared__ df32 coef[2];
  const S* x = static_cast<const S*>(a.a);
  const S* y = static_cast<const S*>(a.b);
  const bool aligned = a.aligned != 0;
  const int64_t nv = (a.n + VW - 1) / VW;  // <= gridDim.x * kPairThreads * kPairVecs (host)
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kPairThreads;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kPairThreads + threadIdx.x;

  // 1. this thread's vectors, held in registers until the combine
  uint4 ra[kPairVecs], rb[kPairVecs];
#pragma unroll
  for (int j = 0; j < kPairVecs; ++j) {
    const int64_t v = t0 + j * stride;
    ra[j] = v < nv ? load_vec_raw<Tag, kLoadStream>(x, v, 0, a.n, aligned) : make_uint4(0u, 0u, 0u, 0u);
    rb[j] = v < nv ? load_vec_raw<Tag, kLoadStream>(y, v, 0, a.n, aligned) : make_uint4(0u, 0u, 0u, 0u);
  }
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < kPairVecs; ++j)
#pragma unroll
    for (int e = 0; e < VW; ++e)
      amax = fmaxf(amax, fmaxf(fabsf(vec_elem<Tag>(ra[j], e)), fabsf(vec_elem<Tag>(rb[j], e))));
  int ex = 0;
  if (amax > 0.f) frexpf(amax, &ex);
  ex = ex < -125 ? -125 : (ex > 125 ? 125 : ex);
  const float sc = ldexpf(1.f, -ex);
  const int ex_sum = amax > 0.f ? ex : kNoExponent;  // threads without data do not set the scale
  df32 sab = {0.f, 0.f}, saa = {0.f, 0.f}, sbb = {0.f, 0.f};
#pragma unroll
  for (int j = 0; j < kPairVecs; ++j)
#pragma unroll
    for (int e = 0; e < VW; ++e) {
      const float u = vec_elem<Tag>(ra[j], e) * sc, w = vec_elem<Tag>(rb[j], e) * sc;
      const float pab = u * w, paa = u * u, pbb = w * w;
      sab = df_add(sab, df32{pab, __fmaf_rn(u, w, -pab)});
      saa = df_add(saa, df32{paa, __fmaf_rn(u, u, -paa)});
      sbb = df_add(sbb, df32{pbb, __fmaf_rn(w, w, -pbb)});
    }
  // the CTA's largest exponent, then its sums in that scale
  const int E = pair_block_max(ex_sum, sh_e);
  df32 cta[3] = {sab, saa, sbb};
  pair_block_sum3(cta, ex_sum, E, sh);
  if (threadIdx.x == 0) {
    float* p = a.partials + 8 * static_cast<size_t>(blockIdx.x);
    p[0] = cta[0].hi;
    p[1] = cta[0].lo;
    p[2] = cta[1].hi;
    p[3] = cta[1].lo;
    p[4] = cta[2].hi;
    p[5] = cta[2].lo;
    p[6] = __int_as_float(E);
  }

  // 2. every CTA's partials are published
  pair_grid_barrier(a.bar, gridDim.x, a.inject_no_arrival != 0, a.spin_budget, a.error);

  // 3. the totals: thread c < gridDim.x (<= kPairThreads) takes CTA c's partials, all
  //    loads at once; the same fixed order in every CTA, so the same totals everywhere
  {
    const int c = threadIdx.x;
    const bool has = c < static_cast<int>(gridDim.x);
    const float* p = a.partials + 8 * static_cast<size_t>(has ? c : 0);
    df32 pab = {0.f, 0.f}, paa = {0.f, 0.f}, pbb = {0.f, 0.f};
    int pe = kNoExponent;
    if (has) {
      pab = {__ldcg(p + 0), __ldcg(p + 1)};
      paa = {__ldcg(p + 2), __ldcg(p + 3)};
      pbb = {__ldcg(p + 4), __ldcg(p + 5)};
      pe = __float_as_int(__ldcg(p + 6));
    }
    const int Eg = pair_block_max(pe, sh_e);
    df32 tot[3] = {pab, paa, pbb};
    pair_block_sum3(tot, pe, Eg, sh);
    if (threadIdx.x == 0) {
      coef[0] = pair_coefficient(tot[0], tot[1]);
      coef[1] = pair_coefficient(tot[0], tot[2]);
    }
  }
  __syncthreads();
  const df32 al = coef[0], be = coef[1];
  S* out = static_cast<S*>(a.out);
#pragma unroll
  for (int j = 0; j < kPairVecs; ++j) {
    const int64_t v = t0 + j * stride;
    if (v >= nv) break;
    float val[VW];
#pragma unroll
    for (int e = 0; e < VW; ++e) {
      const df32 r = df_add(df_mul_f(al, vec_elem<Tag>(ra[j], e)), df_mul_f(be, vec_elem<Tag>(rb[j], e)));
      if constexpr (VW == 4) {
        val[e] = __fadd_rn(r.hi, r.lo);
      } else {
        // bf16: the double-float value rounded once (through fp64, exact for the sum)
        val[e] = __bfloat162float(__double2bfloat16(df_to_double(r)));
      }
    }
    store_vec<Tag, VW>(out, v * VW, 0, a.n, aligned, val);
  }
}

}  // namespace adasum
