// adasum_kernels.cuh -- device code of the GB300 Adasum library (sm_103a).
//
// "Scaling Distributed Training with Adaptive Summation", Section 3: per layer segment,
// the K worker gradients are combined by a binary tree of
//     Adasum(a, b) = (1 - a.b/(2|a|^2)) a + (1 - a.b/(2|b|^2)) b,
// pairs (2i, 2i+1) at every level.  The tree is linear in the leaves, so its result is
// out = sum_k c_k g_k, and every dot product it needs is a quadratic form of the
// segment's Gram matrix.  The kernels here are:
//   gram_*     pass 1: Gram partials of one tile (upper triangle, fp32), one HBM read,
//              with each worker's nonzero bits for the range check
//   reduce_chunks, coef / coef_warp
//              per segment: sum the tile partials (compensated, fixed order), run the
//              tree on the Gram matrix in double-float with its error estimate, emit
//              c_0..c_{K-1} and the recompute flag
//   combine    pass 2: out = sum_k c_k g_k, evaluated as a pairwise tree that mirrors
//              the Adasum tree (so swapping sibling subtrees is bitwise symmetric),
//              optionally followed by a heavy-ball Momentum-SGD step
//   *64        the fp64 recompute of flagged segments
// This path is HBM-bound (a few FMAs per byte), so it is written around coalesced
// 128-bit loads and a grid of tiles that keeps every SM streaming.  The Gram of 8- and
// 16-worker groups uses the tensor cores through mma.sync: bf16 x bf16 products are
// exact in fp32, fp32 values are split exactly into bf16 parts, and the 16x16 Gram of
// a group is a true (tiny) dense contraction.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "adasum_internal.h"
#include "adasum_ptx.cuh"

namespace adasum {

constexpr int kWarps = kThreads / 32;

__host__ __device__ constexpr int tri_count(int K) { return K * (K + 1) / 2; }
// Row-major index of (i, j), i <= j, in the packed upper triangle of a K x K matrix.
__host__ __device__ constexpr int tri_index(int K, int i, int j) {
  return i * K - (i * (i - 1)) / 2 + (j - i);
}

// Unpacks entry e of the packed upper triangle into (i, j), i <= j.  (A closed form, the
// row from the quadratic's root in fp32, measured slower in the coefficient and Gram
// kernels than this loop: 0.1809 -> 0.1823 ms for fp32 K = 16 on the 10,000-segment layout.)
__device__ __forceinline__ void tri_unpack(int K, int e, int& i, int& j) {
  i = 0;
  int rem = e;
  while (rem >= K - i) {
    rem -= K - i;
    ++i;
  }
  j = i + rem;
}

// ------------------------------------------------------------------ element access

struct F32Tag {};
struct BF16Tag {};

template <typename Tag> struct ElemTraits;
template <> struct ElemTraits<F32Tag> {
  using Storage = float;
  static constexpr int kVW = 4;  // elements per 16-byte vector
};
template <> struct ElemTraits<BF16Tag> {
  using Storage = uint16_t;
  static constexpr int kVW = 8;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&p);
}
__device__ __forceinline__ uint16_t float_to_bf16_bits(float x) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&h);
}

// Cache policies: pass 1 reads through the non-coherent path without allocating in L1;
// pass 2 reads and writes with the streaming (evict-first) policy because nothing is
// reused after it.
enum LoadPolicy { kLoadKeep = 0, kLoadStream = 1 };

template <int P>
__device__ __forceinline__ uint4 ld16(const void* p) {
  if constexpr (P == kLoadStream) {
    return __ldcs(reinterpret_cast<const uint4*>(p));
  } else {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
  }
}

// The raw 16-byte vector v (elements [v*VW, v*VW + VW)) of a gradient, with every
// element outside [lo, hi) replaced by +0.  Positions outside [lo, hi) are never
// dereferenced, so partial vectors at buffer ends stay in bounds.
template <typename Tag, int P>
__device__ __forceinline__ uint4 load_vec_raw(const typename ElemTraits<Tag>::Storage* x,
                                              int64_t v, int64_t lo, int64_t hi,
                                              bool aligned) {
  constexpr int VW = ElemTraits<Tag>::kVW;
  if (x == nullptr) return make_uint4(0u, 0u, 0u, 0u);  // a zero (padding) gradient
  const int64_t p0 = v * VW;
  if (aligned && p0 >= lo && p0 + VW <= hi) return ld16<P>(x + p0);
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int e = 0; e < VW; ++e) {
    const int64_t p = p0 + e;
    if (p >= lo && p < hi) {
      if constexpr (VW == 4) {
        w[e] = __float_as_uint(x[p]);
      } else {
        const uint32_t h = static_cast<uint32_t>(x[p]);
        w[e >> 1] |= (e & 1) ? (h << 16) : h;
      }
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Element e (0..VW-1) of a raw vector, widened to fp32.
template <typename Tag>
__device__ __forceinline__ float vec_elem(const uint4& r, int e) {
  const uint32_t w = (e >> (ElemTraits<Tag>::kVW == 8 ? 1 : 0)) == 0   ? r.x
                     : (e >> (ElemTraits<Tag>::kVW == 8 ? 1 : 0)) == 1 ? r.y
                     : (e >> (ElemTraits<Tag>::kVW == 8 ? 1 : 0)) == 2 ? r.z
                                                                         : r.w;
  if constexpr (ElemTraits<Tag>::kVW == 4) {
    return __uint_as_float(w);
  } else {
    return (e & 1) ? bf16_hi(w) : bf16_lo(w);
  }
}

// Nonzero test of a worker's values (for the range check): the OR of their raw bits,
// whose sign bits are cleared at the end (so -0 counts as zero).
template <typename Tag> struct MagBits;
template <> struct MagBits<F32Tag> { static constexpr uint32_t kMask = 0x7FFFFFFFu; };
template <> struct MagBits<BF16Tag> { static constexpr uint32_t kMask = 0x7FFF7FFFu; };
__device__ __forceinline__ uint32_t vec_or(const uint4& r) { return r.x | r.y | r.z | r.w; }

// Appends worker k's nonzero bit to a running mask: m = (m << 1) | (bits != 0), for
// sign-cleared bits (bits + 0x7FFFFFFF has its top bit set exactly when bits >= 1).
__device__ __forceinline__ uint32_t nz_push(uint32_t m, uint32_t bits) {
  return __funnelshift_l(bits + 0x7FFFFFFFu, m, 1);
}

__device__ __forceinline__ uint32_t warp_or_u32(uint32_t v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v |= __shfl_xor_sync(0xFFFFFFFFu, v, off);
  return v;
}

// OR of every thread's mask over the CTA, written to *dst by thread 0.  Called by the
// whole CTA.
__device__ __forceinline__ void block_or_store(uint32_t m, uint32_t* __restrict__ dst) {
  __shared__ uint32_t red[kThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  m = warp_or_u32(m);
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t v = 0u;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) v |= red[w];
    *dst = v;
  }
}

// Kahan-compensated fp32 accumulation: sum - comp tracks the exact running sum to
// about one rounding, whatever the number of terms.
__device__ __forceinline__ void kahan_add(float& sum, float& comp, float x) {
  const float y = __fsub_rn(x, comp);
  const float t = __fadd_rn(sum, y);
  comp = __fsub_rn(__fsub_rn(t, sum), y);
  sum = t;
}

// ------------------------------------------------------- descriptor checks (test build)

// A tile inside the buffers and its segment inside the segment table.
__device__ __forceinline__ bool tile_ok(const StageArgs& a, int tile_id, const TileDesc& t) {
  return ADASUM_CHECK(a.error, tile_id >= 0 && tile_id < a.ntiles && t.start >= 0 && t.len > 0 &&
                                   t.start + t.len <= a.n_total && t.seg >= 0 && t.seg < a.nsegs);
}

// ------------------------------------------------------------- pass 1: Gram (SIMT)

// Sum E per-thread values over the CTA in a fixed order (butterfly within a warp, then
// warps in index order) and write them to dst[0..E).  fp32 throughout: each per-thread
// value already covers a bounded run of products.
template <int E>
__device__ __forceinline__ void block_reduce_store(float (&acc)[E], float* __restrict__ dst) {
  __shared__ float red[kWarps][E];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    float v = acc[e];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
    if (lane == 0) red[warp][e] = v;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kThreads) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s = __fadd_rn(s, red[w][e]);
    dst[e] = s;
  }
}

// Gram partial of one tile with CUDA-core FMAs: every thread owns whole 16-byte
// vectors (VW positions of all Kg workers) and accumulates the Kg(Kg+1)/2 products.
// This thread's products over vectors first, first + step, ... of a tile (acc zeroed),
// and in nz bit k whether worker k had a nonzero value among them.
template <typename Tag, int KG>
__device__ __forceinline__ void gram_accumulate(const StageArgs& a, const TileDesc& t, int q,
                                                int first, int step, float (&acc)[tri_count(KG)],
                                                uint32_t& nz) {
  using S = typename ElemTraits<Tag>::Storage;
  constexpr int VW = ElemTraits<Tag>::kVW;
  constexpr int E = tri_count(KG);
  const S* x[KG];
#pragma unroll
  for (int k = 0; k < KG; ++k) x[k] = static_cast<const S*>(a.in[q * KG + k]);
  const bool aligned = a.aligned != 0;
  const int64_t lo = t.start, hi = t.start + t.len;
  const int64_t v0 = lo / VW, v1 = (hi + VW - 1) / VW;
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  nz = 0u;
  for (int64_t v = v0 + first; v < v1; v += step) {
    uint4 r[KG];
#pragma unroll
    for (int k = 0; k < KG; ++k) r[k] = load_vec_raw<Tag, kLoadKeep>(x[k], v, lo, hi, aligned);
    uint32_t m = 0u;
#pragma unroll
    for (int k = KG - 1; k >= 0; --k) m = nz_push(m, vec_or(r[k]) & MagBits<Tag>::kMask);
    nz |= m;
#pragma unroll
    for (int e = 0; e < VW; ++e) {
      float xe[KG];
#pragma unroll
      for (int k = 0; k < KG; ++k) xe[k] = vec_elem<Tag>(r[k], e);
#pragma unroll
      for (int i = 0; i < KG; ++i)
#pragma unroll
        for (int j = i; j < KG; ++j)
          acc[tri_index(KG, i, j)] = __fmaf_rn(xe[i], xe[j], acc[tri_index(KG, i, j)]);
    }
  }
}

template <typename Tag, int KG>
__device__ __forceinline__ void gram_tile_simt(const StageArgs& a, int tile_id, int q) {
  constexpr int E = tri_count(KG);
  float acc[E];
  uint32_t nz;
  if (!tile_ok(a, tile_id, a.tiles[tile_id])) return;  // (uniform over the CTA)
  gram_accumulate<Tag, KG>(a, a.tiles[tile_id], q, threadIdx.x, kThreads, acc, nz);
  block_reduce_store<E>(acc, a.partials + (static_cast<size_t>(q) * a.ntiles + tile_id) * E);
  block_or_store(nz, a.tile_nz + static_cast<size_t>(q) * a.ntiles + tile_id);
}

// Tile id of this CTA: the CTA kernels run over a.tile_list when the plan splits off
// small tiles (which gram_warp_kernel takes), else over every tile.
__device__ __forceinline__ int cta_tile(const StageArgs& a) {
  return a.tile_list ? a.tile_list[blockIdx.x] : static_cast<int>(blockIdx.x);
}

// (up to 8 workers the 36 accumulators fit in 85 registers: three CTAs per SM)
template <typename Tag, int KG>
__global__ void __launch_bounds__(kThreads, KG <= 8 ? 3 : 1) gram_simt_kernel(const StageArgs a) {
  pdl_enter();
  gram_tile_simt<Tag, KG>(a, cta_tile(a), blockIdx.y);
}

// Gram partials of small tiles, one warp per (tile, group): the lanes' partials are
// summed by the warp's butterfly (a fixed order), with no block-wide reduction, so a
// tile of a few hundred positions costs a warp, not a CTA.
template <typename Tag, int KG>
__global__ void __launch_bounds__(kThreads) gram_warp_kernel(const StageArgs a) {
  pdl_enter();
  constexpr int E = tri_count(KG);
  const int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (w >= a.nsmall) return;  // whole warps only
  const int q = blockIdx.y;
  const int tile_id = a.small_list ? a.small_list[w] : w;
  float acc[E];
  uint32_t nz;
  if (!tile_ok(a, tile_id, a.tiles[tile_id])) return;  // (uniform over the warp)
  gram_accumulate<Tag, KG>(a, a.tiles[tile_id], q, lane, 32, acc, nz);
#pragma unroll
  for (int e = 0; e < E; ++e) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[e] = __fadd_rn(acc[e], __shfl_xor_sync(0xFFFFFFFFu, acc[e], off));
  }
  float* dst = a.partials + (static_cast<size_t>(q) * a.ntiles + tile_id) * E;
#pragma unroll
  for (int e = 0; e < E; ++e)
    if ((e & 31) == lane) dst[e] = acc[e];
  nz = warp_or_u32(nz);
  if (lane == 0) a.tile_nz[static_cast<size_t>(q) * a.ntiles + tile_id] = nz;
}

// --------------------------------------------------- pass 1: Gram (tensor cores, bf16)

// D += A * B for one m16n8k16 bf16 tile with fp32 accumulation.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Lane (g, t) of the MMA fragment layout holds positions of workers g and g + 8: its
// nonzero bits from the ORs of those workers' raw values (sign bits cleared here).
template <typename Tag>
__device__ __forceinline__ uint32_t mma_lane_nz(uint32_t org, uint32_t orh) {
  const int g = (threadIdx.x & 31) >> 2;
  return (((org & MagBits<Tag>::kMask) != 0u) ? 1u << g : 0u) |
         (((orh & MagBits<Tag>::kMask) != 0u) ? 1u << (g + 8) : 0u);
}

// Gram partial of one tile of bf16 gradients on the tensor cores (Kg = 8 or 16).
//
// A warp takes 32 consecutive positions at a time.  Lane (g, t) = (lane/4, lane%4)
// loads positions [8t, 8t+8) of worker g and of worker g+8: 16 bytes each.  Because the
// Gram matrix is a sum over positions, any assignment of positions to the k index of
// the MMA works as long as it is the same for every worker; the one used here puts the
// lane's own elements where the m16n8k16 fragment layout expects row g / row g+8, so
// the same registers serve as the A operand (workers x positions) and as the B operand
// (positions x workers).  Two k-steps of 16 cover the 32 positions; the two n-tiles
// give columns 0-7 and 8-15 of G.
// One warp's share of the Gram of bf16 rows on the tensor cores (8 or 16 workers): the
// 32-position chunks first, first + nw, first + 2 nw, ... of [lo, hi), lane (g, t)
// holding positions [8t, 8t+8) of workers g and g+8 of each chunk, which serve as both
// MMA operands (G = X X^T).  On return s0/e0 and s1/e1 hold the compensated sums of the
// lane's entries (columns 2t, 2t+1 and 8+2t, 9+2t of rows g and g+8), org/orh the raw-bit
// ORs of workers g and g + 8 (range check).
template <int KG>
__device__ __forceinline__ void gram_chunks_mma_bf16(const uint16_t* xg, const uint16_t* xh, int64_t lo, int64_t hi,
                                                     bool aligned, int first, int nw, float (&s0)[4],
                                                     float (&e0)[4], float (&s1)[4], float (&e1)[4],
                                                     uint32_t& org, uint32_t& orh) {
  static_assert(KG == 8 || KG == 16, "tensor-core Gram handles 8 or 16 workers");
  constexpr int U = 4;        // chunks of 32 positions loaded per warp iteration
  constexpr int kFold = 4;    // iterations accumulated in the MMA before a Kahan fold
  const int tq = threadIdx.x & 3;
  const int64_t c0 = lo >> 5, c1 = (hi + 31) >> 5;  // 32-position chunks
  float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 4; ++i) s0[i] = e0[i] = s1[i] = e1[i] = 0.f;
  org = orh = 0u;
  int pending = 0;
  for (int64_t c = c0 + first; c < c1; c += static_cast<int64_t>(nw) * U) {
    uint4 rg[U], rh[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t cu = c + static_cast<int64_t>(u) * nw;
      const int64_t v = cu * 4 + tq;
      if (cu < c1) {
        rg[u] = load_vec_raw<BF16Tag, kLoadKeep>(xg, v, lo, hi, aligned);
        rh[u] = KG == 16 ? load_vec_raw<BF16Tag, kLoadKeep>(xh, v, lo, hi, aligned)
                         : make_uint4(0u, 0u, 0u, 0u);
      } else {
        rg[u] = make_uint4(0u, 0u, 0u, 0u);
        rh[u] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      org |= vec_or(rg[u]);
      orh |= vec_or(rh[u]);
      // (the two accumulators' MMAs alternate, so each waits on its own chain only)
      mma_bf16_16816(d0, rg[u].x, rh[u].x, rg[u].y, rh[u].y, rg[u].x, rg[u].y);
      if constexpr (KG == 16) mma_bf16_16816(d1, rg[u].x, rh[u].x, rg[u].y, rh[u].y, rh[u].x, rh[u].y);
      mma_bf16_16816(d0, rg[u].z, rh[u].z, rg[u].w, rh[u].w, rg[u].z, rg[u].w);
      if constexpr (KG == 16) mma_bf16_16816(d1, rg[u].z, rh[u].z, rg[u].w, rh[u].w, rh[u].z, rh[u].w);
    }
    if (++pending == kFold) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        kahan_add(s0[i], e0[i], d0[i]);
        kahan_add(s1[i], e1[i], d1[i]);
        d0[i] = 0.f;
        d1[i] = 0.f;
      }
      pending = 0;
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    kahan_add(s0[i], e0[i], d0[i]);
    kahan_add(s1[i], e1[i], d1[i]);
  }
}

template <int KG>
__device__ __forceinline__ void gram_tile_mma(const StageArgs& a, int tile_id, int q) {
  static_assert(KG == 8 || KG == 16, "tensor-core Gram handles 8 or 16 workers");
  constexpr int E = tri_count(KG);
  const TileDesc t = a.tiles[tile_id];
  if (!tile_ok(a, tile_id, t)) return;  // (uniform over the CTA)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, tq = lane & 3;
  const uint16_t* xg = static_cast<const uint16_t*>(a.in[q * KG + g]);
  const uint16_t* xh = KG == 16 ? static_cast<const uint16_t*>(a.in[q * KG + g + 8]) : nullptr;
  float s0[4], e0[4], s1[4], e1[4];
  uint32_t org, orh;
  gram_chunks_mma_bf16<KG>(xg, xh, t.start, t.start + t.len, a.aligned != 0, warp, kWarps, s0, e0, s1, e1, org, orh);

  // Each warp now holds its full KG x KG partial, one distinct entry per register:
  // s0[0..1] = G[g][2t..2t+1], s0[2..3] = G[g+8][2t..2t+1], s1 likewise for columns
  // 8 + 2t.  Sum the warps in index order.
  __shared__ float red[kWarps][KG * KG];
  {
    const int r0 = g, r1 = g + 8, cA = 2 * tq;
    red[warp][r0 * KG + cA] = __fsub_rn(s0[0], e0[0]);
    red[warp][r0 * KG + cA + 1] = __fsub_rn(s0[1], e0[1]);
    if constexpr (KG == 16) {
      red[warp][r1 * KG + cA] = __fsub_rn(s0[2], e0[2]);
      red[warp][r1 * KG + cA + 1] = __fsub_rn(s0[3], e0[3]);
      red[warp][r0 * KG + 8 + cA] = __fsub_rn(s1[0], e1[0]);
      red[warp][r0 * KG + 8 + cA + 1] = __fsub_rn(s1[1], e1[1]);
      red[warp][r1 * KG + 8 + cA] = __fsub_rn(s1[2], e1[2]);
      red[warp][r1 * KG + 8 + cA + 1] = __fsub_rn(s1[3], e1[3]);
    }
  }
  __syncthreads();
  float* dst = a.partials + (static_cast<size_t>(q) * a.ntiles + tile_id) * E;
  for (int idx = threadIdx.x; idx < KG * KG; idx += kThreads) {
    const int i = idx / KG, j = idx % KG;
    if (j < i) continue;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s = __fadd_rn(s, red[w][idx]);
    dst[tri_index(KG, i, j)] = s;
  }
  block_or_store(mma_lane_nz<BF16Tag>(org, orh), a.tile_nz + static_cast<size_t>(q) * a.ntiles + tile_id);
}

// 2x of both halves of a packed bf16 pair (exact: x + x).
__device__ __forceinline__ uint32_t bf16x2_twice(uint32_t v) {
  uint32_t r;
  asm("add.rn.bf16x2 %0, %1, %1;" : "=r"(r) : "r"(v));
  return r;
}

// Three bf16 parts of two fp32 values, x = h + m + l exactly: h is x rounded to bf16,
// m the remainder rounded, l what is left (each remainder is exact in fp32, and at most
// 8 significant bits are left for l).  Packed in pairs, as the MMA fragments take them.
__device__ __forceinline__ void split_bf16x3(float x0, float x1, uint32_t& h, uint32_t& m, uint32_t& l) {
  h = pack_bf16x2(x0, x1);
  const float r0 = x0 - bf16_lo(h), r1 = x1 - bf16_hi(h);
  m = pack_bf16x2(r0, r1);
  l = pack_bf16x2(r0 - bf16_lo(m), r1 - bf16_hi(m));
}

// One 32-position chunk of the fp32 tensor-core Gram: lane (g, t) holds positions
// [8t, 8t+8) of workers g (rg) and g + 8 (rh) as two 16-byte vectors each.  Every value
// is split into three bf16 parts (split_bf16x3), and d0 (columns g) and d1 (columns
// g + 8) accumulate R = h.h + m.m + h.(2m) + h.(2l) (see gram_chunks_mma_f32); org and
// orh collect the raw bits (range check).
__device__ __forceinline__ void gram_mma_f32_chunk(const uint4 (&rg)[2], const uint4 (&rh)[2], float (&d0)[4],
                                                   float (&d1)[4], uint32_t& org, uint32_t& orh) {
  org |= vec_or(rg[0]) | vec_or(rg[1]);
  orh |= vec_or(rh[0]) | vec_or(rh[1]);
  // parts of positions (0,1), (2,3), (4,5), (6,7): registers 0..3 as in gram_tile_mma
  uint32_t gh[4], gm[4], gl[4], hh[4], hm[4], hl[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint4 a4 = rg[k >> 1], b4 = rh[k >> 1];
    const float ga = __uint_as_float((k & 1) ? a4.z : a4.x), gb = __uint_as_float((k & 1) ? a4.w : a4.y);
    const float ha = __uint_as_float((k & 1) ? b4.z : b4.x), hb = __uint_as_float((k & 1) ? b4.w : b4.y);
    split_bf16x3(ga, gb, gh[k], gm[k], gl[k]);
    split_bf16x3(ha, hb, hh[k], hm[k], hl[k]);
  }
  // d += A B for A = rows (g, g+8) of part pa, B = columns g (d0) and g+8 (d1) of part
  // pb; the two accumulators' MMAs alternate, so each waits on its own chain only
  auto mmas = [&](const uint32_t (&ag)[4], const uint32_t (&ah)[4], const uint32_t (&bg)[4],
                  const uint32_t (&bh)[4]) {
    mma_bf16_16816(d0, ag[0], ah[0], ag[1], ah[1], bg[0], bg[1]);
    mma_bf16_16816(d1, ag[0], ah[0], ag[1], ah[1], bh[0], bh[1]);
    mma_bf16_16816(d0, ag[2], ah[2], ag[3], ah[3], bg[2], bg[3]);
    mma_bf16_16816(d1, ag[2], ah[2], ag[3], ah[3], bh[2], bh[3]);
  };
  // R = h.h + m.m + h.(2m) + h.(2l): the mirror sum R_ij + R_ji is twice the six
  // products' sum (h.m and m.h, h.l and l.h meet there), and its diagonal R_ii is that
  // sum itself; doubling a bf16 value is exact (doubling h instead, 8 adds for 16,
  // made the kernels spill)
  mmas(gh, hh, gh, hh);
  mmas(gm, hm, gm, hm);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    gm[k] = bf16x2_twice(gm[k]);
    hm[k] = bf16x2_twice(hm[k]);
    gl[k] = bf16x2_twice(gl[k]);
    hl[k] = bf16x2_twice(hl[k]);
  }
  mmas(gh, hh, gm, hm);
  mmas(gh, hh, gl, hl);
}

// One warp's share of the Gram of fp32 rows on the tensor cores (16 workers): the
// 32-position chunks first, first + nw, first + 2 nw, ... of [lo, hi).  Every value is
// split into three bf16 parts (split_bf16x3) and x.y is taken as the six largest of the
// nine part products, h.h + h.m + m.h + m.m + h.l + l.h: the three left out are below
// 2^-23 |x||y| together, the size of one fp32 product's rounding.  Four MMA products
// per chunk carry them: the lane accumulates R = h.h + m.m + h.(2m) + h.(2l), whose
// diagonal is the six products' sum and whose mirror sum R_ij + R_ji is twice it (the
// callers take (R_ij + R_ji) / 2).  The layout, the MMA
// accumulation and the compensated folding are those of gram_tile_mma (lane (g, t) holds
// positions [8t, 8t+8) of workers g and g+8 of each chunk).  On return s0/e0 and s1/e1
// hold the compensated sums of the lane's entries (columns 2t, 2t+1 and 8+2t, 9+2t of
// rows g and g+8).
template <int KG>
__device__ __forceinline__ void gram_chunks_mma_f32(const float* xg, const float* xh, int64_t lo, int64_t hi,
                                                    bool aligned, int first, int nw, float (&s0)[4],
                                                    float (&e0)[4], float (&s1)[4], float (&e1)[4],
                                                    uint32_t& org, uint32_t& orh) {
  static_assert(KG == 16, "16 workers: two n-tiles of the m16n8k16 MMA");
  constexpr int U = 2;        // chunks of 32 positions loaded per warp iteration
  constexpr int kFold = 4;    // iterations accumulated in the MMA before a Kahan fold
  const int lane = threadIdx.x & 31;
  const int tq = lane & 3;
  const int64_t c0 = lo >> 5, c1 = (hi + 31) >> 5;  // 32-position chunks
  float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 4; ++i) s0[i] = e0[i] = s1[i] = e1[i] = 0.f;
  org = orh = 0u;  // raw-bit ORs of workers g and g + 8 (range check)
  int pending = 0;
  for (int64_t c = c0 + first; c < c1; c += static_cast<int64_t>(nw) * U) {
    uint4 rg[U][2], rh[U][2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t cu = c + static_cast<int64_t>(u) * nw;
      const int64_t v = cu * 8 + tq * 2;  // float4 index of positions [32cu + 8t, +8)
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        rg[u][h2] = cu < c1 ? load_vec_raw<F32Tag, kLoadKeep>(xg, v + h2, lo, hi, aligned) : make_uint4(0u, 0u, 0u, 0u);
        rh[u][h2] = cu < c1 ? load_vec_raw<F32Tag, kLoadKeep>(xh, v + h2, lo, hi, aligned) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) gram_mma_f32_chunk(rg[u], rh[u], d0, d1, org, orh);
    if (++pending == kFold) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        kahan_add(s0[i], e0[i], d0[i]);
        kahan_add(s1[i], e1[i], d1[i]);
        d0[i] = 0.f;
        d1[i] = 0.f;
      }
      pending = 0;
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    kahan_add(s0[i], e0[i], d0[i]);
    kahan_add(s1[i], e1[i], d1[i]);
  }
}

// The warp ring of gram_chunks_mma_f32_staged: kGramStages chunks of 16 rows, each row
// 32 positions and 4 floats of padding (a row of 144 bytes puts the 8 lanes of each
// quarter-warp's 16-byte reads, rows g and columns 8t, on distinct banks).
constexpr int kGramStages = 3;
constexpr int kGramStageRow = 36;
constexpr int kGramStageFloats = 16 * kGramStageRow;
// Threads per CTA of the one-warp-per-tile Gram kernels: two warps, so a CTA that holds
// a finished warp retires as soon as its one sibling is done (eight-warp CTAs waited on
// the slowest of eight tiles: the fp32 K = 64 set 0.762 -> 0.753 ms, bf16 K = 64 on its
// layout 0.697 -> 0.682 ms).
constexpr int kGramWarpThreads = 64;
constexpr size_t kGramWarpRingBytes = sizeof(float) * (kGramWarpThreads / 32) * kGramStages * kGramStageFloats;
// CTAs per SM of the staged kernel (its launch bound: 80 registers; at 4 CTAs, 64
// registers spilled and the K = 64 set took 0.891 ms against 0.777)
constexpr int kGramStagedCtas = 3;

// gram_chunks_mma_f32 for one warp alone on [lo, hi) of 16-byte aligned rows, with the
// loads decoupled from the tensor-core work: each chunk's 16 rows x 32 positions are
// copied into the warp's ring (cp.async, 16 bytes a copy, each row's 128 bytes by 8
// lanes) kGramStages - 1 chunks ahead of the chunk being multiplied, so a warp always has
// two chunks in flight without holding them in registers.  The chunks are multiplied in
// order with the same fold every 8 chunks as gram_chunks_mma_f32 with one warp, so the
// two give the same bits.  Rows are read up to the end of the buffers (n_total) and
// never past it (the copy's zero fill); positions outside [lo, hi) are zeroed after the
// read.  Rows of padding workers (null) stay zero in the ring.
__device__ __forceinline__ void gram_chunks_mma_f32_staged(const void* const* rows, int64_t lo, int64_t hi,
                                                           int64_t n_total, float* ring, float (&s0)[4],
                                                           float (&e0)[4], float (&s1)[4], float (&e1)[4],
                                                           uint32_t& org, uint32_t& orh) {
  constexpr int kFoldChunks = 8;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int64_t c0 = lo >> 5, c1 = (hi + 31) >> 5;
  // this lane copies 16-byte vector cv of rows r0, r0 + 4, r0 + 8, r0 + 12 of each chunk
  const int r0 = lane >> 3, cv = lane & 7;
  const float* src[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    src[j] = static_cast<const float*>(rows[r0 + 4 * j]);
    if (src[j] == nullptr) {
#pragma unroll
      for (int st = 0; st < kGramStages; ++st)
        *reinterpret_cast<uint4*>(ring + st * kGramStageFloats + (r0 + 4 * j) * kGramStageRow + cv * 4) =
            make_uint4(0u, 0u, 0u, 0u);
    }
  }
  const uint32_t ring_s = smem_addr(ring);
  auto issue = [&](int64_t c, int slot) {
    if (c < c1) {
      const int64_t p = c * 32 + cv * 4;
      const int64_t left = n_total - p;
      const int bytes = left >= 4 ? 16 : (left > 0 ? static_cast<int>(left) * 4 : 0);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (src[j] == nullptr) continue;
        const uint32_t dst = ring_s + 4u * static_cast<uint32_t>(slot * kGramStageFloats +
                                                                 (r0 + 4 * j) * kGramStageRow + cv * 4);
        cp_async16(dst, bytes > 0 ? src[j] + p : src[j], bytes);
      }
    }
    cp_async_commit();  // (an empty group past the end keeps the wait count uniform)
  };
  float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 4; ++i) s0[i] = e0[i] = s1[i] = e1[i] = 0.f;
  org = orh = 0u;
#pragma unroll
  for (int st = 0; st < kGramStages - 1; ++st) issue(c0 + st, st);
  int pending = 0;
  for (int64_t c = c0; c < c1; ++c) {
    const int i = static_cast<int>(c - c0);
    __syncwarp();  // every lane has read the slot that is refilled next
    issue(c + kGramStages - 1, (i + kGramStages - 1) % kGramStages);
    cp_async_wait<kGramStages - 1>();
    __syncwarp();  // the other lanes' copies of chunk c are visible
    const float* sl = ring + (i % kGramStages) * kGramStageFloats;
    uint4 rg[2], rh[2];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      rg[h2] = *reinterpret_cast<const uint4*>(sl + g * kGramStageRow + 8 * tq + 4 * h2);
      rh[h2] = *reinterpret_cast<const uint4*>(sl + (g + 8) * kGramStageRow + 8 * tq + 4 * h2);
    }
    if (c * 32 < lo || c * 32 + 32 > hi) {  // the segment's first or last chunk
      const int64_t p0 = c * 32 + 8 * tq;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (p0 + e >= lo && p0 + e < hi) continue;
        uint32_t* vg = reinterpret_cast<uint32_t*>(&rg[e >> 2]);
        uint32_t* vh = reinterpret_cast<uint32_t*>(&rh[e >> 2]);
        vg[e & 3] = 0u;
        vh[e & 3] = 0u;
      }
    }
    gram_mma_f32_chunk(rg, rh, d0, d1, org, orh);
    if (++pending == kFoldChunks) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        kahan_add(s0[k], e0[k], d0[k]);
        kahan_add(s1[k], e1[k], d1[k]);
        d0[k] = 0.f;
        d1[k] = 0.f;
      }
      pending = 0;
    }
  }
  cp_async_wait<0>();  // (only empty groups are left)
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    kahan_add(s0[k], e0[k], d0[k]);
    kahan_add(s1[k], e1[k], d1[k]);
  }
}

// A lane's compensated sums into the KG x KG matrix m (row-major), as laid out by the MMA.
__device__ __forceinline__ void store_lane_gram16(float* m, const float (&s0)[4], const float (&e0)[4],
                                                  const float (&s1)[4], const float (&e1)[4]) {
  constexpr int KG = 16;
  const int lane = threadIdx.x & 31;
  const int r0 = lane >> 2, r1 = r0 + 8, cA = 2 * (lane & 3);
  m[r0 * KG + cA] = __fsub_rn(s0[0], e0[0]);
  m[r0 * KG + cA + 1] = __fsub_rn(s0[1], e0[1]);
  m[r1 * KG + cA] = __fsub_rn(s0[2], e0[2]);
  m[r1 * KG + cA + 1] = __fsub_rn(s0[3], e0[3]);
  m[r0 * KG + 8 + cA] = __fsub_rn(s1[0], e1[0]);
  m[r0 * KG + 8 + cA + 1] = __fsub_rn(s1[1], e1[1]);
  m[r1 * KG + 8 + cA] = __fsub_rn(s1[2], e1[2]);
  m[r1 * KG + 8 + cA + 1] = __fsub_rn(s1[3], e1[3]);
}

// Gram partial of one tile of fp32 gradients (16 workers) on the tensor cores, all warps
// of the CTA sharing its chunks (gram_chunks_mma_f32).  The lanes hold R (see there), so
// each off-diagonal entry is the mean of R_ij and R_ji: the six products' sum, and
// symmetric by construction, so permuting the workers permutes the Gram matrix bit for
// bit, as the sibling-swap symmetry needs.
template <int KG>
__device__ __forceinline__ void gram_tile_mma_f32(const StageArgs& a, int tile_id, int q) {
  static_assert(KG == 16, "16 workers");
  constexpr int E = tri_count(KG);
  const TileDesc t = a.tiles[tile_id];
  if (!tile_ok(a, tile_id, t)) return;  // (uniform over the CTA)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2;
  float s0[4], e0[4], s1[4], e1[4];
  uint32_t mg, mh;
  gram_chunks_mma_f32<KG>(static_cast<const float*>(a.in[q * KG + g]), static_cast<const float*>(a.in[q * KG + g + 8]),
                          t.start, t.start + t.len, a.aligned != 0, warp, kWarps, s0, e0, s1, e1, mg, mh);
  __shared__ float red[kWarps][KG * KG];
  store_lane_gram16(red[warp], s0, e0, s1, e1);
  __syncthreads();
  float* dst = a.partials + (static_cast<size_t>(q) * a.ntiles + tile_id) * E;
  for (int idx = threadIdx.x; idx < KG * KG; idx += kThreads) {
    const int i = idx / KG, j = idx % KG;
    if (j < i) continue;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
      s = __fadd_rn(s, i == j ? red[w][idx] : 0.5f * __fadd_rn(red[w][idx], red[w][j * KG + i]));
    dst[tri_index(KG, i, j)] = s;
  }
  block_or_store(mma_lane_nz<F32Tag>(mg, mh), a.tile_nz + static_cast<size_t>(q) * a.ntiles + tile_id);
}

// A warp's Gram partial of one tile from the lanes' compensated sums (m: the warp's
// 256 floats of shared memory): each off-diagonal entry is the mean of its two mirror
// sums, as in gram_tile_mma_f32.
__device__ __forceinline__ void warp_gram16_store(const StageArgs& a, int q, int tile_id, float* m,
                                                  const float (&s0)[4], const float (&e0)[4],
                                                  const float (&s1)[4], const float (&e1)[4], uint32_t mg,
                                                  uint32_t mh) {
  constexpr int KG = 16, E = tri_count(KG);
  const int lane = threadIdx.x & 31;
  store_lane_gram16(m, s0, e0, s1, e1);
  __syncwarp();
  float* dst = a.partials + (static_cast<size_t>(q) * a.ntiles + tile_id) * E;
  for (int e = lane; e < E; e += 32) {
    int i, j;
    tri_unpack(KG, e, i, j);
    dst[e] = i == j ? m[i * KG + i] : 0.5f * __fadd_rn(m[i * KG + j], m[j * KG + i]);
  }
  const uint32_t nz = warp_or_u32(mma_lane_nz<F32Tag>(mg, mh));
  if (lane == 0) a.tile_nz[static_cast<size_t>(q) * a.ntiles + tile_id] = nz;
}

// Gram partials of small tiles of fp32 gradients (16 workers), one warp per (tile,
// group), on the tensor cores (gram_chunks_mma_f32 with the warp alone on the tile):
// rows that are not all 16-byte aligned.
template <int KG>
__global__ void __launch_bounds__(kThreads, 3) gram_warp_mma_f32_kernel(const StageArgs a) {
  pdl_enter();
  static_assert(KG == 16, "16 workers");
  __shared__ float red[kWarps][KG * KG];
  const int wb = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w = blockIdx.x * (blockDim.x >> 5) + wb;
  if (w >= a.nsmall) return;  // whole warps only (no block barrier below)
  const int q = blockIdx.y;
  const int tile_id = a.small_list ? a.small_list[w] : w;
  const TileDesc t = a.tiles[tile_id];
  if (!tile_ok(a, tile_id, t)) return;  // (uniform over the warp)
  const int g = lane >> 2;
  float s0[4], e0[4], s1[4], e1[4];
  uint32_t mg, mh;
  gram_chunks_mma_f32<KG>(static_cast<const float*>(a.in[q * KG + g]), static_cast<const float*>(a.in[q * KG + g + 8]),
                          t.start, t.start + t.len, a.aligned != 0, 0, 1, s0, e0, s1, e1, mg, mh);
  warp_gram16_store(a, q, tile_id, red[wb], s0, e0, s1, e1, mg, mh);
}

// The same for 16-byte aligned rows, staged through each warp's ring in dynamic shared
// memory (gram_chunks_mma_f32_staged; launched with kGramWarpRingBytes).  The ring's
// first slot takes the warp's 16 x 16 sums once the copies have drained.
template <int KG>
__global__ void __launch_bounds__(kThreads, kGramStagedCtas) gram_warp_staged_f32_kernel(const StageArgs a) {
  pdl_enter();
  static_assert(KG == 16, "16 workers");
  extern __shared__ __align__(16) float gram_ring[];
  const int wb = threadIdx.x >> 5;
  const int w = blockIdx.x * (blockDim.x >> 5) + wb;
  if (w >= a.nsmall) return;  // whole warps only (no block barrier below)
  const int q = blockIdx.y;
  const int tile_id = a.small_list ? a.small_list[w] : w;
  const TileDesc t = a.tiles[tile_id];
  if (!tile_ok(a, tile_id, t)) return;  // (uniform over the warp)
  float s0[4], e0[4], s1[4], e1[4];
  uint32_t mg, mh;
  float* ring = gram_ring + wb * kGramStages * kGramStageFloats;
  gram_chunks_mma_f32_staged(a.in + q * KG, t.start, t.start + t.len, a.n_total, ring, s0, e0, s1, e1, mg, mh);
  __syncwarp();  // every lane is done reading the ring
  warp_gram16_store(a, q, tile_id, ring, s0, e0, s1, e1, mg, mh);
}

// Gram partials of small tiles of bf16 gradients (16 workers), one warp per (tile,
// group), on the tensor cores (gram_chunks_mma_bf16 with the warp alone on the tile).
// The bf16 Gram needs no mirror mean: h.h products are symmetric as they stand.
template <int KG>
__global__ void __launch_bounds__(kThreads, 3) gram_warp_mma_bf16_kernel(const StageArgs a) {
  pdl_enter();
  static_assert(KG == 16, "16 workers");
  constexpr int E = tri_count(KG);
  __shared__ float red[kWarps][KG * KG];
  const int wb = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w = blockIdx.x * (blockDim.x >> 5) + wb;
  if (w >= a.nsmall) return;  // whole warps only (no block barrier below)
  const int q = blockIdx.y;
  const int tile_id = a.small_list ? a.small_list[w] : w;
  const TileDesc t = a.tiles[tile_id];
  if (!tile_ok(a, tile_id, t)) return;  // (uniform over the warp)
  const int g = lane >> 2;
  float s0[4], e0[4], s1[4], e1[4];
  uint32_t mg, mh;
  gram_chunks_mma_bf16<KG>(static_cast<const uint16_t*>(a.in[q * KG + g]),
                           static_cast<const uint16_t*>(a.in[q * KG + g + 8]), t.start, t.start + t.len,
                           a.aligned != 0, 0, 1, s0, e0, s1, e1, mg, mh);
  float* m = red[wb];
  store_lane_gram16(m, s0, e0, s1, e1);
  __syncwarp();
  float* dst = a.partials + (static_cast<size_t>(q) * a.ntiles + tile_id) * E;
  for (int e = lane; e < E; e += 32) {
    int i, j;
    tri_unpack(KG, e, i, j);
    dst[e] = m[i * KG + j];
  }
  const uint32_t nz = warp_or_u32(mma_lane_nz<BF16Tag>(mg, mh));
  if (lane == 0) a.tile_nz[static_cast<size_t>(q) * a.ntiles + tile_id] = nz;
}

// Three CTAs per SM (at most 85 registers, a few spilled): its loads' latency is what
// limits it, and 2 -> 3 resident CTAs took the K = 64 set's first-stage Gram from 0.267
// to 0.231 ms per call.
template <int KG>
__global__ void __launch_bounds__(kThreads, 3) gram_mma_f32_kernel(const StageArgs a) {
  pdl_enter();
  gram_tile_mma_f32<KG>(a, cta_tile(a), blockIdx.y);
}

template <int KG>
__global__ void __launch_bounds__(kThreads) gram_mma_bf16_kernel(const StageArgs a) {
  pdl_enter();
  gram_tile_mma<KG>(a, cta_tile(a), blockIdx.y);
}

// Gram partial of one tile with the best engine for the element type and group size.
template <typename Tag, int KG>
__device__ __forceinline__ void gram_tile(const StageArgs& a, int tile_id, int q) {
  if constexpr (ElemTraits<Tag>::kVW == 8 && (KG == 8 || KG == 16)) {
    gram_tile_mma<KG>(a, tile_id, q);
  } else {
    gram_tile_simt<Tag, KG>(a, tile_id, q);
  }
}

// ----------------------------------------------------------- coefficients (per segment)

// Sum the fp32 tile partials of one chunk of at most kChunkTiles tiles (compensated,
// in tile order) into one fp64 value per Gram entry.
// (Partials written by other CTAs are read through L2, never a possibly stale L1.)
// Chunks per CTA of the chunk-sum kernel when chunks are many: most chunks of a layout
// with many short segments hold one tile, and a CTA per chunk would leave most of its
// threads idle.  With few chunks, one per CTA spreads them over the SMs.
constexpr int kChunksPerCta = 8;

// The compensated sum, in slot order, of SLOTS slots p[0], p[E], ... of which the
// first n hold tile partials and the rest read as zero.
template <int SLOTS, int E>
__device__ __forceinline__ void chunk_slots(const float* p, int n, float& sum, float& comp) {
  float v[SLOTS];
#pragma unroll
  for (int t = 0; t < SLOTS; ++t) v[t] = t < n ? __ldcg(p + static_cast<size_t>(t) * E) : 0.f;  // issued together
#pragma unroll
  for (int t = 0; t < SLOTS; ++t) kahan_add(sum, comp, v[t]);
}

// Entry e of a chunk (group q): the compensated sum of its tiles' partials, in tile
// order, as the double-float pair sum - comp (an exact TwoSum of the two).
template <int KG>
__device__ __forceinline__ float2 chunk_entry(const StageArgs& a, const ChunkDesc& ch, int e, int q) {
  constexpr int E = tri_count(KG);
  const float* p = a.partials + (static_cast<size_t>(q) * a.ntiles + ch.first_tile) * E + e;
  // every load issued together, empty slots read as zero; a chunk of at most 16 tiles
  // (a short segment's) takes 16 slots, not 32, since each slot costs four dependent adds
  float sum = 0.f, comp = 0.f;
  if (ch.ntiles <= kChunkTiles / 2)
    chunk_slots<kChunkTiles / 2, E>(p, ch.ntiles, sum, comp);
  else
    chunk_slots<kChunkTiles, E>(p, ch.ntiles, sum, comp);
  const float s = __fsub_rn(sum, comp), bb = __fsub_rn(s, sum);
  const float err = __fadd_rn(__fsub_rn(sum, __fsub_rn(s, bb)), __fsub_rn(-comp, bb));
  return make_float2(s, err);
}

// The OR of a chunk's per-tile nonzero words (range check), group q.
__device__ __forceinline__ uint32_t chunk_nonzero(const StageArgs& a, const ChunkDesc& ch, int q) {
  const uint32_t* p = a.tile_nz + static_cast<size_t>(q) * a.ntiles + ch.first_tile;
  uint32_t m = 0u;
  for (int t = 0; t < ch.ntiles; ++t) m |= __ldcg(p + t);
  return m;
}

__device__ __forceinline__ bool chunk_ok(const StageArgs& a, int c, ChunkDesc& ch) {
  ch = a.chunks[c];
  return ADASUM_CHECK(a.error, c < a.nchunks && ch.first_tile >= 0 && ch.ntiles >= 1 &&
                                   ch.ntiles <= kChunkTiles && ch.first_tile + ch.ntiles <= a.ntiles);
}

// The chunks of multi-chunk segments (a.multi_chunks): CTA b takes entries b * per ...
// (per = the entries over the grid: 1 or kChunksPerCta), every (chunk, entry) pair to one
// thread, and the OR of each chunk's per-tile nonzero words (range check).
template <int KG>
__global__ void __launch_bounds__(kThreads) reduce_chunks_kernel(const StageArgs a) {
  pdl_enter();
  constexpr int E = tri_count(KG);
  const int q = blockIdx.y;
  const int n = a.nmulti;
  const int per = min(kChunksPerCta, (n + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x));
  const int i0 = blockIdx.x * per;
  for (int idx = threadIdx.x; idx < per * E; idx += kThreads) {
    const int i = i0 + idx / E, e = idx % E;
    if (i >= n) continue;
    const int c = a.multi_chunks[i];
    ChunkDesc ch;
    if (!chunk_ok(a, c, ch)) continue;
    a.chunk_sums[(static_cast<size_t>(q) * a.nchunks + c) * E + e] = chunk_entry<KG>(a, ch, e, q);
  }
  if (static_cast<int>(threadIdx.x) < per) {
    const int i = i0 + threadIdx.x;
    ChunkDesc ch;
    if (i < n && chunk_ok(a, a.multi_chunks[i], ch))
      a.chunk_nz[static_cast<size_t>(q) * a.nchunks + a.multi_chunks[i]] = chunk_nonzero(a, ch, q);
  }
}


// Sum over the aligned block of W lanes that contains this lane (butterfly with
// offsets W/2 .. 1); every lane of the block gets the same value.
__device__ __forceinline__ double block_lane_sum(double x, int W) {
  for (int off = W >> 1; off > 0; off >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
  return x;
}

// Sum over the aligned block of W lanes (fp32 version, for the error estimate).
__device__ __forceinline__ float block_lane_sumf(float x, int W) {
  for (int off = W >> 1; off > 0; off >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
  return x;
}

// The Adasum tree of one segment in coefficient space, in fp64, evaluated by one warp:
// lane k < KG owns leaf k (its coefficient c_k).  Every tree node u is
// sum_{k in u} c_k g_k over W = 2^level consecutive leaves; pairing u = [a0, a0+W) with
// v = [a0+W, a0+2W):
//     d = c_u^T G c_v,  pu = c_u^T G c_u,  pv = c_v^T G c_v
//     alpha = 1 - d / (2 pu)   (alpha = 1 when pu == 0: a zero node contributes a plain sum)
//     beta  = 1 - d / (2 pv)
//     c_u *= alpha,  c_v *= beta.
// d is taken as the sum of the two halves' partial sums (one from each side), so
// exchanging u and v gives bitwise the same d.
//
// Alongside, a first-order estimate of the error of the fp32 pass.  Gram entries carry
// errors of about gram_err |g_i||g_j| (independent, so quadratic forms add them in
// quadrature), inputs carry relative errors eps (earlier stages), and the combine
// rounds at each of the log2(K)+1 levels of its pairwise sum.  The estimate follows
// every node's norm and cross term through the tree: when a node's norm is no larger
// than its own error (cancellation), or the estimated relative error of the output
// exceeds the budget, the segment is flagged for the fp64 recompute.  The estimate
// needs a few significant digits only, so it runs in fp32 (GB300's fp64 pipe is narrow)
// on quantities divided by the largest squared leaf norm, which keeps them far from
// fp32's range limits.
//
// Called by all 32 lanes of one warp.  G and eps are in shared memory, c_sh is shared
// scratch of KG doubles.  Returns (in every lane) the estimated relative output error
// (1e30 when ill-conditioned); lane k < KG receives its coefficient in `c`.
template <int KG>
__device__ double coefficient_tree(const double (&G)[KG][KG], const double* eps,
                                   double gram_err, double* c_sh, double& c, bool& ill,
                                   double* P_out = nullptr) {
  static_assert(KG <= 32, "one lane per leaf");
  const int lane = threadIdx.x & 31;
  const bool on = lane < KG;
  const int row = on ? lane : 0;
  double gmax = on ? fmax(G[row][row], 0.0) : 0.0;
  for (int off = 16; off > 0; off >>= 1) gmax = fmax(gmax, __shfl_xor_sync(0xFFFFFFFFu, gmax, off));
  const double inv = gmax > 0.0 ? 1.0 / gmax : 0.0;  // scale of the estimate
  const float ge = static_cast<float>(gram_err);
  const float s2 = on ? static_cast<float>(fmax(G[row][row], 0.0) * inv) : 0.f;  // |g_k|^2, scaled
  const float e = on ? static_cast<float>(eps[row]) : 0.f;
  c = on ? 1.0 : 0.0;
  float dc = 0.f;  // estimated error of c
  bool bad = false;
  if (on) c_sh[lane] = c;
  __syncwarp();
  for (int W = 1; W < KG; W *= 2) {
    const int self0 = (lane / W) * W, sib0 = self0 ^ W;
    double row_self = 0.0, row_sib = 0.0;
    if (on) {
      for (int j = 0; j < W; ++j) {
        row_self = fma(c_sh[self0 + j], G[row][self0 + j], row_self);
        row_sib = fma(c_sh[sib0 + j], G[row][sib0 + j], row_sib);
      }
    }
    const double p_self = block_lane_sum(c * row_self, W);
    const double d_half = block_lane_sum(c * row_sib, W);
    const double d = d_half + __shfl_xor_sync(0xFFFFFFFFu, d_half, W);
    const double dd = 0.5 * d;  // the two halves each hold the full cross term
    const double p_sib = __shfl_xor_sync(0xFFFFFFFFu, p_self, W);
    const float cf = static_cast<float>(c);
    const float S_self = block_lane_sumf(cf * cf * s2, W);
    const float D_self = sqrtf(block_lane_sumf((dc * dc + cf * cf * e * e) * s2, W));
    const float S_sib = __shfl_xor_sync(0xFFFFFFFFu, S_self, W);
    const float D_sib = __shfl_xor_sync(0xFFFFFFFFu, D_self, W);
    const float ps = static_cast<float>(p_self * inv), pb = static_cast<float>(p_sib * inv);
    const float n_self = sqrtf(fmaxf(ps, 0.f)), n_sib = sqrtf(fmaxf(pb, 0.f));
    const float err_p = ge * S_self + 2.f * n_self * D_self;
    const float err_d = ge * sqrtf(S_self * S_sib) + (n_self * D_sib + n_sib * D_self);
    double coef = 1.0;
    float dcoef = 0.f;
    if (p_self != 0.0) {
      coef = 1.0 - dd / (2.0 * p_self);
      const float ap = fabsf(ps), add = fabsf(static_cast<float>(dd * inv));
      dcoef = (err_d + add * err_p / ap) / (2.f * ap);
      if (ps <= err_p) bad = true;
    } else if (S_self > 0.f) {
      bad = true;  // a non-zero subtree cancelled to an exact zero norm
    }
    if (on) {
      dc = fmaf(fabsf(static_cast<float>(coef)), dc, fabsf(cf) * dcoef);
      c *= coef;
    }
    __syncwarp();
    if (on) c_sh[lane] = c;
    __syncwarp();
  }
  double full = 0.0;
  if (on)
    for (int j = 0; j < KG; ++j) full = fma(c_sh[j], G[row][j], full);
  const double P = block_lane_sum(c * full, 32);
  const float cf = static_cast<float>(c);
  const float S = block_lane_sumf(cf * cf * s2, 32);
  const float D = sqrtf(block_lane_sumf((dc * dc + cf * cf * e * e) * s2, 32));
  ill = __any_sync(0xFFFFFFFFu, bad);
  if (P_out) *P_out = P;
  if (S == 0.f) return 0.0;  // every leaf is zero: the output is exactly zero
  int levels = 1;
  for (int k = KG; k > 1; k >>= 1) ++levels;
  const float Pf = static_cast<float>(P * inv);
  const float err_P = ge * S + 2.f * sqrtf(fmaxf(Pf, 0.f)) * D;
  if (Pf <= err_P) {
    ill = true;
    return 1e30;
  }
  const float rel = (D + levels * 5.9604644775390625e-08f * sqrtf(S)) / sqrtf(Pf);
  return ill ? 1e30 : static_cast<double>(rel);
}

// ----------------------------------------------- double-float arithmetic (tree core)
//
// A value hi + lo held in two fp32 numbers, |lo| <= ulp(hi)/2: about 48 significant
// bits from fp32 instructions, which GB300 issues 64 times faster than fp64.  Built from
// the error-free transformations TwoSum (Knuth) and TwoProduct (one FMA), composed as in
// Dekker, "A floating-point technique for extending the available precision" (1971);
// the add is the short ("sloppy") variant, whose error is a few 2^-48 of the operands.
// Every operation is commutative bit for bit, which keeps the tree's sibling symmetry.
struct df32 {
  float hi, lo;
};

__device__ __forceinline__ df32 df_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, err};
}
// requires |a| >= |b| (or a == 0)
__device__ __forceinline__ df32 df_fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ df32 df_add(df32 x, df32 y) {
  const df32 s = df_two_sum(x.hi, y.hi);
  return df_fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo)));
}
__device__ __forceinline__ df32 df_neg(df32 x) { return {-x.hi, -x.lo}; }
__device__ __forceinline__ df32 df_mul(df32 x, df32 y) {
  const float p = __fmul_rn(x.hi, y.hi);
  const float e = __fmaf_rn(x.hi, y.hi, -p);  // exact error of the product
  const float cross = __fadd_rn(__fmul_rn(x.hi, y.lo), __fmul_rn(x.lo, y.hi));
  return df_fast_two_sum(p, __fadd_rn(e, cross));
}
// y * q for a single float q (TwoProduct plus the low part)
__device__ __forceinline__ df32 df_mul_f(df32 y, float q) {
  const float p = __fmul_rn(y.hi, q);
  const float e = __fmaf_rn(y.hi, q, -p);
  return df_fast_two_sum(p, __fmaf_rn(y.lo, q, e));
}
// x / y by long division with fp32 quotient digits (three digits: ~48 bits).  A digit
// only has to be close: the exact remainder carries its error into the next digit, so
// the digits use the fast approximate division (|y| well inside fp32's normal range,
// which the callers' power-of-two scaling provides).
__device__ __forceinline__ df32 df_div(df32 x, df32 y) {
  const float q1 = __fdividef(x.hi, y.hi);
  df32 r = df_add(x, df_neg(df_mul_f(y, q1)));
  const float q2 = __fdividef(r.hi, y.hi);
  r = df_add(r, df_neg(df_mul_f(y, q2)));
  const float q3 = __fdividef(r.hi, y.hi);
  return df_add(df_fast_two_sum(q1, q2), df32{q3, 0.f});
}
__device__ __forceinline__ df32 df_from_double(double v) {
  const float hi = static_cast<float>(v);
  return {hi, static_cast<float>(v - static_cast<double>(hi))};
}
__device__ __forceinline__ double df_to_double(df32 x) {
  return static_cast<double>(x.hi) + static_cast<double>(x.lo);
}
__device__ __forceinline__ df32 df_shfl_xor(df32 x, int off) {
  return {__shfl_xor_sync(0xFFFFFFFFu, x.hi, off), __shfl_xor_sync(0xFFFFFFFFu, x.lo, off)};
}
// Sum over the aligned block of W lanes (butterfly, the same value in every lane).
__device__ __forceinline__ df32 df_block_sum(df32 x, int W) {
  for (int off = W >> 1; off > 0; off >>= 1) x = df_add(x, df_shfl_xor(x, off));
  return x;
}

// Integer mixing for the probe's signs (xorshift-multiply rounds; any well-mixing
// function would do).
__device__ __forceinline__ uint32_t probe_mix(uint32_t x) {
  x ^= x >> 16;
  x *= 0x85EBCA6Bu;
  x ^= x >> 13;
  x *= 0xC2B2AE35u;
  x ^= x >> 16;
  return x;
}

// Shared scratch of coefficient_tree_df<KG> (and of its probe), in floats: two node-Gram
// buffers for each of three fp32 (or two double-float) matrices, three per-node arrays,
// and the leaves' input errors in fp32.
__host__ __device__ constexpr int tree_scratch_floats(int KG) {
  return 3 * ((KG / 2) * (KG / 2) + (KG / 4) * (KG / 4)) + 4 * KG;
}

// Sum over the 32 lanes in the order of the tree itself: siblings (lanes 2i, 2i+1)
// first, then pairs of those, ... -- so swapping the children of any tree node swaps
// the operands of one addition and leaves the sum bitwise unchanged.  Every lane gets it.
__device__ __forceinline__ float tree_lane_sumf(float x) {
  for (int off = 1; off < 32; off <<= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
  return x;
}

// Next level's node Gram entry (p, q), p <= q, from this level's entries of the four
// children a = 2p, b = 2p+1, a' = 2q, b' = 2q+1 with coefficients al, be, al2, be2:
//   H'(p,q) = (al al2 H(a,a') + be be2 H(b,b')) + (al be2 H(a,b') + be al2 H(b,a')).
// The grouping pairs each term with its image under a swap of either node's children,
// and every product is formed coefficient-times-coefficient first, so mirrored trees
// (and the transposed entry) give bitwise the same value.
template <typename T, typename Mul, typename Add>
__device__ __forceinline__ T node_gram_entry(T al, T be, T al2, T be2, T haa, T hbb, T hab, T hba, Mul mul,
                                             Add add) {
  return add(add(mul(mul(al, al2), haa), mul(mul(be, be2), hbb)),
             add(mul(mul(al, be2), hab), mul(mul(be, al2), hba)));
}

// First-order size of the fp32 pass's coefficient error, measured instead of bounded.
// The bound of coefficient_tree_df adds every error term with its worst sign at every
// level; for strongly correlated leaves (near-parallel gradients) that compounds to
// 100-1000x the error the pass really makes.  Here the tree is differentiated (forward
// mode, fp32) along two perturbations E of the Gram matrix of the size the error model
// gives each entry,
//     E_ij = (gram_err s_ij + t_i eps_i + t_j eps_j) |g_i| |g_j|,
// with signs s_ij, t_i = +-1 hashed from the entries' own values (so that permuting
// the leaves permutes E with them), and the output's change |sum_k dc_k g_k| =
// sqrt(dc^T G dc) is returned relative to |out| (the larger of the two).  The tree runs
// on node Gram matrices as in coefficient_tree_df, with their derivatives alongside.
// Called by all 32 lanes of one warp; `scratch` holds the first tree_scratch_floats(KG) -
// KG floats of the tree's scratch, eps the leaves' input errors (fp32, shared).
template <int KG>
__device__ float coefficient_probe(const df32 (&G)[KG][KG], float sc, const float* eps, float ge,
                                   float* scratch) {
  constexpr int M1 = KG / 2, M2 = KG / 4;
  const int lane = threadIdx.x & 31;
  const bool on = lane < KG;
  const int row = on ? lane : 0;
  float* hA = scratch;              // H, T0, T1 of even levels: [3][M1*M1]
  float* hB = hA + 3 * M1 * M1;     // odd levels: [3][M2*M2]
  float* na = hB + 3 * M2 * M2;     // node coefficient and its two derivatives: [3][KG]
  auto g = [&](int i, int j) { return G[i][j].hi * sc; };
  auto tsign = [&](float gkk, int m) {
    return (probe_mix(__float_as_uint(gkk) ^ (0x9E3779B9u * static_cast<uint32_t>(m + 1))) & 1u) ? 1.f : -1.f;
  };
  // leaf-level perturbation E_m(i, j)
  auto pert = [&](int i, int j, int m) {
    const float gii = fmaxf(g(i, i), 0.f), gjj = fmaxf(g(j, j), 0.f);
    const uint32_t h = probe_mix(__float_as_uint(g(i, j)) ^ probe_mix(__float_as_uint(gii * gjj)));
    const float s = (h >> m) & 1u ? 1.f : -1.f;
    const float ti = tsign(gii, m) * eps[i], tj = tsign(gjj, m) * eps[j];
    return (ge * s + (ti + tj)) * (sqrtf(gii) * sqrtf(gjj));
  };
  float c = on ? 1.f : 0.f, t0 = 0.f, t1 = 0.f;  // leaf coefficient and its derivatives
  const float* H = nullptr;  // this level's node Gram and derivatives ([3][m*m]); null: the leaves
  int m = KG;
  for (int lvl = 0; m > 1; ++lvl, m >>= 1) {
    auto h = [&](int k, int i, int j) -> float {
      return H ? H[k * m * m + i * m + j] : (k == 0 ? g(i, j) : pert(i, j, k - 1));
    };
    {
      const int n = lane < m ? lane : 0, sib = n ^ 1;
      const float p = h(0, n, n), d = h(0, n, sib);
      float a = 1.f, a0 = 0.f, a1 = 0.f;
      if (p > 0.f) {
        const float inv2p = 0.5f / p;
        a = 1.f - d * inv2p;
        a0 = (d * h(1, n, n) / p - h(1, n, sib)) * inv2p;
        a1 = (d * h(2, n, n) / p - h(2, n, sib)) * inv2p;
      }
      if (lane < m) {
        na[lane] = a;
        na[KG + lane] = a0;
        na[2 * KG + lane] = a1;
      }
    }
    __syncwarp();
    if (on) {
      const int anc = lane >> lvl;
      const float a = na[anc];
      t0 = fmaf(t0, a, c * na[KG + anc]);
      t1 = fmaf(t1, a, c * na[2 * KG + anc]);
      c *= a;
    }
    const int mh = m / 2;
    float* Hn = (H == hA) ? hB : hA;
    auto mul = [](float x, float y) { return x * y; };
    auto add = [](float x, float y) { return x + y; };
    for (int t = lane; t < mh * (mh + 1) / 2; t += 32) {
      int pi, qi;
      tri_unpack(mh, t, pi, qi);
      const int a = 2 * pi, b = 2 * pi + 1, a2 = 2 * qi, b2 = 2 * qi + 1;
      const float al = na[a], be = na[b], al2 = na[a2], be2 = na[b2];
      const float v = node_gram_entry(al, be, al2, be2, h(0, a, a2), h(0, b, b2), h(0, a, b2), h(0, b, a2), mul, add);
      Hn[pi * mh + qi] = v;
      Hn[qi * mh + pi] = v;
      for (int k = 1; k <= 2; ++k) {
        const float* da = na + k * KG;
        // derivative of every term x y H: (x' y + x y') H + (x y) H'
        auto dterm = [&](int x, int y, int i, int j) {
          return fmaf(da[x] * na[y] + na[x] * da[y], h(0, i, j), (na[x] * na[y]) * h(k, i, j));
        };
        const float dv = (dterm(a, a2, a, a2) + dterm(b, b2, b, b2)) + (dterm(a, b2, a, b2) + dterm(b, a2, b, a2));
        Hn[k * mh * mh + pi * mh + qi] = dv;
        Hn[k * mh * mh + qi * mh + pi] = dv;
      }
    }
    __syncwarp();
    H = Hn;
  }
  // |sum_k dc_k g_k|^2 = dc^T G dc, rows summed pairwise in leaf order
  float r0[KG], r1[KG];
#pragma unroll
  for (int j = 0; j < KG; ++j) {
    const float gj = g(row, j);
    r0[j] = __shfl_sync(0xFFFFFFFFu, t0, j) * gj;
    r1[j] = __shfl_sync(0xFFFFFFFFu, t1, j) * gj;
  }
#pragma unroll
  for (int w = 1; w < KG; w *= 2)
#pragma unroll
    for (int j = 0; j < KG; j += 2 * w) {
      r0[j] += r0[j + w];
      r1[j] += r1[j + w];
    }
  const float q0 = tree_lane_sumf(on ? t0 * r0[0] : 0.f);
  const float q1 = tree_lane_sumf(on ? t1 * r1[0] : 0.f);
  const float P = H ? H[0] : g(0, 0);
  if (!(P > 0.f)) return 1e30f;
  return sqrtf(fmaxf(fmaxf(q0, q1), 0.f) / P);
}

// The Adasum tree of one segment in coefficient space, in double-float arithmetic,
// evaluated by one warp on node Gram matrices.  A node u of the tree is sum_k c_k g_k
// over its leaves; the nodes of one level have the Gram matrix H(u, v) = u . v (the
// leaves' is G).  Pairing u = node 2i with its sibling v = node 2i+1:
//     alpha = 1 - H(u,v) / (2 H(u,u))   (alpha = 1 when H(u,u) == 0: a zero node is a plain sum)
//     beta  = 1 - H(u,v) / (2 H(v,v))
// and the next level's node Gram follows from these coefficients and four entries of H
// (node_gram_entry), so no dot product over the leaves is formed after the first
// level.  Each leaf's coefficient is the product of its ancestors' alpha or beta.  The
// tree runs on G times a power of two that brings the largest squared leaf norm into
// [0.5, 1) (exact, and harmless: the coefficients are scale-invariant); P_out (|out|^2,
// the root's H) is scaled back.  Lane k < KG receives its coefficient in c_out (fp32,
// the double-float value rounded once).
//
// Alongside, a first-order estimate of the error of the fp32 pass.  Gram entries carry
// errors of about gram_err |g_i||g_j| (independent, so quadratic forms add them in
// quadrature), inputs carry relative errors eps (earlier stages), and the combine
// rounds at each of the log2(K)+1 levels of its pairwise sum.  Per node it follows
// S = sum c_k^2 |g_k|^2, the coefficient errors dc_k through R = sum dc_k^2 |g_k|^2 and
// Q = sum |c_k| dc_k |g_k|^2, and E2 = sum c_k^2 eps_k^2 |g_k|^2, with the node's error
// D = sqrt(R + E2).  When a node's norm is no larger than its own error (cancellation),
// or the estimated relative error of the output exceeds the budget even after
// coefficient_probe has measured the coefficient part, the segment is flagged for the
// recompute.  The estimate needs a few significant digits only, so it runs in fp32.
//
// Called by all 32 lanes of one warp.  G and eps are in shared memory (G stored
// symmetric), scratch is shared, tree_scratch_floats(KG) floats.  Returns (in every
// lane) the estimated relative output error (1e30 when ill-conditioned).  Swapping the
// children of any node leaves every result bitwise unchanged.
template <int KG>
__device__ double coefficient_tree_df(const df32 (&G)[KG][KG], const double* eps,
                                      double gram_err, float* scratch, float& c_out, bool& ill,
                                      double* P_out = nullptr) {
  static_assert(KG >= 1 && KG <= 16 && (KG & (KG - 1)) == 0, "a power of two, one lane per leaf");
  constexpr int M1 = KG / 2, M2 = KG / 4;
  const int lane = threadIdx.x & 31;
  const bool on = lane < KG;
  const int row = on ? lane : 0;
  float gmax = on ? fmaxf(G[row][row].hi, 0.f) : 0.f;
  for (int off = 16; off > 0; off >>= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xFFFFFFFFu, gmax, off));
  int ex = 0;
  if (gmax > 0.f) frexpf(gmax, &ex);
  ex = ex < -120 ? -120 : (ex > 120 ? 120 : ex);
  const float sc = ldexpf(1.f, -ex);
  const float ge = static_cast<float>(gram_err);
  df32* hA = reinterpret_cast<df32*>(scratch);  // node Gram of odd levels: [M1][M1]
  df32* hB = hA + M1 * M1;                        // even levels from 2: [M2][M2]
  df32* nc = hB + M2 * M2;                        // this level's node coefficients: [KG]
  // node state (lane n < m holds node n of the current level; the leaves first)
  const float s2 = on ? fmaxf(G[row][row].hi * sc, 0.f) : 0.f;  // |g_k|^2, scaled
  const float e = on ? static_cast<float>(eps[row]) : 0.f;
  float* const epsf = scratch + 3 * (M1 * M1 + M2 * M2) + 3 * KG;  // for the probe
  if (on) epsf[lane] = e;
  float S = s2, Q = 0.f, R = 0.f, E2 = e * e * s2;
  df32 c = {on ? 1.f : 0.f, 0.f};  // lane k < KG: leaf k's coefficient
  bool bad = false;
  const df32* H = nullptr;         // this level's node Gram ([m][m]); null: G
  int m = KG;
  for (int lvl = 0; m > 1; ++lvl, m >>= 1) {
    auto h = [&](int i, int j) -> df32 {
      return H ? H[i * m + j] : df32{G[i][j].hi * sc, G[i][j].lo * sc};
    };
    const bool node = lane < m;
    const int n = node ? lane : 0, sib = n ^ 1;
    const df32 p = h(n, n), d = h(n, sib);
    const float D = sqrtf(R + E2);
    const float S_sib = __shfl_xor_sync(0xFFFFFFFFu, S, 1);
    const float D_sib = __shfl_xor_sync(0xFFFFFFFFu, D, 1);
    const float ps = p.hi, n_self = sqrtf(fmaxf(ps, 0.f)), n_sib = sqrtf(fmaxf(h(sib, sib).hi, 0.f));
    const float err_p = ge * S + 2.f * n_self * D;
    const float err_d = ge * sqrtf(S * S_sib) + (n_self * D_sib + n_sib * D);
    df32 coef = {1.f, 0.f};
    float dcoef = 0.f;
    if (ps != 0.f) {
      coef = df_add(df32{1.f, 0.f}, df_neg(df_div(d, df32{2.f * p.hi, 2.f * p.lo})));
      const float ap = fabsf(ps);
      dcoef = __fdividef(err_d + __fdividef(fabsf(d.hi) * err_p, ap), 2.f * ap);
      if (node && ps <= err_p) bad = true;
    } else if (node && S > 0.f) {
      bad = true;  // a non-zero subtree cancelled to an exact zero norm
    }
    if (node) nc[lane] = coef;
    // the parent's state: node n' (lane n' < m/2) from its children 2n', 2n'+1
    const float a2 = coef.hi * coef.hi, aa = fabsf(coef.hi);
    const float Sc = a2 * S, Qc = fmaf(aa * dcoef, S, a2 * Q);
    const float Rc = fmaf(dcoef * dcoef, S, fmaf(2.f * aa * dcoef, Q, a2 * R)), Ec = a2 * E2;
    const int c0 = (2 * lane) & 31, c1 = (2 * lane + 1) & 31;
    S = __shfl_sync(0xFFFFFFFFu, Sc, c0) + __shfl_sync(0xFFFFFFFFu, Sc, c1);
    Q = __shfl_sync(0xFFFFFFFFu, Qc, c0) + __shfl_sync(0xFFFFFFFFu, Qc, c1);
    R = __shfl_sync(0xFFFFFFFFu, Rc, c0) + __shfl_sync(0xFFFFFFFFu, Rc, c1);
    E2 = __shfl_sync(0xFFFFFFFFu, Ec, c0) + __shfl_sync(0xFFFFFFFFu, Ec, c1);
    __syncwarp();
    if (on) c = df_mul(c, nc[lane >> lvl]);
    const int mh = m / 2;
    df32* Hn = (H == hA) ? hB : hA;
    for (int t = lane; t < mh * (mh + 1) / 2; t += 32) {
      int pi, qi;
      tri_unpack(mh, t, pi, qi);
      const int a = 2 * pi, b = 2 * pi + 1, a2i = 2 * qi, b2i = 2 * qi + 1;
      const df32 v = node_gram_entry(
          nc[a], nc[b], nc[a2i], nc[b2i], h(a, a2i), h(b, b2i), h(a, b2i), h(b, a2i),
          [](df32 x, df32 y) { return df_mul(x, y); }, [](df32 x, df32 y) { return df_add(x, y); });
      Hn[pi * mh + qi] = v;
      Hn[qi * mh + pi] = v;
    }
    __syncwarp();
    H = Hn;
  }
  // root: lane 0 holds its state; H[0] is |out|^2 (scaled)
  S = __shfl_sync(0xFFFFFFFFu, S, 0);
  R = __shfl_sync(0xFFFFFFFFu, R, 0);
  E2 = __shfl_sync(0xFFFFFFFFu, E2, 0);
  const df32 P = H ? H[0] : df32{G[0][0].hi * sc, G[0][0].lo * sc};  // (one leaf: its own norm)
  const float D = sqrtf(R + E2);
  ill = __any_sync(0xFFFFFFFFu, bad);
  c_out = __fadd_rn(c.hi, c.lo);
  if (P_out) *P_out = ldexp(df_to_double(P), ex);
  if (S == 0.f) return 0.0;  // every leaf is zero: the output is exactly zero
  int levels = 1;
  for (int k = KG; k > 1; k >>= 1) ++levels;
  const float Pf = P.hi;
  const float err_P = ge * S + 2.f * sqrtf(fmaxf(Pf, 0.f)) * D;
  if (Pf <= err_P) {
    ill = true;
    return 1e30;
  }
  if (ill) return 1e30;
  const float rnd = levels * 5.9604644775390625e-08f * sqrtf(S);  // the combine's roundings
  float rel = (D + rnd) / sqrtf(Pf);
  if (rel > static_cast<float>(kRelErrBudget)) {
    // The bound asks for a recompute: measure the coefficient error instead (every
    // lane holds the same rel, so the whole warp takes this branch).  The inputs' own
    // errors still reach the output directly, through their coefficients.
    __syncwarp();
    const float probe = coefficient_probe<KG>(G, sc, epsf, ge, scratch);
    rel = fminf(rel, kProbeSafety * probe + (sqrtf(E2) + rnd) / sqrtf(Pf));
  }
  return static_cast<double>(rel);
}

// The linear recursion g[0,k] = Adasum(g[0,k-1], g_k), k = 1 .. kreal-1, in coefficient
// space with the same error estimate as coefficient_tree (u = the running node, v = leaf
// k).  Called by all 32 lanes of one warp; lane k < KG owns leaf k.
template <int KG>
__device__ double coefficient_chain(const double (&G)[KG][KG], const double* eps,
                                    double gram_err, double* c_sh, double& c, bool& ill,
                                    int kreal, double* P_out = nullptr) {
  const int lane = threadIdx.x & 31;
  const bool on = lane < KG;
  const int row = on ? lane : 0;
  const double s = on ? sqrt(fmax(G[row][row], 0.0)) : 0.0;
  const double e = on ? eps[row] : 0.0;
  c = (lane == 0) ? 1.0 : 0.0;
  double dc = 0.0;
  bool bad = false;
  if (on) c_sh[lane] = c;
  __syncwarp();
  for (int k = 1; k < kreal; ++k) {
    const bool in_u = lane < k;
    double row_u = 0.0;
    if (on)
      for (int j = 0; j < k; ++j) row_u = fma(c_sh[j], G[row][j], row_u);
    const double pu = block_lane_sum(in_u ? c * row_u : 0.0, 32);
    const double d = block_lane_sum(in_u ? c * G[row][k] : 0.0, 32);
    const double Su = block_lane_sum(in_u ? c * c * s * s : 0.0, 32);
    const double Du = sqrt(block_lane_sum(in_u ? (dc * dc + c * c * e * e) * s * s : 0.0, 32));
    const double sk = sqrt(fmax(G[k][k], 0.0)), ek = eps[k];
    const double pv = G[k][k], Sv = sk * sk, Dv = ek * sk;
    const double nu = sqrt(fmax(pu, 0.0)), nv = sqrt(fmax(pv, 0.0));
    const double err_pu = gram_err * Su + 2.0 * nu * Du;
    const double err_pv = gram_err * Sv + 2.0 * nv * Dv;
    const double err_d = gram_err * sqrt(Su * Sv) + (nu * Dv + nv * Du);
    double alpha = 1.0, beta = 1.0, dalpha = 0.0, dbeta = 0.0;
    if (pu != 0.0) {
      alpha = 1.0 - d / (2.0 * pu);
      dalpha = (err_d + fabs(d) * err_pu / fabs(pu)) / (2.0 * fabs(pu));
      if (pu <= err_pu) bad = true;
    } else if (Su > 0.0) {
      bad = true;
    }
    if (pv != 0.0) {
      beta = 1.0 - d / (2.0 * pv);
      dbeta = (err_d + fabs(d) * err_pv / fabs(pv)) / (2.0 * fabs(pv));
      if (pv <= err_pv) bad = true;
    } else if (Sv > 0.0) {
      bad = true;
    }
    if (in_u) {
      dc = fma(fabs(alpha), dc, fabs(c) * dalpha);
      c *= alpha;
    } else if (lane == k) {
      dc = dbeta;
      c = beta;
    }
    __syncwarp();
    if (on) c_sh[lane] = c;
    __syncwarp();
  }
  double full = 0.0;
  if (on)
    for (int j = 0; j < KG; ++j) full = fma(c_sh[j], G[row][j], full);
  const double P = block_lane_sum(c * full, 32);
  const double S = block_lane_sum(c * c * s * s, 32);
  const double D = sqrt(block_lane_sum((dc * dc + c * c * e * e) * s * s, 32));
  ill = __any_sync(0xFFFFFFFFu, bad);
  if (P_out) *P_out = P;
  if (S == 0.0) return 0.0;
  int levels = 1;
  for (int k = KG; k > 1; k >>= 1) ++levels;
  const double err_P = gram_err * S + 2.0 * sqrt(fmax(P, 0.0)) * D;
  if (P <= err_P) {
    ill = true;
    return 1e30;
  }
  const double rel = (D + levels * 5.9604644775390625e-08 * sqrt(S)) / sqrt(P);
  return ill ? 1e30 : rel;
}

// Items (segment, worker group) per CTA of the coefficient step when items are many:
// one per warp (coef_warp_kernel), since a tree is a long chain of dependent steps on one
// warp and an SM keeps many of them in flight.  With few items (fewer than a few per SM)
// each CTA takes one (coef_kernel) and all its threads gather the Gram matrix: a long
// segment has many chunk sums.
constexpr int kCoefWarps = 4;

// Shared scratch of one item of the coefficient kernel.
template <int KG>
struct CoefScratch {
  double G[KG][KG];
  df32 Gd[KG][KG];
  double eps[KG];
  double snorm[KG];
  float tree[tree_scratch_floats(KG)];
};

// The Gram matrix of (segment, group) from its chunk sums (double-float, added in chunk
// order; the loads are issued eight at a time) and the input errors, by threads first,
// first + step, ...  The fp64 copy G is filled only for the chain's coefficient step and
// the orthogonality metric's trace.
template <int KG>
__device__ __forceinline__ void coef_gather(const StageArgs& a, const SegDesc& sd, int seg, int q,
                                            CoefScratch<KG>& sh, int first, int step) {
  constexpr int E = tri_count(KG);
  constexpr int U = 8;
  const bool want_fp64 = a.mode == kModeChain || a.diag_sum != nullptr;
  ChunkDesc one = {};
  const bool single = sd.nchunks == 1 && chunk_ok(a, sd.first_chunk, one);
  for (int e = first; e < E; e += step) {
    const float2* p = a.chunk_sums + (static_cast<size_t>(q) * a.nchunks + sd.first_chunk) * E + e;
    df32 sum = {0.f, 0.f};
    int t = 0;
    if (single) {  // the chunk-sum kernel left this segment's one chunk to this kernel
      const float2 v = chunk_entry<KG>(a, one, e, q);
      sum = df_add(sum, df32{v.x, v.y});
      t = 1;
    }
    for (; t + U <= sd.nchunks; t += U) {
      float2 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) v[u] = __ldcg(p + static_cast<size_t>(t + u) * E);
#pragma unroll
      for (int u = 0; u < U; ++u) sum = df_add(sum, df32{v[u].x, v[u].y});
    }
    for (; t < sd.nchunks; ++t) {
      const float2 v = __ldcg(p + static_cast<size_t>(t) * E);
      sum = df_add(sum, df32{v.x, v.y});
    }
    int i, j;
    tri_unpack(KG, e, i, j);
    sh.Gd[i][j] = sh.Gd[j][i] = sum;
    if (want_fp64) sh.G[i][j] = sh.G[j][i] = df_to_double(sum);
  }
  for (int k = first; k < KG; k += step)
    sh.eps[k] = a.in_relerr ? static_cast<double>(a.in_relerr[static_cast<size_t>(q * KG + k) * a.nsegs + seg]) : 0.0;
}

// The tree coefficients of (segment, group) and the conditioning and range checks (see
// coefficient_tree_df), once coef_gather has filled sh.  Called by the 32 lanes of one
// warp.
template <int KG>
__device__ __forceinline__ void coef_tree(const StageArgs& a, const SegDesc& sd, int seg, int q,
                                          CoefScratch<KG>& sh) {
  const int lane = threadIdx.x & 31;
  // the workers with a nonzero value in the segment
  uint32_t seg_nz = 0u;
  ChunkDesc one;
  if (sd.nchunks == 1 && chunk_ok(a, sd.first_chunk, one)) {
    if (lane == 0) seg_nz = chunk_nonzero(a, one, q);
  } else {
    const uint32_t* p = a.chunk_nz + static_cast<size_t>(q) * a.nchunks + sd.first_chunk;
    for (int t = lane; t < sd.nchunks; t += 32) seg_nz |= __ldcg(p + t);
  }
  seg_nz = warp_or_u32(seg_nz);
  double c = 0.0, P = 0.0;
  bool ill = false;
  double rel;
  // (|out|^2 is read back only for the orthogonality metric: fp64 work otherwise saved)
  double* const want_P = a.outnorm2 ? &P : nullptr;
  if (a.mode == kModeChain) {
    rel = coefficient_chain<KG>(sh.G, sh.eps, kGramRelErr, sh.snorm, c, ill, a.Kreal, want_P);
  } else {
    float cf = 0.f;
    rel = coefficient_tree_df<KG>(sh.Gd, sh.eps, kGramRelErr, sh.tree, cf, ill, want_P);
    c = cf;
  }
  if (lane == 0 && a.outnorm2) a.outnorm2[seg] = P;
  if (lane == 0 && a.diag_sum) {
    double tr = 0.0;
    for (int k = 0; k < KG; ++k) tr += sh.G[k][k];
    a.diag_sum[static_cast<size_t>(q) * a.nsegs + seg] = tr;
  }
  if (lane < KG) a.coef[(static_cast<size_t>(q) * a.nsegs + seg) * KG + lane] = static_cast<float>(c);
  // range check (kDiagLoPerPos, kDiagHi), lane k for worker k: a nonzero worker whose
  // squared norm is too small for the segment's length, or too large (NaN compares
  // false: it propagates)
  bool out_of_range = false;
  if (lane < KG && ((seg_nz >> lane) & 1u)) {
    const float d = sh.Gd[lane][lane].hi;  // (fp32 holds both bounds exactly)
    out_of_range = d < static_cast<float>(sd.len) * static_cast<float>(kDiagLoPerPos) ||
                   d > static_cast<float>(kDiagHi);
  }
  out_of_range = __any_sync(0xFFFFFFFFu, out_of_range);
  if (lane == 0) {
    if (a.relerr) a.relerr[static_cast<size_t>(q) * a.nsegs + seg] = static_cast<float>(fmin(rel, 1e30));
    if (a.seg_flag && sd.len > 0 && (ill || !(rel <= kRelErrBudget) || out_of_range)) a.seg_flag[seg] = 1;
  }
}

// The descriptor of item `item` of the (group, listed segment) pairs, checked.
__device__ __forceinline__ bool coef_item(const StageArgs& a, int item, int& seg, int& q, SegDesc& sd) {
  const int nlist = a.seg_list ? a.nseg_list : a.nsegs;
  q = item / nlist;
  const int i = item - q * nlist;
  seg = a.seg_list ? a.seg_list[i] : i;
  sd = a.segs[seg];
  return ADASUM_CHECK(a.error, seg >= 0 && seg < a.nsegs && sd.start >= 0 && sd.start + sd.len <= a.n_total &&
                                   sd.first_chunk >= 0 && sd.first_chunk + sd.nchunks <= a.nchunks);
}

// Few items: CTA b takes item b, all its threads gather, warp 0 runs the tree.  (A
// single kernel holding both layouts needed more registers and made the calls with few
// items measurably slower: ResNet-50, 0.311 -> 0.315 ms.)
template <int KG>
__global__ void __launch_bounds__(32 * kCoefWarps) coef_kernel(const StageArgs a) {
  pdl_enter();
  __shared__ CoefScratch<KG> sh;
  const int items = (a.seg_list ? a.nseg_list : a.nsegs) * a.G;
  int seg, q;
  SegDesc sd;
  if (static_cast<int>(blockIdx.x) >= items || !coef_item(a, blockIdx.x, seg, q, sd)) return;  // (uniform)
  coef_gather<KG>(a, sd, seg, q, sh, threadIdx.x, blockDim.x);
  __syncthreads();
  if (threadIdx.x < 32) coef_tree<KG>(a, sd, seg, q, sh);
}

// Many items: warp w of CTA b takes item b * kCoefWarps + w.
template <int KG>
__global__ void __launch_bounds__(32 * kCoefWarps) coef_warp_kernel(const StageArgs a) {
  pdl_enter();
  __shared__ CoefScratch<KG> sh[kCoefWarps];
  const int warp = threadIdx.x >> 5;
  const int items = (a.seg_list ? a.nseg_list : a.nsegs) * a.G;
  const int item = blockIdx.x * kCoefWarps + warp;
  int seg, q;
  SegDesc sd;
  if (item >= items || !coef_item(a, item, seg, q, sd)) return;  // whole warps
  coef_gather<KG>(a, sd, seg, q, sh[warp], threadIdx.x & 31, 32);
  __syncwarp();
  coef_tree<KG>(a, sd, seg, q, sh[warp]);
}

// ----------------------------------------------------------- pass 2: combine (+ step)

// sum over leaves [LO, LO+CNT) of c_k * x_k[e], as a balanced pairwise tree of
// explicitly rounded products and sums (never contracted into FMAs), so that the value
// is symmetric under swapping the two halves of any subtree.
template <typename Tag, int LO, int CNT, int KG>
__device__ __forceinline__ float tree_combine(const float (&c)[KG], const uint4 (&r)[KG], int e) {
  if constexpr (CNT == 1) {
    return __fmul_rn(c[LO], vec_elem<Tag>(r[LO], e));
  } else {
    return __fadd_rn(tree_combine<Tag, LO, CNT / 2, KG>(c, r, e),
                     tree_combine<Tag, LO + CNT / 2, CNT / 2, KG>(c, r, e));
  }
}

// Store VW fp32 values as elements [p0, p0 + VW) of an output array, only positions in
// [lo, hi); full aligned vectors are written with streaming vector stores.
template <typename OutTag, int VW>
__device__ __forceinline__ void store_vec(typename ElemTraits<OutTag>::Storage* y, int64_t p0,
                                          int64_t lo, int64_t hi, bool aligned,
                                          const float (&val)[VW]) {
  const bool full = aligned && p0 >= lo && p0 + VW <= hi;
  if constexpr (ElemTraits<OutTag>::kVW == 8) {  // bf16 output
    if (full) {
      if constexpr (VW == 8) {
        uint4 w = make_uint4(pack_bf16x2(val[0], val[1]), pack_bf16x2(val[2], val[3]),
                             pack_bf16x2(val[4], val[5]), pack_bf16x2(val[6], val[7]));
        __stcs(reinterpret_cast<uint4*>(y + p0), w);
      } else {
        uint2 w = make_uint2(pack_bf16x2(val[0], val[1]), pack_bf16x2(val[2], val[3]));
        __stcs(reinterpret_cast<uint2*>(y + p0), w);
      }
      return;
    }
#pragma unroll
    for (int e = 0; e < VW; ++e) {
      const int64_t p = p0 + e;
      if (p >= lo && p < hi) y[p] = float_to_bf16_bits(val[e]);
    }
  } else {  // fp32 output
    if (full) {
#pragma unroll
      for (int h = 0; h < VW; h += 4)
        __stcs(reinterpret_cast<float4*>(y + p0 + h),
               make_float4(val[h], val[h + 1], val[h + 2], val[h + 3]));
      return;
    }
#pragma unroll
    for (int e = 0; e < VW; ++e) {
      const int64_t p = p0 + e;
      if (p >= lo && p < hi) y[p] = val[e];
    }
  }
}

// Load VW fp32 values [p0, p0+VW) (positions outside [lo, hi) read as 0).
template <int VW>
__device__ __forceinline__ void load_f32_vec(const float* x, int64_t p0, int64_t lo, int64_t hi,
                                             bool aligned, float (&val)[VW]) {
  if (aligned && p0 >= lo && p0 + VW <= hi) {
#pragma unroll
    for (int h = 0; h < VW; h += 4) {
      const float4 f = __ldcs(reinterpret_cast<const float4*>(x + p0 + h));
      val[h] = f.x;
      val[h + 1] = f.y;
      val[h + 2] = f.z;
      val[h + 3] = f.w;
    }
    return;
  }
#pragma unroll
  for (int e = 0; e < VW; ++e) {
    const int64_t p = p0 + e;
    val[e] = (p >= lo && p < hi) ? x[p] : 0.f;
  }
}

// out = sum_k c_k g_k over one tile; with MOM, also v' = mu v + out, w' = w - lr v'
// (fp32), and out is written only when a.out[q] is not null.
// (Coefficients and flags written by other CTAs are read through L2.)
template <typename InTag, typename OutTag, int KG, bool MOM>
__device__ __forceinline__ void combine_range(const StageArgs& a, int seg, int64_t lo, int64_t hi, int q,
                                              int first, int step) {
  using SI = typename ElemTraits<InTag>::Storage;
  using SO = typename ElemTraits<OutTag>::Storage;
  constexpr int VW = ElemTraits<InTag>::kVW;
  if (!ADASUM_CHECK(a.error, seg >= 0 && seg < a.nsegs && lo >= 0 && lo <= hi && hi <= a.n_total)) return;
  const bool aligned = a.aligned != 0;
  const SI* x[KG];
#pragma unroll
  for (int k = 0; k < KG; ++k) x[k] = static_cast<const SI*>(a.in[q * KG + k]);
  SO* y = static_cast<SO*>(a.out[q]);
  const int64_t v0 = lo / VW, v1 = (hi + VW - 1) / VW;
  // The skip flag and the coefficients are requested together, before the first
  // vectors' loads, and waited on after them: one memory round trip before the stream
  // starts, not three (a warp's short tile is only a few vectors long).
  const int flagged = a.skip_flagged ? __ldcg(a.seg_flag + seg) : 0;
  float c[KG];
  if constexpr (KG == 1) {
    c[0] = 1.f;
  } else {
    const float* cp = a.coef + (static_cast<size_t>(q) * a.nsegs + seg) * KG;
#pragma unroll
    for (int k = 0; k < KG; ++k) c[k] = __ldcg(cp + k);
  }
  if constexpr (MOM) {
    // the next vectors' loads are issued before this vector's w and v are read and
    // written (GPT-style set, K = 8 bf16: 9.08 -> 9.00 ms per step; without the
    // momentum step the same order made the one-warp tiles slower)
    int64_t v = v0 + first;
    uint4 r[KG];
    if (v < v1) {
#pragma unroll
      for (int k = 0; k < KG; ++k) r[k] = load_vec_raw<InTag, kLoadStream>(x[k], v, lo, hi, aligned);
    }
    if (flagged) return;  // left to the recompute
    while (v < v1) {
      float val[VW];
#pragma unroll
      for (int e = 0; e < VW; ++e) val[e] = tree_combine<InTag, 0, KG, KG>(c, r, e);
      const int64_t p0 = v * VW;
      v += step;
      if (v < v1) {
#pragma unroll
        for (int k = 0; k < KG; ++k) r[k] = load_vec_raw<InTag, kLoadStream>(x[k], v, lo, hi, aligned);
      }
      float wv[VW], mv[VW];
      load_f32_vec<VW>(a.master_w, p0, lo, hi, aligned, wv);
      if (a.momentum != nullptr) {  // heavy ball: v' = mu v + A, w' = w - lr v'
        load_f32_vec<VW>(a.momentum, p0, lo, hi, aligned, mv);
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          mv[e] = __fmaf_rn(a.mu, mv[e], val[e]);
          wv[e] = __fmaf_rn(-a.lr, mv[e], wv[e]);
        }
        store_vec<F32Tag, VW>(a.momentum, p0, lo, hi, aligned, mv);
      } else {                      // plain step: w' = w - lr A
#pragma unroll
        for (int e = 0; e < VW; ++e) wv[e] = __fmaf_rn(-a.lr, val[e], wv[e]);
      }
      store_vec<F32Tag, VW>(a.master_w, p0, lo, hi, aligned, wv);
      if (y != nullptr) store_vec<OutTag, VW>(y, p0, lo, hi, aligned, val);
    }
  } else {
    for (int64_t v = v0 + first; v < v1; v += step) {
      uint4 r[KG];
#pragma unroll
      for (int k = 0; k < KG; ++k) r[k] = load_vec_raw<InTag, kLoadStream>(x[k], v, lo, hi, aligned);
      if (flagged) return;  // left to the recompute
      float val[VW];
#pragma unroll
      for (int e = 0; e < VW; ++e) val[e] = tree_combine<InTag, 0, KG, KG>(c, r, e);
      store_vec<OutTag, VW>(y, v * VW, lo, hi, aligned, val);
    }
  }
}

// The tile at entry i of a list of tile ids (all tiles when the list is null), checked.
__device__ __forceinline__ bool list_tile(const StageArgs& a, const int* list, int i, TileDesc& t) {
  const int id = list ? list[i] : i;
  if (!ADASUM_CHECK(a.error, id >= 0 && id < a.ntiles)) return false;
  t = a.tiles[id];
  return true;
}

template <typename InTag, typename OutTag, int KG, bool MOM>
__global__ void __launch_bounds__(kThreads) combine_kernel(const StageArgs a) {
  pdl_enter();
  // a.combine_tiles consecutive tiles per CTA (of a.tile_list when short tiles have a
  // launch of their own), adjacent tiles of one segment merged into one range: the
  // prologue (coefficients, flag) is a dependent L2 round trip, and one long strided
  // loop streams better than several short ones
  const int n = a.tile_list ? a.ntile_list : a.ntiles;
  const int t0 = blockIdx.x * a.combine_tiles;
  const int t1 = min(n, t0 + a.combine_tiles);
  for (int t = t0; t < t1;) {
    TileDesc first;
    if (!list_tile(a, a.tile_list, t, first)) return;  // (uniform over the CTA)
    int64_t hi = first.start + first.len;
    int u = t + 1;
    for (; u < t1; ++u) {
      TileDesc nx;
      if (!list_tile(a, a.tile_list, u, nx) || nx.seg != first.seg || nx.start != hi) break;
      hi = nx.start + nx.len;
    }
    combine_range<InTag, OutTag, KG, MOM>(a, first.seg, first.start, hi, blockIdx.y, threadIdx.x, kThreads);
    t = u;
  }
}

// Short tiles (a.small_list: kSmallTileF32, kSmallTileBF16 or kSmallTileSimt positions at
// most), one warp each: a CTA per tile would leave most of its threads without a vector and run its
// tiles' coefficient loads one after another.
// Each warp takes tiles w, w + W, w + 2W, ... (W the grid's warps: a few per SM,
// warp_tile_grid, in CTAs of kCombineWarpThreads), so warps stay resident across tiles
// instead of a CTA of eight one-tile warps retiring for each eight tiles.
template <typename InTag, typename OutTag, int KG, bool MOM>
__global__ void __launch_bounds__(kThreads) combine_warp_kernel(const StageArgs a) {
  pdl_enter();
  const int wpb = static_cast<int>(blockDim.x) >> 5;
  const int W = static_cast<int>(gridDim.x) * wpb;
  for (int w = blockIdx.x * wpb + (threadIdx.x >> 5); w < a.nsmall; w += W) {  // (whole warps)
    TileDesc t;
    if (!list_tile(a, a.small_list, w, t)) return;
    combine_range<InTag, OutTag, KG, MOM>(a, t.seg, t.start, t.start + t.len, blockIdx.y, threadIdx.x & 31, 32);
  }
}

// ------------------------------------------------------------- flags between CTAs

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}


// ------------------------------------------------ per-worker heavy-ball step (Fig. 3)

// v = mu v + g for one worker (fp32 state; g widened from its storage type).
template <typename Tag>
__global__ void __launch_bounds__(kThreads) local_momentum_kernel(const void* g, float* v,
                                                                  int64_t n, float mu, int aligned) {
  pdl_enter();
  using S = typename ElemTraits<Tag>::Storage;
  constexpr int VW = ElemTraits<Tag>::kVW;
  const S* x = static_cast<const S*>(g);
  const int64_t nv = (n + VW - 1) / VW;
  for (int64_t vi = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; vi < nv;
       vi += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 r = load_vec_raw<Tag, kLoadStream>(x, vi, 0, n, aligned != 0);
    float m[VW], out[VW];
    load_f32_vec<VW>(v, vi * VW, 0, n, aligned != 0, m);
#pragma unroll
    for (int e = 0; e < VW; ++e) out[e] = __fmaf_rn(mu, m[e], vec_elem<Tag>(r, e));
    store_vec<F32Tag, VW>(v, vi * VW, 0, n, aligned != 0, out);
  }
}

// ---------------------------------------------------------------- fp64 recompute path
//
// Segments flagged by coef_kernel are recomputed here entirely in fp64: exact products
// of the stored inputs (fp32 x fp32 and bf16 x bf16 products are exact in fp64), fp64
// Gram sums, the fp64 tree, and an fp64 combine rounded once to the output type.  These
// kernels walk the flagged lists with a small persistent grid and return at once when
// the lists are empty, which is the normal case.

enum Kind { kKindF32 = 0, kKindBF16 = 1, kKindF64 = 2 };

template <int IN>
__device__ __forceinline__ double load_f64(const void* base, int64_t i) {
  if (base == nullptr) return 0.0;  // a zero (padding) gradient
  if constexpr (IN == kKindF32) return static_cast<double>(static_cast<const float*>(base)[i]);
  if constexpr (IN == kKindBF16)
    return static_cast<double>(bf16_bits_to_float(static_cast<const uint16_t*>(base)[i]));
  return static_cast<const double*>(base)[i];
}

// Builds the lists of flagged tiles and segments (order of the lists is irrelevant:
// every tile and segment is computed on its own).
static __global__ void collect_kernel(const StageArgs a) {
  pdl_enter();
  for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < a.nsegs; s += gridDim.x * blockDim.x) {
    if (!a.seg_flag[s]) continue;
    const SegDesc sd = a.segs[s];
    if (sd.ntiles == 0) continue;
    if (sd.len <= kTinySeg) {
      a.list_tiny[atomicAdd(&a.list_count[2], 1)] = s;
      continue;
    }
    if (a.oc_vecs > 0) {  // small enough for the on-chip kernel's recompute
      const int vw = a.oc_vw;
      const int64_t nv = (sd.start + sd.len + vw - 1) / vw - sd.start / vw;
      if ((nv + a.oc_cmax - 1) / a.oc_cmax <= a.oc_vecs) {
        a.oc_list[atomicAdd(a.oc_count, 1)] = s;
        continue;
      }
    }
    const int base = atomicAdd(&a.list_count[0], sd.ntiles);
    for (int t = 0; t < sd.ntiles; ++t) a.list_tiles[base + t] = sd.first_tile + t;
    a.list_segs[atomicAdd(&a.list_count[1], 1)] = s;
  }
}

// The orthogonality metric of every segment: |A|^2 / sum_k |g_k|^2 (NaN when 0/0).
static __global__ void orthogonality_kernel(const double* outnorm2, const double* diag_sum,
                                            int groups, int nsegs, float* ortho) {
  pdl_enter();
  for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < nsegs; s += gridDim.x * blockDim.x) {
    double den = 0.0;
    for (int q = 0; q < groups; ++q) den += diag_sum[static_cast<size_t>(q) * nsegs + s];
    ortho[s] = den == 0.0 ? __int_as_float(0x7FC00000) : static_cast<float>(outnorm2[s] / den);
  }
}

// Sum over the warp in a fixed butterfly order (every lane gets the same value).
__device__ __forceinline__ double warp_sum64(double v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
  return v;
}

// Vector-space fp64 recompute of a flagged segment of at most 32 positions: one warp,
// lane j holds position j of every node.  The tree is evaluated depth first (leaves
// left to right, a node is formed as soon as both children exist), which visits the
// same pairs (2i, 2i+1) at every level as the level-by-level definition.  Norms are
// recomputed from the node values themselves, as in the definition.
template <int IN, int OUT, bool MOM>
__global__ void __launch_bounds__(kThreads) tiny64_kernel(const StageArgs a) {
  pdl_enter();
  constexpr int kMaxDepth = 10;  // log2(kMaxK) + 2
  const int lane = threadIdx.x & 31;
  const int wid = (blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * kThreads) >> 5;
  const int count = a.list_count[2];
  for (int li = wid; li < count; li += nwarps) {
    const SegDesc sd = a.segs[a.list_tiny[li]];
    if (!ADASUM_CHECK(a.error, sd.start >= 0 && sd.len <= 32 && sd.start + sd.len <= a.n_total)) continue;
    const int n = static_cast<int>(sd.len);
    const int64_t p = sd.start + lane;
    const bool on = lane < n;
    double val[kMaxDepth];
    int lvl[kMaxDepth];
    int top = 0;
    for (int k = 0; k < a.Ktotal; ++k) {
      val[top] = on ? load_f64<IN>(a.in[k], p) : 0.0;
      lvl[top] = 0;
      ++top;
      // the chain folds every new leaf into the running node; the tree merges equal levels
      while (top >= 2 && (a.mode == kModeChain || lvl[top - 1] == lvl[top - 2])) {
        const double x = val[top - 2], y = val[top - 1];
        const double d = warp_sum64(x * y), pa = warp_sum64(x * x), pb = warp_sum64(y * y);
        const double alpha = 1.0 - (pa == 0.0 ? 0.0 : d / (2.0 * pa));
        const double beta = 1.0 - (pb == 0.0 ? 0.0 : d / (2.0 * pb));
        val[top - 2] = alpha * x + beta * y;
        lvl[top - 2] += 1;
        --top;
      }
    }
    const double nrm2 = warp_sum64(val[0] * val[0]);
    if (lane == 0 && a.outnorm2) a.outnorm2[a.list_tiny[li]] = nrm2;
    if (!on) continue;
    const double yv = val[0];
    if constexpr (MOM) {
      double v = yv;
      if (a.momentum != nullptr) {
        v = static_cast<double>(a.mu) * static_cast<double>(a.momentum[p]) + yv;
        a.momentum[p] = static_cast<float>(v);
      }
      a.master_w[p] = static_cast<float>(static_cast<double>(a.master_w[p]) - static_cast<double>(a.lr) * v);
      if (a.out[0] == nullptr) continue;
    }
    if constexpr (OUT == kKindF32) {
      static_cast<float*>(a.out[0])[p] = static_cast<float>(yv);
    } else {
      __nv_bfloat16 h = __double2bfloat16(yv);
      static_cast<uint16_t*>(a.out[0])[p] = *reinterpret_cast<uint16_t*>(&h);
    }
  }
}

// The largest |input| of every flagged segment, as 1024 + its binary exponent (atomic
// max over the segment's tiles; 0 stays for an all-zero segment).  The recompute's Gram
// scales its segment by the matching power of two.
template <int IN>
__global__ void __launch_bounds__(kThreads) segmax_kernel(const StageArgs a) {
  pdl_enter();
  __shared__ float wmax[kWarps];
  const int count = a.list_count[0];
  const int K = a.G * a.Kg;
  for (int li = blockIdx.x; li < count; li += gridDim.x) {
    const TileDesc t = a.tiles[a.list_tiles[li]];
    if (!tile_ok(a, a.list_tiles[li], t)) continue;  // (uniform over the CTA)
    float m = 0.f;
    for (int k = 0; k < K; ++k) {
      if (a.in[k] == nullptr) continue;
      for (int p = threadIdx.x; p < t.len; p += kThreads)
        m = fmaxf(m, fabsf(static_cast<float>(load_f64<IN>(a.in[k], t.start + p))));
    }
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      float mm = 0.f;
      for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, wmax[w]);
      if (mm > 0.f) {
        int ex = 0;
        frexpf(mm, &ex);
        atomicMax(a.seg_exp + t.seg, 1024 + ex);
      }
    }
    __syncthreads();
  }
}

// Gram matrix of every flagged tile, in double-float arithmetic: fp32 and bf16 inputs
// are exact fp32 numbers, so every product is exact (TwoProduct) and only the sums round,
// at about 2^-48.  The tile is staged through shared memory 64 positions at a time,
// scaled by the segment's power of two (exact) so that the squares stay inside fp32's
// range; thread e owns Gram entry e.  The partial is scaled back and stored in fp64.
template <int IN, int KG>
__global__ void __launch_bounds__(kThreads) gram64_kernel(const StageArgs a) {
  pdl_enter();
  constexpr int E = tri_count(KG);
  constexpr int P = 64;
  __shared__ df32 xs[KG][P];
  const int q = blockIdx.y;
  const int count = a.list_count[0];
  int ei = 0, ej = 0;
  if (threadIdx.x < E) tri_unpack(KG, threadIdx.x, ei, ej);
  for (int li = blockIdx.x; li < count; li += gridDim.x) {
    const int tile_id = a.list_tiles[li];
    const TileDesc t = a.tiles[tile_id];
    if (!tile_ok(a, tile_id, t)) continue;  // (uniform over the CTA)
    const int enc = a.seg_exp[t.seg];
    int ex = enc > 0 ? enc - 1024 : 0;
    ex = ex < -125 ? -125 : (ex > 125 ? 125 : ex);
    df32 se = {0.f, 0.f}, so = {0.f, 0.f};
    for (int64_t p0 = t.start; p0 < t.start + t.len; p0 += P) {
      const int64_t left = t.start + t.len - p0;
      const int np = left < P ? static_cast<int>(left) : P;
      __syncthreads();
      for (int idx = threadIdx.x; idx < KG * P; idx += kThreads) {
        const int k = idx / P, p = idx % P;
        const double v = p < np ? ldexp(load_f64<IN>(a.in[q * KG + k], p0 + p), -ex) : 0.0;
        xs[k][p] = IN == kKindF64 ? df_from_double(v) : df32{static_cast<float>(v), 0.f};
      }
      __syncthreads();
      if (threadIdx.x < E) {
        for (int p = 0; p + 1 < np; p += 2) {
          se = df_add(df_mul(xs[ei][p], xs[ej][p]), se);
          so = df_add(df_mul(xs[ei][p + 1], xs[ej][p + 1]), so);
        }
        if (np & 1) se = df_add(df_mul(xs[ei][np - 1], xs[ej][np - 1]), se);
      }
    }
    if (threadIdx.x < E)
      a.partials64[(static_cast<size_t>(q) * a.ntiles + tile_id) * E + threadIdx.x] =
          ldexp(df_to_double(df_add(se, so)), 2 * ex);
    __syncthreads();
  }
}

// fp64 coefficients of every flagged segment (plain tree, no error estimate needed).
template <int KG>
__global__ void __launch_bounds__(128) coef64_kernel(const StageArgs a) {
  pdl_enter();
  constexpr int E = tri_count(KG);
  __shared__ double G[KG][KG];
  __shared__ double zeros[KG];
  __shared__ double snorm[KG];
  const int q = blockIdx.y;
  const int count = a.list_count[1];
  for (int k = threadIdx.x; k < KG; k += blockDim.x) zeros[k] = 0.0;
  for (int li = blockIdx.x; li < count; li += gridDim.x) {
    const int seg = a.list_segs[li];
    const SegDesc sd = a.segs[seg];
    if (!ADASUM_CHECK(a.error, seg >= 0 && seg < a.nsegs && sd.first_tile >= 0 &&
                                   sd.first_tile + sd.ntiles <= a.ntiles))
      continue;  // (uniform over the CTA)
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      double sum = 0.0;
      const double* p = a.partials64 + (static_cast<size_t>(q) * a.ntiles + sd.first_tile) * E + e;
      for (int t = 0; t < sd.ntiles; ++t) sum += p[static_cast<size_t>(t) * E];
      int i, j;
      tri_unpack(KG, e, i, j);
      G[i][j] = sum;
      G[j][i] = sum;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      double c = 0.0, P = 0.0;
      bool ill = false;
      if (a.mode == kModeChain)
        coefficient_chain<KG>(G, zeros, 0.0, snorm, c, ill, a.Kreal, &P);
      else
        coefficient_tree<KG>(G, zeros, 0.0, snorm, c, ill, &P);
      if (threadIdx.x == 0 && a.outnorm2) a.outnorm2[seg] = P;
      if (threadIdx.x < KG) a.coef64[(static_cast<size_t>(q) * a.nsegs + seg) * KG + threadIdx.x] = c;
    }
  }
}

template <int IN, int LO, int CNT, int KG>
__device__ __forceinline__ double tree_combine64(const double (&c)[KG], const StageArgs& a, int q,
                                                 int64_t p) {
  if constexpr (CNT == 1) {
    return c[LO] * load_f64<IN>(a.in[q * KG + LO], p);
  } else {
    return tree_combine64<IN, LO, CNT / 2, KG>(c, a, q, p) +
           tree_combine64<IN, LO + CNT / 2, CNT / 2, KG>(c, a, q, p);
  }
}

// fp64 combine of every flagged tile (plus the fp64 heavy-ball step when requested).
template <int IN, int OUT, int KG, bool MOM>
__global__ void __launch_bounds__(kThreads) combine64_kernel(const StageArgs a) {
  pdl_enter();
  const int q = blockIdx.y;
  const int count = a.list_count[0];
  for (int li = blockIdx.x; li < count; li += gridDim.x) {
    const TileDesc t = a.tiles[a.list_tiles[li]];
    if (!tile_ok(a, a.list_tiles[li], t)) continue;  // (uniform over the CTA)
    double c[KG];
    if constexpr (KG == 1) {
      c[0] = 1.0;
    } else {
      const double* cp = a.coef64 + (static_cast<size_t>(q) * a.nsegs + t.seg) * KG;
#pragma unroll
      for (int k = 0; k < KG; ++k) c[k] = cp[k];
    }
    for (int64_t p = t.start + threadIdx.x; p < t.start + t.len; p += kThreads) {
      const double y = tree_combine64<IN, 0, KG, KG>(c, a, q, p);
      if constexpr (MOM) {
        double v = y;
        if (a.momentum != nullptr) {
          v = static_cast<double>(a.mu) * static_cast<double>(a.momentum[p]) + y;
          a.momentum[p] = static_cast<float>(v);
        }
        a.master_w[p] = static_cast<float>(static_cast<double>(a.master_w[p]) - static_cast<double>(a.lr) * v);
        if (a.out[q] == nullptr) continue;
      }
      if constexpr (OUT == kKindF64) {
        static_cast<double*>(a.out[q])[p] = y;
      } else if constexpr (OUT == kKindF32) {
        static_cast<float*>(a.out[q])[p] = static_cast<float>(y);
      } else {
        __nv_bfloat16 h = __double2bfloat16(y);
        static_cast<uint16_t*>(a.out[q])[p] = *reinterpret_cast<uint16_t*>(&h);
      }
    }
  }
}

}  // namespace adasum
