// adasum_onchip.cuh -- the small-segment path (sm_103a): one segment per CTA or per
// thread-block cluster, every worker's slice of the segment read from HBM once into
// shared memory (bulk copies), and the whole Adasum tree evaluated on chip; and, for
// segments of at most 32 positions, one warp (or a group of 8 or 16 of its lanes) per
// segment.
//
// "Scaling Distributed Training with Adaptive Summation", Section 3: each layer is
// combined on its own by the binary tree of Adasum(a, b) = (1 - a.b/(2|a|^2)) a +
// (1 - a.b/(2|b|^2)) b over the K workers.  Small layers are where the tiled route pays
// for its structure: a Gram tile, a chunk reduction, a coefficient launch and a combine
// tile per layer, and a second HBM read of every input.  Here a segment's K x n block
// lives in shared memory from the moment it arrives until its output is written:
//
//   load     K rows of the segment (this CTA's share of its positions) by bulk copy
//   stage 1  Gram matrix of every 16-worker group from shared memory (register-blocked
//            fp32 FMAs), summed over the cluster through distributed shared memory in
//            CTA order; each group's coefficient tree (double-float, with the fp32 error
//            estimate) evaluated once, by one CTA of the cluster, and shared
//   stage 2  (K > 16) the tree's top levels over the group results, kept in registers
//   store    out = the tree's value, written once
//
// A segment whose error estimate flags it is recomputed right there in vector space,
// level by level as the definition reads (pairs (2i, 2i+1), dot products summed over the
// cluster, alpha/beta, combine), in double-float arithmetic, with the level values in the
// same shared memory.  Every CTA of a cluster reads the same sums in the same order, so
// all of them reach bitwise-identical decisions and follow the same control flow.
//
// The only wait that is not a hardware barrier is the bulk-copy completion, bounded by a
// clock budget (bit 2 of the device error word reports a timeout).
#pragma once

#include "adasum_kernels.cuh"
#include "adasum_ptx.cuh"

namespace adasum {

constexpr int kOnchipThreads = 256;
constexpr int kOnchipWarps = kOnchipThreads / 32;
constexpr int kOnchipRedBytes = kOnchipThreads * 16 * 4;  // per-thread 4x4 partials
constexpr int kOnchipMaxCluster = 16;

__host__ __device__ constexpr int onchip_row_bytes(int P) { return P * 4 + 16; }
__host__ __device__ constexpr int onchip_dynamic_smem(int K) {
  return K * onchip_row_bytes(onchip_positions(K)) + kOnchipRedBytes;
}

// Pairwise tree sum of c_k * y_k over CNT leaves from LO (explicit roundings, as in
// tree_combine), for values already in fp32 registers.
template <int LO, int CNT, int N>
__device__ __forceinline__ float tree_combine_f(const float (&c)[N], const float (&y)[N]) {
  if constexpr (CNT == 1) {
    return __fmul_rn(c[LO], y[LO]);
  } else {
    return __fadd_rn(tree_combine_f<LO, CNT / 2, N>(c, y), tree_combine_f<LO + CNT / 2, CNT / 2, N>(c, y));
  }
}

template <typename S>
__device__ __forceinline__ float elem_f32(const S* x, int64_t p) {
  if constexpr (sizeof(S) == 4) {
    return x[p];
  } else {
    return bf16_bits_to_float(x[p]);
  }
}

// Element g of an output array from a double-float value times 2^ex, rounded once
// (bf16 through its exact fp64 sum, so that it too is rounded once).
template <typename S>
__device__ __forceinline__ void store_df(S* out, int64_t g, df32 y, int ex) {
  if constexpr (sizeof(S) == 4) {
    out[g] = ldexpf(__fadd_rn(y.hi, y.lo), ex);
  } else {
    __nv_bfloat16 h = __double2bfloat16(ldexp(df_to_double(y), ex));
    out[g] = *reinterpret_cast<uint16_t*>(&h);
  }
}

// Exponent e with amax * 2^-e in [0.5, 1) (0 for amax == 0), kept where 2^-e is a normal
// fp32 number.  Scaling a segment's values by 2^-e is exact and the tree is
// scale-invariant; it keeps the squares of the double-float paths inside fp32's range.
__device__ __forceinline__ int scale_exponent(float amax) {
  int ex = 0;
  if (amax > 0.f) frexpf(amax, &ex);
  return ex < -125 ? -125 : (ex > 125 ? 125 : ex);
}

// Entry e of every CTA's copy of buf (the cluster's partials after an exchange), summed
// in rank order.  All loads are issued before the first add, so the distributed shared
// memory latency is paid once, not once per CTA.
__device__ __forceinline__ void cluster_kahan_sum(const float* buf, int e, uint32_t C, float& sum,
                                                  float& comp) {
  float v[kOnchipMaxCluster];
#pragma unroll
  for (int r = 0; r < kOnchipMaxCluster; ++r) v[r] = static_cast<uint32_t>(r) < C ? map_rank(buf, r)[e] : 0.f;
  sum = 0.f;
  comp = 0.f;
#pragma unroll
  for (int r = 0; r < kOnchipMaxCluster; ++r) kahan_add(sum, comp, v[r]);
}
__device__ __forceinline__ df32 cluster_df_sum(const df32* buf, int e, uint32_t C) {
  df32 v[kOnchipMaxCluster];
#pragma unroll
  for (int r = 0; r < kOnchipMaxCluster; ++r)
    v[r] = static_cast<uint32_t>(r) < C ? map_rank(buf, r)[e] : df32{0.f, 0.f};
  df32 s = v[0];
#pragma unroll
  for (int r = 1; r < kOnchipMaxCluster; ++r) s = df_add(s, v[r]);
  return s;
}
__device__ __forceinline__ df32 df_warp_sum(df32 x) { return df_block_sum(x, 32); }
__device__ __forceinline__ void cta_or_cluster_sync(uint32_t C) {
  if (C > 1) {
    cluster_sync_all();
  } else {
    __syncthreads();
  }
}

template <typename InTag, int KG1, int NG>
__global__ void __launch_bounds__(kOnchipThreads, 2) onchip_kernel(const OnchipArgs a) {
  pdl_enter();
  using S = typename ElemTraits<InTag>::Storage;
  constexpr int VW = ElemTraits<InTag>::kVW;
  constexpr int K = KG1 * NG;
  static_assert(K <= kOnchipMaxK && (NG == 1 || KG1 == kMaxGroup), "groups of 16, then one top stage");
  constexpr int E1 = tri_count(KG1);
  constexpr int E2 = tri_count(NG);
  constexpr int B = KG1 < 4 ? KG1 : 4;        // register block: B x B Gram entries
  constexpr int NBS = KG1 / B;                // blocks per side of a group's Gram
  constexpr int NBG = NBS * (NBS + 1) / 2;    // upper-triangle blocks per group
  constexpr int NB = NG * NBG;
  constexpr int SL = kOnchipThreads / NB;     // position slices per block
  constexpr int kXch1 = NG * E1 * 4;
  constexpr int kXchD = (K / 2) * 3 * 8;
  constexpr int kXch = (kXch1 > kXchD ? kXch1 : kXchD) + 16;

  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ df32 G1[NG][KG1][KG1];
  __shared__ df32 G2[NG][NG];
  __shared__ double zeros[KG1];
  __shared__ double rel1[NG];
  __shared__ df32 ab[K / 2][2];
  __shared__ float coef1[NG][KG1];
  __shared__ float coef2[NG];
  // results of the trees this CTA evaluates (group q belongs to CTA q % C), read by the
  // whole cluster
  __shared__ float tcoef[NG][KG1];
  __shared__ double trel[NG];
  __shared__ int tflag[NG];
  __shared__ float t2coef[NG];
  __shared__ int t2flag;
  __shared__ __align__(16) unsigned char xch[2][kXch];
  __shared__ int flag;
  __shared__ uint32_t knz[K];   // OR of every worker's raw bits in this CTA's share
  __shared__ __align__(8) uint64_t bar;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = a.P;
  const int rs = onchip_row_bytes(P);
  unsigned char* data = smem;                              // K rows of rs bytes
  float* red = reinterpret_cast<float*>(smem + K * rs);   // [SL][NB][B*B]; the trees' scratch after
  static_assert(NG * tree_scratch_floats(KG1) * 4 <= kOnchipRedBytes, "tree scratch fits the Gram's");

  const uint32_t C = cluster_nctarank(), rank = cluster_ctarank();
  // cluster i takes list entries i, i + nclusters, ... (all CTAs of a cluster the same)
  const int nclusters = static_cast<int>(gridDim.x / C);
  const int nitems = a.dev_count != nullptr ? *a.dev_count : nclusters;
  if (static_cast<int>(cluster_id_x()) >= nitems) return;  // whole clusters
  const bool aligned = a.aligned != 0;
  int xi = 0;  // exchange counter (buffers alternate)
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  if (tid < KG1) zeros[tid] = 0.0;
  uint32_t phase = 0;
  for (int item = static_cast<int>(cluster_id_x()); item < nitems; item += nclusters, phase ^= 1u) {
  if (tid == 0) flag = 0;
  __syncthreads();
  const SegDesc sd = a.segs[a.list[item]];
  const int64_t s0 = sd.start, s1 = sd.start + sd.len;
  const int64_t vs0 = s0 / VW, vs1 = (s1 + VW - 1) / VW;
  const int64_t chunk = (vs1 - vs0 + C - 1) / C;
  if (!ADASUM_CHECK(a.error, sd.start >= 0 && sd.len >= 0 && s1 <= a.n_total && chunk * VW <= P)) {
    phase ^= 1u;  // nothing was armed for this entry: keep the barrier phase
    continue;     // (uniform over the cluster: every CTA reads the same descriptor)
  }
  const int64_t cv0 = min(vs1, vs0 + static_cast<int64_t>(rank) * chunk);
  const int64_t cv1 = min(vs1, cv0 + chunk);
  const int nvec = static_cast<int>(cv1 - cv0);            // <= P / VW (host guarantees)
  const int64_t iv0 = max(cv0, (s0 + VW - 1) / VW), iv1 = min(cv1, s1 / VW);  // whole vectors
  const bool bulk = aligned && iv1 > iv0;

  // ---------------------------------------------------------------- load
  if (warp == 0) {
    if (lane == 0) {
      uint32_t bytes = 0;
      if (bulk)
        for (int k = 0; k < K; ++k)
          if (a.in[k] != nullptr) bytes += static_cast<uint32_t>(iv1 - iv0) * 16u;
      mbar_arrive_expect_tx(&bar, bytes + (a.inject_extra_tx ? 16u : 0u));
    }
    __syncwarp();
    if (bulk)
      for (int k = lane; k < K; k += 32)
        if (a.in[k] != nullptr)
          bulk_g2s(data + k * rs + (iv0 - cv0) * 16, static_cast<const S*>(a.in[k]) + iv0 * VW,
                   static_cast<uint32_t>(iv1 - iv0) * 16u, &bar);
  }
  // partial vectors at the segment's ends, zero rows, and everything when unaligned
  for (int idx = tid; idx < K * nvec; idx += kOnchipThreads) {
    const int k = idx / nvec, j = idx - k * nvec;
    const int64_t v = cv0 + j;
    const S* x = static_cast<const S*>(a.in[k]);
    if (bulk && x != nullptr && v >= iv0 && v < iv1) continue;
    *reinterpret_cast<uint4*>(data + k * rs + j * 16) = load_vec_raw<InTag, kLoadKeep>(x, v, s0, s1, aligned);
  }
  if (!mbar_wait(&bar, phase, a.spin_budget, a.error)) mbar_wait(&bar, phase, a.spin_budget, a.error);
  if (a.recompute_only && tid == 0) flag = 1;
  __syncthreads();
  if (!a.recompute_only) {
    // range check of the fp32 pass (kDiagLoPerPos, kDiagHi), completed with the trees:
    // which workers have a nonzero value in this CTA's share, TPR threads per row
    {
      constexpr int TPR = K >= 8 ? kOnchipThreads / K : 32;
      const int k = tid / TPR, j = tid % TPR;
      uint32_t b = 0u;
      if (k < K)
        for (int v = j; v < nvec; v += TPR) b |= vec_or(*reinterpret_cast<const uint4*>(data + k * rs + v * 16));
#pragma unroll
      for (int off = TPR / 2; off > 0; off >>= 1) b |= __shfl_xor_sync(0xFFFFFFFFu, b, off);
      if (k < K && j == 0) knz[k] = b & MagBits<InTag>::kMask;
    }

    // ---------------------------------------------------------------- stage 1: Gram
    if (tid < NB * SL) {
      const int slice = tid % SL, blk = tid / SL;
      const int q = blk / NBG;
      int bi, bj;
      tri_unpack(NBS, blk % NBG, bi, bj);
      const unsigned char* rowp = data + (q * KG1 + bi * B) * rs;
      const unsigned char* colp = data + (q * KG1 + bj * B) * rs;
      float acc[B][B];
#pragma unroll
      for (int i = 0; i < B; ++i)
#pragma unroll
        for (int j = 0; j < B; ++j) acc[i][j] = 0.f;
      for (int v = slice; v < nvec; v += SL) {
        uint4 rr[B], cc[B];
#pragma unroll
        for (int i = 0; i < B; ++i) {
          rr[i] = *reinterpret_cast<const uint4*>(rowp + i * rs + v * 16);
          cc[i] = *reinterpret_cast<const uint4*>(colp + i * rs + v * 16);
        }
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          float xr[B], xc[B];
#pragma unroll
          for (int i = 0; i < B; ++i) {
            xr[i] = vec_elem<InTag>(rr[i], e);
            xc[i] = vec_elem<InTag>(cc[i], e);
          }
#pragma unroll
          for (int i = 0; i < B; ++i)
#pragma unroll
            for (int j = 0; j < B; ++j) acc[i][j] = __fmaf_rn(xr[i], xc[j], acc[i][j]);
        }
      }
#pragma unroll
      for (int i = 0; i < B; ++i)
#pragma unroll
        for (int j = 0; j < B; ++j) red[(slice * NB + blk) * (B * B) + i * B + j] = acc[i][j];
    }
    __syncthreads();
    {
      float* xg = reinterpret_cast<float*>(xch[xi & 1]);
      for (int e = tid; e < NB * B * B; e += kOnchipThreads) {
        float sum = 0.f, comp = 0.f;
        for (int s = 0; s < SL; ++s) kahan_add(sum, comp, red[s * NB * B * B + e]);
        const int blk = e / (B * B), ij = e % (B * B);
        const int q = blk / NBG;
        int bi, bj;
        tri_unpack(NBS, blk % NBG, bi, bj);
        const int i = bi * B + ij / B, j = bj * B + ij % B;
        if (i <= j) xg[q * E1 + tri_index(KG1, i, j)] = __fsub_rn(sum, comp);
      }
      cta_or_cluster_sync(C);
      // the Gram matrices of this CTA's groups: compensated sums over the cluster, CTA order
      for (int e = tid; e < NG * E1; e += kOnchipThreads) {
        const int q = e / E1;
        if (static_cast<uint32_t>(q) % C != rank) continue;
        float sum = xg[e], comp = 0.f;
        if (C > 1) cluster_kahan_sum(xg, e, C, sum, comp);
        const df32 g = df_fast_two_sum(sum, -comp);  // the compensated sum, as a double-float
        int i, j;
        tri_unpack(KG1, e % E1, i, j);
        G1[q][i][j] = g;
        G1[q][j][i] = g;
      }
      ++xi;
    }
    __syncthreads();
    {
      // warp w of CTA r evaluates group w * C + r
      const int q = warp * static_cast<int>(C) + static_cast<int>(rank);
      if (q < NG) {
        float c = 0.f;
        bool ill = false;
        const double rel = coefficient_tree_df<KG1>(G1[q], zeros, kGramRelErr, red + q * tree_scratch_floats(KG1), c, ill);
        if (lane < KG1) tcoef[q][lane] = c;
        // range check, lane i for worker i of the group: a nonzero value anywhere in the
        // cluster's share and a squared norm too small for the segment's length, or too
        // large, sends the segment to the recompute (NaN compares false: it propagates)
        bool out_of_range = false;
        if (lane < KG1) {
          uint32_t nz = knz[q * KG1 + lane];
          for (uint32_t r = 0; r < C; ++r)
            if (r != rank) nz |= *map_rank(&knz[q * KG1 + lane], r);
          const double d = df_to_double(G1[q][lane][lane]);
          out_of_range = nz != 0u && (d < static_cast<double>(sd.len) * kDiagLoPerPos || d > kDiagHi);
        }
        out_of_range = __any_sync(0xFFFFFFFFu, out_of_range);
        if (lane == 0) {
          trel[q] = rel;
          tflag[q] = (ill || !(rel <= kRelErrBudget) || out_of_range) ? 1 : 0;
        }
      }
    }
    cta_or_cluster_sync(C);
    if (tid < NG * KG1) {
      const int q = tid / KG1, k = tid % KG1;
      coef1[q][k] = *map_rank(&tcoef[q][k], static_cast<uint32_t>(q) % C);
    }
    if (tid < NG) {
      rel1[tid] = *map_rank(&trel[tid], static_cast<uint32_t>(tid) % C);
      if (*map_rank(&tflag[tid], static_cast<uint32_t>(tid) % C)) flag = 1;
    }
    __syncthreads();

  }  // fp32 pass: stage-1 Gram and trees
  S* const out = static_cast<S*>(a.out);
  if (!flag) {
    if constexpr (NG == 1) {
      float c[KG1];
#pragma unroll
      for (int k = 0; k < KG1; ++k) c[k] = coef1[0][k];
      for (int v = tid; v < nvec; v += kOnchipThreads) {
        uint4 r[KG1];
#pragma unroll
        for (int k = 0; k < KG1; ++k) r[k] = *reinterpret_cast<const uint4*>(data + k * rs + v * 16);
        float val[VW];
#pragma unroll
        for (int e = 0; e < VW; ++e) val[e] = tree_combine<InTag, 0, KG1, KG1>(c, r, e);
        store_vec<InTag, VW>(out, (cv0 + v) * VW, s0, s1, aligned, val);
      }
    } else {
      // ---------------------------------------------------------------- stage 2
      // nvec <= P / VW <= kOnchipThreads when K >= 32: one vector per thread at most.
      const bool mine = tid < nvec;
      float y[VW][NG];
#pragma unroll
      for (int q = 0; q < NG; ++q) {
        float c[KG1];
#pragma unroll
        for (int k = 0; k < KG1; ++k) c[k] = coef1[q][k];
        uint4 r[KG1];
#pragma unroll
        for (int k = 0; k < KG1; ++k)
          r[k] = mine ? *reinterpret_cast<const uint4*>(data + (q * KG1 + k) * rs + tid * 16)
                      : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int e = 0; e < VW; ++e) y[e][q] = tree_combine<InTag, 0, KG1, KG1>(c, r, e);
      }
      float acc2[E2];
#pragma unroll
      for (int e = 0; e < E2; ++e) acc2[e] = 0.f;
#pragma unroll
      for (int e = 0; e < VW; ++e)
#pragma unroll
        for (int i = 0; i < NG; ++i)
#pragma unroll
          for (int j = i; j < NG; ++j)
            acc2[tri_index(NG, i, j)] = __fmaf_rn(y[e][i], y[e][j], acc2[tri_index(NG, i, j)]);
      float* xg = reinterpret_cast<float*>(xch[xi & 1]);
      block_reduce_store<E2>(acc2, xg);
      cta_or_cluster_sync(C);
      ++xi;
      if (rank == 0) {  // the top tree: CTA 0 of the cluster
        if (tid < E2) {
          float sum = xg[tid], comp = 0.f;
          if (C > 1) cluster_kahan_sum(xg, tid, C, sum, comp);
          const df32 g = df_fast_two_sum(sum, -comp);
          int i, j;
          tri_unpack(NG, tid, i, j);
          G2[i][j] = g;
          G2[j][i] = g;
        }
        __syncthreads();
        if (warp == 0) {
          float c = 0.f;
          bool ill = false;
          const double rel = coefficient_tree_df<NG>(G2, rel1, kGramRelErr, red, c, ill);  // (red is free after stage 1)
          if (lane < NG) t2coef[lane] = c;
          if (lane == 0) t2flag = (ill || !(rel <= kRelErrBudget)) ? 1 : 0;
        }
      }
      cta_or_cluster_sync(C);
      if (tid < NG) coef2[tid] = *map_rank(&t2coef[tid], 0u);
      if (tid == 0 && *map_rank(&t2flag, 0u)) flag = 1;
      __syncthreads();
      if (!flag && mine) {
        float c2[NG];
#pragma unroll
        for (int q = 0; q < NG; ++q) c2[q] = coef2[q];
        float val[VW];
#pragma unroll
        for (int e = 0; e < VW; ++e) val[e] = tree_combine_f<0, NG, NG>(c2, y[e]);
        store_vec<InTag, VW>(out, (cv0 + tid) * VW, s0, s1, aligned, val);
      }
    }
  }

  if (flag) {
    // ------------------------------------------------------- recompute (double-float)
    // The definition, level by level, in double-float arithmetic (about 48 significant
    // bits; GB300's fp64 pipe is 64 times narrower than its fp32 pipe).  Level 0 reads the
    // leaves: dot products from shared memory, the combine from global memory, so the
    // shared block is free to take the level values, one double-float (8 bytes) per
    // position -- level-0 node i in the bytes of data rows 2i and 2i+1.  Later levels
    // combine in place, position by position; node j of level l >= 1 lives in row
    // j * 2^(l-1).
    if (rank == 0 && tid == 0) atomicAdd(a.recomputed, 1);
    const int npos = nvec * VW;
    const int64_t p0 = cv0 * VW;
    const int rsd = 2 * rs / 8;  // row stride in double-floats
    df32* rows = reinterpret_cast<df32*>(data);
    int stride = 1;              // rows between consecutive nodes (level >= 1)
    // the segment's largest |value| over the cluster sets the power-of-two scale
    float amax = 0.f;
    for (int idx = tid; idx < K * nvec; idx += kOnchipThreads) {
      const uint4 x = *reinterpret_cast<const uint4*>(data + (idx / nvec) * rs + (idx % nvec) * 16);
#pragma unroll
      for (int e = 0; e < VW; ++e) amax = fmaxf(amax, fabsf(vec_elem<InTag>(x, e)));
    }
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    float* xm = reinterpret_cast<float*>(xch[xi & 1]);
    if (lane == 0) xm[warp] = amax;
    cta_or_cluster_sync(C);
    amax = 0.f;
    for (uint32_t r = 0; r < C; ++r)
      for (int w = 0; w < kOnchipWarps; ++w) amax = fmaxf(amax, map_rank(xm, r)[w]);
    ++xi;
    const int ex = scale_exponent(amax);
    const float sc = ldexpf(1.f, -ex);
    for (int m = K; m > 1; m /= 2) {
      const bool leaves = m == K;
      df32* xd = reinterpret_cast<df32*>(xch[xi & 1]);
      for (int i = warp; i < m / 2; i += kOnchipWarps) {
        df32 d = {0.f, 0.f}, pa = {0.f, 0.f}, pb = {0.f, 0.f};
        if (leaves) {
          const unsigned char* ra = data + (2 * i) * rs;
          const unsigned char* rb = data + (2 * i + 1) * rs;
          for (int v = lane; v < nvec; v += 32) {
            const uint4 x = *reinterpret_cast<const uint4*>(ra + v * 16);
            const uint4 y = *reinterpret_cast<const uint4*>(rb + v * 16);
#pragma unroll
            for (int e = 0; e < VW; ++e) {
              const df32 xe = {vec_elem<InTag>(x, e) * sc, 0.f}, ye = {vec_elem<InTag>(y, e) * sc, 0.f};
              d = df_add(df_mul(xe, ye), d);
              pa = df_add(df_mul(xe, xe), pa);
              pb = df_add(df_mul(ye, ye), pb);
            }
          }
        } else {
          const df32* ra = rows + static_cast<size_t>(2 * i) * stride * rsd;
          const df32* rb = rows + static_cast<size_t>(2 * i + 1) * stride * rsd;
          for (int p = lane; p < npos; p += 32) {
            const df32 xe = ra[p], ye = rb[p];
            d = df_add(df_mul(xe, ye), d);
            pa = df_add(df_mul(xe, xe), pa);
            pb = df_add(df_mul(ye, ye), pb);
          }
        }
        d = df_warp_sum(d);
        pa = df_warp_sum(pa);
        pb = df_warp_sum(pb);
        if (lane == 0) {
          xd[3 * i] = d;
          xd[3 * i + 1] = pa;
          xd[3 * i + 2] = pb;
        }
      }
      cta_or_cluster_sync(C);
      for (int i = tid; i < m / 2; i += kOnchipThreads) {
        const df32 d = C > 1 ? cluster_df_sum(xd, 3 * i, C) : xd[3 * i];
        const df32 pa = C > 1 ? cluster_df_sum(xd, 3 * i + 1, C) : xd[3 * i + 1];
        const df32 pb = C > 1 ? cluster_df_sum(xd, 3 * i + 2, C) : xd[3 * i + 2];
        const df32 one = {1.f, 0.f};
        ab[i][0] = pa.hi == 0.f ? one : df_add(one, df_neg(df_div(d, df32{2.f * pa.hi, 2.f * pa.lo})));
        ab[i][1] = pb.hi == 0.f ? one : df_add(one, df_neg(df_div(d, df32{2.f * pb.hi, 2.f * pb.lo})));
      }
      ++xi;
      __syncthreads();
      for (int idx = tid; idx < (m / 2) * npos; idx += kOnchipThreads) {
        const int i = idx / npos, p = idx - i * npos;
        const df32 al = ab[i][0], be = ab[i][1];
        if (leaves) {
          const int64_t g = p0 + p;
          const bool in = g >= s0 && g < s1;
          const S* ga = static_cast<const S*>(a.in[2 * i]);
          const S* gb = static_cast<const S*>(a.in[2 * i + 1]);
          const df32 xa = {(in && ga != nullptr) ? elem_f32(ga, g) * sc : 0.f, 0.f};
          const df32 xb = {(in && gb != nullptr) ? elem_f32(gb, g) * sc : 0.f, 0.f};
          rows[static_cast<size_t>(i) * rsd + p] = df_add(df_mul(al, xa), df_mul(be, xb));
        } else {
          df32* ra = rows + static_cast<size_t>(2 * i) * stride * rsd;
          const df32* rb = rows + static_cast<size_t>(2 * i + 1) * stride * rsd;
          ra[p] = df_add(df_mul(al, ra[p]), df_mul(be, rb[p]));
        }
      }
      if (!leaves) stride *= 2;
      __syncthreads();
    }
    for (int p = tid; p < npos; p += kOnchipThreads) {
      const int64_t g = p0 + p;
      if (g < s0 || g >= s1) continue;
      store_df(out, g, rows[p], ex);
    }
  }
  // The next entry's bulk copies overwrite this CTA's shared memory: its own reads come
  // first (proxy fence), and no CTA moves on (or leaves) while another may still read it.
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  cta_or_cluster_sync(C);
  }  // list entries
}

// ------------------------------------------------------------------ tiny segments
//
// Segments of at most kTinyDirect positions: a warp, or an aligned group of 8 or 16 of
// its lanes, per segment, lane j holding position j of every node, the tree evaluated on
// the values themselves in double-float arithmetic -- no Gram matrix, no error
// estimate, no second pass.  No block barriers: the warps' latencies overlap.

// One node: Adasum of two nodes held one position per lane, the dot products summed
// over aligned groups of gw lanes (one segment per group; every lane calls it).  Out of
// line: a 64-leaf tree makes 63 calls, and one copy of the code keeps the instruction
// cache warm for all the warps of an SM.
__device__ __noinline__ df32 tiny_node(df32 xa, df32 xb, int gw) {
  const df32 d = df_block_sum(df_mul(xa, xb), gw);
  const df32 pa = df_block_sum(df_mul(xa, xa), gw);
  const df32 pb = df_block_sum(df_mul(xb, xb), gw);
  const df32 one = {1.f, 0.f};
  const df32 al = pa.hi == 0.f ? one : df_add(one, df_neg(df_div(d, df32{2.f * pa.hi, 2.f * pa.lo})));
  const df32 be = pb.hi == 0.f ? one : df_add(one, df_neg(df_div(d, df32{2.f * pb.hi, 2.f * pb.lo})));
  return df_add(df_mul(al, xa), df_mul(be, xb));
}

// The subtree over leaves [LO, LO + CNT) of values already in registers.
template <int LO, int CNT, int KP>
__device__ __forceinline__ df32 tiny_subtree(const float (&v)[KP], int gw) {
  if constexpr (CNT == 1) {
    return df32{v[LO], 0.f};
  } else {
    const df32 left = tiny_subtree<LO, CNT / 2, KP>(v, gw);
    const df32 right = tiny_subtree<LO + CNT / 2, CNT / 2, KP>(v, gw);
    return tiny_node(left, right, gw);
  }
}

// List entry e, checked; false (after recording a failed check) when the entry is not
// one the kernel may touch.
__device__ __forceinline__ bool tiny_entry(const TinyArgs& a, int e, SegDesc& sd) {
  sd = a.segs[a.list[e]];
  return ADASUM_CHECK(a.error, sd.start >= 0 && sd.len <= kTinyDirect && sd.start + sd.len <= a.n_total);
}

// K = KP leaves (a power of two up to 64).  A warp takes 4 segments of at most 8
// positions, or 2 of at most 16, or 1 (lane groups of gw = 8, 16 or 32; list order:
// count8, count16, the rest).  Every value is loaded at once into registers, read once,
// prescaled by the power of two of its segment's largest |value|, and the tree runs from
// registers (its pairs (2i, 2i+1) at every level).  Sums over a group equal the sums over
// the whole warp of the one-segment layout: the other lanes hold zeros, and adding a zero
// is exact (it can only turn an exact -0 into +0).
template <typename InTag, int KP>
__global__ void __launch_bounds__(kOnchipThreads) tiny_reg_kernel(const TinyArgs a) {
  pdl_enter();
  using S = typename ElemTraits<InTag>::Storage;
  const int lane = threadIdx.x & 31;
  const int w = blockIdx.x * kOnchipWarps + (threadIdx.x >> 5);
  const int w8 = (a.count8 + 3) / 4, w16 = (a.count16 + 1) / 2;
  const int c32 = a.count - a.count8 - a.count16;
  if (w >= w8 + w16 + c32) return;  // whole warps only
  int gw, e, end;
  if (w < w8) {
    gw = 8;
    e = 4 * w + (lane >> 3);
    end = a.count8;
  } else if (w < w8 + w16) {
    gw = 16;
    e = a.count8 + 2 * (w - w8) + (lane >> 4);
    end = a.count8 + a.count16;
  } else {
    gw = 32;
    e = a.count8 + a.count16 + (w - w8 - w16);
    end = a.count;
  }
  SegDesc sd = {};
  const bool seg_ok = e < end && tiny_entry(a, e, sd);  // (lanes of a group agree)
  const int pos = lane & (gw - 1);
  const int64_t p = sd.start + pos;
  const bool on = seg_ok && pos < sd.len;
  float v[KP];
#pragma unroll
  for (int k = 0; k < KP; ++k) {
    const S* x = static_cast<const S*>(a.in[k]);
    v[k] = (on && x != nullptr) ? elem_f32(x, p) : 0.f;
  }
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < KP; ++k) amax = fmaxf(amax, fabsf(v[k]));
  for (int off = gw >> 1; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
  const int ex = scale_exponent(amax);
  const float sc = ldexpf(1.f, -ex);
#pragma unroll
  for (int k = 0; k < KP; ++k) v[k] *= sc;
  const df32 r = tiny_subtree<0, KP, KP>(v, gw);
  if (on) store_df(static_cast<S*>(a.out), p, r, ex);
}

// Any K (a power of two up to kMaxK): a max pass over the inputs, then the leaves read
// again left to right and a node formed as soon as both of its children exist (depth
// first), which visits the same pairs (2i, 2i+1) at every level as the level-by-level
// definition.
template <typename InTag>
__global__ void __launch_bounds__(kOnchipThreads) tiny_df_kernel(const TinyArgs a) {
  pdl_enter();
  using S = typename ElemTraits<InTag>::Storage;
  constexpr int kMaxDepth = 10;  // log2(kMaxK) + 2
  const int lane = threadIdx.x & 31;
  const int w = blockIdx.x * kOnchipWarps + (threadIdx.x >> 5);
  if (w >= a.count) return;  // whole warps only
  SegDesc sd;
  if (!tiny_entry(a, w, sd)) return;
  const int64_t p = sd.start + lane;
  const bool on = lane < sd.len;
  float amax = 0.f;
  for (int k = 0; k < a.K; ++k) {
    const S* x = static_cast<const S*>(a.in[k]);
    if (on && x != nullptr) amax = fmaxf(amax, fabsf(elem_f32(x, p)));
  }
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
  const int ex = scale_exponent(amax);
  const float sc = ldexpf(1.f, -ex);
  df32 val[kMaxDepth];
  int lvl[kMaxDepth];
  int top = 0;
  for (int k = 0; k < a.K; ++k) {
    const S* x = static_cast<const S*>(a.in[k]);
    val[top] = {(on && x != nullptr) ? elem_f32(x, p) * sc : 0.f, 0.f};
    lvl[top] = 0;
    ++top;
    while (top >= 2 && lvl[top - 1] == lvl[top - 2]) {
      val[top - 2] = tiny_node(val[top - 2], val[top - 1], 32);
      lvl[top - 2] += 1;
      --top;
    }
  }
  if (on) store_df(static_cast<S*>(a.out), p, val[0], ex);
}





}  // namespace adasum
