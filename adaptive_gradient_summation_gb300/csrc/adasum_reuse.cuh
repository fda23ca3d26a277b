// adasum_reuse.cuh -- the single-stage tiled route with the second read served from L2:
// one persistent kernel, one CTA per SM, for 8 or 16 workers of bf16 gradients.
//
// "Scaling Distributed Training with Adaptive Summation", Section 3: the combine of a
// layer needs its dot products and norms over the whole layer first ("cannot be
// performed in a streaming manner"), so every input is read twice -- once for the
// Gram matrix, once for out = sum_k c_k g_k.  The three-kernel route reads everything
// for the Gram pass, then everything again for the combine, so no second read can hit
// the 126 MB L2.  Here the work is one sequence of steps that every CTA follows on its
// own share of positions:
//
//   G steps  Gram partials of a run of segments (forward), tensor cores as in
//            gram_tile_mma; the part of each unit that will be read again soon is loaded
//            with the L2 evict_last policy, the rest with evict_first
//   C steps  the combine of a unit whose Gram finished a few tens of MB earlier, in
//            REVERSE position order (the most recently read bytes first, still in L2),
//            loads with evict_first, outputs with streaming stores
//
// Segment finishing runs beside the streaming, never in its way:
//   - when a CTA has seen its last position of a segment, its streaming warps add the
//     CTA's partial Gram matrix into the segment's exact fixed-point accumulators
//     (integer atomic adds, so the sum is the same whatever the order of arrival, and
//     the results are bitwise reproducible) and count the contribution;
//   - a finisher warp on every CTA (segments dealt round robin) waits for the count,
//     converts the exact sum to double, runs the coefficient tree (coefficient_tree_df,
//     with its error estimate and the range check) and publishes the coefficients;
//   - a C step waits (bounded) for its segments' coefficients.
// Flagged segments are skipped by the combine and left to the recompute path.
#pragma once

#include "adasum_kernels.cuh"

namespace adasum {

constexpr int kReuseWarps = kReuseThreads / 32;
constexpr int kStreamWarps = kReuseWarps - 1;          // warps 0..14 stream, warp 15 finishes
constexpr int kStreamThreads = kStreamWarps * 32;
constexpr int kAccBase = -160;                          // digit d weighs 2^(32 d - 160)

// ------------------------------------------------------------ cache-policy loads

__device__ __forceinline__ uint64_t l2_policy_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint4 ld16_policy(const void* p, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
}
// bf16 vector v of x masked to [lo, hi), as load_vec_raw, with an L2 policy on full loads.
__device__ __forceinline__ uint4 load_bf16_policy(const uint16_t* x, int64_t v, int64_t lo, int64_t hi,
                                                  bool aligned, uint64_t pol) {
  if (x == nullptr) return make_uint4(0u, 0u, 0u, 0u);
  const int64_t p0 = v * 8;
  if (aligned && p0 >= lo && p0 + 8 <= hi) return ld16_policy(x + p0, pol);
  return load_vec_raw<BF16Tag, kLoadKeep>(x, v, lo, hi, aligned);
}

// ------------------------------------------------------------ exact accumulation

// Adds the fp32 value x exactly to the digits acc[0..kAccDigits): x = m 2^e with m a
// 24-bit integer, split over the two digits its bits fall into (every fp32 number, down
// to the smallest subnormal, is covered).  Integer adds are exact and commute, so the
// accumulated value does not depend on the order in which contributions arrive.
__device__ __forceinline__ void acc_add_exact(long long* acc, float x) {
  const uint32_t b = __float_as_uint(x);
  const int bexp = static_cast<int>((b >> 23) & 0xFFu);
  if ((b & 0x7FFFFFFFu) == 0u || bexp == 0xFF) return;  // zero (Inf/NaN: see the range check)
  const uint32_t m = (b & 0x7FFFFFu) | (bexp ? 0x800000u : 0u);
  const int e = (bexp ? bexp : 1) - 150;                 // x = m 2^e
  const int off = e - kAccBase;                          // >= 0 for every fp32 value
  const int d = off >> 5, r = off & 31;
  const uint64_t w = static_cast<uint64_t>(m) << r;      // < 2^55
  long long lo = static_cast<long long>(w & 0xFFFFFFFFull), hi = static_cast<long long>(w >> 32);
  if (b >> 31) {
    lo = -lo;
    hi = -hi;
  }
  if (lo) atomicAdd(reinterpret_cast<unsigned long long*>(acc + d), static_cast<unsigned long long>(lo));
  if (hi) atomicAdd(reinterpret_cast<unsigned long long*>(acc + d + 1), static_cast<unsigned long long>(hi));
}

// The exact sum held by the digits, rounded to fp64 (a fixed function of the exact value:
// the digits are first brought to their unique normal form, 0 <= d_i < 2^32 below the
// top one, which carries the sign).  The digits are then read from the top down
// (Horner): a negative value has a top digit of -1 above lower digits close to 2^32, and
// adding them from the bottom up would cancel all but the leading bits away; from the top
// the running value stays the exact integer until it is large, then rounds relatively.
__device__ __forceinline__ double acc_value(const long long* acc) {
  long long d[kAccDigits];
#pragma unroll
  for (int i = 0; i < kAccDigits; ++i) d[i] = __ldcg(acc + i);
#pragma unroll
  for (int i = 0; i + 1 < kAccDigits; ++i) {
    const long long carry = d[i] >> 32;  // arithmetic shift: floor division by 2^32
    d[i] -= carry * (1ll << 32);
    d[i + 1] += carry;
  }
  double v = static_cast<double>(d[kAccDigits - 1]);
#pragma unroll
  for (int i = kAccDigits - 2; i >= 0; --i) v = fma(v, 4294967296.0, static_cast<double>(d[i]));
  return ldexp(v, kAccBase);
}

// ------------------------------------------------------------ schedule

// Bounded waits: the budget is in SM clock cycles; a wait that runs out sets bit 0 of
// the status word, and from then on every wait of the launch gives up at once (so a
// lost contribution costs one budget, not one per waiter).
__device__ __forceinline__ bool gave_up(const int* error) {
  return (*reinterpret_cast<const volatile int*>(error) & 1) != 0;
}

__device__ __forceinline__ bool bounded_wait_ge(const int* p, int target, long long budget, int* error) {
  if (ld_acquire_gpu(p) >= target) return true;
  const long long t0 = clock64();
  while (ld_acquire_gpu(p) < target) {
    if (clock64() - t0 > budget || gave_up(error)) {
      atomicOr(error, 1);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

// Bounded wait on a shared-memory word of this CTA.
__device__ __forceinline__ bool bounded_wait_shared(const volatile int* p, int target, long long budget,
                                                    int* error) {
  if (*p == target) return true;
  const long long t0 = clock64();
  while (*p != target) {
    if (clock64() - t0 > budget || gave_up(error)) {
      atomicOr(error, 1);
      return false;
    }
  }
  return true;
}

// ------------------------------------------------------------ the kernel

template <int KG>
__global__ void __launch_bounds__(kReuseThreads, 1) reuse_kernel(const ReuseArgs a) {
  static_assert(KG == 8 || KG == 16, "tensor-core Gram of 8 or 16 workers");
  constexpr int E = tri_count(KG);
  constexpr int U = 4;  // 32-position chunks per warp iteration
  // a CTA's partial is gathered warp by warp: two buffers used by alternate flushes;
  // epoch[b] is the flush number the buffer may take next, arrive[b] the warps in it
  __shared__ float red[2][kStreamWarps][KG * KG];
  __shared__ uint32_t nzred[2][kStreamWarps];
  __shared__ int arrive[2], epoch[2];
  __shared__ df32 Gd[KG][KG];
  __shared__ double zeros[KG];
  __shared__ float tree_sh[tree_scratch_floats(KG)];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x, ncta = gridDim.x;
  if (threadIdx.x < 2) {
    arrive[threadIdx.x] = 0;
    epoch[threadIdx.x] = threadIdx.x;
  }
  __syncthreads();

  if (warp == kStreamWarps) {
    // ------------------------------------------------------------ finisher warp
    if (lane < KG) zeros[lane] = 0.0;
    __syncwarp();
    for (int s = cta; s < a.nsegs; s += ncta) {
      const int want = a.contrib[s];
      if (want == 0) continue;  // empty, or not on this route
      bool ok = true;
      if (lane == 0) ok = bounded_wait_ge(a.count + s, want, a.spin_budget, a.error);
      ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
      (void)ld_acquire_gpu(a.count + s);  // every lane's own acquire of the partial sums
      const SegDesc sd = a.segs[s];
      if (ok) {
        for (int e = lane; e < E; e += 32) {
          int i, j;
          tri_unpack(KG, e, i, j);
          const df32 g = df_from_double(acc_value(a.acc + (static_cast<size_t>(s) * E + e) * kAccDigits));
          Gd[i][j] = g;
          Gd[j][i] = g;
        }
        __syncwarp();
        float c = 0.f;
        bool ill = false;
        const double rel = coefficient_tree_df<KG>(Gd, zeros, kGramRelErr, tree_sh, c, ill);
        // range check (kDiagLoPerPos, kDiagHi): lane k for worker k
        const uint32_t nz = __ldcg(a.seg_nz + s);
        bool oor = false;
        if (lane < KG && ((nz >> lane) & 1u)) {
          const double d = df_to_double(Gd[lane][lane]);
          oor = d < static_cast<double>(sd.len) * kDiagLoPerPos || d > kDiagHi;
        }
        oor = __any_sync(0xFFFFFFFFu, oor);
        if (lane < KG) a.coef[static_cast<size_t>(s) * KG + lane] = c;
        if (lane == 0 && (ill || !(rel <= kRelErrBudget) || oor)) a.seg_flag[s] = 1;
      } else if (lane == 0) {
        a.seg_flag[s] = 1;  // a bounded wait gave up: leave the segment to the recompute
      }
      __threadfence();
      __syncwarp();
      if (lane == 0) st_release_gpu(a.ready + s, 1);
      __syncwarp();
    }
    return;
  }

  // -------------------------------------------------------------- streaming warps
  const int g = lane >> 2, tq = lane & 3;
  const uint16_t* xg = static_cast<const uint16_t*>(a.in[g]);
  const uint16_t* xh = KG == 16 ? static_cast<const uint16_t*>(a.in[g + 8]) : nullptr;
  const bool aligned = a.aligned != 0;
  const uint64_t pol_last = l2_policy_last(), pol_first = l2_policy_first();
  // the open segment's partial (kept across steps until this CTA's last position of it)
  float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
  float e0[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
  uint32_t org = 0u, orh = 0u;
  int pending = 0;
  int nflush = 0;  // this CTA's flushes so far (every streaming warp counts the same)

  for (int si = 0; si < a.nsteps; ++si) {
    const ReuseStep st = a.steps[si];
    int64_t sa, sb;
    reuse_share(st.p0, st.p1, cta, ncta, sa, sb);
    if (sb <= sa) continue;
    if (st.kind == 0) {
      // ---------------------------------------------------------------- Gram step
      for (int s = st.seg_lo; s < st.seg_hi; ++s) {
        const SegDesc sd = a.segs[s];
        if (sd.start >= sb) break;
        const int64_t lo = max(sa, sd.start), hi = min(sb, sd.start + sd.len);
        if (hi <= lo || sd.ntiles == 0) continue;
        if (!ADASUM_CHECK(a.error, sd.start >= 0 && sd.start + sd.len <= a.n_total)) continue;
        const int64_t c0 = lo >> 5, c1 = (hi + 31) >> 5;
        for (int64_t c = c0 + warp; c < c1; c += kStreamWarps * U) {
          uint4 rg[U], rh[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int64_t cu = c + static_cast<int64_t>(u) * kStreamWarps;
            const int64_t v = cu * 4 + tq;
            const uint64_t pol = (cu << 5) >= st.keep_from ? pol_last : pol_first;
            if (cu < c1) {
              rg[u] = load_bf16_policy(xg, v, lo, hi, aligned, pol);
              rh[u] = KG == 16 ? load_bf16_policy(xh, v, lo, hi, aligned, pol) : make_uint4(0u, 0u, 0u, 0u);
            } else {
              rg[u] = make_uint4(0u, 0u, 0u, 0u);
              rh[u] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            org |= vec_or(rg[u]);
            orh |= vec_or(rh[u]);
            mma_bf16_16816(d0, rg[u].x, rh[u].x, rg[u].y, rh[u].y, rg[u].x, rg[u].y);
            mma_bf16_16816(d0, rg[u].z, rh[u].z, rg[u].w, rh[u].w, rg[u].z, rg[u].w);
            if constexpr (KG == 16) {
              mma_bf16_16816(d1, rg[u].x, rh[u].x, rg[u].y, rh[u].y, rh[u].x, rh[u].y);
              mma_bf16_16816(d1, rg[u].z, rh[u].z, rg[u].w, rh[u].w, rh[u].z, rh[u].w);
            }
          }
          if (++pending == 4) {
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
        if (a.flush_step[static_cast<size_t>(s) * ncta + cta] != si) continue;  // more of it later
        // This CTA's last positions of segment s: the warp leaves its partial in the
        // buffer of this flush; the last warp to do so adds the CTA's sum to the exact
        // accumulators and counts the contribution.  No barrier across the warps.
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          kahan_add(s0[i], e0[i], d0[i]);
          kahan_add(s1[i], e1[i], d1[i]);
        }
        const int b = nflush & 1;
        bool ok = true;
        if (a.serial_flush) {
          // (test build) the same sums behind a barrier of the streaming warps
          float* m = red[b][warp];
          const int r0 = g, r1 = g + 8, cA = 2 * tq;
          m[r0 * KG + cA] = __fsub_rn(s0[0], e0[0]);
          m[r0 * KG + cA + 1] = __fsub_rn(s0[1], e0[1]);
          if constexpr (KG == 16) {
            m[r1 * KG + cA] = __fsub_rn(s0[2], e0[2]);
            m[r1 * KG + cA + 1] = __fsub_rn(s0[3], e0[3]);
            m[r0 * KG + 8 + cA] = __fsub_rn(s1[0], e1[0]);
            m[r0 * KG + 8 + cA + 1] = __fsub_rn(s1[1], e1[1]);
            m[r1 * KG + 8 + cA] = __fsub_rn(s1[2], e1[2]);
            m[r1 * KG + 8 + cA + 1] = __fsub_rn(s1[3], e1[3]);
          }
          const uint32_t nzl = warp_or_u32(mma_lane_nz<BF16Tag>(org, orh));
          if (lane == 0) nzred[b][warp] = nzl;
          asm volatile("bar.sync 1, %0;" ::"n"(kStreamThreads) : "memory");
          if (warp == 0) {
            for (int e = lane; e < E; e += 32) {
              int i, j;
              tri_unpack(KG, e, i, j);
              float v = 0.f;
#pragma unroll
              for (int w = 0; w < kStreamWarps; ++w) v = __fadd_rn(v, red[b][w][i * KG + j]);
              acc_add_exact(a.acc + (static_cast<size_t>(s) * E + e) * kAccDigits, v);
            }
            if (lane == 0) {
              uint32_t nz = 0u;
#pragma unroll
              for (int w = 0; w < kStreamWarps; ++w) nz |= nzred[b][w];
              if (nz) atomicOr(a.seg_nz + s, nz);
            }
            __threadfence();
            __syncwarp();
            if (lane == 0) atomicAdd(a.count + s, 1);
          }
          asm volatile("bar.sync 1, %0;" ::"n"(kStreamThreads) : "memory");
          ok = false;  // done
        } else {
          if (lane == 0) ok = bounded_wait_shared(&epoch[b], nflush, a.spin_budget, a.error);
          ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        }
        if (ok) {
          float* m = red[b][warp];
          const int r0 = g, r1 = g + 8, cA = 2 * tq;
          m[r0 * KG + cA] = __fsub_rn(s0[0], e0[0]);
          m[r0 * KG + cA + 1] = __fsub_rn(s0[1], e0[1]);
          if constexpr (KG == 16) {
            m[r1 * KG + cA] = __fsub_rn(s0[2], e0[2]);
            m[r1 * KG + cA + 1] = __fsub_rn(s0[3], e0[3]);
            m[r0 * KG + 8 + cA] = __fsub_rn(s1[0], e1[0]);
            m[r0 * KG + 8 + cA + 1] = __fsub_rn(s1[1], e1[1]);
            m[r1 * KG + 8 + cA] = __fsub_rn(s1[2], e1[2]);
            m[r1 * KG + 8 + cA + 1] = __fsub_rn(s1[3], e1[3]);
          }
          const uint32_t nzl = warp_or_u32(mma_lane_nz<BF16Tag>(org, orh));
          if (lane == 0) nzred[b][warp] = nzl;
          __threadfence_block();
          __syncwarp();
          int last = 0;
          if (lane == 0) last = atomicAdd(&arrive[b], 1) == kStreamWarps - 1;
          last = __shfl_sync(0xFFFFFFFFu, last, 0);
          if (last) {
            __threadfence_block();
            for (int e = lane; e < E; e += 32) {
              int i, j;
              tri_unpack(KG, e, i, j);
              float v = 0.f;
#pragma unroll
              for (int w = 0; w < kStreamWarps; ++w) v = __fadd_rn(v, red[b][w][i * KG + j]);
              acc_add_exact(a.acc + (static_cast<size_t>(s) * E + e) * kAccDigits, v);
            }
            if (lane == 0) {
              uint32_t nz = 0u;
#pragma unroll
              for (int w = 0; w < kStreamWarps; ++w) nz |= nzred[b][w];
              if (nz) atomicOr(a.seg_nz + s, nz);
            }
            __threadfence();
            __syncwarp();
            if (lane == 0) {
              atomicAdd(a.count + s, 1);
              arrive[b] = 0;
              __threadfence_block();
              atomicExch(&epoch[b], nflush + 2);  // the buffer may take flush nflush + 2
            }
            __syncwarp();
          }
        }
        ++nflush;
#pragma unroll
        for (int i = 0; i < 4; ++i) d0[i] = d1[i] = s0[i] = s1[i] = e0[i] = e1[i] = 0.f;
        org = orh = 0u;
        pending = 0;
      }
    } else {
      // ------------------------------------------------------------- combine step
      uint16_t* y = static_cast<uint16_t*>(a.out);
      for (int s = st.seg_hi - 1; s >= st.seg_lo; --s) {
        const SegDesc sd = a.segs[s];
        if (sd.start + sd.len <= sa) {
          if (sd.len > 0) break;
          continue;
        }
        const int64_t lo = max(sa, sd.start), hi = min(sb, sd.start + sd.len);
        if (hi <= lo || sd.ntiles == 0) continue;
        if (!ADASUM_CHECK(a.error, sd.start >= 0 && sd.start + sd.len <= a.n_total)) continue;
        bool ok = true;
        if (lane == 0) ok = bounded_wait_ge(a.ready + s, 1, a.spin_budget, a.error);
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        (void)ld_acquire_gpu(a.ready + s);  // every lane's own acquire of the coefficients
        if (!ok || __ldcg(a.seg_flag + s)) continue;  // left to the recompute path
        float c[KG];
#pragma unroll
        for (int k = 0; k < KG; ++k) c[k] = __ldcg(a.coef + static_cast<size_t>(s) * KG + k);
        const int64_t v0 = lo / 8, v1 = (hi + 7) / 8;
        for (int64_t v = v1 - 1 - threadIdx.x; v >= v0; v -= kStreamThreads) {
          uint4 r[KG];
#pragma unroll
          for (int k = 0; k < KG; ++k)
            r[k] = load_bf16_policy(static_cast<const uint16_t*>(a.in[k]), v, lo, hi, aligned, pol_first);
          float val[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) val[e] = tree_combine<BF16Tag, 0, KG, KG>(c, r, e);
          store_vec<BF16Tag, 8>(y, v * 8, lo, hi, aligned, val);
        }
      }
    }
  }
}

}  // namespace adasum
