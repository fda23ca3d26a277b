// adasum_stream.cuh -- the streaming single-stage kernel (sm_103a): one cooperative
// persistent launch, one CTA per SM, a producer warp that streams tiles into a shared
// memory ring with bulk copies (cp.async.bulk + mbarrier), and eight consumer warps that
// compute Gram partials (tensor cores for bf16 groups of 8 and 16) or combine tiles out
// of shared memory.
//
// Why: the Adasum combine of a segment needs the segment's whole Gram matrix before its
// first output element, so every input byte is read twice.  The second read is cheap
// only if it hits L2, and on GB300 re-reads hit only while the working set between the
// two reads stays under about 64 MB.  The schedule therefore groups segments into small
// waves and gives every CTA the same static interleave:
//     Gram tiles of wave w,  then combine tiles of wave w-1 (newest first),  ...
// so a tile's second read comes about one wave after its first.  The producer keeps
// loading across task boundaries, so the consumers never wait on a cold pipeline.
//
// Status: correct (parity and determinism tests pass on GB300) but not yet fast: on
// the BERT-Large K=16 set it runs at 4-5x the time of the three-kernel route, because a
// CTA's share of one wave is only ~100 KB while each segment costs it a partial flush
// and each combine task waits for the segment's coefficients, which the last-arriving
// CTA computes on the critical path.  It is selected only with ADASUM_ROUTE=stream.
//
// Determinism: the schedule is static, each CTA accumulates its tiles of a segment in a
// fixed order and writes one partial per (segment, CTA); the CTA whose partial completes
// a segment (last arriver) sums the partials in a fixed CTA order, runs the fp64
// coefficient tree and publishes the coefficients with a release store.  Combine tiles
// wait for that flag with acquire loads under a clock budget (never an unbounded spin).
#pragma once

#include "adasum_kernels.cuh"
#include "adasum_ptx.cuh"

namespace adasum {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kStreamThreads = kConsumers + 32;  // warp 0 produces, warps 1..8 consume
constexpr int kStages = 3;
constexpr int kRowPad = 64;                      // bytes between rows: spreads smem banks

// Arguments of the streaming kernel beyond StageArgs.
struct StreamArgs {
  const int* task_ptr;      // [G+1] CSR offsets of each CTA's task list
  const int* tasks;         // tile id (Gram) or tile id | 0x80000000 (combine)
  const int* seg_c0;        // [nsegs] CTA of each segment's first tile (round robin)
  float* slots;             // [nsegs][E][G] per-(segment, CTA) Gram partials (entry-major)
  int* seg_count;           // [nsegs] tiles accumulated so far
  int* seg_ready;           // [nsegs] coefficients published
  int* error;               // device status word
  long long spin_budget;    // clock64 cycles of any single wait
  int stage_pos;            // positions per stage (P)
  int row_bytes;            // bytes per smem row (P * element size + kRowPad)
  int inject_no_ready;      // test hook: never publish
};

// Barrier among the consumer warps only (the producer warp never joins it).
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}
// Consumer barrier that also returns the AND of `ok` over all consumer threads, so a
// wait that gave up in one thread stops every consumer at the same point.
__device__ __forceinline__ bool consumers_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, %2, p;\n"
      " selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(ok ? 1u : 0u), "n"(kConsumers)
      : "memory");
  return r != 0;
}

// Bounded wait (one thread) for a segment's published coefficients: 1 when published.
__device__ __forceinline__ int wait_ready_stream(const StreamArgs& s, int seg) {
  if (ld_acquire_gpu(s.seg_ready + seg)) return 1;
  const long long t0 = clock64();
  for (;;) {
    __nanosleep(64);
    if (ld_acquire_gpu(s.seg_ready + seg)) return 1;
    if (clock64() - t0 > s.spin_budget) {
      atomicOr(s.error, 1);
      return 0;
    }
  }
}

// ------------------------------------------------------------------ producer

// Loads tile `tile_id` into a stage: rows k = 0..Kg-1, row k holds positions
// [b, b + P) of worker k, b = 32-aligned start of the tile.  The 16-byte-aligned interior
// goes by bulk copy; the ragged ends and, for Gram tiles, the zero padding up to the
// tile's 32-position chunk boundaries are written by the producer lanes.
template <typename Tag, int KG>
__device__ __forceinline__ void produce_tile(const StageArgs& a, const StreamArgs& s, int tile_id,
                                             bool gram, char* stage, uint64_t* full) {
  using S = typename ElemTraits<Tag>::Storage;
  constexpr int ES = sizeof(S);
  constexpr int VW = 16 / ES;
  const int lane = threadIdx.x & 31;
  const TileDesc t = a.tiles[tile_id];
  const int64_t lo = t.start, hi = t.start + t.len;
  const int64_t b = lo & ~int64_t(31);
  int64_t lo16 = (lo + VW - 1) / VW * VW, hi16 = hi / VW * VW;
  if (!a.aligned || hi16 <= lo16) {
    lo16 = hi;  // no bulk part: everything by hand
    hi16 = hi;
  }
  // ragged ends and zero padding
  const int64_t z0 = gram ? b : lo;                       // chunk-aligned span for Gram tiles
  const int64_t z1 = gram ? ((hi + 31) & ~int64_t(31)) : hi;
  for (int k = 0; k < KG; ++k) {
    const S* src = static_cast<const S*>(a.in[k]);
    S* row = reinterpret_cast<S*>(stage + k * s.row_bytes);
    for (int64_t p = z0 + lane; p < lo16; p += 32) row[p - b] = (p >= lo) ? src[p] : S(0);
    for (int64_t p = hi16 + lane; p < z1; p += 32) row[p - b] = (p < hi) ? src[p] : S(0);
  }
  __syncwarp();
  if (lane == 0) {
    const uint32_t bytes = static_cast<uint32_t>((hi16 - lo16) * ES);
    mbar_arrive_expect_tx(full, bytes * KG);
    if (bytes > 0)
      for (int k = 0; k < KG; ++k)
        bulk_g2s(stage + k * s.row_bytes + (lo16 - b) * ES,
                 static_cast<const S*>(a.in[k]) + lo16, bytes, full);
  }
}

// ------------------------------------------------------------------ consumers: Gram

// Per-warp Gram accumulators of the current segment.
struct GramAcc {
  float d0[4], d1[4], s0[4], s1[4], e0[4], e1[4];
  int pending;
  __device__ void clear() {
#pragma unroll
    for (int i = 0; i < 4; ++i) d0[i] = d1[i] = s0[i] = s1[i] = e0[i] = e1[i] = 0.f;
    pending = 0;
  }
  __device__ void fold() {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      kahan_add(s0[i], e0[i], d0[i]);
      kahan_add(s1[i], e1[i], d1[i]);
      d0[i] = 0.f;
      d1[i] = 0.f;
    }
    pending = 0;
  }
};

// Tensor-core Gram of one staged bf16 tile (Kg = 8 or 16), accumulated into `acc`.
// Chunk c of 32 positions: lane (g, t) reads 16 bytes of rows g and g+8 at 8t; the
// fragment mapping is the one of gram_tile_mma (the Gram matrix is a sum over
// positions, so any position order common to all rows works).
template <int KG>
__device__ __forceinline__ void consume_gram_mma(const TileDesc& t, const char* stage, int row_bytes,
                                                 GramAcc& acc) {
  const int lane = threadIdx.x & 31, cw = (threadIdx.x >> 5) - 1;
  const int g = lane >> 2, tq = lane & 3;
  const int64_t b = t.start & ~int64_t(31);
  const int nch = static_cast<int>(((t.start + t.len + 31) & ~int64_t(31)) - b) >> 5;
  const char* rg = stage + g * row_bytes;
  const char* rh = stage + (g + 8) * row_bytes;
  for (int c = cw; c < nch; c += kConsumerWarps) {
    const uint4 x = *reinterpret_cast<const uint4*>(rg + c * 64 + tq * 16);
    const uint4 y = KG == 16 ? *reinterpret_cast<const uint4*>(rh + c * 64 + tq * 16)
                             : make_uint4(0u, 0u, 0u, 0u);
    mma_bf16_16816(acc.d0, x.x, y.x, x.y, y.y, x.x, x.y);
    mma_bf16_16816(acc.d0, x.z, y.z, x.w, y.w, x.z, x.w);
    if constexpr (KG == 16) {
      mma_bf16_16816(acc.d1, x.x, y.x, x.y, y.y, y.x, y.y);
      mma_bf16_16816(acc.d1, x.z, y.z, x.w, y.w, y.z, y.w);
    }
    if (++acc.pending == 16) acc.fold();
  }
}

// CUDA-core Gram of one staged tile: every consumer thread owns whole 16-byte vectors.
template <typename Tag, int KG>
__device__ __forceinline__ void consume_gram_simt(const TileDesc& t, const char* stage, int row_bytes,
                                                  float (&acc)[tri_count(KG)]) {
  using S = typename ElemTraits<Tag>::Storage;
  constexpr int VW = ElemTraits<Tag>::kVW;
  const int64_t b = t.start & ~int64_t(31);
  const int nv = static_cast<int>((((t.start + t.len + 31) & ~int64_t(31)) - b) / VW);
  for (int v = threadIdx.x - 32; v < nv; v += kConsumers) {
    uint4 r[KG];
#pragma unroll
    for (int k = 0; k < KG; ++k) r[k] = *reinterpret_cast<const uint4*>(stage + k * row_bytes + v * 16);
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

// ------------------------------------------------------------------ consumers: finisher

// The CTA whose partial completes segment `seg`: sum the contributing CTAs' partials in
// a fixed order, run the coefficient tree, publish.  Consumer warps only.
template <int KG>
__device__ __forceinline__ void finish_segment(const StageArgs& a, const StreamArgs& s, int seg) {
  constexpr int E = tri_count(KG);
  __shared__ df32 G[KG][KG];
  __shared__ double eps[KG];
  __shared__ float tree_sh[tree_scratch_floats(KG)];
  const int ct = threadIdx.x - 32, lane = threadIdx.x & 31, cw = (threadIdx.x >> 5) - 1;
  const SegDesc sd = a.segs[seg];
  const int nctas = static_cast<int>(gridDim.x);
  const int ncontrib = sd.ntiles < nctas ? sd.ntiles : nctas;
  const int c0 = s.seg_c0[seg];
  // warp cw sums entries cw, cw+8, ...: lane l takes contributors l, l+32, ... (all its
  // loads issued together), then a fixed butterfly -- the same order on every run
  constexpr int kMaxPerLane = 8;  // up to 256 CTAs
  for (int e = cw; e < E; e += kConsumerWarps) {
    const float* row = s.slots + (static_cast<size_t>(seg) * E + e) * nctas;
    float v[kMaxPerLane];
#pragma unroll
    for (int r = 0; r < kMaxPerLane; ++r) {
      const int j = lane + 32 * r;
      v[r] = j < ncontrib ? __ldcg(row + (c0 + j) % nctas) : 0.f;
    }
    double sum = 0.0;
#pragma unroll
    for (int r = 0; r < kMaxPerLane; ++r) sum += static_cast<double>(v[r]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
    if (lane == 0) {
      int i, jj;
      tri_unpack(KG, e, i, jj);
      G[i][jj] = G[jj][i] = df_from_double(sum);
    }
  }
  for (int k = ct; k < KG; k += kConsumers) eps[k] = 0.0;
  consumers_sync();
  if (ct < 32) {
    float c = 0.f;
    bool ill = false;
    const double rel = coefficient_tree_df<KG>(G, eps, kGramRelErr, tree_sh, c, ill);
    if (ct < KG) a.coef[static_cast<size_t>(seg) * KG + ct] = static_cast<float>(c);
    if (ct == 0) {
      if (a.relerr) a.relerr[seg] = static_cast<float>(fmin(rel, 1e30));
      if (ill || !(rel <= kRelErrBudget)) a.seg_flag[seg] = 1;
      __threadfence();
      if (!s.inject_no_ready) st_release_gpu(s.seg_ready + seg, 1);
    }
  }
  consumers_sync();
}

// Writes this CTA's accumulated partial of `seg` (ntiles of its tiles) and, when it
// completes the segment, finishes it.  Consumer warps only.
template <typename Tag, int KG, bool MMA>
__device__ __forceinline__ void flush_segment(const StageArgs& a, const StreamArgs& s, int seg, int ntiles,
                                              GramAcc& acc, float (&simt)[tri_count(KG)]) {
  constexpr int E = tri_count(KG);
  constexpr int RED = MMA ? KG * KG : E;
  __shared__ float red[kConsumerWarps][RED];
  __shared__ int last;
  const int lane = threadIdx.x & 31, cw = (threadIdx.x >> 5) - 1, ct = threadIdx.x - 32;
  if constexpr (MMA) {
    acc.fold();
    const int g = lane >> 2, cA = 2 * (lane & 3);
    red[cw][g * KG + cA] = __fsub_rn(acc.s0[0], acc.e0[0]);
    red[cw][g * KG + cA + 1] = __fsub_rn(acc.s0[1], acc.e0[1]);
    if constexpr (KG == 16) {
      red[cw][(g + 8) * KG + cA] = __fsub_rn(acc.s0[2], acc.e0[2]);
      red[cw][(g + 8) * KG + cA + 1] = __fsub_rn(acc.s0[3], acc.e0[3]);
      red[cw][g * KG + 8 + cA] = __fsub_rn(acc.s1[0], acc.e1[0]);
      red[cw][g * KG + 8 + cA + 1] = __fsub_rn(acc.s1[1], acc.e1[1]);
      red[cw][(g + 8) * KG + 8 + cA] = __fsub_rn(acc.s1[2], acc.e1[2]);
      red[cw][(g + 8) * KG + 8 + cA + 1] = __fsub_rn(acc.s1[3], acc.e1[3]);
    }
    acc.clear();
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      float v = simt[e];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
      if (lane == 0) red[cw][e] = v;
      simt[e] = 0.f;
    }
  }
  consumers_sync();
  float* slot = s.slots + static_cast<size_t>(seg) * E * gridDim.x + blockIdx.x;
  for (int idx = ct; idx < RED; idx += kConsumers) {
    int e = idx;
    if constexpr (MMA) {
      const int i = idx / KG, j = idx % KG;
      if (j < i) continue;
      e = tri_index(KG, i, j);
    }
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) sum = __fadd_rn(sum, red[w][idx]);
    slot[static_cast<size_t>(e) * gridDim.x] = sum;
  }
  __threadfence();
  consumers_sync();
  if (ct == 0) last = atomicAdd(s.seg_count + seg, ntiles) + ntiles == a.segs[seg].ntiles;
  consumers_sync();
  if (last) {
    __threadfence();
    finish_segment<KG>(a, s, seg);
  }
}

// ------------------------------------------------------------------ consumers: combine

template <typename InTag, typename OutTag, int KG, bool MOM>
__device__ __forceinline__ void consume_combine(const StageArgs& a, const TileDesc& t, const char* stage,
                                                int row_bytes, const float (&c)[KG]) {
  using SO = typename ElemTraits<OutTag>::Storage;
  constexpr int VW = ElemTraits<InTag>::kVW;
  const bool aligned = a.aligned != 0;
  SO* y = static_cast<SO*>(a.out[0]);
  const int64_t lo = t.start, hi = t.start + t.len;
  const int64_t b = lo & ~int64_t(31);
  const int64_t v0 = lo / VW, v1 = (hi + VW - 1) / VW;
  for (int64_t v = v0 + (threadIdx.x - 32); v < v1; v += kConsumers) {
    const int off = static_cast<int>(v * VW - b) * static_cast<int>(sizeof(typename ElemTraits<InTag>::Storage));
    uint4 r[KG];
#pragma unroll
    for (int k = 0; k < KG; ++k) r[k] = *reinterpret_cast<const uint4*>(stage + k * row_bytes + off);
    float val[VW];
#pragma unroll
    for (int e = 0; e < VW; ++e) val[e] = tree_combine<InTag, 0, KG, KG>(c, r, e);
    const int64_t p0 = v * VW;
    if constexpr (MOM) {
      float wv[VW], mv[VW];
      load_f32_vec<VW>(a.momentum, p0, lo, hi, aligned, mv);
      load_f32_vec<VW>(a.master_w, p0, lo, hi, aligned, wv);
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        mv[e] = __fmaf_rn(a.mu, mv[e], val[e]);
        wv[e] = __fmaf_rn(-a.lr, mv[e], wv[e]);
      }
      store_vec<F32Tag, VW>(a.momentum, p0, lo, hi, aligned, mv);
      store_vec<F32Tag, VW>(a.master_w, p0, lo, hi, aligned, wv);
      if (y != nullptr) store_vec<OutTag, VW>(y, p0, lo, hi, aligned, val);
    } else {
      store_vec<OutTag, VW>(y, p0, lo, hi, aligned, val);
    }
  }
}

// ------------------------------------------------------------------ the kernel

template <typename InTag, int KG, bool MOM>
__global__ void __launch_bounds__(kStreamThreads, 1) stream_kernel(const StageArgs a, const StreamArgs s) {
  constexpr bool kMMA = ElemTraits<InTag>::kVW == 8 && (KG == 8 || KG == 16);
  extern __shared__ __align__(128) char smem[];
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
  __shared__ float coef_sh[KG];
  __shared__ int seg_ok;   // coefficients published and the segment not flagged
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int stage_bytes = KG * s.row_bytes;
  const int t0 = s.task_ptr[blockIdx.x], t1 = s.task_ptr[blockIdx.x + 1];

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ---------------- producer
    int n_issued = 0;
    for (int i = t0; i < t1; ++i) {
      const int n = i - t0, st = n % kStages;
      if (n >= kStages) {
        // lane 0 waits; the whole warp follows its verdict
        int ok = 1;
        if (lane == 0) ok = mbar_wait(&empty[st], ((n / kStages) - 1) & 1, s.spin_budget, s.error);
        if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
      }
      const int task = s.tasks[i];
      produce_tile<InTag, KG>(a, s, task & 0x7FFFFFFF, task >= 0, smem + st * stage_bytes, &full[st]);
      n_issued = n + 1;
    }
    // Do not leave while bulk copies into this CTA's shared memory are in flight: the
    // last kStages stages were all issued by this warp; wait (bounded) for each.
    if (lane == 0)
      for (int n = n_issued - kStages > 0 ? n_issued - kStages : 0; n < n_issued; ++n)
        mbar_wait(&full[n % kStages], (n / kStages) & 1, s.spin_budget, s.error);
    return;
  }

  // ---------------- consumers
  GramAcc acc;
  acc.clear();
  float simt[tri_count(KG)];
#pragma unroll
  for (int e = 0; e < tri_count(KG); ++e) simt[e] = 0.f;
  int cur_seg = -1, cur_n = 0;   // Gram segment being accumulated and its tile count
  int coef_seg = -1;             // segment whose coefficients are in coef_sh
  float c[KG];
#pragma unroll
  for (int k = 0; k < KG; ++k) c[k] = 0.f;
  for (int i = t0; i < t1; ++i) {
    const int n = i - t0, st = n % kStages;
    const int task = s.tasks[i];
    const bool gram = task >= 0;
    const int tile_id = task & 0x7FFFFFFF;
    const TileDesc t = a.tiles[tile_id];
    if (!consumers_all(mbar_wait(&full[st], (n / kStages) & 1, s.spin_budget, s.error))) break;
    const char* stage = smem + st * stage_bytes;
    if (gram) {
      if constexpr (kMMA) consume_gram_mma<KG>(t, stage, s.row_bytes, acc);
      else consume_gram_simt<InTag, KG>(t, stage, s.row_bytes, simt);
      ++cur_n;
      cur_seg = t.seg;
    } else {
      // one thread waits for the segment and reads its flag and coefficients; the
      // decision is then taken by every consumer from shared memory, uniformly
      if (t.seg != coef_seg) {
        if (threadIdx.x == 32) {
          const int ok = wait_ready_stream(s, t.seg);
          seg_ok = ok && !__ldcg(a.seg_flag + t.seg);
          for (int k = 0; k < KG; ++k) coef_sh[k] = __ldcg(a.coef + static_cast<size_t>(t.seg) * KG + k);
        }
        consumers_sync();
#pragma unroll
        for (int k = 0; k < KG; ++k) c[k] = coef_sh[k];
        coef_seg = t.seg;
      }
      if (seg_ok) consume_combine<InTag, InTag, KG, MOM>(a, t, stage, s.row_bytes, c);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    // flush the Gram partial when the next task is not a Gram tile of the same segment
    if (gram) {
      bool next_same = false;
      if (i + 1 < t1) {
        const int nt = s.tasks[i + 1];
        next_same = nt >= 0 && a.tiles[nt].seg == cur_seg;
      }
      if (!next_same) {
        flush_segment<InTag, KG, kMMA>(a, s, cur_seg, cur_n, acc, simt);
        cur_n = 0;
        cur_seg = -1;
      }
    }
  }
}

}  // namespace adasum
