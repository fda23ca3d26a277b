// adasum_internal.h -- declarations shared by the host side (adasum_api.cu) and the
// kernel translation units of the GB300 Adasum library.  Not part of the public ABI.
//
// Method ("Scaling Distributed Training with Adaptive Summation", Section 3): per layer
// segment, K worker gradients are combined by a binary tree of the pair operator
//     Adasum(a, b) = (1 - a.b/(2|a|^2)) a + (1 - a.b/(2|b|^2)) b.
// Every node of the tree is a linear combination of the leaves, so the whole tree
// result is  out = sum_k c_k g_k,  and every dot product the tree needs is a quadratic
// form in the segment's Gram matrix G_ij = g_i . g_j.  The library therefore runs
//   pass 1  Gram partials per tile          (one read of the K inputs)
//   coef    per segment: reduce partials, run the tree on G in fp64 -> c_0..c_{K-1}
//   pass 2  out = sum_k c_k g_k per tile     (second read of the K inputs, one write)
// which is the same tree, in the same order, evaluated in coefficient space.  Groups
// of at most 16 workers form one stage; larger K runs stages of 16-leaf subtrees whose
// fp32 results feed the next stage (the tree's top levels).
#pragma once

#include <cstdint>

namespace adasum {

// Bits of the device status word (adasum_get_last_error): a bounded wait gave up, or
// (test build only) an index check failed.
constexpr int kErrTimeoutMask = 0xF;
constexpr int kErrBounds = 0x10;

// Device-side index checks, compiled in with -DADASUM_BOUNDS_CHECK (the test build): a
// failed check sets kErrBounds in the status word and the caller skips the access.  It
// never traps.  Without the flag every check is `true` and costs nothing.
#ifdef ADASUM_BOUNDS_CHECK
#define ADASUM_CHECK(err, cond) ((cond) ? true : (atomicOr((err), kErrBounds), false))
#else
#define ADASUM_CHECK(err, cond) true
#endif

constexpr int kMaxK = 256;        // largest worker count accepted
constexpr int kMaxGroup = 16;     // workers combined in one Gram stage
constexpr int kThreads = 256;     // threads per CTA of the tile kernels

enum Dtype : int { kF32 = 0, kBF16 = 1 };

// One tile: a contiguous run of positions inside one segment.
struct TileDesc {
  int64_t start;   // first position (absolute index into the flat gradient)
  int32_t len;     // positions in the tile (> 0)
  int32_t seg;     // owning segment
};

// One segment (layer) of the flat gradient.
struct SegDesc {
  int64_t start;
  int64_t len;
  int32_t first_tile;   // index of its first tile
  int32_t ntiles;       // 0 for an empty segment
  int32_t first_chunk;  // its tiles' partial Gram matrices are summed in chunks
  int32_t nchunks;
};

// A run of at most kChunkTiles consecutive tiles of one segment.
struct ChunkDesc {
  int32_t first_tile;
  int32_t ntiles;
};
constexpr int kChunkTiles = 32;
// Tiles of at most this many positions get their Gram partial, and with groups of 8 or
// more workers their combine, from one warp: 16-worker groups (the tensor-core warp
// Gram) with fp32 / bf16 inputs, and smaller groups (the SIMT warp Gram).  Measured on a
// layout of 10,000 segments of 1..4096 positions: 512 and 2048 against 1024 took fp32
// K = 64 from 0.900 to 0.889 ms and bf16 K = 64 from 0.876 to 0.864 ms; 2048 made bf16
// K = 8 slower (0.124 -> 0.135 ms).
constexpr int kSmallTileF32 = 512;
// 256-thread CTAs per SM, for each of grid.y's groups, of the short-tile combine's grid, whose
// warps loop over the tiles (each warp takes every W-th tile).  Measured on the
// 10,000-segment layout against one CTA per eight tiles: fp32 K = 64 0.768 -> 0.764 ms,
// bf16 K = 64 0.758 -> 0.733 ms.  8 per SM gained less (0.766 ms).  A single wave of
// the CTAs that fit, for the combine and the warp Grams alike, measured 0.801 ms: with
// 15 tiles of unequal length per warp, warps sat idle at the end.  The warp Grams keep one
// CTA per eight tiles.  The CTAs are two warps (kCombineWarpThreads; the grid holds as
// many warps as four 256-thread CTAs per SM), so a warp that has run out of tiles holds
// its registers only until its one sibling is done: fp32 K = 64 0.768 -> 0.762 ms, bf16
// K = 64 0.727 -> 0.696 ms against eight-warp CTAs; one-warp CTAs measured the same.
constexpr int kWarpTileCtasPerSm = 4;
constexpr int kCombineWarpThreads = 64;
inline int warp_tile_grid(int ntiles, int num_sms) {
  const int wpb = kCombineWarpThreads / 32;
  const int need = (ntiles + wpb - 1) / wpb;
  const int cap = kWarpTileCtasPerSm * (kThreads / kCombineWarpThreads) * (num_sms > 0 ? num_sms : 1);
  return need < cap ? need : cap;
}
constexpr int kSmallTileBF16 = 2048;
constexpr int kSmallTileSimt = 1024;

// Arguments of one stage: G independent groups of Kg workers each, over the same
// segments and tiles.  Group q reads in[q*Kg + k], k < Kg, and writes out[q].
struct StageArgs {
  const void* in[kMaxK];
  void* out[kMaxK / kMaxGroup];
  int64_t n_total;   // positions of every input and output (bounds checks)
  int* error;        // device status word (bounds checks)
  int Kg;          // workers per group: 1, 2, 4, 8 or 16
  int G;           // groups
  int aligned;     // every in/out pointer is 16-byte aligned
  int ntiles;
  int nsegs;
  int nchunks;
  const TileDesc* tiles;
  const SegDesc* segs;
  const ChunkDesc* chunks;
  float* partials;   // [G][ntiles][E] Gram partials, E = Kg(Kg+1)/2 (upper triangle)
  float2* chunk_sums; // [G][nchunks][E] compensated sums of the partials of each chunk, as
                      //   double-float (hi, lo) pairs (chunks of multi-chunk segments only)
  const int* multi_chunks;  // the chunks of segments with more than one chunk
  int nmulti;
  // Range check of the fp32 pass (kDiagLoPerPos, kDiagHi): bit k set when worker k has a
  // nonzero value in the tile / chunk (-0 counts as zero).
  uint32_t* tile_nz;   // [G][ntiles]
  uint32_t* chunk_nz;  // [G][nchunks] (chunks of multi-chunk segments only)
  float* coef;       // [G][nsegs][Kg] tree coefficients
  // Fused heavy-ball step (final stage of adasum_reduce_momentum_sgd only).
  float* master_w;
  float* momentum;
  float lr;
  float mu;

  // Conditioning check and fp64 recompute (see coef_kernel).
  int* seg_flag;              // [nsegs] 1: the segment is recomputed in fp64
  float* relerr;              // [G][nsegs] estimated relative error of this stage's output
  const float* in_relerr;     // [G*Kg][nsegs] same, of this stage's inputs (null = exact)
  int skip_flagged;           // combine: leave flagged segments to the fp64 path
  const int* seg_list;        // coef: the segments to run (null: all nsegs)
  int nseg_list;
  const int* tile_list;       // Gram CTA kernels: the tiles to run (null: all ntiles)
  int ntile_list;
  const int* small_list;      // small tiles, one warp each (gram_warp_kernel); null when
                              // every tile is small (entry i is then tile i)
  int nsmall;
  int combine_tiles;          // consecutive tiles per combine CTA (>= 1; up to 4 while the
                              //   grid keeps 16 CTAs per SM)
  int num_sms;                // SMs of the device (launch shapes)

  // fp64 path (only the segments listed by collect_kernel).
  double* partials64;         // [G][ntiles][E]
  double* coef64;             // [G][nsegs][Kg]
  int* list_tiles;            // flagged tiles, list_count[0] of them
  int* list_segs;             // flagged segments, list_count[1] of them
  int* list_tiny;             // flagged segments of at most kTinySeg positions, list_count[2]
  int* list_count;            // [3]
  int* seg_exp;               // [nsegs] 1024 + exponent of the segment's largest |input| (0: all zero)
  // Flagged segments that fit the on-chip kernel's clusters of oc_cmax CTAs (plain
  // reductions of up to 64 workers) are listed for its recompute instead of the fp64 path.
  int oc_vecs;                // 16-byte vectors per CTA (0: none go there)
  int oc_vw;                  // elements per 16-byte vector
  int oc_cmax;                // cluster size of the recompute launch
  int* oc_list;               // [nsegs]
  int* oc_count;              // [1]
  int Ktotal;                 // all workers (the tiny-segment recompute runs the whole tree)
  int in_f64;                 // stage inputs are fp64 intermediates
  int out_f64;                // stage outputs are fp64 intermediates

  // Combination order: kModeTree (binary tree, pairs (2i, 2i+1) per level) or kModeChain
  // (g[0,k] = Adasum(g[0,k-1], g_k), left to right).  Kreal workers are real; a null
  // input pointer is a zero gradient (worker counts are padded to a power of two with
  // them, which is exact: an unpaired node meets a zero node and Adasum(x, 0) = x).
  int mode;
  int Kreal;

  // Orthogonality metric (optional): |A|^2 of the final stage per segment, and the sum of
  // the first stage's Gram diagonals per (group, segment).
  double* outnorm2;           // [nsegs], final stage only
  double* diag_sum;           // [G][nsegs], first stage only
};
enum Mode : int { kModeTree = 0, kModeChain = 1 };

// Gram-entry error model of the fp32 pass, relative to |g_i| |g_j|: products and
// bounded-length fp32 sums, then compensated sums (a typical-case constant).
constexpr double kGramRelErr = 4.0 * 5.9604644775390625e-08;   // 4 u, u = 2^-24
// Range of the fp32 pass.  Products are exact in the Gram kernels except below 2^-126,
// where a product may be flushed to zero (the tensor cores) or rounded to a subnormal:
// at most n 2^-126 over a segment of n positions.  For every nonzero worker k the fp32
// pass therefore needs its squared norm G_kk >= n 2^-96, which keeps what may be lost
// below 2^-30 G_kk (and a worker whose squares all vanish, G_kk = 0, is still seen, by
// its nonzero bit); and G_kk <= 2^80, which keeps every product and partial sum far from
// fp32's overflow.  A segment outside is flagged like an ill-conditioned one and
// recomputed by a path that scales by a power of two first.
constexpr double kDiagLoPerPos = 0x1p-96;
constexpr double kDiagHi = 0x1p80;
// Estimated relative output error above which a segment is recomputed in fp64.  The
// estimate is a conservative first-order bound: over random, correlated and nearly
// cancelling test sets the realised error of the fp32 pass stayed below 0.16 times it,
// so an estimate of 2.5e-5 keeps the realised error below 4e-6.
constexpr double kRelErrBudget = 2.5e-5;
// Factor on the measured coefficient error (coefficient_probe) where it replaces the
// bound: the measurement follows one direction of the error model at a time, so it is
// taken 4x.  Over random, correlated, parallel and partly cancelling sets the realised
// error stayed below 0.08 times the resulting estimate.
constexpr float kProbeSafety = 4.f;
// Flagged segments of at most this many positions are recomputed in vector space (the
// tree level by level on the values themselves, one warp per segment): there, nodes can
// cancel almost exactly, which a Gram-matrix quadratic form cannot follow even in fp64.
constexpr int kTinySeg = 32;

// Small-segment kernel (adasum_onchip.cuh): one segment per CTA or thread-block cluster,
// its K x n block held in shared memory, the whole tree evaluated on chip.
constexpr int kOnchipMaxK = 64;
// Shared memory per CTA for the block: K rows of P positions of 4 bytes each.
constexpr int kOnchipDataBytes = 80 * 1024;
__host__ __device__ constexpr int onchip_positions(int K) { return kOnchipDataBytes / (4 * K); }

struct OnchipArgs {
  const void* in[kOnchipMaxK];  // K leaves (K a power of two); null = a zero gradient
  void* out;
  const SegDesc* segs;
  const int* list;              // the segments of this launch, taken in turn by its clusters
  int P;                        // positions per CTA, onchip_positions(K)
  int aligned;                  // every in/out pointer is 16-byte aligned
  int* error;                   // device status word (bit 2: a bulk-copy wait gave up)
  int64_t n_total;              // positions of every input and the output (bounds checks)
  int* recomputed;              // segments recomputed in double-float
  long long spin_budget;        // clock64 cycles of the bulk-copy wait
  int inject_extra_tx;          // test hook: expect 16 bytes that never arrive
  const int* dev_count;         // when set: the list's length (else one entry per cluster)
  int recompute_only;           // skip the fp32 pass (segments the fp32 pass flagged)
};

// Two workers, one segment (adasum_pair.cuh): one cooperative kernel with one grid
// barrier, double-float sums and combine, every thread holding up to kPairVecs 16-byte
// vectors of each input in registers; segments of up to min(co-resident CTAs,
// kPairThreads) * kPairThreads * kPairVecs vectors.
constexpr int kPairThreads = 512;
constexpr int kPairVecs = 4;
struct PairArgs {
  const void* a;
  const void* b;
  void* out;                    // may be a or b
  int64_t n;
  int aligned;                  // a, b and out are 16-byte aligned
  float* partials;              // [grid][8]: each CTA's double-float sums and exponent
  unsigned* bar;                // [2]: grid barrier (arrivals, generation), zero when allocated
  int* error;                   // device status word (bit 8: the grid barrier gave up)
  long long spin_budget;        // clock64 cycles of the barrier wait
  int inject_no_arrival;        // test hook: wait at the barrier without arriving
};

// Segments of at most kTinyDirect positions (adasum_onchip.cuh): a warp or a lane group
// each, the tree on the values themselves in double-float arithmetic.
constexpr int kTinyDirect = 32;
struct TinyArgs {
  const void* in[kMaxK];  // K leaves (K a power of two); null = a zero gradient
  void* out;
  const SegDesc* segs;
  const int* list;        // the segments: count8 of <= 8 positions, then count16 of <= 16,
                          // then the rest
  int count;
  int count8, count16;
  int K;
  int64_t n_total;        // positions of every input and the output (bounds checks)
  int* error;             // device status word (bounds checks)
};

// Launchers, one translation unit per input element type (compiled in parallel).
// Each enqueues one kernel on `stream` and returns its cudaError_t as int (0 = ok);
// `name` receives a static string naming the kernel, for the optional profiler.
int launch_gram_f32(const StageArgs& a, void* stream, const char** name);
int launch_gram_bf16(const StageArgs& a, void* stream, const char** name);
// Gram partials of a.small_list's tiles, one warp per (tile, group).
int launch_gram_warp(const StageArgs& a, int in_dtype, void* stream, const char** name);
int launch_coef(const StageArgs& a, void* stream, const char** name);
int launch_combine_f32in(const StageArgs& a, int out_dtype, int momentum, int warp, void* stream,
                         const char** name);
int launch_combine_bf16in(const StageArgs& a, int out_dtype, int momentum, int warp, void* stream,
                          const char** name);
// Partial-Gram chunk sums (segments with many tiles), then coefficients.
int launch_reduce_chunks(const StageArgs& a, void* stream, const char** name);
// Small-segment kernel: `count` clusters of C CTAs over a.list[0..count).
int launch_onchip(const OnchipArgs& a, int dtype, int K, int count, int C, void* stream,
                  const char** name);
// Largest cluster size (1..16, a power of two) the small-segment kernel can run with.
int onchip_max_cluster(int dtype, int K);
int onchip_resident_clusters(int dtype, int K, int C);
// CTAs of the fused pair kernel that fit on the current device at once (0: none).
int pair_fused_max_grid(int dtype);
int launch_pair_fused(const PairArgs& a, int dtype, int grid, void* stream, const char** name);
// Tiny segments (the warp kernel).
int launch_tiny_df(const TinyArgs& a, int dtype, void* stream, const char** name);
// fp64 path: build the flagged lists, then Gram / coefficients / combine over them.
int launch_collect(const StageArgs& a, int grid, void* stream, const char** name);
// v = mu v + g for one worker (grad in `dtype`, state fp32).
int launch_local_momentum(const void* g, int dtype, float* v, int64_t n, float mu, int aligned,
                          int num_sms, void* stream, const char** name);
// ortho[s] = outnorm2[s] / sum_q diag_sum[q][s] (NaN when the sum is 0).
int launch_orthogonality(const double* outnorm2, const double* diag_sum, int groups, int nsegs,
                         float* ortho, void* stream, const char** name);
int launch_tiny64(const StageArgs& a, int in_dtype, int out_dtype, int momentum, int grid,
                  void* stream, const char** name);
int launch_segmax(const StageArgs& a, int in_dtype, int grid, void* stream, const char** name);
int launch_gram64(const StageArgs& a, int in_dtype, int grid, void* stream, const char** name);
int launch_coef64(const StageArgs& a, int grid, void* stream, const char** name);
int launch_combine64(const StageArgs& a, int in_dtype, int out_dtype, int momentum, int grid,
                     void* stream, const char** name);

}  // namespace adasum
