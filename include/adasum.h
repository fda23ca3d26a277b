/*
 * adasum.h -- C ABI of the GB300 Adasum library (libadasum_gb300.so).
 *
 * Adasum ("Scaling Distributed Training with Adaptive Summation", Maleki et al., arXiv
 * 2006.02924) combines the gradients of K data-parallel workers.  For two gradients
 * (Section 3, Equations 1-2 and the average of the two emulated SGD orders):
 *
 *     Adasum(a, b) = (1 - a.b / (2 |a|^2)) a + (1 - a.b / (2 |b|^2)) b
 *
 * with a zero-norm operand's quotient taken as 0 (its coefficient is 1).  K gradients
 * are combined as a binary tree over workers (Section 3, recursive application): level
 * 0 combines pairs (2i, 2i+1), every further level pairs the previous level's results
 * the same way, log2(K) levels in all.  Every layer segment of the flat gradient is
 * combined on its own, with its own dot products and norms (Section 3, after Figure 1).
 *
 * On one GPU the K worker gradients are K device buffers.  All entry points:
 *   - take DEVICE pointers for gradient, output and optimizer-state buffers and HOST
 *     pointers for the small descriptor arrays (the pointer list and the offsets);
 *     the library copies the descriptor arrays before it returns, so the caller may
 *     free or reuse them at once;
 *   - are asynchronous and stream-ordered on `stream` (a cudaStream_t; NULL means the
 *     legacy default stream).  They return once the work is enqueued.  A call whose
 *     segment layout (offsets, K, dtype) was seen by an earlier call on the device, and
 *     whose workspace need that call already met, enqueues only memsets and kernels, so
 *     it can be captured in a CUDA graph (the first call with a new layout uploads its
 *     plan synchronously and may grow the workspace: make it before capturing);
 *   - never modify the gradient buffers (unless `out` is one of them) and never
 *     allocate or free caller memory; the library keeps its own per-device workspace,
 *     grown on demand with cudaMalloc and reused by later calls (see Workspace below);
 *   - throw nothing across the ABI: every failure is a status code.  Argument errors
 *     are detected on the host before anything is enqueued; device-side conditions
 *     (a bounded wait that ran out) are reported by adasum_get_last_error() once the
 *     stream has been synchronised;
 *   - propagate NaN and Inf rather than check for them.
 *
 * Element types: ADASUM_F32 (fp32 storage and fp32 math) and ADASUM_BF16 (bf16 storage,
 * fp32 math: inputs are widened exactly, every intermediate is fp32, the final result is
 * rounded once to bf16, to nearest even).  Dot products and norms are accumulated from
 * fp32 products (exact for bf16 inputs) in fp32 partial sums of bounded length, then
 * combined across warps and tiles with compensated fp32 sums, in a fixed order, so
 * results are bitwise reproducible run to run.  The tree coefficients are computed in
 * double-float arithmetic (pairs of fp32 values, about 48 significant bits); segments of
 * at most 32 positions, and segments whose error estimate flags them, are evaluated in
 * vector space in double-float or fp64 (see adasum_recomputed_segments).
 *
 * Range: the fp32 pass is used for a segment while every worker with a nonzero value in
 * it has a squared norm between n * 2^-96 and 2^80 (n: the segment's length): then what
 * fp32 loses to underflow (products below 2^-126) stays below 2^-30 of that norm and
 * nothing overflows.  A segment outside that range (a worker with tiny or huge values,
 * including one whose squares all vanish in fp32) is detected and recomputed by a path
 * that first scales the segment by a power of two, so any magnitude fp32 or bf16 can
 * hold is combined to the stated accuracy.  The remaining limit: inside one segment, workers whose
 * largest magnitudes differ by more than a factor of about 2^60 lose the smaller
 * worker's precision (one power of two scales the whole segment).
 *
 * Alignment: buffers aligned to 16 bytes take the vectorised path; others are accepted
 * and take a scalar-load path inside the same kernels (slower, same results).
 *
 * Workspace: each device gets one library-owned workspace, reused across calls.  Calls
 * that overlap on the GPU (different streams without ordering between them) must not
 * share a device; order them with events or use one stream.  adasum_release_workspace()
 * frees it (after synchronising the device).
 *
 * Thread safety: the entry points may be called from several host threads; calls are
 * serialised inside the library.
 */
#ifndef ADASUM_GB300_H
#define ADASUM_GB300_H

#include <stdint.h>

#if defined(__GNUC__)
#define ADASUM_API __attribute__((visibility("default")))
#else
#define ADASUM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *adasum_stream_t;

typedef enum {
  ADASUM_F32 = 0,  /* fp32 storage, fp32 math */
  ADASUM_BF16 = 1  /* bf16 storage, fp32 math */
} adasum_dtype_t;

typedef enum {
  ADASUM_OK = 0,
  ADASUM_ERR_INVALID_ARG = 1,  /* null pointer, bad offsets, bad dtype, n < 0, ... */
  ADASUM_ERR_UNSUPPORTED = 2,  /* K outside [1, 256] (chain: [1, 16]), size limits */
  ADASUM_ERR_ALIAS = 3,        /* an output overlaps an input other than as allowed */
  ADASUM_ERR_NO_MEMORY = 4,    /* the workspace could not be grown */
  ADASUM_ERR_CUDA = 5,         /* a CUDA runtime call failed (launch, copy, ...) */
  ADASUM_ERR_TIMEOUT = 6,      /* a device-side bounded wait gave up */
  ADASUM_ERR_BOUNDS = 7        /* test build only (-DADASUM_BOUNDS_CHECK): a device-side index
                                  check found an access outside the call's buffers and
                                  skipped it; the product library never reports it */
} adasum_status_t;

/* Largest worker count accepted. */
#define ADASUM_MAX_K 256

/*
 * adasum_reduce -- Adasum of K worker gradients, per segment, as a binary tree.
 *
 *   grads        host array of K device pointers; grads[k] points to N = seg_offsets[L]
 *                elements of `dtype` (worker k's flat gradient).  1 <= K <= ADASUM_MAX_K;
 *                K = 1 copies grads[0] to out.  When K is not a power of two, every
 *                level still pairs (2i, 2i+1) and an unpaired last node moves up
 *                unchanged (the same as padding with zero gradients, since
 *                Adasum(x, 0) = x).
 *   seg_offsets  host array of L+1 int64 offsets, seg_offsets[0] = 0, non-decreasing;
 *                segment s is positions [seg_offsets[s], seg_offsets[s+1]).  Empty
 *                segments are allowed.  L = 0 (or N = 0) is a no-op.
 *   out          device pointer to N elements of `dtype`.  It may be exactly equal to
 *                one of the grads[k] (in-place); any other overlap with a gradient
 *                buffer is ADASUM_ERR_ALIAS.
 * Result: out[p] for p in segment s is the tree combination of g_0..g_{K-1} restricted
 * to segment s.
 */
ADASUM_API adasum_status_t adasum_reduce(const void *const *grads, int K, const int64_t *seg_offsets,
                              int L, adasum_dtype_t dtype, void *out,
                              adasum_stream_t stream);

/*
 * adasum_reduce_host -- adasum_reduce end to end from HOST memory: the K gradients are
 * copied to the device, combined, and the result copied back, in one call that returns
 * once host_out holds the result.  The paper exposes Adasum as an option of the
 * allreduce a training script already calls (Section 3, the Horovod allreduce and
 * DistributedOptimizer option); this is that single call for gradients held in host
 * memory, with the transfers inside it.
 *
 *   host_grads   host array of K HOST pointers, each to N = seg_offsets[L] elements of
 *                `dtype`.  Page-locked memory (cudaHostAlloc, cudaHostRegister) is copied
 *                asynchronously at full speed; pageable memory works, more slowly.
 *   seg_offsets, L, dtype, K   as for adasum_reduce.
 *   host_out     HOST pointer to N elements; it may be exactly one of host_grads[k]; any
 *                other overlap is ADASUM_ERR_ALIAS.
 *   stream       the copies start after the work already enqueued on it (which may still
 *                be writing the inputs).
 * Pipelining: whole segments are grouped into about 1 GiB of input (a longer segment is a
 * group of its own) and groups go through two device staging slots of the library
 * workspace (grown with cudaMalloc) on three library streams, so the copy of group i+1
 * to the device, the combine of group i and the copy of group i-1 back overlap.  One
 * cudaMemcpyAsync per worker row and group.
 * Blocking: returns when the result is in host_out; on any error, only after every copy
 * it started has finished, so the caller may free its buffers at once.
 * Errors: as adasum_reduce; a device pointer given as a host buffer is
 * ADASUM_ERR_INVALID_ARG.
 */
ADASUM_API adasum_status_t adasum_reduce_host(const void *const *host_grads, int K,
                                              const int64_t *seg_offsets, int L,
                                              adasum_dtype_t dtype, void *host_out,
                                              adasum_stream_t stream);

/*
 * adasum_reduce_orthogonality -- adasum_reduce, and per segment the orthogonality metric
 * of the paper's Figure 1 (Section 3):
 *
 *     ortho[s] = |Adasum(g_0..g_{K-1})|^2 / sum_k |g_k|^2     over segment s,
 *
 * which is 1 for mutually orthogonal gradients and 1/K for K parallel gradients of equal
 * norm.  ortho is a DEVICE array of L floats; an all-zero (or empty) segment gives NaN.
 * |A|^2 is the fp64 quadratic form of the final coefficients in the segment's Gram
 * matrix (the fp64 recompute's, for recomputed segments), not the rounded output.
 */
ADASUM_API adasum_status_t adasum_reduce_orthogonality(const void *const *grads, int K,
                                                       const int64_t *seg_offsets, int L,
                                                       adasum_dtype_t dtype, void *out,
                                                       float *ortho, adasum_stream_t stream);

/*
 * adasum_reduce_chain -- the linear recursion of the same section of the paper,
 * g[0,n+1] = Adasum(g[0,n], g_{n+1}): workers are folded in one at a time, left to
 * right, instead of pairwise up a tree.  Same arguments and conventions as
 * adasum_reduce; 1 <= K <= 16 (ADASUM_ERR_UNSUPPORTED above).
 */
ADASUM_API adasum_status_t adasum_reduce_chain(const void *const *grads, int K,
                                               const int64_t *seg_offsets, int L,
                                               adasum_dtype_t dtype, void *out,
                                               adasum_stream_t stream);

/*
 * adasum_pair -- Adasum(a, b) of two device vectors of n elements (one segment).
 * Equivalent to adasum_reduce with K = 2 and L = 1.  The combine is evaluated
 * symmetrically, so adasum_pair(a, b) and adasum_pair(b, a) agree bit for bit.
 * Pairs that the GPU's co-resident CTAs hold in registers (about 1.2M fp32 or 5M bf16
 * elements on a GB300) run as one cooperative kernel: the three dot products in
 * double-float arithmetic with exact products, and the output the double-float value of
 * alpha a + beta b rounded once (that value lies within about 2^-48 (|alpha a| + |beta b|)
 * of the exact one).  Longer pairs take the tiled route, within the stated tolerances.
 */
ADASUM_API adasum_status_t adasum_pair(const void *a, const void *b, int64_t n, adasum_dtype_t dtype,
                            void *out, adasum_stream_t stream);

/*
 * adasum_reduce_momentum_sgd -- adasum_reduce followed, in the same pass over the data,
 * by one heavy-ball Momentum-SGD step on fp32 master weights:
 *
 *     A  = Adasum tree of the K gradients (fp32, not rounded to the gradient dtype)
 *     v' = mu * v + A,     w' = w - lr * v'
 *
 * The paper applies Adasum to the optimizer's output when a distributed optimizer is
 * used (Section 3, Figure 3); this entry point is the allreduce-then-step form the paper
 * also exposes, and for zero initial momentum its first step equals that ordering
 * because the tree is scale-equivariant.
 *   master_w, momentum  device fp32 arrays of N elements, updated in place.  They must
 *                       not overlap each other, the gradients or out.
 *   out_or_null         optional device pointer to N elements of `grad_dtype` receiving A
 *                       (rounded to grad_dtype); NULL skips that write.
 */
ADASUM_API adasum_status_t adasum_reduce_momentum_sgd(const void *const *grads, int K,
                                           const int64_t *seg_offsets, int L,
                                           adasum_dtype_t grad_dtype, float *master_w,
                                           float *momentum, float lr, float mu,
                                           void *out_or_null, adasum_stream_t stream);

/*
 * adasum_local_momentum_reduce -- Adasum after the optimizer (paper, Section 3 and
 * Figure 3): every worker first takes its own heavy-ball step on its own momentum,
 *
 *     v_k' = mu * v_k + g_k                       (per worker, fp32 state, in place)
 *
 * proposes the update -lr * v_k', and the proposals are combined by the Adasum tree and
 * applied:  w' = w + Adasum(-lr v_0', ..., -lr v_{K-1}') = w - lr * Adasum(v_0', ...).
 * (Adasum is scale-equivariant.)  With zero initial momenta the first step equals
 * adasum_reduce_momentum_sgd's.
 *   grads     K device pointers, N elements of grad_dtype each (not modified)
 *   momenta   host array of K device pointers to fp32 states of N elements, updated
 *   master_w  device fp32 weights of N elements, updated
 * The states must not overlap each other, the gradients or the weights.
 */
ADASUM_API adasum_status_t adasum_local_momentum_reduce(const void *const *grads, int K,
                                                        const int64_t *seg_offsets, int L,
                                                        adasum_dtype_t grad_dtype,
                                                        float *const *momenta, float *master_w,
                                                        float lr, float mu,
                                                        adasum_stream_t stream);

/*
 * adasum_get_last_error -- the sticky device-side status of the current device
 * (ADASUM_OK, ADASUM_ERR_TIMEOUT, or in the test build ADASUM_ERR_BOUNDS), read after
 * the caller has synchronised the stream
 * of the calls in question.  Reading clears it.  Host-side failures are returned by the
 * entry points themselves and are not repeated here.
 */
ADASUM_API adasum_status_t adasum_get_last_error(void);

/* adasum_status_string -- a static, human-readable name for a status code. */
ADASUM_API const char *adasum_status_string(adasum_status_t status);

/*
 * adasum_release_workspace -- synchronise the current device and free the library's
 * workspace on it.  Later calls grow a new one.
 */
ADASUM_API adasum_status_t adasum_release_workspace(void);

/*
 * adasum_version -- library version as 10000*major + 100*minor + patch.
 */
ADASUM_API int adasum_version(void);

/*
 * adasum_pair_noalloc -- adasum_pair for callers that cannot allocate device memory.
 *
 * The paper has no counterpart to this entry point: it is a deployment variant of the
 * two-worker combine, not a different method.
 *
 * Who needs it: code that must not call cudaMalloc when it reduces -- for example a
 * process whose framework allocator already holds nearly all of the GPU's memory (a new
 * cudaMalloc fails, or makes the framework release and re-fragment its pool), a
 * latency-sensitive loop that cannot afford the device synchronisation cudaMalloc and
 * cudaFree imply, or a serving process that fixes its memory footprint at start-up.
 * The other entry points grow a library workspace with cudaMalloc on first use; this
 * one allocates nothing, ever.  The caller passes inputs and output as for adasum_pair.
 *
 * Scratch: a fixed file-scope device array of 64 KiB (plus a few bytes) inside the
 * library, present on every GPU that loads the library until the process exits.  The
 * first call on a device looks up that array's device address (cudaGetSymbolAddress,
 * with the device current); make that first call before any stream capture.  Every
 * call reuses the same array: calls that overlap on the GPU (different streams with no
 * ordering between them) race and give wrong results; order them.  Each call writes
 * every scratch slot it reads before reading it, so no state carries over between calls.
 *
 * Limits and errors: 0 <= n <= ADASUM_NOALLOC_MAX_N, else ADASUM_ERR_INVALID_ARG (n < 0)
 * or ADASUM_ERR_UNSUPPORTED (n too large); out may equal a or b, other overlap is
 * ADASUM_ERR_ALIAS; argument errors are found before anything is enqueued.
 * ADASUM_ERR_CUDA reports a failure of one of the call's own three launches (an error
 * left pending by other code on the thread is neither reported nor cleared here).
 * It runs the fp32 pass only: unlike adasum_pair it does not detect and recompute
 * ill-conditioned (strongly cancelling) inputs in fp64, and it needs the largest |a_i|
 * and |b_i| inside about [2^-40, 2^40], where their squares stay normal fp32 numbers
 * (outside it the result is not checked).
 */
#define ADASUM_NOALLOC_MAX_N 33554432
ADASUM_API adasum_status_t adasum_pair_noalloc(const void *a, const void *b, int64_t n,
                                               adasum_dtype_t dtype, void *out,
                                               adasum_stream_t stream);

/* ---- Instrumentation (used by the benchmark; not needed for normal use) ---------- */

/*
 * adasum_debug_workspace_guards -- for the test build of the library only
 * (libadasum_gb300_test.so, compiled with -DADASUM_TEST_HOOKS): every region of the
 * workspace is followed by a 256-byte guard band, filled with a pattern by each call;
 * this synchronises the current device and returns how many guard bytes of the last
 * call's layout lost the pattern (0: every kernel wrote only inside its regions).  The
 * product library has no guard bands and returns -1.
 */
ADASUM_API int64_t adasum_debug_workspace_guards(void);

/*
 * adasum_recomputed_segments -- synchronises the current device and returns how many
 * segments the last call on it recomputed in fp64 (-1 on a CUDA error).
 *
 * Every call first runs the fp32 pass; its per-segment coefficient step also estimates,
 * in fp64 from the Gram matrix, the relative error the fp32 pass will reach (Gram
 * rounding, error amplification through cancelling tree nodes, combine rounding).
 * Segments whose estimate exceeds 2.5e-5, or whose tree has a node norm at or below its
 * own error, are recomputed from the inputs entirely in fp64 and written over.
 */
ADASUM_API int64_t adasum_recomputed_segments(void);

/* Aggregated timing of one kernel kind. */
typedef struct {
  char name[64];      /* kernel kind, e.g. "gram_mma<bf16,16>" */
  int64_t launches;   /* launches recorded since the last collect */
  double total_ms;    /* summed device time between CUDA events around each launch */
  double total_bytes; /* summed algorithmic bytes of those launches: the input each must
                         read and the output it must write (0 for kernels whose work is
                         known only on the device, such as the recompute of flagged
                         segments) */
} adasum_kernel_stat_t;

/*
 * adasum_launch_count -- number of kernels this library has launched in this process.
 */
ADASUM_API int64_t adasum_launch_count(void);

/*
 * adasum_profile_enable -- when `on` is nonzero, every later launch is bracketed by two
 * CUDA events recorded on the launch stream.  Costs two event records per launch.
 */
ADASUM_API adasum_status_t adasum_profile_enable(int on);

/*
 * adasum_profile_collect -- waits for the recorded events, aggregates them per kernel
 * kind into `stats` (at most `max_stats` entries, in first-seen order), clears the
 * record, and returns the number of kinds seen (which may exceed max_stats).
 */
ADASUM_API int adasum_profile_collect(adasum_kernel_stat_t *stats, int max_stats);

#ifdef __cplusplus
}
#endif

#endif /* ADASUM_GB300_H */
