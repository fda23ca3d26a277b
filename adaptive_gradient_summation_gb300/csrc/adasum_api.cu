// adasum_api.cu -- host side of the C ABI declared in include/adasum.h.
//
// Validation, tiling plans, the per-device workspace, stage scheduling and launches.
// "Scaling Distributed Training with Adaptive Summation", Section 3: the K worker
// gradients are combined per layer segment by a binary tree of the Adasum pair
// operator.  The device computes it in coefficient space (see adasum_internal.h):
// for every stage, pass 1 (Gram partials per tile) -> coefficients per segment ->
// pass 2 (out = sum_k c_k g_k).  Trees of more than 16 leaves run as stages: 16-leaf
// subtrees first (fp32 intermediates in the workspace), then the tree over their roots.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cstdlib>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <functional>
#include <list>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/adasum.h"
#include "adasum_internal.h"

namespace adasum {
namespace {

constexpr int kVersion = 100;  // 0.1.0

int elem_size(int dt) { return dt == kBF16 ? 2 : 4; }

// Switches for tests and comparisons.  Only a library built with -DADASUM_TEST_HOOKS
// (the test build) reads them from the environment; the product library reads no
// environment variable and always takes the defaults.
const char* hook(const char* name) {
#ifdef ADASUM_TEST_HOOKS
  return std::getenv(name);
#else
  (void)name;
  return nullptr;
#endif
}

// A positive integer switch, else `dflt`.
int64_t env_int(const char* name, int64_t dflt) {
  const char* v = hook(name);
  if (v == nullptr) return dflt;
  const long long x = std::atoll(v);
  return x > 0 ? x : dflt;
}

// An on/off switch: "0" is off, anything else on, unset `dflt`.
bool env_on(const char* name, bool dflt) {
  const char* v = hook(name);
  if (v == nullptr || *v == '\0') return dflt;
  return std::strcmp(v, "0") != 0;
}


// NVTX range over one phase of a call (what the host enqueues in it), for profilers
// that collect NVTX ranges; inactive otherwise.
struct Range {
  explicit Range(const char* name) { nvtxRangePushA(name); }
  void next(const char* name) {  // ends this phase and starts the next
    nvtxRangePop();
    nvtxRangePushA(name);
  }
  ~Range() { nvtxRangePop(); }
  Range(const Range&) = delete;
  Range& operator=(const Range&) = delete;
};

// Test build: every workspace region is followed by a guard band filled with a pattern
// at the start of each call; adasum_debug_workspace_guards counts the bytes that lost it.
constexpr size_t kGuardBytes = 256;
constexpr unsigned char kGuardByte = 0xA5;

// ------------------------------------------------------------------------ profiler

struct ProfRecord {
  const char* name;
  cudaEvent_t start, stop;
  double bytes;  // algorithmic bytes of the launch (0: not rated)
};

std::mutex g_mu;                   // serialises every entry point
std::atomic<int64_t> g_launches{0};
bool g_profiling = false;
std::vector<ProfRecord> g_prof_pending;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t pool_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// ----------------------------------------------------------------------- workspace

// A tiling plan: tiles never straddle segments; inside a segment, tile boundaries sit
// on multiples of 32 positions (so 16-byte vectors never straddle two tiles) except at
// the segment's own ends.
struct Plan {
  std::vector<int64_t> offsets;
  int Kg0 = 0;        // workers per group in the first stage
  int dtype = 0;
  int ntiles = 0;
  int nsegs = 0;
  int nchunks = 0;
  TileDesc* d_tiles = nullptr;
  SegDesc* d_segs = nullptr;
  ChunkDesc* d_chunks = nullptr;
  // the chunks of segments with more than one (the chunk-sum kernel's work; a segment of
  // one chunk is summed by the coefficient kernel from its tile partials)
  int nmulti = 0;
  int* d_multi = nullptr;
  // small segments: held on chip (grouped by cluster size 1, 2, 4, 8, 16) or, up to
  // kTinyDirect positions, on the warp kernel; neither gets tiles.  The coefficient kernel
  // then runs over the list of the remaining (tiled) segments.
  int onchip_K = 0;  // padded worker count the grouping was made for (0: none)
  int onchip_cmax = 0;
  bool onchip_force = false;
  int onchip_count[5] = {0, 0, 0, 0, 0};
  int onchip_first[5] = {0, 0, 0, 0, 0};
  int* d_onchip = nullptr;
  bool tiny_on = false;
  int tiny_count = 0;
  int tiny_c8 = 0, tiny_c16 = 0;  // d_tiny: segments of <= 8 positions, then <= 16, then the rest
  int* d_tiny = nullptr;
  int ncoef = 0;
  int* d_coef_list = nullptr;
  // three-kernel route: short tiles (kSmallTileF32, kSmallTileBF16, kSmallTileSimt) take
  // the warp Gram kernel
  // (lists empty when there are none)
  bool warp_tiles = true;
  int nbig = 0, nsmall = 0;
  int* d_big = nullptr;
  int* d_small = nullptr;
  // positions each launch covers (for the profiler's algorithmic bytes): all tiles, the
  // CTA Gram's and the warp Gram's tiles, each fast-pass launch's and the tiny kernel's
  // segments
  int64_t pos_tiles = 0, pos_big = 0, pos_small = 0, pos_tiny = 0;
  int64_t pos_onchip[5] = {0, 0, 0, 0, 0};
  // tiled segments the on-chip kernel could recompute if flagged (clusters of rc_cmax
  // CTAs), and whether any tiled segment is too long for it (else the fp64 path, which
  // only ever receives those, is not launched)
  int rc_cmax = 0;
  int rc_count = 0;
  bool need64 = true;
};

// A stream of the workspace with the two events that fork it from the caller's stream
// and join it back (created on first use, destroyed by adasum_release_workspace).
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;

  // `side` waits for everything enqueued on `caller` so far.
  adasum_status_t fork_from(cudaStream_t caller) {
    if (stream == nullptr) {
      if (cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking) != cudaSuccess ||
          cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&join, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        return ADASUM_ERR_CUDA;
      }
    }
    if (cudaEventRecord(fork, caller) != cudaSuccess || cudaStreamWaitEvent(stream, fork, 0) != cudaSuccess)
      return ADASUM_ERR_CUDA;
    return ADASUM_OK;
  }
  void destroy() {
    if (stream) cudaStreamDestroy(stream);
    if (fork) cudaEventDestroy(fork);
    if (join) cudaEventDestroy(join);
    stream = nullptr;
    fork = join = nullptr;
  }
};

// Device staging of adasum_reduce_host: two slots, each holding K input rows and one
// output row of the largest segment group, and three streams (host-to-device copies,
// reductions, device-to-host copies) with the events that order them.
struct HostPipe {
  void* buf = nullptr;
  size_t cap = 0;
  cudaStream_t in = nullptr, compute = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, h2d[2] = {nullptr, nullptr}, reduced[2] = {nullptr, nullptr},
              d2h[2] = {nullptr, nullptr};

  adasum_status_t init() {
    if (in != nullptr) return ADASUM_OK;
    bool ok = cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&compute, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&start, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; i < 2 && ok; ++i)
      ok = cudaEventCreateWithFlags(&h2d[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&reduced[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&d2h[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      destroy();
      return ADASUM_ERR_CUDA;
    }
    return ADASUM_OK;
  }
  void destroy() {
    for (cudaStream_t* st : {&in, &compute, &out}) {
      if (*st) cudaStreamDestroy(*st);
      *st = nullptr;
    }
    for (cudaEvent_t* e : {&start, &h2d[0], &h2d[1], &reduced[0], &reduced[1], &d2h[0], &d2h[1]}) {
      if (*e) cudaEventDestroy(*e);
      *e = nullptr;
    }
    if (buf) cudaFree(buf);
    buf = nullptr;
    cap = 0;
  }
};

struct Workspace {
  int device = -1;
  void* buf = nullptr;
  size_t cap = 0;
  std::list<Plan> plans;            // most recently used first
  int* last_flag_counts = nullptr;  // device counters of the last call's fp64 lists
  int* d_error = nullptr;           // device status word (bounded waits), kept for good
  // two more streams, each forked from and joined back into the caller's stream within
  // a call: [0] the tiny-segment kernel, [1] the recompute of flagged segments
  SideStream side[2];
  // the fused pair kernel's partials, grid-barrier words and four zero counters
  // (allocated and zeroed on its first use)
  void* pair_buf = nullptr;
  HostPipe host;                    // staging of adasum_reduce_host
  std::vector<size_t> guards;       // test build: guard-band offsets of the last call
};

std::vector<Workspace> g_ws;

Workspace& workspace_for(int device) {
  for (auto& w : g_ws)
    if (w.device == device) return w;
  g_ws.push_back(Workspace{});
  g_ws.back().device = device;
  return g_ws.back();
}

void free_plan(Plan& p) {
  if (p.d_tiles) cudaFree(p.d_tiles);
  if (p.d_segs) cudaFree(p.d_segs);
  if (p.d_chunks) cudaFree(p.d_chunks);
  if (p.d_multi) cudaFree(p.d_multi);
  if (p.d_onchip) cudaFree(p.d_onchip);
  if (p.d_tiny) cudaFree(p.d_tiny);
  if (p.d_coef_list) cudaFree(p.d_coef_list);
  if (p.d_big) cudaFree(p.d_big);
  if (p.d_small) cudaFree(p.d_small);
  p.d_big = nullptr;
  p.d_small = nullptr;
  p.d_onchip = nullptr;
  p.d_tiny = nullptr;
  p.d_coef_list = nullptr;
  p.d_tiles = nullptr;
  p.d_segs = nullptr;
  p.d_chunks = nullptr;
  p.d_multi = nullptr;
}

// Input bytes per tile of the tiled passes.
constexpr int64_t kTileBytes = int64_t(256) << 10;
// When segments that fit one tile but are longer than this many positions hold at least
// a quarter of the tiled positions, each of them is cut into tiles of this many
// positions on the 32-position grid, all of them short tiles (one warp for the Gram and,
// with 8 or more workers per group, for the combine).  A whole-CTA tile of a few
// thousand positions leaves most of its warps waiting on the slowest one and on the
// block reduction.  Measured on a layout of 10,000 segments of 1..4096 positions: fp32
// K = 16 took 0.227 ms uncut, 0.193 cut at 512 positions (0.198 at 256); bf16 K = 16
// 0.237 ms uncut, 0.187 cut at 1024 (0.193 at 512); K = 64 0.873 -> 0.835 ms (fp32) and
// 0.841 -> 0.766 ms (bf16).  On the BERT-Large set such segments hold almost none of the
// positions, and cutting them measured slower (3.340 -> 3.362 ms): their 318 short tiles
// then take a warp launch of their own.
constexpr int64_t kSplitTileF32 = 512;
constexpr int64_t kSplitTileBF16 = 1024;

int64_t tile_positions(int Kg, int dtype, int64_t N, int num_sms) {
  // About kTileBytes of input per tile, but enough tiles to give every SM a few.
  const int64_t bytes_per_pos = static_cast<int64_t>(Kg) * elem_size(dtype);
  int64_t T = kTileBytes / bytes_per_pos;
  const int64_t want = std::max<int64_t>(1, N / (4 * static_cast<int64_t>(num_sms)));
  T = std::min(T, want);
  T = std::max<int64_t>(256, std::min<int64_t>(T, 65536));
  return (T + 255) / 256 * 256;
}

template <typename T>
adasum_status_t upload(T** dst, const std::vector<T>& v) {
  if (cudaMalloc(dst, std::max<size_t>(1, v.size()) * sizeof(T)) != cudaSuccess) {
    cudaGetLastError();
    *dst = nullptr;
    return ADASUM_ERR_NO_MEMORY;
  }
  // Synchronous copy: a plan is immutable once built, so no later call can race with it.
  if (!v.empty() && cudaMemcpy(*dst, v.data(), v.size() * sizeof(T), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return ADASUM_ERR_CUDA;
  }
  return ADASUM_OK;
}

adasum_status_t get_plan(Workspace& ws, const int64_t* offs, int L, int Kg0, int dtype,
                         int onchip_K, int onchip_cmax, bool onchip_force, int rc_cmax, bool tiny_on,
                         bool warp_tiles, Plan** out) {
  for (auto it = ws.plans.begin(); it != ws.plans.end(); ++it) {
    if (it->Kg0 == Kg0 && it->dtype == dtype && it->onchip_K == onchip_K &&
        it->onchip_cmax == onchip_cmax && it->onchip_force == onchip_force && it->rc_cmax == rc_cmax &&
        it->tiny_on == tiny_on && it->warp_tiles == warp_tiles &&
        it->offsets.size() == static_cast<size_t>(L + 1) &&
        std::memcmp(it->offsets.data(), offs, sizeof(int64_t) * (L + 1)) == 0) {
      ws.plans.splice(ws.plans.begin(), ws.plans, it);
      *out = &ws.plans.front();
      return ADASUM_OK;
    }
  }
  int num_sms = 148;
  cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, ws.device);
  const int64_t N = offs[L];
  const int64_t T = tile_positions(Kg0, dtype, N, num_sms);
  std::vector<TileDesc> tiles;
  std::vector<SegDesc> segs(L);
  std::vector<ChunkDesc> chunks;
  std::vector<int> onchip[5], tiny;
  int rc_count = 0;
  bool need64 = false;
  const int64_t VW = dtype == kF32 ? 4 : 8;
  // the on-chip fast pass (onchip_cmax > 0): segments it may hold, in 16-byte vectors
  int64_t onchip_vecs = (onchip_K > 0 && onchip_cmax > 0) ? onchip_positions(onchip_K) / VW : 0;
  if (onchip_vecs > 0) {
    // The on-chip kernel pays off when small segments are numerous enough to fill the
    // GPU by themselves (each CTA is latency-bound and takes half an SM); a few small
    // segments ride along in the tiled passes at no measurable cost.
    int64_t eligible = 0;
    for (int s = 0; s < L; ++s) {
      const int64_t lo = offs[s], hi = offs[s + 1];
      const int64_t nv = (hi + VW - 1) / VW - lo / VW;
      if (hi - lo > (tiny_on ? kTinyDirect : 0) && (nv + onchip_cmax - 1) / onchip_cmax <= onchip_vecs) ++eligible;
    }
    if (!onchip_force && eligible < 4 * static_cast<int64_t>(num_sms)) onchip_vecs = 0;
  }
  // whether segments that fit one tile are cut into short tiles (kSplitTileF32)
  const int64_t Ts = dtype == kF32 ? kSplitTileF32 : kSplitTileBF16;
  bool split = false;
  if (warp_tiles) {
    int64_t tiled = 0, cut = 0;
    for (int s = 0; s < L; ++s) {
      const int64_t n = offs[s + 1] - offs[s];
      if (n > kTinyDirect) tiled += n;
      if (n > Ts && n <= T) cut += n;
    }
    split = cut > 0 && 4 * cut >= tiled;
  }
  for (int s = 0; s < L; ++s) {
    const int64_t lo = offs[s], hi = offs[s + 1];
    segs[s].start = lo;
    segs[s].len = hi - lo;
    segs[s].first_tile = static_cast<int32_t>(tiles.size());
    bool small = false;
    if (hi > lo && tiny_on && hi - lo <= kTinyDirect) {
      tiny.push_back(s);
      small = true;
    }
    if (hi > lo && !small && onchip_vecs > 0) {
      // the smallest cluster whose CTAs hold the segment's 16-byte vectors
      const int64_t nv = (hi + VW - 1) / VW - lo / VW;
      for (int c = 0, C = 1; C <= onchip_cmax && c < 5; ++c, C *= 2) {
        if ((nv + C - 1) / C <= onchip_vecs) {
          onchip[c].push_back(s);
          small = true;
          break;
        }
      }
    }
    if (hi > lo && !small) {
      const int64_t nv = (hi + VW - 1) / VW - lo / VW;
      if (rc_cmax > 0 && (nv + rc_cmax - 1) / rc_cmax <= onchip_positions(onchip_K) / VW)
        ++rc_count;
      else
        need64 = true;
    }
    if (hi > lo && !small) {
      const int64_t base = lo / 32 * 32;
      const int64_t step = (split && hi - lo <= T && hi - lo > Ts) ? Ts : T;
      for (int64_t b = base; b < hi; b += step) {
        const int64_t t0 = std::max(lo, b), t1 = std::min(hi, b + step);
        if (t1 <= t0) continue;
        tiles.push_back(TileDesc{t0, static_cast<int32_t>(t1 - t0), s});
      }
    }
    segs[s].ntiles = static_cast<int32_t>(tiles.size()) - segs[s].first_tile;
    segs[s].first_chunk = static_cast<int32_t>(chunks.size());
    for (int32_t t = 0; t < segs[s].ntiles; t += kChunkTiles)
      chunks.push_back(ChunkDesc{segs[s].first_tile + t, std::min(kChunkTiles, segs[s].ntiles - t)});
    segs[s].nchunks = static_cast<int32_t>(chunks.size()) - segs[s].first_chunk;
  }
  if (tiles.size() > static_cast<size_t>(INT32_MAX / 2)) return ADASUM_ERR_UNSUPPORTED;
  if (ws.plans.size() >= 32) {  // (a pipelined caller keeps one plan per segment group)
    free_plan(ws.plans.back());
    ws.plans.pop_back();
  }
  Plan p;
  p.offsets.assign(offs, offs + L + 1);
  p.Kg0 = Kg0;
  p.dtype = dtype;
  p.ntiles = static_cast<int>(tiles.size());
  p.nsegs = L;
  p.nchunks = static_cast<int>(chunks.size());
  p.onchip_K = onchip_K;
  p.onchip_cmax = onchip_cmax;
  p.onchip_force = onchip_force;
  p.rc_cmax = rc_cmax;
  p.rc_count = rc_count;
  p.need64 = need64 || !tiny_on;
  p.tiny_on = tiny_on;
  p.tiny_count = static_cast<int>(tiny.size());
  // the warp kernel packs 4 segments of <= 8 positions, or 2 of <= 16, into a warp
  std::stable_partition(tiny.begin(), tiny.end(), [&](int s) { return offs[s + 1] - offs[s] <= 8; });
  std::stable_partition(tiny.begin(), tiny.end(), [&](int s) { return offs[s + 1] - offs[s] <= 16; });
  p.tiny_c8 = p.tiny_c16 = 0;
  for (int s : tiny) {
    const int64_t n = offs[s + 1] - offs[s];
    if (n <= 8) ++p.tiny_c8;
    else if (n <= 16) ++p.tiny_c16;
  }
  std::vector<int> onchip_all, coef_list;
  for (int c = 0; c < 5; ++c) {
    p.onchip_first[c] = static_cast<int>(onchip_all.size());
    p.onchip_count[c] = static_cast<int>(onchip[c].size());
    onchip_all.insert(onchip_all.end(), onchip[c].begin(), onchip[c].end());
  }
  const bool any_small = !onchip_all.empty() || !tiny.empty();
  if (any_small)
    for (int s = 0; s < L; ++s)
      if (segs[s].ntiles > 0) coef_list.push_back(s);
  p.ncoef = static_cast<int>(coef_list.size());
  std::vector<int> big, small_tiles;
  if (warp_tiles) {
    const int small_tile = Kg0 < kMaxGroup ? kSmallTileSimt : (dtype == kF32 ? kSmallTileF32 : kSmallTileBF16);
    for (int t = 0; t < static_cast<int>(tiles.size()); ++t)
      (tiles[t].len <= small_tile ? small_tiles : big).push_back(t);
    // a few small tiles cost nothing inside the CTA launch; a separate warp launch pays
    // its own latency, worth it only when small tiles are numerous
    if (small_tiles.size() < 2 * static_cast<size_t>(num_sms)) {
      small_tiles.clear();
      big.clear();
    }
  }
  p.warp_tiles = warp_tiles;
  p.nbig = static_cast<int>(big.size());
  p.nsmall = static_cast<int>(small_tiles.size());
  for (const TileDesc& t : tiles) p.pos_tiles += t.len;
  for (int t : small_tiles) p.pos_small += tiles[t].len;
  p.pos_big = p.pos_tiles - p.pos_small;
  for (int s : tiny) p.pos_tiny += offs[s + 1] - offs[s];
  for (int c = 0; c < 5; ++c)
    for (int s : onchip[c]) p.pos_onchip[c] += offs[s + 1] - offs[s];
  adasum_status_t st = upload(&p.d_tiles, tiles);
  if (!st && p.nsmall > 0) st = upload(&p.d_big, big);
  if (!st && p.nsmall > 0) st = upload(&p.d_small, small_tiles);
  if (!st && !onchip_all.empty()) st = upload(&p.d_onchip, onchip_all);
  if (!st && !tiny.empty()) st = upload(&p.d_tiny, tiny);
  if (!st && any_small) st = upload(&p.d_coef_list, coef_list);
  if (!st) st = upload(&p.d_segs, segs);
  if (!st) st = upload(&p.d_chunks, chunks);
  {
    std::vector<int> multi;
    for (int s2 = 0; s2 < L; ++s2)
      if (segs[s2].nchunks > 1)
        for (int c = 0; c < segs[s2].nchunks; ++c) multi.push_back(segs[s2].first_chunk + c);
    p.nmulti = static_cast<int>(multi.size());
    if (!st && !multi.empty()) st = upload(&p.d_multi, multi);
  }
  if (st) {
    free_plan(p);
    return st;
  }
  ws.plans.push_front(std::move(p));
  *out = &ws.plans.front();
  return ADASUM_OK;
}

adasum_status_t ensure_capacity(Workspace& ws, size_t bytes) {
  if (bytes <= ws.cap) return ADASUM_OK;
  if (ws.buf) {
    cudaDeviceSynchronize();  // earlier calls may still use the old buffer
    cudaFree(ws.buf);
    ws.buf = nullptr;
    ws.cap = 0;
    ws.last_flag_counts = nullptr;
  }
  const size_t rounded = (bytes + (size_t(1) << 21) - 1) & ~((size_t(1) << 21) - 1);
  if (cudaMalloc(&ws.buf, rounded) != cudaSuccess) {
    cudaGetLastError();
    ws.buf = nullptr;
    return ADASUM_ERR_NO_MEMORY;
  }
  ws.cap = rounded;
  return ADASUM_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Host-side fault injection for the error-path tests (test build only):
// ADASUM_FAULT_INJECT=alloc makes the next workspace growth fail as if cudaMalloc had;
// ADASUM_FAULT_INJECT=timeout makes the small-segment kernel expect 16 bulk-copy bytes
// that are never sent and the fused pair kernel wait at a barrier no CTA arrives at,
// with their bounded waits shortened, so the waits run out and the device status
// reports ADASUM_ERR_TIMEOUT.
bool inject_alloc_failure() {
  const char* v = hook("ADASUM_FAULT_INJECT");
  return v != nullptr && std::strcmp(v, "alloc") == 0;
}
bool inject_timeout() {
  const char* v = hook("ADASUM_FAULT_INJECT");
  return v != nullptr && std::strcmp(v, "timeout") == 0;
}

int record_launch(int rc, const char* name, cudaEvent_t start, cudaStream_t stream, double bytes) {
  if (rc != 0) return rc;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (g_profiling && start) {
    cudaEvent_t stop = pool_event();
    cudaEventRecord(stop, stream);
    g_prof_pending.push_back(ProfRecord{name, start, stop, bytes});
  }
  return 0;
}

cudaEvent_t maybe_start(cudaStream_t stream) {
  if (!g_profiling) return nullptr;
  cudaEvent_t e = pool_event();
  cudaEventRecord(e, stream);
  return e;
}

// Launch wrapper: counts launches and, when profiling, brackets them with events and
// records the launch's algorithmic bytes (the input it must read and the output it must
// write; 0 for kernels whose work depends on what earlier kernels found).
template <typename F>
adasum_status_t launch_one(cudaStream_t stream, F&& f, double bytes = 0.0) {
  const char* name = "";
  cudaEvent_t e = maybe_start(stream);
  const int rc = f(&name);
  return record_launch(rc, name, e, stream, bytes) ? ADASUM_ERR_CUDA : ADASUM_OK;
}

// fp32 pass of one stage (all groups): Gram partials, chunk sums, coefficients with the
// conditioning check, then `before_combine` (when given), then the combine (flagged
// segments are skipped and left to the recompute).
// bytes: the algorithmic bytes of the CTA Gram, the warp Gram, the CTA combine and the
// warp combine launches (the warp launches take the short tiles when they have a list).
adasum_status_t run_stage(StageArgs& a, int in_dtype, int out_dtype, int momentum, cudaStream_t stream,
                          const std::function<adasum_status_t()>& before_combine, const double (&bytes)[4]) {
  if (a.ntiles == 0)  // every segment went to the small-segment kernels
    return before_combine ? before_combine() : ADASUM_OK;
  if (a.Kg > 1) {
    if (a.tile_list == nullptr || a.ntile_list > 0) {
      if (adasum_status_t st = launch_one(stream, [&](const char** n) {
            return in_dtype == kBF16 ? launch_gram_bf16(a, stream, n) : launch_gram_f32(a, stream, n);
          }, bytes[0]))
        return st;
    }
    if (a.nsmall > 0) {
      if (adasum_status_t st = launch_one(stream, [&](const char** n) {
            return launch_gram_warp(a, in_dtype, stream, n);
          }, bytes[1]))
        return st;
    }
    if (a.nmulti > 0)
      if (adasum_status_t st = launch_one(stream, [&](const char** n) {
            return launch_reduce_chunks(a, stream, n);
          }))
        return st;
    if (adasum_status_t st = launch_one(stream, [&](const char** n) { return launch_coef(a, stream, n); }))
      return st;
  }
  if (before_combine)
    if (adasum_status_t st = before_combine()) return st;
  // Short tiles get a warp each when groups have 8 or more workers; with fewer, the
  // per-tile work is small and one CTA over every tile measured faster.
  StageArgs c = a;
  const bool warp_combine = a.nsmall > 0 && a.Kg >= 8;
  if (!warp_combine) {
    c.tile_list = nullptr;
    c.ntile_list = 0;
    c.nsmall = 0;
  }
  const int n = c.tile_list ? c.ntile_list : c.ntiles;
  c.combine_tiles = static_cast<int>(
      std::max<int64_t>(1, std::min<int64_t>(4, n / (16 * static_cast<int64_t>(std::max(1, c.num_sms))))));
  for (int warp = 0; warp < 2; ++warp) {
    if (warp ? c.nsmall == 0 : n == 0) continue;
    const double b = warp ? bytes[3] : (warp_combine ? bytes[2] : bytes[2] + bytes[3]);
    if (adasum_status_t st = launch_one(stream, [&](const char** nm) {
          return in_dtype == kBF16 ? launch_combine_bf16in(c, out_dtype, momentum, warp, stream, nm)
                                   : launch_combine_f32in(c, out_dtype, momentum, warp, stream, nm);
        }, b))
      return st;
  }
  return ADASUM_OK;
}

// fp64 pass of one stage over the flagged lists.
adasum_status_t run_stage64(StageArgs& a, int in_dtype, int out_dtype, int momentum, int grid,
                            cudaStream_t stream) {
  if (a.Kg > 1) {
    if (adasum_status_t st = launch_one(stream, [&](const char** n) {
          return launch_gram64(a, in_dtype, grid, stream, n);
        }))
      return st;
    if (adasum_status_t st = launch_one(stream, [&](const char** n) {
          return launch_coef64(a, grid, stream, n);
        }))
      return st;
  }
  return launch_one(stream, [&](const char** n) {
    return launch_combine64(a, in_dtype, out_dtype, momentum, grid, stream, n);
  });
}

// Carves the workspace: returns the byte offset of a region of `bytes` and advances.
struct Carver {
  size_t off = 0;
  std::vector<size_t> guards;  // test build: a guard band after every region
  size_t take(size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
#ifdef ADASUM_TEST_HOOKS
    guards.push_back(off);
    off += kGuardBytes;
#endif
    return at;
  }
};

// The device status word of the workspace (bounded waits), created on first use.
adasum_status_t ensure_error_word(Workspace& ws) {
  if (ws.d_error != nullptr) return ADASUM_OK;
  if (cudaMalloc(&ws.d_error, sizeof(int)) != cudaSuccess || cudaMemset(ws.d_error, 0, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    ws.d_error = nullptr;
    return ADASUM_ERR_NO_MEMORY;
  }
  return ADASUM_OK;
}

// Adasum(a, b) over one segment by the fused pair kernel (adasum_pair.cuh).  Returns
// false, having enqueued nothing, when the kernel cannot run on this device or the
// segment is longer than its CTAs hold; else sets *status.
bool run_pair_fused(Workspace& ws, const void* a, const void* b, int64_t n, int dtype, void* out,
                    cudaStream_t stream, adasum_status_t* status) {
  const int cap = std::min(pair_fused_max_grid(dtype), kPairThreads);
  const int64_t vw = dtype == kF32 ? 4 : 8;
  const int64_t nv = (n + vw - 1) / vw;
  const int64_t per_cta = static_cast<int64_t>(kPairThreads) * kPairVecs;
  if (cap <= 0 || nv > cap * per_cta) return false;  // more than the registers of the CTAs hold
  // one layout for every call (partials of up to kPairThreads CTAs, then the barrier
  // words and the zero counters), so that the barrier's state stays where it was
  const size_t part_bytes = align_up(static_cast<size_t>(kPairThreads) * 8 * sizeof(float), 256);
  if (ws.pair_buf == nullptr) {
    const size_t bytes = part_bytes + 256;
    if (cudaMalloc(&ws.pair_buf, bytes) != cudaSuccess || cudaMemset(ws.pair_buf, 0, bytes) != cudaSuccess) {
      cudaGetLastError();
      if (ws.pair_buf) cudaFree(ws.pair_buf);
      ws.pair_buf = nullptr;
      *status = ADASUM_ERR_NO_MEMORY;
      return true;
    }
  }
  if (adasum_status_t st = ensure_error_word(ws)) {
    *status = st;
    return true;
  }
  const int grid = static_cast<int>(std::max<int64_t>(1, (nv + per_cta - 1) / per_cta));
  char* base = static_cast<char*>(ws.pair_buf);
  PairArgs pa;
  std::memset(&pa, 0, sizeof pa);
  pa.a = a;
  pa.b = b;
  pa.out = out;
  pa.n = n;
  pa.aligned = aligned16(a) && aligned16(b) && aligned16(out) ? 1 : 0;
  pa.partials = reinterpret_cast<float*>(base);
  pa.bar = reinterpret_cast<unsigned*>(base + part_bytes);
  pa.error = ws.d_error;
  pa.spin_budget = 2000000000LL;  // about one second of SM clock
  if (inject_timeout()) {
    pa.inject_no_arrival = 1;
    pa.spin_budget = 200000LL;
  }
  *status = launch_one(stream, [&](const char** nm) { return launch_pair_fused(pa, dtype, grid, stream, nm); },
                       3.0 * static_cast<double>(n) * static_cast<double>(elem_size(dtype)));
  ws.last_flag_counts = reinterpret_cast<int*>(base + part_bytes + 64);  // zeros: nothing is recomputed
  return true;
}

adasum_status_t reduce_impl(const void* const* grads_in, int K, const int64_t* offs, int L,
                            int dtype, void* out, float* master_w, float* momentum,
                            float lr, float mu, cudaStream_t stream, bool chain = false,
                            float* ortho = nullptr) {
  const bool mom = master_w != nullptr;
  if (dtype != kF32 && dtype != kBF16) return ADASUM_ERR_INVALID_ARG;
  if (L < 0 || (L > 0 && offs == nullptr) || K < 1 || grads_in == nullptr)
    return ADASUM_ERR_INVALID_ARG;
  if (K > ADASUM_MAX_K || (chain && K > kMaxGroup)) return ADASUM_ERR_UNSUPPORTED;
  // Pad the worker list to a power of two with zero (null) gradients: exact for the
  // tree (an unpaired node meets a zero node, Adasum(x, 0) = x); the chain ignores them.
  const int Kreal = K;
  int P2 = 1;
  while (P2 < K) P2 *= 2;
  if (ortho != nullptr && P2 == 1) P2 = 2;  // a zero partner: Adasum(g, 0) = g, and a Gram pass
  std::vector<const void*> padded(grads_in, grads_in + K);
  padded.resize(P2, nullptr);
  const void* const* grads = padded.data();
  K = P2;
  if (L == 0) return ADASUM_OK;
  if (offs[0] != 0) return ADASUM_ERR_INVALID_ARG;
  for (int s = 0; s < L; ++s)
    if (offs[s + 1] < offs[s]) return ADASUM_ERR_INVALID_ARG;
  const int64_t N = offs[L];
  if (N == 0) return ADASUM_OK;
  if (!mom && out == nullptr) return ADASUM_ERR_INVALID_ARG;  // (momentum null: plain step)
  for (int k = 0; k < Kreal; ++k)
    if (grads[k] == nullptr) return ADASUM_ERR_INVALID_ARG;
  const size_t es = elem_size(dtype);
  const size_t nbytes = static_cast<size_t>(N) * es;
  if (out) {
    for (int k = 0; k < Kreal; ++k)
      if (out != grads[k] && overlaps(out, nbytes, grads[k], nbytes)) return ADASUM_ERR_ALIAS;
  }
  if (mom) {
    const size_t fb = static_cast<size_t>(N) * sizeof(float);
    const size_t mb = momentum ? fb : 0;
    if (overlaps(master_w, fb, momentum, mb)) return ADASUM_ERR_ALIAS;
    for (int k = 0; k < Kreal; ++k)
      if (overlaps(master_w, fb, grads[k], nbytes) || overlaps(momentum, mb, grads[k], nbytes))
        return ADASUM_ERR_ALIAS;
    if (out && (overlaps(master_w, fb, out, nbytes) || overlaps(momentum, mb, out, nbytes)))
      return ADASUM_ERR_ALIAS;
  }
  if (!mom && Kreal == 1 && out == grads[0] && ortho == nullptr) return ADASUM_OK;  // in-place copy

  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) {
    cudaGetLastError();
    return ADASUM_ERR_CUDA;
  }
  Workspace& ws = workspace_for(device);
  int num_sms = 148;
  cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device);

  // Two workers and one segment whose inputs fit well inside L2: one fused kernel
  // (ADASUM_PAIR_FUSED=0 switches it off, for comparisons).
  if (K == 2 && Kreal == 2 && L == 1 && !mom && !chain && ortho == nullptr &&
      env_on("ADASUM_PAIR_FUSED", true)) {
    adasum_status_t st = ADASUM_OK;
    if (run_pair_fused(ws, grads[0], grads[1], N, dtype, out, stream, &st)) return st;
  }

  // Stage structure: groups of at most 16 workers; K=1 is a single pass-2 "copy".
  std::vector<int> kg;  // workers per group, per stage
  for (int rem = K; rem > 1;) {
    const int g = std::min(rem, kMaxGroup);
    kg.push_back(g);
    rem /= g;
  }
  if (kg.empty()) kg.push_back(1);
  std::vector<int> groups(kg.size());
  {
    int rem = K;
    for (size_t s = 0; s < kg.size(); ++s) {
      rem /= kg[s];
      groups[s] = rem;
    }
  }

  // Plain reductions: segments of at most kTinyDirect positions go to the warp kernel,
  // the rest to the tiles; the on-chip kernel recomputes the flagged ones that fit a
  // cluster.  The on-chip kernel's fp32 fast pass (every level of a small segment on chip
  // in one pass) measured slower than the tiled route at every worker count and dtype on
  // the 10,000-segment layout, so the product library does not use it; the test build
  // turns it on with ADASUM_ONCHIP_FAST=1 (segments that fit 2 CTAs, or
  // ADASUM_ONCHIP_MAX_CLUSTER, when they are numerous) or ADASUM_ONCHIP=force (every
  // segment it holds, whatever their number, unless ADASUM_ONCHIP_FAST=0).
  // (ADASUM_TINY=0 and ADASUM_ONCHIP=0 switch the warp kernel and the on-chip kernel off,
  // for comparisons; ADASUM_WARP_GRAM=0 keeps every tile on the CTA Gram kernels.)
  const bool plain = !mom && !chain && ortho == nullptr && K >= 2;
  const bool tiny_on = plain && env_on("ADASUM_TINY", true);
  int onchip_K = 0, onchip_cmax = 0;
  const char* onchip_env = hook("ADASUM_ONCHIP");
  const bool onchip_force = onchip_env != nullptr && std::strcmp(onchip_env, "force") == 0;
  if (plain && K <= kOnchipMaxK && env_on("ADASUM_ONCHIP", true) &&
      env_on("ADASUM_ONCHIP_FAST", onchip_force)) {
    onchip_cmax = std::min<int>(onchip_max_cluster(dtype, K), env_int("ADASUM_ONCHIP_MAX_CLUSTER", 2));
    if (onchip_cmax >= 1) onchip_K = K;
  }
  // flagged tiled segments that fit are recomputed by the on-chip kernel
  const int rc_cmax = (plain && K <= kOnchipMaxK && env_on("ADASUM_ONCHIP", true)) ? onchip_max_cluster(dtype, K) : 0;
  Plan* plan = nullptr;
  Range phase("adasum:plan");
  if (adasum_status_t st = get_plan(ws, offs, L, kg[0], dtype, rc_cmax > 0 ? K : onchip_K, onchip_cmax,
                                    onchip_force, rc_cmax, tiny_on, env_on("ADASUM_WARP_GRAM", true), &plan))
    return st;

  phase.next("adasum:workspace");
  // Workspace layout.
  size_t max_e_tiles = 0, max_e_chunks = 0, max_coef = 0, max_g = 1, max_g_tiles = 0, max_g_chunks = 0;
  for (size_t s = 0; s < kg.size(); ++s) {
    const size_t E = static_cast<size_t>(kg[s]) * (kg[s] + 1) / 2;
    max_e_tiles = std::max(max_e_tiles, groups[s] * plan->ntiles * E);
    max_e_chunks = std::max(max_e_chunks, groups[s] * plan->nchunks * E);
    max_g_tiles = std::max(max_g_tiles, static_cast<size_t>(groups[s]) * plan->ntiles);
    max_g_chunks = std::max(max_g_chunks, static_cast<size_t>(groups[s]) * plan->nchunks);
    max_coef = std::max(max_coef, static_cast<size_t>(groups[s]) * L * kg[s]);
    max_g = std::max(max_g, static_cast<size_t>(groups[s]));
  }
  const size_t inter32 = align_up(static_cast<size_t>(N) * sizeof(float), 256);
  const size_t inter64 = align_up(static_cast<size_t>(N) * sizeof(double), 256);
  Carver cv;
  // One zeroed int region per call: segment flags, the 3 fp64-list counters and the
  // small-segment kernel's recompute counter, the recompute's segment scales, and the
  // count of flagged segments listed for the on-chip recompute.
  const size_t n_ints = 2 * static_cast<size_t>(L) + 5;
  const size_t o_flags = cv.take(n_ints * sizeof(int));
  const size_t o_part = cv.take(max_e_tiles * sizeof(float));
  const size_t o_chunk = cv.take(max_e_chunks * sizeof(double));
  const size_t o_tnz = cv.take(max_g_tiles * sizeof(uint32_t));
  const size_t o_cnz = cv.take(max_g_chunks * sizeof(uint32_t));
  const size_t o_coef = cv.take(max_coef * sizeof(float));
  const size_t o_rel0 = cv.take(max_g * L * sizeof(float));
  const size_t o_rel1 = cv.take(max_g * L * sizeof(float));
  const size_t o_part64 = cv.take(max_e_tiles * sizeof(double));
  const size_t o_coef64 = cv.take(max_coef * sizeof(double));
  const size_t o_ltiles = cv.take(static_cast<size_t>(plan->ntiles) * sizeof(int));
  const size_t o_lsegs = cv.take(static_cast<size_t>(L) * sizeof(int));
  const size_t o_ltiny = cv.take(static_cast<size_t>(L) * sizeof(int));
  const size_t o_oclist = cv.take(plan->rc_cmax > 0 ? static_cast<size_t>(L) * sizeof(int) : 0);
  const size_t o_onorm = cv.take(ortho ? static_cast<size_t>(L) * sizeof(double) : 0);
  const size_t o_diag = cv.take(ortho ? static_cast<size_t>(groups[0]) * L * sizeof(double) : 0);
  // Stage outputs of every non-final stage: fp32 (fast pass) and fp64 (recompute).
  std::vector<size_t> off32(kg.size(), 0), off64(kg.size(), 0);
  for (size_t s = 0; s + 1 < kg.size(); ++s) {
    off32[s] = cv.take(groups[s] * inter32);
    off64[s] = cv.take(groups[s] * inter64);
  }
  const size_t total = cv.off;
  if (total > ws.cap && inject_alloc_failure()) return ADASUM_ERR_NO_MEMORY;
  if (adasum_status_t st = ensure_capacity(ws, total)) return st;
  char* base = static_cast<char*>(ws.buf);
  int* seg_flag = reinterpret_cast<int*>(base + o_flags);
  int* list_count = seg_flag + L;
  int* seg_exp = list_count + 4;  // the fp64 recompute's per-segment scale
  int* oc_count = seg_exp + L;   // flagged segments listed for the on-chip recompute
  if (adasum_status_t st = ensure_error_word(ws)) return st;

  bool all_aligned = aligned16(out) && (!mom || (aligned16(master_w) && aligned16(momentum)));
  // (aligned16(nullptr) is true: absent buffers do not force the scalar path)
  for (int k = 0; k < Kreal; ++k) all_aligned = all_aligned && aligned16(grads[k]);

  if (cudaMemsetAsync(seg_flag, 0, n_ints * sizeof(int), stream) != cudaSuccess)
    return ADASUM_ERR_CUDA;
#ifdef ADASUM_TEST_HOOKS
  ws.guards = cv.guards;
  for (size_t g : ws.guards)
    if (cudaMemsetAsync(base + g, kGuardByte, kGuardBytes, stream) != cudaSuccess) return ADASUM_ERR_CUDA;
#endif

  auto make_args = [&](size_t s) {
    StageArgs a;
    std::memset(&a, 0, sizeof a);
    a.n_total = N;
    a.error = ws.d_error;
    a.Kg = kg[s];
    a.G = groups[s];
    a.aligned = all_aligned ? 1 : 0;
    a.ntiles = plan->ntiles;
    a.nsegs = plan->nsegs;
    a.nchunks = plan->nchunks;
    a.tiles = plan->d_tiles;
    a.segs = plan->d_segs;
    a.chunks = plan->d_chunks;
    a.multi_chunks = plan->d_multi;
    a.nmulti = plan->nmulti;
    a.partials = reinterpret_cast<float*>(base + o_part);
    a.chunk_sums = reinterpret_cast<float2*>(base + o_chunk);
    a.tile_nz = reinterpret_cast<uint32_t*>(base + o_tnz);
    a.chunk_nz = reinterpret_cast<uint32_t*>(base + o_cnz);
    a.coef = reinterpret_cast<float*>(base + o_coef);
    a.seg_flag = seg_flag;
    a.partials64 = reinterpret_cast<double*>(base + o_part64);
    a.coef64 = reinterpret_cast<double*>(base + o_coef64);
    a.list_tiles = reinterpret_cast<int*>(base + o_ltiles);
    a.list_segs = reinterpret_cast<int*>(base + o_lsegs);
    a.list_tiny = reinterpret_cast<int*>(base + o_ltiny);
    a.list_count = list_count;
    a.Ktotal = chain ? Kreal : K;
    a.seg_exp = seg_exp;
    // up to 4 tiles (1 MiB) per combine CTA while the grid keeps 16 CTAs per SM
    a.combine_tiles = 1;  // (set per launch by run_stage)
    a.num_sms = num_sms;
    if (plan->rc_cmax > 0) {
      a.oc_vecs = onchip_positions(K) / (dtype == kF32 ? 4 : 8);
      a.oc_vw = dtype == kF32 ? 4 : 8;
      a.oc_cmax = plan->rc_cmax;
      a.oc_list = reinterpret_cast<int*>(base + o_oclist);
      a.oc_count = oc_count;
    }
    a.seg_list = plan->d_coef_list;
    a.nseg_list = plan->ncoef;
    if (plan->nsmall > 0) {
      a.tile_list = plan->d_big;
      a.ntile_list = plan->nbig;
      a.small_list = plan->nbig > 0 ? plan->d_small : nullptr;  // (null: every tile, in order)
      a.nsmall = plan->nsmall;
    }
    a.mode = chain ? kModeChain : kModeTree;
    a.Kreal = Kreal;
    const bool last = s + 1 == kg.size();
    if (last && mom) {
      a.master_w = master_w;
      a.momentum = momentum;
      a.lr = lr;
      a.mu = mu;
    }
    if (ortho != nullptr) {
      if (last) a.outnorm2 = reinterpret_cast<double*>(base + o_onorm);
      if (s == 0) a.diag_sum = reinterpret_cast<double*>(base + o_diag);
    }
    return a;
  };

  // Work on the workspace's side streams is joined back into `stream` before the call
  // returns, on every path (errors included): the guard records each forked side
  // stream's join event and makes `stream` wait for it.
  struct JoinGuard {
    cudaStream_t caller;
    SideStream* forked[2] = {nullptr, nullptr};
    adasum_status_t join(int i) {
      if (forked[i] == nullptr) return ADASUM_OK;
      SideStream& sd = *forked[i];
      forked[i] = nullptr;
      if (cudaEventRecord(sd.join, sd.stream) != cudaSuccess || cudaStreamWaitEvent(caller, sd.join, 0) != cudaSuccess)
        return ADASUM_ERR_CUDA;
      return ADASUM_OK;
    }
    adasum_status_t fork(SideStream& sd, int i) {
      if (adasum_status_t st = sd.fork_from(caller)) return st;
      forked[i] = &sd;
      return ADASUM_OK;
    }
    ~JoinGuard() {
      join(0);
      join(1);
    }
  } joins{stream};

  phase.next("adasum:small segments");
  // Small segments: whole tree on chip, one launch per cluster size.
  if (plan->onchip_K > 0) {
    OnchipArgs oa;
    std::memset(&oa, 0, sizeof oa);
    for (int k = 0; k < K; ++k) oa.in[k] = grads[k];
    oa.out = out;
    oa.segs = plan->d_segs;
    oa.P = onchip_positions(K);
    oa.aligned = all_aligned ? 1 : 0;
    oa.error = ws.d_error;
    oa.n_total = N;
    oa.recomputed = list_count + 3;
    oa.spin_budget = 2000000000LL;  // about one second of SM clock
    if (inject_timeout()) {
      oa.inject_extra_tx = 1;
      oa.spin_budget = 200000LL;
    }
    for (int c = 0; c < 5; ++c) {
      if (plan->onchip_count[c] == 0) continue;
      oa.list = plan->d_onchip + plan->onchip_first[c];
      if (adasum_status_t st = launch_one(stream, [&](const char** n) {
            return launch_onchip(oa, dtype, K, plan->onchip_count[c], 1 << c, stream, n);
          }, static_cast<double>(plan->pos_onchip[c]) * (Kreal + 1) * es))
        return st;
    }
  }

  // Tiny segments: the warp kernel, on side stream 0.  The launch is a wave of
  // compute-bound warps, so it runs beside the tiled passes (bandwidth-bound) instead of
  // ahead of them.  (It is forked after the on-chip fast pass when the test build runs
  // that: forked before, its CTAs held registers the on-chip CTAs need.)
  if (plan->tiny_count > 0) {
    if (adasum_status_t st = joins.fork(ws.side[0], 0)) return st;
    TinyArgs ta;
    std::memset(&ta, 0, sizeof ta);
    for (int k = 0; k < K; ++k) ta.in[k] = grads[k];
    ta.out = out;
    ta.segs = plan->d_segs;
    ta.list = plan->d_tiny;
    ta.count = plan->tiny_count;
    ta.count8 = plan->tiny_c8;
    ta.count16 = plan->tiny_c16;
    ta.K = K;
    ta.n_total = N;
    ta.error = ws.d_error;
    cudaStream_t side = ws.side[0].stream;
    if (adasum_status_t st = launch_one(side, [&](const char** n) { return launch_tiny_df(ta, dtype, side, n); },
                                        static_cast<double>(plan->pos_tiny) * (Kreal + 1) * es))
      return st;
  }

  // Recompute of the flagged segments, enqueued on `ts` (usually nothing is flagged and
  // every kernel returns at once).  It needs the last stage's flags and nothing that the
  // last combine writes: that combine skips the flagged segments, and these kernels write
  // only the flagged segments' elements (edges masked per element), so the two run
  // concurrently.
  auto enqueue_recompute = [&](cudaStream_t ts) -> adasum_status_t {
    Range recompute_range("adasum:recompute");
    // (the lists' lengths are on the device: enough CTAs for many flagged tiles, the
    // surplus returns at once)
    const int grid64 = std::max(1, std::min(plan->ntiles, 16 * num_sms));
    {
      StageArgs a = make_args(0);
      if (adasum_status_t st = launch_one(ts, [&](const char** n) {
            return launch_collect(a, std::max(1, std::min((L + kThreads - 1) / kThreads, 4 * num_sms)),
                                  ts, n);
          }))
        return st;
    }
    // flagged segments that fit: the on-chip kernel's recompute, one launch of clusters of
    // rc_cmax CTAs, no more than fit on the device at once (the list's length is on the
    // device; each cluster takes every rc_clusters-th entry, surplus clusters return at once)
    if (plan->rc_count > 0) {
      const int resident = onchip_resident_clusters(dtype, K, plan->rc_cmax);
      const int rc_clusters = std::max(1, std::min(plan->rc_count, resident));
      OnchipArgs oa;
      std::memset(&oa, 0, sizeof oa);
      for (int k = 0; k < K; ++k) oa.in[k] = grads[k];
      oa.out = out;
      oa.segs = plan->d_segs;
      oa.P = onchip_positions(K);
      oa.aligned = all_aligned ? 1 : 0;
      oa.error = ws.d_error;
    oa.n_total = N;
      oa.recomputed = list_count + 3;
      oa.spin_budget = 2000000000LL;
      oa.list = reinterpret_cast<int*>(base + o_oclist);
      oa.dev_count = oc_count;
      oa.recompute_only = 1;
      if (adasum_status_t st = launch_one(ts, [&](const char** n) {
            return launch_onchip(oa, dtype, K, rc_clusters, plan->rc_cmax, ts, n);
          }))
        return st;
    }
    // the fp64 path, for flagged segments too long for the on-chip kernel (not launched
    // when there are none)
    if (!plan->need64) return ADASUM_OK;
    {
      // the scale of every flagged segment's Gram (from the stage-0 inputs)
      StageArgs a = make_args(0);
      for (int k = 0; k < K; ++k) a.in[k] = grads[k];
      if (adasum_status_t st = launch_one(ts, [&](const char** n) {
            return launch_segmax(a, dtype, grid64, ts, n);
          }))
        return st;
    }
    if (!plan->tiny_on) {  // (with the warp kernel on, no tiled segment is that short)
      // flagged segments of at most kTinySeg positions: the whole tree, vector space
      StageArgs a = make_args(kg.size() - 1);
      for (int k = 0; k < K; ++k) a.in[k] = grads[k];
      a.out[0] = out;
      if (adasum_status_t st = launch_one(ts, [&](const char** n) {
            return launch_tiny64(a, dtype, dtype, mom ? 1 : 0, grid64, ts, n);
          }))
        return st;
    }
    for (size_t s = 0; s < kg.size(); ++s) {
      const bool last = s + 1 == kg.size();
      StageArgs a = make_args(s);
      if (s == 0) {
        for (int k = 0; k < K; ++k) a.in[k] = grads[k];
      } else {
        for (int i = 0; i < groups[s] * kg[s]; ++i)
          a.in[i] = base + off64[s - 1] + i * inter64;
        a.in_f64 = 1;
      }
      if (last) {
        a.out[0] = out;
      } else {
        for (int q = 0; q < groups[s]; ++q)
          a.out[q] = base + off64[s] + q * inter64;
        a.out_f64 = 1;
      }
      const int in_dt = s == 0 ? dtype : kF32;
      const int out_dt = last ? dtype : kF32;
      if (adasum_status_t st = run_stage64(a, in_dt, out_dt, (last && mom) ? 1 : 0, grid64, ts))
        return st;
    }
    return ADASUM_OK;
  };
  // side stream 1: forked once the last stage's coefficients (and flags) are known
  auto fork_recompute = [&]() -> adasum_status_t {
    if (adasum_status_t st = joins.fork(ws.side[1], 1)) return st;
    return enqueue_recompute(ws.side[1].stream);
  };
  phase.next("adasum:stages");
  for (size_t s = 0; s < kg.size(); ++s) {
    const bool last = s + 1 == kg.size();
    StageArgs a = make_args(s);
    if (s == 0) {
      for (int k = 0; k < K; ++k) a.in[k] = grads[k];
    } else {
      for (int i = 0; i < groups[s] * kg[s]; ++i) a.in[i] = base + off32[s - 1] + i * inter32;
      a.in_relerr = reinterpret_cast<float*>(base + ((s - 1) % 2 ? o_rel1 : o_rel0));
    }
    if (last) {
      a.out[0] = out;
    } else {
      for (int q = 0; q < groups[s]; ++q) a.out[q] = base + off32[s] + q * inter32;
    }
    a.relerr = reinterpret_cast<float*>(base + (s % 2 ? o_rel1 : o_rel0));
    a.skip_flagged = 1;
    const int in_dt = s == 0 ? dtype : kF32;
    const int out_dt = last ? dtype : kF32;
    // algorithmic bytes: each tile's inputs once, and the combine's outputs (or the
    // momentum step's w and v, read and written)
    const double es_in = static_cast<double>(elem_size(in_dt)), es_out = static_cast<double>(elem_size(out_dt));
    const double nin = static_cast<double>(groups[s]) * kg[s];
    const double big = static_cast<double>(plan->nsmall > 0 ? plan->pos_big : plan->pos_tiles);
    const double out_b = (!last || out != nullptr) ? groups[s] * es_out : 0.0;
    const double mom_b = (last && mom) ? (momentum != nullptr ? 16.0 : 8.0) : 0.0;
    const double per_pos = nin * es_in + out_b + mom_b;  // the combine's bytes per position
    const double small = static_cast<double>(plan->nsmall > 0 ? plan->pos_small : 0);
    const double bytes[4] = {big * nin * es_in, small * nin * es_in, big * per_pos, small * per_pos};
    if (adasum_status_t st = run_stage(a, in_dt, out_dt, (last && mom) ? 1 : 0, stream,
                                       last ? fork_recompute : std::function<adasum_status_t()>(), bytes))
      return st;
  }

  if (ortho != nullptr) {
    if (adasum_status_t st = joins.join(1)) return st;  // the recompute's norms
    if (adasum_status_t st = launch_one(stream, [&](const char** n) {
          return launch_orthogonality(reinterpret_cast<double*>(base + o_onorm),
                                      reinterpret_cast<double*>(base + o_diag), groups[0], L,
                                      ortho, stream, n);
        }))
      return st;
  }
  ws.last_flag_counts = list_count;
  return ADASUM_OK;
}

// Input bytes (all K workers) per segment group of adasum_reduce_host; a longer segment
// is a group of its own.
constexpr int64_t kHostGroupBytes = int64_t(1) << 30;

adasum_status_t reduce_host_impl(const void* const* host_grads, int K, const int64_t* offs, int L,
                                 int dtype, void* host_out, cudaStream_t stream) {
  if (dtype != kF32 && dtype != kBF16) return ADASUM_ERR_INVALID_ARG;
  if (L < 0 || (L > 0 && offs == nullptr) || K < 1 || host_grads == nullptr) return ADASUM_ERR_INVALID_ARG;
  if (K > ADASUM_MAX_K) return ADASUM_ERR_UNSUPPORTED;
  if (L == 0) return ADASUM_OK;
  if (offs[0] != 0) return ADASUM_ERR_INVALID_ARG;
  for (int s = 0; s < L; ++s)
    if (offs[s + 1] < offs[s]) return ADASUM_ERR_INVALID_ARG;
  const int64_t N = offs[L];
  if (N == 0) return ADASUM_OK;
  if (host_out == nullptr) return ADASUM_ERR_INVALID_ARG;
  const size_t es = elem_size(dtype);
  const size_t nbytes = static_cast<size_t>(N) * es;
  for (int k = 0; k < K; ++k) {
    if (host_grads[k] == nullptr) return ADASUM_ERR_INVALID_ARG;
    if (host_out != host_grads[k] && overlaps(host_out, nbytes, host_grads[k], nbytes)) return ADASUM_ERR_ALIAS;
  }
  // every buffer must be host memory (pinned, pageable or managed); a device pointer is
  // an argument error
  for (int k = 0; k <= K; ++k) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, k < K ? host_grads[k] : host_out) != cudaSuccess) {
      cudaGetLastError();
      return ADASUM_ERR_CUDA;
    }
    if (attr.type == cudaMemoryTypeDevice) return ADASUM_ERR_INVALID_ARG;
  }
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) {
    cudaGetLastError();
    return ADASUM_ERR_CUDA;
  }
  Workspace& ws = workspace_for(device);
  HostPipe& hp = ws.host;
  if (adasum_status_t st = hp.init()) return st;

  // groups of whole segments, about kHostGroupBytes of input each
  std::vector<std::pair<int, int>> groups;
  const int64_t row = static_cast<int64_t>(K) * static_cast<int64_t>(es);
  int64_t slot_pos = 0;
  for (int a = 0; a < L;) {
    int b = a + 1;
    while (b < L && (offs[b + 1] - offs[a]) * row <= kHostGroupBytes) ++b;
    groups.emplace_back(a, b);
    slot_pos = std::max(slot_pos, offs[b] - offs[a]);
    a = b;
  }
  const size_t row_bytes = align_up(static_cast<size_t>(slot_pos) * es, 256);
  const size_t slot_bytes = row_bytes * static_cast<size_t>(K + 1);
  if (2 * slot_bytes > hp.cap) {
    if (hp.buf) {
      cudaDeviceSynchronize();  // earlier calls may still use the old staging
      cudaFree(hp.buf);
      hp.buf = nullptr;
      hp.cap = 0;
    }
    if (cudaMalloc(&hp.buf, 2 * slot_bytes) != cudaSuccess) {
      cudaGetLastError();
      hp.buf = nullptr;
      return ADASUM_ERR_NO_MEMORY;
    }
    hp.cap = 2 * slot_bytes;
  }

  // Work starts after everything already on the caller's stream (which may still be
  // writing the host inputs).  Whatever happens, every copy has finished when the call
  // returns, so the caller may reuse or free its host buffers at once.
  struct Drain {
    HostPipe& hp;
    ~Drain() {
      cudaStreamSynchronize(hp.in);
      cudaStreamSynchronize(hp.compute);
      cudaStreamSynchronize(hp.out);
    }
  } drain{hp};
  if (cudaEventRecord(hp.start, stream) != cudaSuccess || cudaStreamWaitEvent(hp.in, hp.start, 0) != cudaSuccess)
    return ADASUM_ERR_CUDA;
  std::vector<const void*> slot_in(K);
  std::vector<int64_t> goffs;
  for (size_t i = 0; i < groups.size(); ++i) {
    const int a = groups[i].first, b = groups[i].second, slot = static_cast<int>(i & 1);
    const int64_t p0 = offs[a], p1 = offs[b];
    if (p1 == p0) continue;
    const size_t gbytes = static_cast<size_t>(p1 - p0) * es;
    char* base = static_cast<char*>(hp.buf) + slot * slot_bytes;
    // host -> device, once the reduction of the group that last used the slot is done
    if (i >= 2 && cudaStreamWaitEvent(hp.in, hp.reduced[slot], 0) != cudaSuccess) return ADASUM_ERR_CUDA;
    for (int k = 0; k < K; ++k) {
      slot_in[k] = base + k * row_bytes;
      if (cudaMemcpyAsync(base + k * row_bytes, static_cast<const char*>(host_grads[k]) + p0 * es, gbytes,
                          cudaMemcpyHostToDevice, hp.in) != cudaSuccess)
        return ADASUM_ERR_CUDA;
    }
    if (cudaEventRecord(hp.h2d[slot], hp.in) != cudaSuccess) return ADASUM_ERR_CUDA;
    // the reduction, once the inputs are in and the slot's last result has left
    void* slot_out = base + K * row_bytes;
    if (cudaStreamWaitEvent(hp.compute, hp.h2d[slot], 0) != cudaSuccess) return ADASUM_ERR_CUDA;
    if (i >= 2 && cudaStreamWaitEvent(hp.compute, hp.d2h[slot], 0) != cudaSuccess) return ADASUM_ERR_CUDA;
    Range group_range("adasum_reduce_host:group");
    goffs.assign(offs + a, offs + b + 1);
    for (int64_t& o : goffs) o -= p0;
    if (adasum_status_t st = reduce_impl(slot_in.data(), K, goffs.data(), b - a, dtype, slot_out, nullptr,
                                         nullptr, 0.f, 0.f, hp.compute))
      return st;
    if (cudaEventRecord(hp.reduced[slot], hp.compute) != cudaSuccess) return ADASUM_ERR_CUDA;
    // device -> host
    if (cudaStreamWaitEvent(hp.out, hp.reduced[slot], 0) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<char*>(host_out) + p0 * es, slot_out, gbytes, cudaMemcpyDeviceToHost,
                        hp.out) != cudaSuccess ||
        cudaEventRecord(hp.d2h[slot], hp.out) != cudaSuccess)
      return ADASUM_ERR_CUDA;
  }
  if (cudaStreamSynchronize(hp.out) != cudaSuccess) return ADASUM_ERR_CUDA;
  return ADASUM_OK;
}

}  // namespace
}  // namespace adasum

using namespace adasum;

extern "C" {

adasum_status_t adasum_reduce_host(const void* const* host_grads, int K, const int64_t* seg_offsets,
                                   int L, adasum_dtype_t dtype, void* host_out, adasum_stream_t stream) {
  std::lock_guard<std::mutex> lock(g_mu);
  Range range("adasum_reduce_host");
  return reduce_host_impl(host_grads, K, seg_offsets, L, static_cast<int>(dtype), host_out,
                          reinterpret_cast<cudaStream_t>(stream));
}

adasum_status_t adasum_reduce(const void* const* grads, int K, const int64_t* seg_offsets,
                              int L, adasum_dtype_t dtype, void* out,
                              adasum_stream_t stream) {
  std::lock_guard<std::mutex> lock(g_mu);
  Range range("adasum_reduce");
  return reduce_impl(grads, K, seg_offsets, L, static_cast<int>(dtype), out, nullptr,
                     nullptr, 0.f, 0.f, reinterpret_cast<cudaStream_t>(stream));
}

adasum_status_t adasum_local_momentum_reduce(const void* const* grads, int K,
                                             const int64_t* seg_offsets, int L,
                                             adasum_dtype_t grad_dtype, float* const* momenta,
                                             float* master_w, float lr, float mu,
                                             adasum_stream_t stream) {
  if (grads == nullptr || momenta == nullptr || master_w == nullptr || K < 1 || L < 0 ||
      (L > 0 && seg_offsets == nullptr))
    return ADASUM_ERR_INVALID_ARG;
  if (grad_dtype != ADASUM_F32 && grad_dtype != ADASUM_BF16) return ADASUM_ERR_INVALID_ARG;
  if (K > ADASUM_MAX_K) return ADASUM_ERR_UNSUPPORTED;
  if (L == 0 || seg_offsets[L] == 0) return ADASUM_OK;
  const int64_t N = seg_offsets[L];
  const size_t gb = static_cast<size_t>(N) * (grad_dtype == ADASUM_BF16 ? 2 : 4);
  const size_t fb = static_cast<size_t>(N) * sizeof(float);
  for (int k = 0; k < K; ++k) {
    if (grads[k] == nullptr || momenta[k] == nullptr) return ADASUM_ERR_INVALID_ARG;
    if (overlaps(momenta[k], fb, master_w, fb)) return ADASUM_ERR_ALIAS;
    for (int j = 0; j < K; ++j)
      if (overlaps(momenta[k], fb, grads[j], gb) || (j != k && overlaps(momenta[k], fb, momenta[j], fb)))
        return ADASUM_ERR_ALIAS;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  Range range("adasum_local_momentum_reduce");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int device = 0, num_sms = 148;
  if (cudaGetDevice(&device) != cudaSuccess) return ADASUM_ERR_CUDA;
  cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device);
  // every worker's own heavy-ball step on its own state
  for (int k = 0; k < K; ++k) {
    const int aligned = aligned16(grads[k]) && aligned16(momenta[k]);
    if (adasum_status_t st = launch_one(s, [&](const char** n) {
          return launch_local_momentum(grads[k], static_cast<int>(grad_dtype), momenta[k], N, mu,
                                       aligned, num_sms, s, n);
        }))
      return st;
  }
  // Adasum of the proposed updates -lr v_k' = -lr Adasum(v_k'), applied: w -= lr A(v')
  std::vector<const void*> vs(momenta, momenta + K);
  return reduce_impl(vs.data(), K, seg_offsets, L, kF32, nullptr, master_w, nullptr, lr, 0.f, s);
}

adasum_status_t adasum_reduce_orthogonality(const void* const* grads, int K,
                                            const int64_t* seg_offsets, int L,
                                            adasum_dtype_t dtype, void* out, float* ortho,
                                            adasum_stream_t stream) {
  if (ortho == nullptr && L > 0) return ADASUM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  Range range("adasum_reduce_orthogonality");
  return reduce_impl(grads, K, seg_offsets, L, static_cast<int>(dtype), out, nullptr, nullptr, 0.f,
                     0.f, reinterpret_cast<cudaStream_t>(stream), false, ortho);
}

adasum_status_t adasum_reduce_chain(const void* const* grads, int K, const int64_t* seg_offsets,
                                    int L, adasum_dtype_t dtype, void* out, adasum_stream_t stream) {
  std::lock_guard<std::mutex> lock(g_mu);
  Range range("adasum_reduce_chain");
  return reduce_impl(grads, K, seg_offsets, L, static_cast<int>(dtype), out, nullptr, nullptr, 0.f,
                     0.f, reinterpret_cast<cudaStream_t>(stream), true);
}

adasum_status_t adasum_pair(const void* a, const void* b, int64_t n, adasum_dtype_t dtype,
                            void* out, adasum_stream_t stream) {
  if (n < 0 || a == nullptr || b == nullptr) return ADASUM_ERR_INVALID_ARG;
  const void* g[2] = {a, b};
  const int64_t offs[2] = {0, n};
  std::lock_guard<std::mutex> lock(g_mu);
  Range range("adasum_pair");
  return reduce_impl(g, 2, offs, 1, static_cast<int>(dtype), out, nullptr, nullptr, 0.f,
                     0.f, reinterpret_cast<cudaStream_t>(stream));
}

adasum_status_t adasum_reduce_momentum_sgd(const void* const* grads, int K,
                                           const int64_t* seg_offsets, int L,
                                           adasum_dtype_t grad_dtype, float* master_w,
                                           float* momentum, float lr, float mu,
                                           void* out_or_null, adasum_stream_t stream) {
  if (master_w == nullptr || momentum == nullptr) {
    // Nothing to update is only fine when there is nothing at all to do.
    if (L > 0 && seg_offsets != nullptr && seg_offsets[L] > 0) return ADASUM_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  Range range("adasum_reduce_momentum_sgd");
  if (master_w == nullptr) return ADASUM_OK;
  return reduce_impl(grads, K, seg_offsets, L, static_cast<int>(grad_dtype), out_or_null,
                     master_w, momentum, lr, mu, reinterpret_cast<cudaStream_t>(stream));
}

adasum_status_t adasum_get_last_error(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (cudaGetLastError() != cudaSuccess) return ADASUM_ERR_CUDA;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return ADASUM_ERR_CUDA;
  Workspace& ws = workspace_for(device);
  if (ws.d_error == nullptr) return ADASUM_OK;
  int h = 0;
  if (cudaMemcpy(&h, ws.d_error, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(ws.d_error, 0, sizeof h) != cudaSuccess)
    return ADASUM_ERR_CUDA;
  if (h & kErrBounds) return ADASUM_ERR_BOUNDS;
  return h ? ADASUM_ERR_TIMEOUT : ADASUM_OK;
}

const char* adasum_status_string(adasum_status_t s) {
  switch (s) {
    case ADASUM_OK: return "ADASUM_OK";
    case ADASUM_ERR_INVALID_ARG: return "ADASUM_ERR_INVALID_ARG";
    case ADASUM_ERR_UNSUPPORTED: return "ADASUM_ERR_UNSUPPORTED";
    case ADASUM_ERR_ALIAS: return "ADASUM_ERR_ALIAS";
    case ADASUM_ERR_NO_MEMORY: return "ADASUM_ERR_NO_MEMORY";
    case ADASUM_ERR_CUDA: return "ADASUM_ERR_CUDA";
    case ADASUM_ERR_TIMEOUT: return "ADASUM_ERR_TIMEOUT";
    case ADASUM_ERR_BOUNDS: return "ADASUM_ERR_BOUNDS";
  }
  return "ADASUM_ERR_UNKNOWN";
}

adasum_status_t adasum_release_workspace(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return ADASUM_ERR_CUDA;
  Workspace& ws = workspace_for(device);
  if (cudaDeviceSynchronize() != cudaSuccess) return ADASUM_ERR_CUDA;
  if (ws.buf) cudaFree(ws.buf);
  ws.buf = nullptr;
  ws.cap = 0;
  ws.last_flag_counts = nullptr;
  for (auto& p : ws.plans) free_plan(p);
  ws.plans.clear();
  for (auto& s : ws.side) s.destroy();
  if (ws.pair_buf) cudaFree(ws.pair_buf);
  ws.pair_buf = nullptr;
  ws.host.destroy();
  return ADASUM_OK;
}

int adasum_version(void) { return kVersion; }

int64_t adasum_debug_workspace_guards(void) {
#ifdef ADASUM_TEST_HOOKS
  std::lock_guard<std::mutex> lock(g_mu);
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return -1;
  Workspace& ws = workspace_for(device);
  if (cudaDeviceSynchronize() != cudaSuccess || ws.buf == nullptr) return -1;
  int64_t bad = 0;
  unsigned char h[kGuardBytes];
  for (size_t g : ws.guards) {
    if (g + kGuardBytes > ws.cap || cudaMemcpy(h, static_cast<char*>(ws.buf) + g, kGuardBytes,
                                               cudaMemcpyDeviceToHost) != cudaSuccess)
      return -1;
    for (size_t i = 0; i < kGuardBytes; ++i) bad += h[i] != kGuardByte;
  }
  return bad;
#else
  return -1;
#endif
}

int64_t adasum_recomputed_segments(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return -1;
  Workspace& ws = workspace_for(device);
  if (ws.last_flag_counts == nullptr) return 0;
  int counts[4] = {0, 0, 0, 0};
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(counts, ws.last_flag_counts, sizeof counts, cudaMemcpyDeviceToHost) != cudaSuccess)
    return -1;
  return static_cast<int64_t>(counts[1]) + counts[2] + counts[3];
}

int64_t adasum_launch_count(void) { return g_launches.load(); }

adasum_status_t adasum_profile_enable(int on) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_profiling = on != 0;
  return ADASUM_OK;
}

int adasum_profile_collect(adasum_kernel_stat_t* stats, int max_stats) {
  std::lock_guard<std::mutex> lock(g_mu);
  std::vector<adasum_kernel_stat_t> agg;
  for (auto& r : g_prof_pending) {
    float ms = 0.f;
    cudaEventSynchronize(r.stop);
    cudaEventElapsedTime(&ms, r.start, r.stop);
    adasum_kernel_stat_t* slot = nullptr;
    for (auto& s : agg)
      if (std::strncmp(s.name, r.name, sizeof s.name) == 0) slot = &s;
    if (!slot) {
      agg.push_back(adasum_kernel_stat_t{});
      slot = &agg.back();
      std::strncpy(slot->name, r.name, sizeof slot->name - 1);
    }
    slot->launches += 1;
    slot->total_ms += ms;
    slot->total_bytes += r.bytes;
    g_event_pool.push_back(r.start);
    g_event_pool.push_back(r.stop);
  }
  g_prof_pending.clear();
  const int n = std::min<int>(max_stats, static_cast<int>(agg.size()));
  for (int i = 0; i < n; ++i) stats[i] = agg[i];
  return static_cast<int>(agg.size());
}

}  // extern "C"
