// Host side of the GB300 angular-correlation library: the C ABI declared in include/acf.h.
//
// One acf_histogram call = catalog conversion (one or two launches) -> pair kernel (persistent
// blocks, one resident set per SM) -> merge kernel, all on the context's stream with no host
// synchronisation. See acf_kernels.cuh for the device side.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/acf.h"
#include "acf_kernels.cuh"

using namespace acf;

namespace {

constexpr int kK = 4;                          // i-galaxies per thread (32 * kK == kJT)
constexpr int kMaxEntries = 49152;             // entries a code may address (the shared-memory plan
                                               // binds first: 41,216 beside 512 threads' tiles)
constexpr size_t kWarpTileBytes = 2 * kJT * sizeof(float4);  // one warp's double-buffered j-tile
constexpr size_t kMaxSmem = 232448 - 2048;  // dynamic shared memory per block: 227 KB less the pair kernel's static arrays
constexpr int kMaxTimed = 4096;

struct Plan {
  BinParams bp;
  double w_rad = 0.0;
  int exact = 0;
  float exact_lo = 0.f;
  int map = kDirect;
  int method = kChordPoly;
  int layout = kLane;
  int threads = 256;
  size_t smem = 0;
  bool grouped = false;  // exact mode 2 with the block-shared histogram: group records, no queue
};

struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
};

// A call that repeats with the same arguments, options, stream and workspace replays a CUDA graph
// of its launches instead of launching each kernel (see GraphCache).
struct CallKey {
  int entry = 0;  // 1 acf_correlate, 2 acf_histogram, 3 acf_correlate_host
  const void* p[8] = {};
  long long n[2] = {};
  double w = 0.0;
  int nbins = 0;
  cudaStream_t stream = nullptr;
  const void* ws = nullptr;
  size_t ws_bytes = 0;
  const void* io = nullptr;  // acf_correlate_host's device staging
  size_t io_bytes = 0;
  // the options that shape the launches
  int threads = 0, ctas = 0, method = 0, layout = 0, exact = 0, range_forms = 0, unit_groups = 0, timing = 0;
  long long units_per_launch = 0, exact_queue = 0;
  double exact_below_deg = 0.0;
  bool operator==(const CallKey& o) const {
    return entry == o.entry && std::equal(p, p + 8, o.p) && n[0] == o.n[0] && n[1] == o.n[1] && w == o.w &&
           nbins == o.nbins && stream == o.stream && ws == o.ws && ws_bytes == o.ws_bytes && io == o.io &&
           io_bytes == o.io_bytes && threads == o.threads &&
           ctas == o.ctas && method == o.method && layout == o.layout && exact == o.exact &&
           range_forms == o.range_forms && unit_groups == o.unit_groups && timing == o.timing &&
           units_per_launch == o.units_per_launch &&
           exact_queue == o.exact_queue && exact_below_deg == o.exact_below_deg;
  }
};
// What a call leaves for acf_get_info on the host side (restored when a graph stands in for it).
struct CallInfo {
  unsigned int* last_counters = nullptr;
  long long last_qcap = 0, grid = 0, threads = 0, ctas = 0, chunks = 0, layout = 0, map = 0, entries = 0, smem = 0,
            pairs = 0, flush = 0, groups = 0;
};
struct CachedGraph {
  CallKey key;
  cudaGraph_t graph = nullptr;  // kept while its event nodes are rebound on every launch
  cudaGraphExec_t exec = nullptr;
  long long launches = 0;    // kernels in the graph
  unsigned long long used = 0;  // last use (for eviction)
  CallInfo info;             // the captured call's
  // kernel timing: the graph's event-record nodes and, for each, which of the call's events it is
  std::vector<std::pair<cudaGraphNode_t, int>> ev_nodes;
  int ev_count = 0;
  void release() {
    if (exec) cudaGraphExecDestroy(exec);
    if (graph) cudaGraphDestroy(graph);
    exec = nullptr;
    graph = nullptr;
    ev_nodes.clear();
    ev_count = 0;
  }
};
constexpr int kGraphSlots = 4;

}  // namespace

struct acf_ctx {
  int device = 0;
  cudaStream_t stream = nullptr;
  int num_sms = 0;
  std::string err;
  Workspace ws;     // vectors + per-block partial rows
  Workspace io;     // device staging for acf_correlate_host
  // options
  int opt_threads = 0, opt_ctas = 0, opt_method = kChordPoly, opt_layout = 0, opt_timing = 0;
  long long opt_units_per_launch = 0;
  long long opt_workspace_limit = 0;   // bytes a workspace may grow to (0: no limit)
  long long inject_launch_error = 0;   // fault injection: the n-th kernel launch from now reports an error
  int opt_exact = 2;              // 0 off, 1 near 0 and 180 degrees, 2 everywhere
  double opt_exact_below_deg = 20.0;
  int opt_range_forms = 1;        // 1: cheaper forms where the caps bound the separations
  int opt_pair_bins_form = 0;     // acf_pair_bins: 0 full-range chord form, 1 the range forms by own u.v
  int opt_unit_groups = 0;        // j-groups per work unit: 0 automatic, 4 (chunk pairs) or 1 (small problems)
  long long opt_exact_queue = 0;  // exact-mode queue records: 0 automatic, else this many (tests of overflow)
  int opt_graphs = 1;             // 1: repeated calls replay a CUDA graph of their launches
  // graph replay: calls seen once (captured when they repeat) and the captured graphs
  CallKey seen[kGraphSlots];
  int seen_next = 0;
  CachedGraph graphs[kGraphSlots];
  unsigned long long graph_clock = 0;
  long long graph_replays = 0;    // calls served by a graph
  bool capturing = false;         // the library is capturing a call (see run_graphed)
  CallInfo info() const {
    return CallInfo{last_counters, last_qcap, info_grid,  info_threads, info_ctas, info_chunks, info_layout,
                    info_map,      info_entries, info_smem, info_pairs, info_flush, info_groups};
  }
  void set_info(const CallInfo& i) {
    last_counters = i.last_counters;
    last_qcap = i.last_qcap;
    info_grid = i.grid;
    info_threads = i.threads;
    info_ctas = i.ctas;
    info_chunks = i.chunks;
    info_layout = i.layout;
    info_map = i.map;
    info_entries = i.entries;
    info_smem = i.smem;
    info_pairs = i.pairs;
    info_flush = i.flush;
    info_groups = i.groups;
  }
  unsigned int* last_counters = nullptr;  // device counters of the last histogram (ticket, slots, moved, flagged)
  long long last_qcap = 0;
  // info about the last histogram
  long long info_grid = 0, info_threads = 0, info_ctas = 0, info_chunks = 0, info_layout = 0, info_map = 0,
            info_entries = 0, info_smem = 0, info_pairs = 0, info_flush = 0, info_groups = 0;
  long long kernel_launches = 0;  // kernels this context has launched, over its lifetime
  // kernel timing
  std::vector<cudaEvent_t> ev;  // pairs (start, stop)
  int ev_used = 0;
};

namespace {

int fail(acf_ctx* c, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (c) c->err = buf;
  return code;
}

int cuda_fail(acf_ctx* c, cudaError_t e, const char* what) {
  return fail(c, ACF_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

#define ACF_CUDA(c, call)                                  \
  do {                                                     \
    cudaError_t e_ = (call);                               \
    if (e_ != cudaSuccess) return cuda_fail((c), e_, #call); \
  } while (0)

// Check a kernel launch just made on context c and count it. With the option
// "inject_launch_error" n, the n-th launch from then on is reported as failed (host-side fault
// injection: the launch itself ran normally and nothing touches the device).
#define ACF_LAUNCHED(c)                                                                                   \
  do {                                                                                                    \
    ACF_CUDA((c), cudaGetLastError());                                                                    \
    ++(c)->kernel_launches;                                                                               \
    if ((c)->inject_launch_error > 0 && --(c)->inject_launch_error == 0)                                  \
      return fail((c), ACF_ERR_CUDA, "injected launch failure (option inject_launch_error) after launch %lld", \
                  (c)->kernel_launches);                                                                  \
  } while (0)

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int ensure(acf_ctx* c, Workspace& w, size_t bytes) {
  if (bytes <= w.bytes) return ACF_OK;
  const size_t limit = c->opt_workspace_limit > 0 ? (size_t)c->opt_workspace_limit : SIZE_MAX;
  if (bytes > limit)
    return fail(c, ACF_ERR_NOMEM, "a workspace of %zu bytes exceeds the limit of %zu bytes (option workspace_limit)",
                bytes, limit);
  size_t want = std::min(std::max(bytes, w.bytes + w.bytes / 2), limit);
  if (w.ptr) {
    ACF_CUDA(c, cudaStreamSynchronize(c->stream));
    ACF_CUDA(c, cudaFree(w.ptr));
    w.ptr = nullptr;
    w.bytes = 0;
  }
  cudaError_t e = cudaMalloc(&w.ptr, want);
  if (e != cudaSuccess) {
    cudaGetLastError();
    w.ptr = nullptr;
    return fail(c, ACF_ERR_NOMEM, "cudaMalloc of %zu bytes failed: %s", want, cudaGetErrorString(e));
  }
  w.bytes = want;
  return ACF_OK;
}

// Work out the bin map, the shared-memory layout and the polynomial for one binning.
int make_plan(acf_ctx* c, double w_deg, int nbins, Plan& pl) {
  if (!(w_deg > 0.0) || !std::isfinite(w_deg)) return fail(c, ACF_ERR_ARG, "bin_width_deg must be finite and > 0");
  if (nbins <= 0) return fail(c, ACF_ERR_ARG, "nbins must be > 0");
  const double pi = 3.14159265358979323846;
  const double w_rad = w_deg * pi / 180.0;
  const double P = 180.0 / w_deg;  // bins in half a turn
  BinParams& bp = pl.bp;
  std::memset(&bp, 0, sizeof bp);
  bp.nbins = nbins;
  bp.inv_w = (float)(1.0 / w_rad);
  pl.method = c->opt_method;
  pl.w_rad = w_rad;
  const double pr = std::rint(P);
  const bool integral = std::fabs(P - pr) <= 1e-9 * std::max(1.0, P) && pr >= 4.0;
  // direct map: every code is floor(theta / w) exactly, in [0, P - 1] (near-side chords reach at
  // most P/2 + 1); two spare entries
  const long long direct_entries = integral ? (long long)pr + 2 : -1;
  if (pl.method == kChordPoly && integral && direct_entries <= kMaxEntries) {
    pl.map = kDirect;
    bp.entries = (int)direct_entries;
    bp.magic_far = (float)(8388608.0 + pr);
    bp.clamp_c = (float)(bp.entries - 1);
    // the dot form needs 2^23 + P/2 to be an integer
    bp.mid = (c->opt_range_forms && std::fmod(pr, 2.0) == 0.0) ? 1 : 0;
    bp.magic_mid = (float)(8388608.0 + pr / 2.0);
    for (int k = 0; k < kRTerms; ++k) bp.rc[k] = (float)(kR[k] / w_rad);
  } else {
    pl.map = kClamp;
    const double fp = std::floor(P * (1.0 + 1e-6)) + 1.0;  // indices the clamp-free range can reach
    const long long entries = (long long)std::min<double>((double)nbins, fp);
    if (entries > kMaxEntries)
      return fail(c, ACF_ERR_UNSUPPORTED, "histogram of %lld entries exceeds the %d-entry shared-memory plan",
                  entries, kMaxEntries);
    bp.entries = (int)entries;
    bp.clamp_c = (float)(entries - 1);
  }
  bp.small = c->opt_range_forms ? 1 : 0;
  // Exact mode: S fractional bits in the bin code make a window of 2^-S bins around every edge,
  // wider than the fp32 path's error there.
  pl.exact = (pl.method == kChordPoly) ? c->opt_exact : 0;
  pl.exact_lo = (float)(c->opt_exact_below_deg * pi / 180.0);
  if (pl.exact) {
    // Worst-case fp32 error of each form (every rounding aligned): the full-range chord <= 1.25e-6
    // rad (near 90 degrees), the short chord (theta' <= 72 deg) <= 1.05e-6, the dot form (55..125
    // deg) <= 6e-7. Mode 1 only re-decides separations within exact_lo of 0 or 180 degrees, where
    // the chord's error is err1(lo) (vectors, chord rounding ~ tan(theta'/2), polynomial, sqrt and
    // 1/w ~ theta'). Each form's S is the largest whose window 2^-S bins covers its bound.
    const double lo = std::min(c->opt_exact_below_deg, 90.0) * pi / 180.0;
    const double err1 = 1.2e-7 / std::cos(lo / 2) + 6e-7 * std::tan(lo / 2) + 5e-8 + 3.5e-7 * lo;
    const double err_full = (pl.exact == 2) ? 1.25e-6 : err1;
    const double err_small = (pl.exact == 2) ? 1.05e-6 : err1;
    const double err_mid = (pl.exact == 2) ? 6e-7 : err1;
    const int room = (int)std::floor(std::log2(8.0e6 / ((double)bp.entries + 2.0)));  // (entries+2) << S < 2^23
    auto shift_for = [&](double err) {
      return std::max(0, std::min((int)std::floor(std::log2(w_rad / err)), room));
    };
    const int S = shift_for(err_full), Ss = shift_for(err_small), Sm = shift_for(err_mid);
    bp.fine_shift = S;
    bp.fine_shift_small = Ss;
    bp.fine_shift_mid = Sm;
    bp.inv_w_f = (float)(std::ldexp(1.0, S) / w_rad);
    bp.inv_w_fs = (float)(std::ldexp(1.0, Ss) / w_rad);
    // fine codes carry a bias of one fine unit (see BinParams)
    bp.magic_f = 8388609.0f;
    if (pl.map == kDirect) {
      bp.magic_far_f = (float)(8388609.0 + std::ldexp(pr, S));
      bp.magic_far_fs = (float)(8388609.0 + std::ldexp(pr, Ss));
      bp.magic_mid_f = (float)(8388609.0 + std::ldexp(pr / 2.0, Sm));
      for (int k = 0; k < kRTerms; ++k) bp.rc_f[k] = (float)(std::ldexp(kR[k], Sm) / w_rad);
    }
    bp.clamp_f = (float)std::ldexp((double)bp.clamp_c + 0.5, S);
    bp.clamp_fs = (float)std::ldexp((double)bp.clamp_c + 0.5, Ss);
  }
  bp.kmax = (int)std::min<double>((double)nbins - 1.0, std::floor(P + 1e-9));
  // exact zone, as histogram entries: everything (mode 2), or separations within exact_lo of
  // 0 or 180 degrees (mode 1): entries <= L or >= floor(P) - L - 1 (both maps index entries by bin)
  bp.zone0 = 0u; bp.span0 = 0xFFFFFFFFu; bp.zone1 = 0u; bp.span1 = 0u;
  if (pl.exact == 1) {
    // L + 2 bins stay within exact_lo, so every zone pair sits in a j-group the caps mark for
    // re-decision (and bin by the chord form) whatever the grouping, and the set of re-decided
    // pairs is order-independent
    const long long L = std::max<long long>(0, (long long)std::floor(c->opt_exact_below_deg / w_deg) - 2);
    bp.zone0 = 0u;
    bp.span0 = (unsigned)L;
    bp.zone1 = (unsigned)std::max<long long>(0, (long long)std::floor(P + 1e-9) - L - 1);
    bp.span1 = 0xFFFFFFFFu - bp.zone1;
  }
  // Shared memory = every warp's double-buffered j-tile (4 KB per warp) + the histogram: 32
  // lane-private copies when they fit beside the tiles of at least 16 warps, else one block-shared
  // copy. 1024 threads (32 warps, one block per SM) when everything fits, else 512.
  const size_t lane_hist = (size_t)bp.entries * 32 * 4;
  const size_t block_hist = (size_t)((bp.entries * 4 + 15) & ~15);
  // (option 3, built with -DACF_U16_HIST=1 and exact mode 0 only: two copies of 16-bit counters)
  const size_t block16_hist = (size_t)((2 * ((bp.entries + 1) / 2) * 4 + 15) & ~15);
  int layout = c->opt_layout;
  if (layout == 0) layout = (lane_hist + 16 * kWarpTileBytes <= kMaxSmem) ? kLane : kBlock;
  if (layout == kBlock16 && (!ACF_U16_HIST || pl.exact))
    return fail(c, ACF_ERR_UNSUPPORTED, "layout 3 (16-bit counters) needs a build with ACF_U16_HIST and exact mode 0");
  const size_t hist_bytes = (layout == kLane) ? lane_hist : (layout == kBlock16 ? block16_hist : block_hist);
  int threads = c->opt_threads;
  if (threads == 0) threads = (hist_bytes + 32 * kWarpTileBytes <= kMaxSmem) ? 1024 : 512;
  if (threads != 512 && threads != 1024) return fail(c, ACF_ERR_ARG, "threads must be 512 or 1024");
  pl.layout = layout;
  pl.threads = threads;
  pl.grouped = layout == kBlock && pl.exact == 2 && pl.method == kChordPoly;
  pl.smem = hist_bytes + (size_t)(threads / 32) * kWarpTileBytes;
  if (pl.smem > kMaxSmem)
    return fail(c, ACF_ERR_UNSUPPORTED, "%s histogram of %d entries with %d threads needs %zu bytes of shared memory",
                layout == kLane ? "lane-private" : (layout == kBlock16 ? "16-bit block-shared" : "block-shared"),
                bp.entries, threads, pl.smem);
  return ACF_OK;
}

typedef void (*PairKernelFn)(const PairParams);

// small: units of one 32-galaxy j-group (lane-private layout, 1024 threads, chord method only)
PairKernelFn pick_kernel(const Plan& pl, bool small) {
  // the block-shared histogram in exact mode 2 takes the build without the plain loops
  const int layout = (pl.layout == kBlock && pl.exact == 2 && pl.method == kChordPoly) ? kBlockExact : pl.layout;
  if (small) {
    if (pl.threads == 1024 && layout == kLane && pl.method == kChordPoly)
      return pl.map == kDirect ? pair_kernel<kK, 1024, kLane, kDirect, kChordPoly, 1>
                               : pair_kernel<kK, 1024, kLane, kClamp, kChordPoly, 1>;
    return nullptr;
  }
#define ACF_PICK(T, L, M, X) \
  if (pl.threads == T && layout == L && pl.map == M && pl.method == X) return pair_kernel<kK, T, L, M, X>;
  ACF_PICK(1024, kLane, kDirect, kChordPoly)
  ACF_PICK(1024, kLane, kClamp, kChordPoly)
  ACF_PICK(1024, kBlock, kDirect, kChordPoly)
  ACF_PICK(1024, kBlock, kClamp, kChordPoly)
  ACF_PICK(1024, kBlockExact, kDirect, kChordPoly)
  ACF_PICK(1024, kBlockExact, kClamp, kChordPoly)
  ACF_PICK(512, kLane, kDirect, kChordPoly)
  ACF_PICK(512, kLane, kClamp, kChordPoly)
  ACF_PICK(512, kBlock, kDirect, kChordPoly)
  ACF_PICK(512, kBlock, kClamp, kChordPoly)
  ACF_PICK(512, kBlockExact, kDirect, kChordPoly)
  ACF_PICK(512, kBlockExact, kClamp, kChordPoly)
#if ACF_U16_HIST
  ACF_PICK(1024, kBlock16, kDirect, kChordPoly)
  ACF_PICK(1024, kBlock16, kClamp, kChordPoly)
  ACF_PICK(512, kBlock16, kDirect, kChordPoly)
  ACF_PICK(512, kBlock16, kClamp, kChordPoly)
#endif
  ACF_PICK(1024, kLane, kClamp, kDotAcos)
  ACF_PICK(1024, kBlock, kClamp, kDotAcos)
  ACF_PICK(512, kLane, kClamp, kDotAcos)
  ACF_PICK(512, kBlock, kClamp, kDotAcos)
  ACF_PICK(1024, kLane, kClamp, kDotFastAcos)
  ACF_PICK(1024, kBlock, kClamp, kDotFastAcos)
  ACF_PICK(512, kLane, kClamp, kDotFastAcos)
  ACF_PICK(512, kBlock, kClamp, kDotFastAcos)
#undef ACF_PICK
  return nullptr;
}

// Device buffers of one histogram call, carved out of one scratch region.
struct CatBufs {
  float4* v = nullptr;       // unit vectors in spatial order (fp32)
  DsVec* ds = nullptr;       // double-single vectors (v and what fp32 leaves of the fp64 components)
  double4_32a* v64 = nullptr;    // the same in fp64 (exact re-decision)
  float4* cap32 = nullptr;   // caps of 32-galaxy groups (4 per 128-chunk)
  float4* cap128 = nullptr;  // caps of 128-galaxy chunks
  unsigned int* key0 = nullptr;    // sort: cell keys in input order, at the end the order
  unsigned int* key1 = nullptr;    // sort: keys after the first pass
  unsigned int* idx1 = nullptr;    // sort: input indices after the first pass
  unsigned int* counts = nullptr;  // sort: digit counts per tile, then their offsets
};
struct Scratch {
  unsigned int* counters = nullptr;    // [0] unit ticket, [1] queue spill records handed out (this launch),
                                       // [2] moved pairs, [3] flagged pairs, [4] flagged pairs without a
                                       // record slot, [5] pairs the fix-up redid in fp64;
                                       // bytes 64..135: pairs per path (u64)
  CatBufs a, b;                        // b only for cross-correlations
  unsigned long long* partial = nullptr;
  unsigned long long* delta = nullptr; // exact mode: count moves of the exact re-decision, per bin
  double* T = nullptr;                 // exact mode: edge tables, nbins + 1 each
  double* U = nullptr;
  float2* Tds = nullptr;               // the same as double-single (hi, lo) pairs
  float2* Uds = nullptr;
  int* kd = nullptr;                   // the last bin re-decided with T (difference chord)
  uint2* qhdr = nullptr;               // exact mode: flag records, headers ..
  uint4* qmask = nullptr;              // .. and lane ballots
  unsigned int* qused = nullptr;       // per pair-kernel warp: records of its queue region in use
  long long qcap = 0;
  unsigned int* gbal = nullptr;        // exact mode with group records: lane ballots and records of
  GroupRecord* grec = nullptr;         // .. gunits units (4 groups of 32 lanes each)
  long long gunits = 0;
};

// the fix-up's shared moves and tables at most: several 256-thread blocks per SM still fit, since the
// kernel waits on loads and needs every warp it can get
constexpr size_t kFixupSmemMax = 24 * 1024;
constexpr long long kQueueCapMin = 1ll << 20;  // flag records the workspace can hold: 24 MB ..
constexpr long long kQueueCapMax = 1ll << 28;  // .. 6 GB
constexpr size_t kRecordBytes = sizeof(uint2) + sizeof(uint4);
constexpr size_t kGroupUnitBytes = 4 * sizeof(unsigned int) + kJT * sizeof(GroupRecord);  // group records of a unit

// Lay the buffers out from `base` (nullptr: only measure). Returns the bytes needed.
size_t carve(char* base, long long n, long long nj, bool sym, long long grid, int nbins, long long qcap, long long gunits,
             Scratch* s) {
  size_t off = 0;
  auto take = [&](size_t bytes) -> char* {
    char* p = base ? base + off : nullptr;
    off += align256(bytes);
    return p;
  };
  auto cat = [&](long long m, CatBufs& cb) {
    const long long ch = (m + 127) / 128;
    const long long tiles = (m + kSortTile - 1) / kSortTile;
    cb.key0 = reinterpret_cast<unsigned int*>(take((size_t)m * 4));
    cb.key1 = reinterpret_cast<unsigned int*>(take((size_t)m * 4));
    cb.idx1 = reinterpret_cast<unsigned int*>(take((size_t)m * 4));
    cb.counts = reinterpret_cast<unsigned int*>(take((size_t)tiles * kSortDigits * 4));
    cb.v = reinterpret_cast<float4*>(take((size_t)m * 16));
    cb.ds = reinterpret_cast<DsVec*>(take((size_t)m * sizeof(DsVec)));
    cb.v64 = reinterpret_cast<double4_32a*>(take((size_t)m * 32));
    cb.cap32 = reinterpret_cast<float4*>(take((size_t)ch * 4 * 16));
    cb.cap128 = reinterpret_cast<float4*>(take((size_t)ch * 16));
  };
  Scratch t;
  Scratch& r = s ? *s : t;
  r.counters = reinterpret_cast<unsigned int*>(take(256));
  cat(n, r.a);
  if (!sym) cat(nj, r.b);
  r.partial = reinterpret_cast<unsigned long long*>(take((size_t)grid * (size_t)nbins * 8));
  r.delta = reinterpret_cast<unsigned long long*>(take((size_t)nbins * 8));
  r.T = reinterpret_cast<double*>(take((size_t)(nbins + 1) * 8));
  r.U = reinterpret_cast<double*>(take((size_t)(nbins + 1) * 8));
  r.Tds = reinterpret_cast<float2*>(take((size_t)(nbins + 1) * 8));
  r.Uds = reinterpret_cast<float2*>(take((size_t)(nbins + 1) * 8));
  r.kd = reinterpret_cast<int*>(take(sizeof(int)));
  r.qcap = qcap;
  r.qused = reinterpret_cast<unsigned int*>(take((size_t)grid * 32 * 4));  // up to 32 warps per block
  r.qhdr = reinterpret_cast<uint2*>(take((size_t)qcap * sizeof(uint2)));
  r.qmask = reinterpret_cast<uint4*>(take((size_t)qcap * sizeof(uint4)));
  r.gunits = gunits;
  r.gbal = reinterpret_cast<unsigned int*>(take((size_t)gunits * 4 * sizeof(unsigned int)));
  r.grec = reinterpret_cast<GroupRecord*>(take((size_t)gunits * kJT * sizeof(GroupRecord)));
  return off;
}

// Unit vectors of one or two catalogs in spatial order (a stable radix sort on the cell key: low 8
// bits, then high 7; then the fp64 vectors in that order), with their caps. Both catalogs of a
// cross-correlation go through the same eight launches (blockIdx.y selects the catalog).
int prepare_catalogs(acf_ctx* c, int count, const float* const ra[2], const float* const dec[2], const long long n[2],
                     const CatBufs* const cb[2]) {
  PrepBatch b;
  std::memset(&b, 0, sizeof b);
  int tiles_max = 0;
  long long n_max = 0;
  for (int k = 0; k < count; ++k) {
    PrepCat& C = b.c[k];
    C.ra = ra[k];
    C.dec = dec[k];
    C.n = n[k];
    C.tiles = (int)((n[k] + kSortTile - 1) / kSortTile);
    C.key0 = cb[k]->key0;
    C.key1 = cb[k]->key1;
    C.idx1 = cb[k]->idx1;
    C.counts = cb[k]->counts;
    C.v = cb[k]->v;
    C.ds = cb[k]->ds;
    C.v64 = cb[k]->v64;
    C.cap32 = cb[k]->cap32;
    C.cap128 = cb[k]->cap128;
    tiles_max = std::max(tiles_max, C.tiles);
    n_max = std::max(n_max, n[k]);
  }
  const dim3 tiles_grid((unsigned)tiles_max, (unsigned)count), one(1, (unsigned)count);
  sort_count_kernel<true><<<tiles_grid, kSortThreads, 0, c->stream>>>(b, 0);
  ACF_LAUNCHED(c);
  scan_kernel<<<one, 1024, 0, c->stream>>>(b);
  ACF_LAUNCHED(c);
  sort_scatter_kernel<false><<<tiles_grid, kSortThreads, 0, c->stream>>>(b, 0);
  ACF_LAUNCHED(c);
  sort_count_kernel<false><<<tiles_grid, kSortThreads, 0, c->stream>>>(b, 8);
  ACF_LAUNCHED(c);
  scan_kernel<<<one, 1024, 0, c->stream>>>(b);
  ACF_LAUNCHED(c);
  sort_scatter_kernel<true><<<tiles_grid, kSortThreads, 0, c->stream>>>(b, 8);
  ACF_LAUNCHED(c);
  const long long vblocks = std::min<long long>((n_max + 255) / 256, (long long)c->num_sms * 8 / count);
  vectors_kernel<<<dim3((unsigned)std::max<long long>(vblocks, 1), (unsigned)count), 256, 0, c->stream>>>(b);
  ACF_LAUNCHED(c);
  const long long warps = (n_max + 127) / 128;
  caps_kernel<<<dim3((unsigned)((warps * 32 + 255) / 256), (unsigned)count), 256, 0, c->stream>>>(b);
  ACF_LAUNCHED(c);
  return ACF_OK;
}

struct Launch {
  PairKernelFn fn = nullptr;
  int ctas = 0;
  long long grid = 0, units = 0, rows = 0, cols = 0, per_launch = 0;
  bool small = false;  // units of one j-group (four per chunk pair)
};

// Below this many chunk-pair units per resident warp a problem takes units of one j-group.
constexpr double kSmallUnitsPerWarp = 2.0;

// Persistent grid: every SM gets as many blocks as can be resident (one, normally).
int plan_launch(acf_ctx* c, const Plan& pl, long long ni, long long nj, bool sym, Launch& L) {
  L.rows = (ni + kJT - 1) / kJT;
  L.cols = (nj + kJT - 1) / kJT;
  const long long chunk_units = sym ? L.rows * L.cols - L.rows * (L.rows - 1) / 2 : L.rows * L.cols;
  // few chunk pairs for the warps of the whole GPU: four units per chunk pair, if a kernel exists
  const bool few = chunk_units < kSmallUnitsPerWarp * c->num_sms * (pl.threads / 32);
  L.small = (c->opt_unit_groups == 1 || (c->opt_unit_groups == 0 && few)) && pick_kernel(pl, true) != nullptr;
  L.fn = pick_kernel(pl, L.small);
  if (!L.fn) return fail(c, ACF_ERR_UNSUPPORTED, "no kernel for this plan");
  ACF_CUDA(c, cudaFuncSetAttribute(L.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem));
  int occ = 0;
  ACF_CUDA(c, cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, L.fn, pl.threads, pl.smem));
  if (occ <= 0) return fail(c, ACF_ERR_UNSUPPORTED, "pair kernel cannot be resident (smem %zu)", pl.smem);
  L.ctas = c->opt_ctas > 0 ? std::min(c->opt_ctas, occ) : occ;
  L.units = L.small ? 4 * chunk_units : chunk_units;
  L.grid = std::min<long long>((long long)c->num_sms * L.ctas, std::max<long long>(L.units, 1));
  // One unit adds at most kK*kJT*inc to a lane-private 32-bit counter (32 times that to a
  // block-shared one). Even if one block took every unit of a launch, no counter may wrap, so
  // large problems are split into launches that add into the same block rows.
  const double inc = sym ? 2.0 : 1.0;
  const double per_unit = (pl.layout == kLane ? 1.0 : 32.0) * kK * (L.small ? 32 : kJT) * inc;
  L.per_launch = (long long)std::floor(4294967295.0 / per_unit);
  if (c->opt_units_per_launch > 0) L.per_launch = std::min(L.per_launch, c->opt_units_per_launch);
  return ACF_OK;
}

// Every pair a launch flagged near an edge is re-decided exactly; its count moves if the bin differs.
// The per-bin moves (int32 per block) and, when they fit too, the double-single edge tables go to
// shared memory if small.
int launch_fixup(acf_ctx* c, const Plan& pl, const Launch& L, const PairParams& p, const Scratch& sc,
                 const CatBufs& ci, const CatBufs& cj) {
  const long long regions = L.grid * (pl.threads / 32);
  const int nb = pl.bp.nbins;
  const size_t moves = ((size_t)nb * 4 + 15) & ~(size_t)15, tables = (size_t)(nb + 1) * 16;
  const int level = moves + tables <= kFixupSmemMax ? 2 : (moves <= kFixupSmemMax ? 1 : 0);
  const size_t fsmem = level == 2 ? moves + tables : (level == 1 ? moves : 0);
  constexpr int fwpb = kFixupThreads / 32;  // warps per block
  // per-j records: one warp per region; group records: enough warps for the batches of groups,
  // as many blocks as are resident at once (they take batches from a ticket)
  const long long ngroups = (p.unit_end - p.unit_begin) * 4;
  // group records: kFixupBatch groups per ticket where a lane's 128 pairs of a group hold a flag
  // more often than not (probability ~ 1 - (1 - 2^(1 - S))^128, S the short chord's fine bits:
  // 0.87 at 0.01 deg bins), else 32
  const double prec = 1.0 - std::pow(1.0 - std::ldexp(1.0, 1 - pl.bp.fine_shift_small), 128.0);
  const int gbatch = prec > 0.5 ? kFixupBatch : 32;
  const long long fwarps = pl.grouped ? std::min<long long>((ngroups + gbatch - 1) / gbatch,
                                                            (long long)c->num_sms * ACF_FIXUP_MINB * fwpb)
                                      : regions;
  const unsigned fblocks = (unsigned)std::max<long long>(1, (fwarps + fwpb - 1) / fwpb);
  FixupParams f;
  f.qhdr = sc.qhdr;
  f.qmask = sc.qmask;
  f.qused = sc.qused;
  f.qspill = sc.counters + 1;
  f.regions = (unsigned)regions;
  f.qbatch = p.qbatch;
  f.qcap = p.qcap;
  f.ds_i = ci.ds;
  f.ds_j = cj.ds;
  f.vi = ci.v64;
  f.vj = cj.v64;
  f.T = sc.T;
  f.U = sc.U;
  f.Tds = sc.Tds;
  f.Uds = sc.Uds;
  f.kd = sc.kd;
  f.bp = pl.bp;
  f.inc = p.inc;
  f.delta = sc.delta;
  f.moved = sc.counters + 2;
  f.redone = sc.counters + 5;
  f.flagged = sc.counters + 3;
  f.gbal = sc.gbal;
  f.grec = sc.grec;
  f.ngroups = pl.grouped ? (unsigned long long)ngroups : 0ull;
  f.gticket = sc.counters + 1;  // (the spill counter of per-j records; zero before every pair launch)
#define ACF_FIXUP(M, SM, G) fixup_kernel<M, SM, G><<<fblocks, kFixupThreads, fsmem, c->stream>>>(f)
#define ACF_FIXUP_LEVELS(M, G)      \
  if (level == 2) ACF_FIXUP(M, 2, G); \
  else if (level == 1) ACF_FIXUP(M, 1, G); \
  else ACF_FIXUP(M, 0, G);
  if (pl.map == kDirect) {
    if (!pl.grouped) { ACF_FIXUP_LEVELS(kDirect, 0) }
    else if (gbatch == kFixupBatch) { ACF_FIXUP_LEVELS(kDirect, kFixupBatch) }
    else { ACF_FIXUP_LEVELS(kDirect, 32) }
  } else {
    if (!pl.grouped) { ACF_FIXUP_LEVELS(kClamp, 0) }
    else if (gbatch == kFixupBatch) { ACF_FIXUP_LEVELS(kClamp, kFixupBatch) }
    else { ACF_FIXUP_LEVELS(kClamp, 32) }
  }
#undef ACF_FIXUP_LEVELS
#undef ACF_FIXUP
  ACF_LAUNCHED(c);
  return ACF_OK;
}

// The pair kernel (one or more launches) and the merge for prepared catalogs.
int histogram_vectors(acf_ctx* c, const CatBufs& ci, long long ni, const CatBufs& cj, long long nj, bool sym,
                      const Plan& pl, const Launch& L, const Scratch& sc, uint64_t* out) {
  unsigned long long* partial = sc.partial;
  unsigned int* ticket = sc.counters;
  ACF_CUDA(c, cudaMemsetAsync(sc.counters, 0, 256, c->stream));  // ticket, queue, path counters
  // exact mode needs its queue (per-j records) or its group records
  const bool exact_on = pl.exact && (pl.grouped ? sc.gunits > 0 : sc.qcap > 0);
  if (exact_on) ACF_CUDA(c, cudaMemsetAsync(sc.delta, 0, (size_t)pl.bp.nbins * 8, c->stream));
  PairParams p;
  p.exact_mode = exact_on ? pl.exact : 0;
  p.exact_lo = pl.exact_lo;
  p.qhdr = sc.qhdr;
  p.qmask = sc.qmask;
  p.qspill = sc.counters + 1;
  p.qused = sc.qused;
  p.qflagged = sc.counters + 3;
  p.qoverflow = sc.counters + 4;
  p.qcap = (unsigned int)std::min<long long>(sc.qcap, 0xFFFFFFFFll);
  // each warp owns a region of the queue: two thirds of the queue spread over the warps of a launch,
  // at least what a warp records on average (the queue is drained after every launch). Warps that
  // record more append to the spill region through one global counter, which all warps contend
  // for, so the regions must hold nearly everything.
  p.qbatch = (unsigned int)std::min<long long>((long long)p.qcap * 2 / 3 / std::max<long long>(L.grid * (pl.threads / 32), 1),
                                               0x7FFFFFFFll);
  p.path_pairs = reinterpret_cast<unsigned long long*>(sc.counters + 16);
  p.gbal = sc.gbal;
  p.grec = sc.grec;
  if (pl.grouped && sc.gunits < std::min(L.units, L.per_launch))
    return fail(c, ACF_ERR_UNSUPPORTED, "group records for %lld units, a launch takes %lld", sc.gunits,
                std::min(L.units, L.per_launch));
  p.vi = ci.v;
  p.vj = cj.v;
  p.icap32 = ci.cap32;
  p.jcap32 = cj.cap32;
  p.igroups = (ni + 31) / 32;
  p.ni = ni;
  p.nj = nj;
  p.rows = L.rows;
  p.cols = L.cols;
  p.sym = sym ? 1 : 0;
  p.inc = sym ? 2u : 1u;
  p.partial = partial;
  p.ticket = ticket;
  p.bp = pl.bp;
  int launches = 0;
  for (long long ub = 0; ub < L.units; ub += L.per_launch, ++launches) {
    p.unit_begin = ub;
    p.unit_end = std::min(L.units, ub + L.per_launch);
    p.accumulate = ub > 0 ? 1 : 0;
    if (ub > 0) ACF_CUDA(c, cudaMemsetAsync(ticket, 0, 8, c->stream));  // ticket and queue slots
    // kernel_timing 1: events around the pair kernel; 2: around the fix-up
    const bool timed = c->opt_timing && c->ev_used + 2 <= (int)c->ev.size();
    // (while the library captures the call, external records: event nodes of the graph)
    const unsigned rec = c->capturing ? cudaEventRecordExternal : cudaEventRecordDefault;
    if (timed && c->opt_timing == 1)
      ACF_CUDA(c, cudaEventRecordWithFlags(c->ev[c->ev_used], c->stream, rec));
    L.fn<<<(unsigned)L.grid, pl.threads, pl.smem, c->stream>>>(p);
    ACF_LAUNCHED(c);
    if (timed && c->opt_timing == 1) {
      ACF_CUDA(c, cudaEventRecordWithFlags(c->ev[c->ev_used + 1], c->stream, rec));
      c->ev_used += 2;
    }
    if (p.exact_mode) {
      if (timed && c->opt_timing == 2)
        ACF_CUDA(c, cudaEventRecordWithFlags(c->ev[c->ev_used], c->stream, rec));
      const int frc = launch_fixup(c, pl, L, p, sc, ci, cj);
      if (frc) return frc;
      if (timed && c->opt_timing == 2) {
        ACF_CUDA(c, cudaEventRecordWithFlags(c->ev[c->ev_used + 1], c->stream, rec));
        c->ev_used += 2;
      }
    }
  }
#ifdef ACF_DEBUG_BOUNDS
  {
    DebugRecord r;
    ACF_CUDA(c, cudaStreamSynchronize(c->stream));
    ACF_CUDA(c, cudaMemcpyFromSymbol(&r, g_debug, sizeof r));
    if (r.count) {
      DebugRecord z{};
      ACF_CUDA(c, cudaMemcpyToSymbol(g_debug, &z, sizeof z));
      return fail(c, ACF_ERR_CUDA,
                  "bounds check: %u violations; first kind %d a=%lld b=%lld f=[%.9g %.9g %.9g %.9g %.9g %.9g %.9g %.9g]",
                  r.count, r.kind, r.a, r.b, r.f[0], r.f[1], r.f[2], r.f[3], r.f[4], r.f[5], r.f[6], r.f[7]);
    }
  }
#endif
  const unsigned long long self = sym ? (unsigned long long)ni : 0ull;
  const int mblocks = (pl.bp.nbins + 31) / 32;
  merge_kernel<<<mblocks, 32 * kMergeWarps, 0, c->stream>>>(partial, (int)L.grid, pl.bp.nbins, self,
                                                             p.exact_mode ? sc.delta : nullptr,
                                                             reinterpret_cast<unsigned long long*>(out));
  ACF_LAUNCHED(c);
  c->last_counters = sc.counters;
  c->last_qcap = p.exact_mode ? (pl.grouped ? sc.gunits : (long long)p.qcap) : 0;
  c->info_grid = L.grid;
  c->info_groups = L.small ? 1 : 4;
  c->info_threads = pl.threads;
  c->info_ctas = L.ctas;
  c->info_chunks = L.units;
  c->info_layout = pl.layout;
  c->info_map = pl.map;
  c->info_entries = pl.bp.entries;
  c->info_smem = (long long)pl.smem;
  c->info_pairs = sym ? ni * (ni - 1) / 2 : ni * nj;
  c->info_flush = launches;
  return ACF_OK;
}

// Everything after argument checks and workspace layout: prepare the catalogs, pair, merge,
// and (exact mode) re-decide the flagged pairs.
int run_pipeline(acf_ctx* c, const float* ra, const float* dec, long long n, const float* ra2, const float* dec2,
                 long long nj, bool sym, const Plan& pl, const Launch& L, const Scratch& sc, uint64_t* out) {
  const float* const ras[2] = {ra, ra2};
  const float* const decs[2] = {dec, dec2};
  const long long ns[2] = {n, nj};
  const CatBufs* const cbs[2] = {&sc.a, &sc.b};
  int rc = prepare_catalogs(c, sym ? 1 : 2, ras, decs, ns, cbs);
  if (rc) return rc;
  if (pl.exact && (sc.qcap > 0 || sc.gunits > 0)) {
    edge_table_kernel<<<(pl.bp.nbins + 256) / 256, 256, 0, c->stream>>>(pl.w_rad, pl.bp.nbins, pl.bp.kmax, sc.T, sc.U,
                                                                         sc.Tds, sc.Uds, sc.kd);
    ACF_LAUNCHED(c);
  }
  return histogram_vectors(c, sc.a, n, sym ? sc.a : sc.b, nj, sym, pl, L, sc, out);
}

// Exact-mode queue records for a histogram of `units` work units: every computed pair may be flagged
// with probability up to 2^(1-S) (S of the full-range chord, the smallest), and a record holds at
// least one flagged pair: twice that. A record stands for one warp and one j, so there are never more
// than pairs / 128 of them: where flags are that dense, one and a half times that. Within bounds.
// Overflow is not an error: those pairs keep their fp32 bin, and "exact_overflow" counts them.
long long queue_slots(const acf_ctx* c, const Plan& pl, long long units) {
  // the queue is drained after every launch: it holds one launch's flagged pairs
  if (!pl.exact || pl.grouped) return 0;
  if (c->opt_exact_queue > 0) return c->opt_exact_queue;
  const double pairs = (double)units * kJT * kJT;
  const double want = std::min(4.0 * pairs * std::ldexp(1.0, -pl.bp.fine_shift), 1.5 * pairs / kJT);
  return (long long)std::min<double>(kQueueCapMax, std::max<double>(kQueueCapMin, want));
}

// Group records (exact mode 2, block-shared histogram): every unit of a launch has its slots, so
// they never overflow.
long long group_units(const Plan& pl, long long units) { return pl.grouped ? units : 0; }

int launch_omega(acf_ctx* c, const uint64_t* dd, const uint64_t* dr, const uint64_t* rr, int32_t nbins, int64_t n_d,
                 int64_t n_r, double* omega) {
  const double nd = (double)n_d, nr = (double)n_r;
  const double f_dd = (nr * nr) / (nd * nd), f_dr = (nr * nr) / (nd * nr);
  const int threads = 256;
  const int blocks = std::min((nbins + threads - 1) / threads, 4096);
  omega_kernel<<<blocks, threads, 0, c->stream>>>(reinterpret_cast<const unsigned long long*>(dd),
                                                   reinterpret_cast<const unsigned long long*>(dr),
                                                   reinterpret_cast<const unsigned long long*>(rr), nbins, f_dd, f_dr,
                                                   omega);
  ACF_LAUNCHED(c);
  return ACF_OK;
}

// DD, DR, RR and omega from device catalogs: each catalog is sorted and converted once, the
// edge tables built once, then the three histograms run back to back on the same workspace.
int correlate_impl(acf_ctx* c, const float* ra_d, const float* dec_d, int64_t n_d, const float* ra_r,
                   const float* dec_r, int64_t n_r, double w_deg, int32_t nbins, uint64_t* dd, uint64_t* dr,
                   uint64_t* rr, double* omega) {
  if (!ra_d || !dec_d || !ra_r || !dec_r || !dd || !dr || !rr || !omega)
    return fail(c, ACF_ERR_ARG, "correlate: NULL pointer");
  if (n_d <= 0 || n_r <= 0) return fail(c, ACF_ERR_ARG, "correlate: n_d and n_r must be > 0");
  if (n_d > 2147483647ll || n_r > 2147483647ll) return fail(c, ACF_ERR_UNSUPPORTED, "catalogs are limited to 2^31-1 galaxies");
  Plan pl;
  int rc = make_plan(c, w_deg, nbins, pl);
  if (rc) return rc;
  ACF_CUDA(c, cudaSetDevice(c->device));
  Launch Ldd, Ldr, Lrr;
  if ((rc = plan_launch(c, pl, n_d, n_d, true, Ldd)) || (rc = plan_launch(c, pl, n_d, n_r, false, Ldr)) ||
      (rc = plan_launch(c, pl, n_r, n_r, true, Lrr)))
    return rc;
  const long long grid = std::max(Ldd.grid, std::max(Ldr.grid, Lrr.grid));
  const long long units = std::max(std::min(Ldd.units, Ldd.per_launch),
                                   std::max(std::min(Ldr.units, Ldr.per_launch), std::min(Lrr.units, Lrr.per_launch)));
  const long long qcap = queue_slots(c, pl, units), gunits = group_units(pl, units);
  rc = ensure(c, c->ws, carve(nullptr, n_d, n_r, false, grid, nbins, qcap, gunits, nullptr));
  if (rc) return rc;
  Scratch sc;
  carve(static_cast<char*>(c->ws.ptr), n_d, n_r, false, grid, nbins, qcap, gunits, &sc);
  {
    const float* const ras[2] = {ra_d, ra_r};
    const float* const decs[2] = {dec_d, dec_r};
    const long long ns[2] = {n_d, n_r};
    const CatBufs* const cbs[2] = {&sc.a, &sc.b};
    if ((rc = prepare_catalogs(c, 2, ras, decs, ns, cbs))) return rc;
  }
  if (pl.exact && (sc.qcap > 0 || sc.gunits > 0)) {
    edge_table_kernel<<<(pl.bp.nbins + 256) / 256, 256, 0, c->stream>>>(pl.w_rad, pl.bp.nbins, pl.bp.kmax, sc.T, sc.U,
                                                                         sc.Tds, sc.Uds, sc.kd);
    ACF_LAUNCHED(c);
  }
  if ((rc = histogram_vectors(c, sc.a, n_d, sc.a, n_d, true, pl, Ldd, sc, dd)) ||
      (rc = histogram_vectors(c, sc.a, n_d, sc.b, n_r, false, pl, Ldr, sc, dr)) ||
      (rc = histogram_vectors(c, sc.b, n_r, sc.b, n_r, true, pl, Lrr, sc, rr)))
    return rc;
  return launch_omega(c, dd, dr, rr, nbins, n_d, n_r, omega);
}

int histogram_impl(acf_ctx* c, const float* ra, const float* dec, int64_t n, const float* ra2, const float* dec2,
                   int64_t n2, double w_deg, int32_t nbins, uint64_t* out) {
  if (!c) return ACF_ERR_ARG;
  if (n < 0) return fail(c, ACF_ERR_ARG, "n must be >= 0");
  if (n > 2147483647ll || n2 > 2147483647ll) return fail(c, ACF_ERR_UNSUPPORTED, "catalogs are limited to 2^31-1 galaxies");
  if (!out) return fail(c, ACF_ERR_ARG, "out is NULL");
  const bool sym = (ra2 == nullptr && dec2 == nullptr) || (ra2 == ra && dec2 == dec && n2 == n);
  if (!sym && n2 < 0) return fail(c, ACF_ERR_ARG, "n2 must be >= 0");
  if (!sym && ((ra2 == nullptr) != (dec2 == nullptr))) return fail(c, ACF_ERR_ARG, "ra2 and dec2 must both be set");
  const int64_t nj = sym ? n : n2;
  Plan pl;
  int rc = make_plan(c, w_deg, nbins, pl);
  if (rc) return rc;
  ACF_CUDA(c, cudaSetDevice(c->device));
  if (n == 0 || nj == 0) {
    ACF_CUDA(c, cudaMemsetAsync(out, 0, sizeof(uint64_t) * (size_t)nbins, c->stream));
    return ACF_OK;
  }
  if (!ra || !dec || (!sym && (!ra2 || !dec2))) return fail(c, ACF_ERR_ARG, "catalog pointer is NULL");
  Launch L;
  rc = plan_launch(c, pl, n, nj, sym, L);
  if (rc) return rc;
  const long long units = std::min(L.units, L.per_launch);
  const long long qcap = queue_slots(c, pl, units), gunits = group_units(pl, units);
  rc = ensure(c, c->ws, carve(nullptr, n, nj, sym, L.grid, nbins, qcap, gunits, nullptr));
  if (rc) return rc;
  Scratch sc;
  carve(static_cast<char*>(c->ws.ptr), n, nj, sym, L.grid, nbins, qcap, gunits, &sc);
  return run_pipeline(c, ra, dec, n, ra2, dec2, nj, sym, pl, L, sc, out);
}

// Graph replay of repeated calls. A call is eligible when the option is on, no launch-error
// injection is asked for, the context has a stream of its own (the legacy default stream cannot be
// captured) and the caller is not capturing that stream. The first call with a key runs as usual
// (and sizes the workspace); when the same key comes again the call is captured into a graph (its
// kernels do not run while it is captured), instantiated and launched, and later calls with that
// key launch the graph. The results are those of the call: the graph holds the same launches with
// the same arguments, and they read the inputs' current contents. With kernel timing on, the timing
// events the call records are event nodes of the graph; before every launch they are pointed at the
// next free events, so acf_kernel_times sees each launch as if the call had run kernel by kernel.
// run() is the call.
template <class Run>
int run_graphed(acf_ctx* c, CallKey key, Run run) {
  bool eligible = c->opt_graphs && c->inject_launch_error == 0 && c->stream != nullptr && c->stream != cudaStreamLegacy &&
                  c->stream != cudaStreamPerThread;
  if (eligible) {
    ACF_CUDA(c, cudaSetDevice(c->device));
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    ACF_CUDA(c, cudaStreamIsCapturing(c->stream, &st));
    eligible = st == cudaStreamCaptureStatusNone;
  }
  if (!eligible) return run();
  key.stream = c->stream;
  key.threads = c->opt_threads;
  key.ctas = c->opt_ctas;
  key.method = c->opt_method;
  key.layout = c->opt_layout;
  key.exact = c->opt_exact;
  key.range_forms = c->opt_range_forms;
  key.unit_groups = c->opt_unit_groups;
  key.timing = c->opt_timing;
  key.units_per_launch = c->opt_units_per_launch;
  key.exact_queue = c->opt_exact_queue;
  key.exact_below_deg = c->opt_exact_below_deg;
  key.ws = c->ws.ptr;
  key.ws_bytes = c->ws.bytes;
  key.io = c->io.ptr;
  key.io_bytes = c->io.bytes;
  // launch a cached graph, its timing events (if any) pointed at the next free ones; false when the
  // timing record is full (the call then runs kernel by kernel, which stops recording)
  auto launch = [&](CachedGraph& g, int& rc) -> bool {
    rc = ACF_OK;
    if (g.ev_count) {
      if (c->ev_used + g.ev_count > (int)c->ev.size()) return false;
      for (const auto& nr : g.ev_nodes) {
        const cudaError_t e = cudaGraphExecEventRecordNodeSetEvent(g.exec, nr.first, c->ev[c->ev_used + nr.second]);
        if (e != cudaSuccess) {
          rc = cuda_fail(c, e, "cudaGraphExecEventRecordNodeSetEvent");
          return true;
        }
      }
    }
    const cudaError_t e = cudaGraphLaunch(g.exec, c->stream);
    if (e != cudaSuccess) {
      rc = cuda_fail(c, e, "cudaGraphLaunch");
      return true;
    }
    c->ev_used += g.ev_count;
    g.used = ++c->graph_clock;
    c->kernel_launches += g.launches;
    ++c->graph_replays;
    c->set_info(g.info);
    return true;
  };
  for (CachedGraph& g : c->graphs)
    if (g.exec && g.key == key) {
      int rc = ACF_OK;
      if (launch(g, rc)) return rc;
      return run();
    }
  int seen = -1;
  for (int k = 0; k < kGraphSlots; ++k)
    if (c->seen[k] == key) seen = k;
  if (seen < 0) {
    const int rc = run();
    if (rc == ACF_OK) {
      key.ws = c->ws.ptr;  // as the call left the workspace
      key.ws_bytes = c->ws.bytes;
      c->seen[c->seen_next] = key;
      c->seen_next = (c->seen_next + 1) % kGraphSlots;
    }
    return rc;
  }
  c->seen[seen] = CallKey();  // captured once, whatever the outcome
  const long long before = c->kernel_launches;
  const int ev_start = c->ev_used;
  if (cudaStreamBeginCapture(c->stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    return run();
  }
  c->capturing = true;
  const int rc = run();
  c->capturing = false;
  CachedGraph ng;
  const cudaError_t e = cudaStreamEndCapture(c->stream, &ng.graph);
  ng.ev_count = c->ev_used - ev_start;
  c->ev_used = ev_start;  // the captured records did not happen
  bool ok = rc == ACF_OK && e == cudaSuccess && ng.graph;
  if (ok && ng.ev_count) {
    // the event-record nodes, and which of the call's events each one records
    size_t nn = 0;
    ok = cudaGraphGetNodes(ng.graph, nullptr, &nn) == cudaSuccess;
    std::vector<cudaGraphNode_t> nodes(nn);
    if (ok && nn) ok = cudaGraphGetNodes(ng.graph, nodes.data(), &nn) == cudaSuccess;
    for (size_t k = 0; ok && k < nn; ++k) {
      cudaGraphNodeType t;
      ok = cudaGraphNodeGetType(nodes[k], &t) == cudaSuccess;
      if (!ok || t != cudaGraphNodeTypeEventRecord) continue;
      cudaEvent_t ev = nullptr;
      ok = cudaGraphEventRecordNodeGetEvent(nodes[k], &ev) == cudaSuccess;
      int rel = -1;
      for (int i = 0; ok && i < ng.ev_count; ++i)
        if (c->ev[ev_start + i] == ev) rel = i;
      ok = ok && rel >= 0;
      if (ok) ng.ev_nodes.emplace_back(nodes[k], rel);
    }
    ok = ok && (int)ng.ev_nodes.size() == ng.ev_count;
  }
  if (ok && cudaGraphInstantiate(&ng.exec, ng.graph, 0) != cudaSuccess) ng.exec = nullptr;
  if (!ok || !ng.exec) {
    // not capturable after all (or the call failed while captured): run it as usual
    ng.release();
    cudaGetLastError();
    c->kernel_launches = before;
    return run();
  }
  if (!ng.ev_count) {
    cudaGraphDestroy(ng.graph);  // nothing to rebind: the instantiated graph is all that is needed
    ng.graph = nullptr;
  }
  CachedGraph* slot = &c->graphs[0];
  for (CachedGraph& g : c->graphs)
    if (!g.exec || (slot->exec && g.used < slot->used)) slot = &g;
  slot->release();
  ng.key = key;
  ng.launches = c->kernel_launches - before;
  ng.info = c->info();
  c->kernel_launches = before;  // launch() counts them
  *slot = ng;
  ng.graph = nullptr;  // (ownership moved to the slot)
  ng.exec = nullptr;
  int lrc = ACF_OK;
  if (launch(*slot, lrc)) return lrc;
  return run();
}

}  // namespace

extern "C" {

#ifdef ACF_DEBUG_BOUNDS
const char* acf_version(void) { return "acf 0.1 sm_103a bounds-checked"; }
#else
const char* acf_version(void) { return "acf 0.1 sm_103a"; }
#endif

int acf_plan_info(double bin_width_deg, int32_t nbins, int32_t exact, int64_t* info) {
  if (!info || exact < 0 || exact > 2) return ACF_ERR_ARG;
  acf_ctx host;  // default options and no device: make_plan only reads options
  host.opt_exact = exact;
  Plan pl;
  const int rc = make_plan(&host, bin_width_deg, nbins, pl);
  if (rc) return rc;
  const BinParams& bp = pl.bp;
  const int64_t v[ACF_PLAN_INFO_FIELDS] = {pl.map,           bp.entries,           pl.layout,          pl.threads,
                                           (int64_t)pl.smem, pl.exact ? bp.fine_shift : 0,
                                           pl.exact ? bp.fine_shift_small : 0,
                                           pl.exact ? bp.fine_shift_mid : 0, bp.mid, bp.small, bp.kmax, pl.exact};
  for (int k = 0; k < ACF_PLAN_INFO_FIELDS; ++k) info[k] = v[k];
  return ACF_OK;
}

int acf_create(acf_ctx** out, int device, void* cuda_stream) {
  if (!out) return ACF_ERR_ARG;
  *out = nullptr;
  acf_ctx* c = new (std::nothrow) acf_ctx();
  if (!c) return ACF_ERR_NOMEM;
  c->device = device;
  c->stream = static_cast<cudaStream_t>(cuda_stream);
  cudaError_t e = cudaSetDevice(device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess) {
    delete c;
    return ACF_ERR_CUDA;
  }
  *out = c;
  return ACF_OK;
}

void acf_destroy(acf_ctx* c) {
  if (!c) return;
  cudaSetDevice(c->device);
  cudaStreamSynchronize(c->stream);
  if (c->ws.ptr) cudaFree(c->ws.ptr);
  if (c->io.ptr) cudaFree(c->io.ptr);
  for (cudaEvent_t e : c->ev) cudaEventDestroy(e);
  for (CachedGraph& g : c->graphs) g.release();
  delete c;
}

const char* acf_last_error(const acf_ctx* c) { return c ? c->err.c_str() : "null context"; }

int acf_set_stream(acf_ctx* c, void* s) {
  if (!c) return ACF_ERR_ARG;
  ACF_CUDA(c, cudaSetDevice(c->device));
  ACF_CUDA(c, cudaStreamSynchronize(c->stream));
  c->stream = static_cast<cudaStream_t>(s);
  return ACF_OK;
}

int acf_histogram(acf_ctx* c, const float* ra, const float* dec, int64_t n, const float* ra2, const float* dec2,
                  int64_t n2, double w_deg, int32_t nbins, uint64_t* out) {
  if (!c) return ACF_ERR_ARG;
  CallKey k;
  k.entry = 2;
  const void* p[8] = {ra, dec, ra2, dec2, out, nullptr, nullptr, nullptr};
  std::copy(p, p + 8, k.p);
  k.n[0] = n;
  k.n[1] = n2;
  k.w = w_deg;
  k.nbins = nbins;
  return run_graphed(c, k, [&] { return histogram_impl(c, ra, dec, n, ra2, dec2, n2, w_deg, nbins, out); });
}

int acf_omega(acf_ctx* c, const uint64_t* dd, const uint64_t* dr, const uint64_t* rr, int32_t nbins, int64_t n_d,
              int64_t n_r, double* omega) {
  if (!c) return ACF_ERR_ARG;
  if (!dd || !dr || !rr || !omega) return fail(c, ACF_ERR_ARG, "omega: NULL pointer");
  if (nbins <= 0 || n_d <= 0 || n_r <= 0) return fail(c, ACF_ERR_ARG, "omega: nbins, n_d, n_r must be > 0");
  ACF_CUDA(c, cudaSetDevice(c->device));
  return launch_omega(c, dd, dr, rr, nbins, n_d, n_r, omega);
}

int acf_correlate(acf_ctx* c, const float* ra_d, const float* dec_d, int64_t n_d, const float* ra_r,
                  const float* dec_r, int64_t n_r, double w_deg, int32_t nbins, uint64_t* dd, uint64_t* dr, uint64_t* rr,
                  double* omega) {
  if (!c) return ACF_ERR_ARG;
  CallKey k;
  k.entry = 1;
  const void* p[8] = {ra_d, dec_d, ra_r, dec_r, dd, dr, rr, omega};
  std::copy(p, p + 8, k.p);
  k.n[0] = n_d;
  k.n[1] = n_r;
  k.w = w_deg;
  k.nbins = nbins;
  return run_graphed(c, k, [&] { return correlate_impl(c, ra_d, dec_d, n_d, ra_r, dec_r, n_r, w_deg, nbins, dd, dr, rr, omega); });
}

int acf_correlate_host(acf_ctx* c, const float* ra_d, const float* dec_d, int64_t n_d, const float* ra_r,
                       const float* dec_r, int64_t n_r, double w_deg, int32_t nbins, uint64_t* dd, uint64_t* dr,
                       uint64_t* rr, double* omega) {
  if (!c) return ACF_ERR_ARG;
  if (!ra_d || !dec_d || !ra_r || !dec_r || !dd || !dr || !rr || !omega)
    return fail(c, ACF_ERR_ARG, "correlate: NULL pointer");
  if (n_d <= 0 || n_r <= 0) return fail(c, ACF_ERR_ARG, "correlate: n_d and n_r must be > 0");
  if (nbins <= 0) return fail(c, ACF_ERR_ARG, "nbins must be > 0");
  ACF_CUDA(c, cudaSetDevice(c->device));
  const size_t bd = align256((size_t)n_d * 4), br = align256((size_t)n_r * 4), bh = align256((size_t)nbins * 8);
  int rc = ensure(c, c->io, 2 * bd + 2 * br + 4 * bh);
  if (rc) return rc;
  char* p = static_cast<char*>(c->io.ptr);
  float* d_ra_d = reinterpret_cast<float*>(p);
  float* d_dec_d = reinterpret_cast<float*>(p + bd);
  float* d_ra_r = reinterpret_cast<float*>(p + 2 * bd);
  float* d_dec_r = reinterpret_cast<float*>(p + 2 * bd + br);
  char* h = p + 2 * bd + 2 * br;
  uint64_t* d_dd = reinterpret_cast<uint64_t*>(h);
  uint64_t* d_dr = reinterpret_cast<uint64_t*>(h + bh);
  uint64_t* d_rr = reinterpret_cast<uint64_t*>(h + 2 * bh);
  double* d_om = reinterpret_cast<double*>(h + 3 * bh);
  auto body = [&]() -> int {
    ACF_CUDA(c, cudaMemcpyAsync(d_ra_d, ra_d, (size_t)n_d * 4, cudaMemcpyHostToDevice, c->stream));
    ACF_CUDA(c, cudaMemcpyAsync(d_dec_d, dec_d, (size_t)n_d * 4, cudaMemcpyHostToDevice, c->stream));
    ACF_CUDA(c, cudaMemcpyAsync(d_ra_r, ra_r, (size_t)n_r * 4, cudaMemcpyHostToDevice, c->stream));
    ACF_CUDA(c, cudaMemcpyAsync(d_dec_r, dec_r, (size_t)n_r * 4, cudaMemcpyHostToDevice, c->stream));
    const int rc2 = correlate_impl(c, d_ra_d, d_dec_d, n_d, d_ra_r, d_dec_r, n_r, w_deg, nbins, d_dd, d_dr, d_rr, d_om);
    if (rc2) return rc2;
    ACF_CUDA(c, cudaMemcpyAsync(dd, d_dd, (size_t)nbins * 8, cudaMemcpyDeviceToHost, c->stream));
    ACF_CUDA(c, cudaMemcpyAsync(dr, d_dr, (size_t)nbins * 8, cudaMemcpyDeviceToHost, c->stream));
    ACF_CUDA(c, cudaMemcpyAsync(rr, d_rr, (size_t)nbins * 8, cudaMemcpyDeviceToHost, c->stream));
    ACF_CUDA(c, cudaMemcpyAsync(omega, d_om, (size_t)nbins * 8, cudaMemcpyDeviceToHost, c->stream));
    return ACF_OK;
  };
  // with page-locked host buffers the copies can sit in a graph with the kernels (pageable ones
  // cannot be captured)
  const void* hp[8] = {ra_d, dec_d, ra_r, dec_r, dd, dr, rr, omega};
  bool pinned = true;
  for (const void* q : hp) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, q) != cudaSuccess) {
      cudaGetLastError();
      pinned = false;
    } else if (at.type != cudaMemoryTypeHost) {
      pinned = false;
    }
  }
  if (pinned) {
    CallKey k;
    k.entry = 3;
    std::copy(hp, hp + 8, k.p);
    k.n[0] = n_d;
    k.n[1] = n_r;
    k.w = w_deg;
    k.nbins = nbins;
    rc = run_graphed(c, k, body);
  } else {
    rc = body();
  }
  if (rc) return rc;
  ACF_CUDA(c, cudaStreamSynchronize(c->stream));
  return ACF_OK;
}

int acf_pair_bins(acf_ctx* c, const float* ra1, const float* dec1, const float* ra2, const float* dec2, int64_t n,
                  double w_deg, int32_t nbins, int32_t* bins) {
  if (!c) return ACF_ERR_ARG;
  if (n < 0) return fail(c, ACF_ERR_ARG, "n must be >= 0");
  Plan pl;
  int rc = make_plan(c, w_deg, nbins, pl);
  if (rc) return rc;
  if (n == 0) return ACF_OK;
  if (!ra1 || !dec1 || !ra2 || !dec2 || !bins) return fail(c, ACF_ERR_ARG, "pair_bins: NULL pointer");
  ACF_CUDA(c, cudaSetDevice(c->device));
  const int threads = 256;
  const long long blocks = std::min<long long>((n + threads - 1) / threads, (long long)c->num_sms * 32);
  if (pl.method == kDotFastAcos)
    pair_bins_kernel<kClamp, kDotFastAcos><<<(unsigned)blocks, threads, 0, c->stream>>>(ra1, dec1, ra2, dec2, n, pl.bp,
                                                                                      c->opt_pair_bins_form, bins);
  else if (pl.method == kDotAcos)
    pair_bins_kernel<kClamp, kDotAcos><<<(unsigned)blocks, threads, 0, c->stream>>>(ra1, dec1, ra2, dec2, n, pl.bp,
                                                                                  c->opt_pair_bins_form, bins);
  else if (pl.map == kDirect)
    pair_bins_kernel<kDirect, kChordPoly><<<(unsigned)blocks, threads, 0, c->stream>>>(ra1, dec1, ra2, dec2, n, pl.bp,
                                                                                  c->opt_pair_bins_form, bins);
  else
    pair_bins_kernel<kClamp, kChordPoly><<<(unsigned)blocks, threads, 0, c->stream>>>(ra1, dec1, ra2, dec2, n, pl.bp,
                                                                                  c->opt_pair_bins_form, bins);
  ACF_LAUNCHED(c);
  return ACF_OK;
}

int acf_set_option(acf_ctx* c, const char* key, int64_t v) {
  if (!c || !key) return ACF_ERR_ARG;
  if (!strcmp(key, "threads")) {
    if (v != 0 && v != 512 && v != 1024) return fail(c, ACF_ERR_ARG, "threads must be 0, 512 or 1024");
    c->opt_threads = (int)v;
  } else if (!strcmp(key, "ctas_per_sm")) {
    if (v < 0 || v > 8) return fail(c, ACF_ERR_ARG, "ctas_per_sm must be 0..8");
    c->opt_ctas = (int)v;
  } else if (!strcmp(key, "bin_method")) {
    if (v != kChordPoly && v != kDotAcos && v != kDotFastAcos) return fail(c, ACF_ERR_ARG, "bin_method must be 0, 1 or 2");
    c->opt_method = (int)v;
  } else if (!strcmp(key, "layout")) {
    if (v < 0 || v > 3) return fail(c, ACF_ERR_ARG, "layout must be 0, 1, 2 or 3");
    c->opt_layout = (int)v;
  } else if (!strcmp(key, "exact")) {
    if (v < 0 || v > 2) return fail(c, ACF_ERR_ARG, "exact must be 0, 1 or 2");
    c->opt_exact = (int)v;
  } else if (!strcmp(key, "exact_below_deg")) {
    if (v < 0 || v > 180) return fail(c, ACF_ERR_ARG, "exact_below_deg must be 0..180");
    c->opt_exact_below_deg = (double)v;
  } else if (!strcmp(key, "range_forms")) {
    if (v != 0 && v != 1) return fail(c, ACF_ERR_ARG, "range_forms must be 0 or 1");
    c->opt_range_forms = (int)v;
  } else if (!strcmp(key, "pair_bins_form")) {
    if (v != 0 && v != 1) return fail(c, ACF_ERR_ARG, "pair_bins_form must be 0 or 1");
    c->opt_pair_bins_form = (int)v;
  } else if (!strcmp(key, "units_per_launch")) {
    if (v < 0) return fail(c, ACF_ERR_ARG, "units_per_launch must be >= 0");
    c->opt_units_per_launch = v;
  } else if (!strcmp(key, "unit_groups")) {
    if (v != 0 && v != 1 && v != 4) return fail(c, ACF_ERR_ARG, "unit_groups must be 0, 1 or 4");
    c->opt_unit_groups = (int)v;
  } else if (!strcmp(key, "exact_queue")) {
    if (v < 0 || v > kQueueCapMax) return fail(c, ACF_ERR_ARG, "exact_queue must be 0..2^28");
    c->opt_exact_queue = v;
  } else if (!strcmp(key, "graphs")) {
    if (v != 0 && v != 1) return fail(c, ACF_ERR_ARG, "graphs must be 0 or 1");
    c->opt_graphs = (int)v;
  } else if (!strcmp(key, "workspace_limit")) {
    if (v < 0) return fail(c, ACF_ERR_ARG, "workspace_limit must be >= 0");
    c->opt_workspace_limit = v;
  } else if (!strcmp(key, "inject_launch_error")) {
    if (v < 0) return fail(c, ACF_ERR_ARG, "inject_launch_error must be >= 0");
    c->inject_launch_error = v;
  } else if (!strcmp(key, "kernel_timing")) {
    if (v < 0 || v > 2) return fail(c, ACF_ERR_ARG, "kernel_timing must be 0, 1 or 2");
    c->opt_timing = (int)v;
    if (c->opt_timing && c->ev.empty()) {
      ACF_CUDA(c, cudaSetDevice(c->device));
      c->ev.resize(2 * kMaxTimed);
      for (auto& e : c->ev) ACF_CUDA(c, cudaEventCreate(&e));
    }
    c->ev_used = 0;
  } else {
    return fail(c, ACF_ERR_ARG, "unknown option '%s'", key);
  }
  return ACF_OK;
}

int acf_get_info(const acf_ctx* c, const char* key, int64_t* v) {
  if (!c || !key || !v) return ACF_ERR_ARG;
  struct {
    const char* k;
    long long val;
  } t[] = {{"grid", c->info_grid},       {"threads", c->info_threads},   {"ctas_per_sm", c->info_ctas},
           {"units", c->info_chunks},   {"layout", c->info_layout},     {"bin_map", c->info_map},
           {"hist_entries", c->info_entries}, {"smem_bytes", c->info_smem}, {"pairs_evaluated", c->info_pairs},
           {"launches", c->info_flush},  {"kernel_launches", c->kernel_launches},
           {"graph_replays", c->graph_replays},
           {"unit_groups", c->info_groups}};
  for (auto& e : t)
    if (!strcmp(e.k, key)) {
      *v = e.val;
      return ACF_OK;
    }
  const char* path_keys[9] = {"pairs_fixed",  "pairs_general",   "pairs_fixed_exact", "pairs_general_exact",
                               "pairs_masked", "pairs_mid",       "pairs_mid_exact",   "pairs_small",
                               "pairs_small_exact"};
  for (int k = 0; k < 9; ++k)
    if (!strcmp(key, path_keys[k])) {
      // synchronises the stream; pairs the last histogram call evaluated on each pair-kernel path
      unsigned long long h[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
      if (c->last_counters) {
        if (cudaSetDevice(c->device) != cudaSuccess || cudaStreamSynchronize(c->stream) != cudaSuccess ||
            cudaMemcpy(h, c->last_counters + 16, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess)
          return ACF_ERR_CUDA;
      }
      *v = (long long)h[k];
      return ACF_OK;
    }
  if (!strcmp(key, "exact_flagged") || !strcmp(key, "exact_moved") || !strcmp(key, "exact_overflow") ||
      !strcmp(key, "exact_redone_fp64")) {
    // synchronises the stream; counts of the last histogram call
    unsigned int h[6] = {0, 0, 0, 0, 0, 0};
    if (c->last_counters && c->last_qcap > 0) {
      if (cudaSetDevice(c->device) != cudaSuccess || cudaStreamSynchronize(c->stream) != cudaSuccess ||
          cudaMemcpy(h, c->last_counters, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess)
        return ACF_ERR_CUDA;
    }
    if (!strcmp(key, "exact_flagged")) *v = h[3];
    else if (!strcmp(key, "exact_moved")) *v = h[2];
    else if (!strcmp(key, "exact_redone_fp64")) *v = h[5];
    else *v = h[4];  // slots requested past the end, over all launches
    return ACF_OK;
  }
  return ACF_ERR_ARG;
}

int acf_fp32_peak(acf_ctx* c, int64_t iters, double* ffma_per_s, float* thread0) {
  if (!c || !ffma_per_s || iters <= 0) return ACF_ERR_ARG;
  ACF_CUDA(c, cudaSetDevice(c->device));
  const int blocks = c->num_sms * 2, threads = 1024;
  float* out = nullptr;
  ACF_CUDA(c, cudaMallocAsync(reinterpret_cast<void**>(&out), (size_t)blocks * threads * sizeof(float), c->stream));
  cudaEvent_t e0, e1;
  ACF_CUDA(c, cudaEventCreate(&e0));
  ACF_CUDA(c, cudaEventCreate(&e1));
  const float a = 0.9999999f, b = 1e-7f;
  fma_peak_kernel<<<blocks, threads, 0, c->stream>>>(a, b, iters / 8 + 1, out);  // warm-up
  ACF_LAUNCHED(c);
  ACF_CUDA(c, cudaEventRecord(e0, c->stream));
  fma_peak_kernel<<<blocks, threads, 0, c->stream>>>(a, b, iters, out);
  ACF_LAUNCHED(c);
  ACF_CUDA(c, cudaEventRecord(e1, c->stream));
  ACF_CUDA(c, cudaEventSynchronize(e1));
  float ms = 0.f;
  ACF_CUDA(c, cudaEventElapsedTime(&ms, e0, e1));
  if (thread0) ACF_CUDA(c, cudaMemcpyAsync(thread0, out, sizeof(float), cudaMemcpyDeviceToHost, c->stream));
  ACF_CUDA(c, cudaFreeAsync(out, c->stream));
  ACF_CUDA(c, cudaStreamSynchronize(c->stream));
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  *ffma_per_s = (double)blocks * threads * (double)iters * kFmaChains / (ms * 1e-3);
  return ACF_OK;
}

int acf_kernel_times(acf_ctx* c, float* ms, int32_t cap, int32_t* count) {
  if (!c || !count || (cap > 0 && !ms)) return ACF_ERR_ARG;
  *count = 0;
  if (!c->opt_timing) return fail(c, ACF_ERR_ARG, "kernel_timing is off");
  ACF_CUDA(c, cudaSetDevice(c->device));
  ACF_CUDA(c, cudaStreamSynchronize(c->stream));
  const int pairs = c->ev_used / 2;
  int k = 0;
  for (; k < pairs && k < cap; ++k) ACF_CUDA(c, cudaEventElapsedTime(&ms[k], c->ev[2 * k], c->ev[2 * k + 1]));
  *count = k;
  c->ev_used = 0;
  return ACF_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------------------------
// acf_histogram_noalloc: the histogram with its scratch in a fixed, statically sized device
// array instead of the context's workspace, for callers that cannot allocate device memory.
//
// The array below is what every GPU that loads this library reserves for it, until the process
// exits. In host code its name is only a host-side stand-in for the device symbol; the device
// address is looked up once per device with cudaGetSymbolAddress (with that device current) and
// that address is what the kernels receive.

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};
unsigned long long g_noalloc_ctx_id[kMaxDevices] = {};  // the context the cached address belongs to

// Unique ID of the calling thread's current CUDA context (0 if it cannot be read). A device reset
// (cudaDeviceReset) destroys the primary context and a new one gets a new ID, even if the driver
// hands out the same handle again. The two driver functions are resolved through the runtime, so
// the library does not link the driver library itself.
unsigned long long current_context_id() {
  typedef int (*GetCurrentFn)(void**);
  typedef int (*GetIdFn)(void*, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static bool resolved = false;
  if (!resolved) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) == cudaSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) == cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess && q2 == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<GetCurrentFn>(f1);
      get_id = reinterpret_cast<GetIdFn>(f2);
    }
    resolved = true;
  }
  void* ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != 0 || !ctx || get_id(ctx, &id) != 0) return 0;
  return id;
}

// Device address of the static scratch on `device` (which must be current). Looked up on the first
// call on a device, and again whenever that device's context has changed since (after a device
// reset the module is loaded anew, possibly elsewhere).
int noalloc_scratch(acf_ctx* c, int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return fail(c, ACF_ERR_UNSUPPORTED, "device %d out of range", device);
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  const unsigned long long id = current_context_id();
  if (!g_noalloc_ptr[device] || id == 0 || id != g_noalloc_ctx_id[device]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(c, e, "cudaGetSymbolAddress(g_noalloc_scratch)");
    g_noalloc_ptr[device] = p;
    g_noalloc_ctx_id[device] = id;
  }
  *out = g_noalloc_ptr[device];
  return ACF_OK;
}

}  // namespace

extern "C" int acf_histogram_noalloc(acf_ctx* c, const float* ra, const float* dec, int64_t n, const float* ra2,
                                     const float* dec2, int64_t n2, double w_deg, int32_t nbins, uint64_t* out) {
  if (!c) return ACF_ERR_ARG;
  if (n < 0) return fail(c, ACF_ERR_ARG, "n must be >= 0");
  if (n > 2147483647ll || n2 > 2147483647ll) return fail(c, ACF_ERR_UNSUPPORTED, "catalogs are limited to 2^31-1 galaxies");
  if (!out) return fail(c, ACF_ERR_ARG, "out is NULL");
  const bool sym = (ra2 == nullptr && dec2 == nullptr) || (ra2 == ra && dec2 == dec && n2 == n);
  if (!sym && n2 < 0) return fail(c, ACF_ERR_ARG, "n2 must be >= 0");
  if (!sym && ((ra2 == nullptr) != (dec2 == nullptr))) return fail(c, ACF_ERR_ARG, "ra2 and dec2 must both be set");
  const int64_t nj = sym ? n : n2;
  Plan pl;
  int rc = make_plan(c, w_deg, nbins, pl);
  if (rc) return rc;
  ACF_CUDA(c, cudaSetDevice(c->device));
  if (n == 0 || nj == 0) {
    ACF_CUDA(c, cudaMemsetAsync(out, 0, sizeof(uint64_t) * (size_t)nbins, c->stream));
    return ACF_OK;
  }
  if (!ra || !dec || (!sym && (!ra2 || !dec2))) return fail(c, ACF_ERR_ARG, "catalog pointer is NULL");
  Launch L;
  rc = plan_launch(c, pl, n, nj, sym, L);
  if (rc) return rc;
  const size_t need = carve(nullptr, n, nj, sym, L.grid, nbins, 0, 0, nullptr);
  // the exact-mode queue (or the group records) takes whatever the static array has left (minus the
  // alignment of its two parts); group records take fewer units per launch to fit
  const long long left = need + 1024 < kNoAllocScratchBytes ? (long long)(kNoAllocScratchBytes - need - 1024) : 0;
  const long long qcap = pl.exact && !pl.grouped ? left / (long long)kRecordBytes : 0;
  const long long gunits = pl.grouped ? std::min(std::min(L.units, L.per_launch), left / (long long)kGroupUnitBytes) : 0;
  if (pl.grouped && gunits < 1 && need <= kNoAllocScratchBytes)
    return fail(c, ACF_ERR_UNSUPPORTED,
                "acf_histogram_noalloc: the static array has no room left for the exact mode's group records "
                "(%zu of %zu bytes taken); use acf_histogram or exact mode 0", need, kNoAllocScratchBytes);
  if (pl.grouped) L.per_launch = std::min(L.per_launch, gunits);
  if (need > kNoAllocScratchBytes)
    return fail(c, ACF_ERR_UNSUPPORTED,
                "acf_histogram_noalloc needs %zu bytes of scratch but its static array holds %zu "
                "(about 93 bytes per galaxy of each catalog plus (%lld blocks + 2) x nbins x 8 bytes); use acf_histogram",
                need, kNoAllocScratchBytes, L.grid);
  void* scratch = nullptr;
  rc = noalloc_scratch(c, c->device, &scratch);
  if (rc) return rc;
  // Every byte the kernels read is rewritten first: the ticket and cell counters are cleared,
  // the preparation kernels write the vectors and caps, and the pair kernel zeroes its rows.
  Scratch sc;
  carve(static_cast<char*>(scratch), n, nj, sym, L.grid, nbins, std::max(qcap, 0ll), std::max(gunits, 0ll), &sc);
  return run_pipeline(c, ra, dec, n, ra2, dec2, nj, sym, pl, L, sc, out);
}
