// Device code of the GB300 angular-correlation library (sm_103a, CUDA cores).
//
// The method is that of "CUDA Deep Dive: 10B Galaxy Pairs on an RTX 5080": bin the angular
// separation theta of every ordered pair of two galaxy catalogs (section "The problem"), using
// DD/RR symmetry (section "L1"), per-galaxy precomputation (section "L2"), a register i-tile
// against a shared-memory j-tile (section "L3") and whole-tile diagonal skipping (section "L5").
// What differs from the page, and why:
//   * each galaxy becomes an fp32 unit vector once (built in fp64), so a pair costs a dot product
//     instead of a cosine of the RA difference;
//   * catalogs are sorted along a Hilbert curve over cube-map cells, and each run of 32 sorted
//     galaxies gets a cap (centre, radius); from two caps the kernel knows the range of separations
//     of a (warp, j-group) block of pairs and picks the cheapest exact-enough form for it;
//   * below 55 and above 125 degrees the separation is taken from the CHORD, not from arccos of the
//     dot product: with s = sign(u.v), q = |u - s v|^2 = 4 sin^2(theta'/2), theta' = theta
//     (s = +1) or pi - theta (s = -1), theta' <= 90 deg; q keeps full relative precision at small
//     and near-antipodal separations, where arccos of an fp32 dot product loses up to ~3e-4 rad.
//     theta'^2 = q * P(q) with a polynomial P (degree 5 where theta' < 72 deg, else 7), then one
//     sqrt.approx;
//   * between 55 and 125 degrees the dot product itself is precise enough: theta = pi/2 - d R(d^2)
//     with a degree-4 polynomial R and no square root (11 instead of 18 instructions per pair);
//   * the bin index comes from exact float rounding (one fma rounded toward zero onto 2^23 + c)
//     instead of acos, multiply and float-to-int conversion;
//   * each histogram lives in shared memory as 32 lane-private copies (word = bin*32 + lane), so a
//     warp's 32 increments always hit 32 different banks and the shared-memory atomic unit
//     retires one warp instruction per clock; very fine binnings fall back to one block-shared
//     copy;
//   * persistent blocks whose warps take 128 x 128-pair work units from a global ticket (only the
//     upper triangle for DD/RR); per-block counts go to per-block uint64 rows that a final kernel
//     reduces;
//   * in exact mode (the default), pairs whose fast code lies within a fine unit of a bin edge are
//     queued and re-decided after every launch: in double-single fp32 where that settles them,
//     else in fp64.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace acf {

constexpr int kJT = 128;  // j-galaxies per shared-memory chunk
#ifndef ACF_JJ_UNROLL
#define ACF_JJ_UNROLL 4
#endif
constexpr int kJJUnroll = ACF_JJ_UNROLL;
#ifndef ACF_JJ_UNROLL_FINE
#define ACF_JJ_UNROLL_FINE 2
#endif
constexpr int kJJUnrollFine = ACF_JJ_UNROLL_FINE;  // j-loop unroll of the exact-mode (fine code) loops
#ifndef ACF_JJ_UNROLL_FINE2
#define ACF_JJ_UNROLL_FINE2 2
#endif
constexpr int kJJUnrollFine2 = ACF_JJ_UNROLL_FINE2;  // and of the two-code (fixed-sign chord) ones
// (with a queue push per flagged pair both measured slower unrolled twice: that push code no longer
// fit the instruction cache; with one flag record per j it does, and twice is faster: 4.02 against
// 4.23 ms per 100k DR-sized launch, 2.47 against 2.55 ms per fine-binning launch)
// Flag test per j: 1 = OR of per-pair tests "biased fraction bits above bit 0 all zero"; 0 = a
// running minimum of the biased fractions compared with 1 (measured alternative: 12.62 against
// 12.47 ms of pair kernels per 100k step)
#ifndef ACF_FLAG_PRED
#define ACF_FLAG_PRED 1
#endif
// Fix-up: the blocks per SM its registers must allow (it waits on loads and wants every warp it can
// get).
#ifndef ACF_FIXUP_MINB
#define ACF_FIXUP_MINB 4
#endif
#ifndef ACF_JJ_BATCH
#define ACF_JJ_BATCH 2
#endif
// j-galaxies per step of the hot loops: their tile loads first, then every code, then every atomic
// (the atomics' memory clobber would otherwise keep the next tile load behind them)
constexpr int kJJBatch = ACF_JJ_BATCH;
#ifndef ACF_J_SHUFFLE
#define ACF_J_SHUFFLE 0  // 1: j-vectors broadcast by warp shuffles instead of shared-memory loads
#endif
#ifndef ACF_ASM_LOP3
#define ACF_ASM_LOP3 1  // write the two sign-bit logic ops as explicit lop3 (2 ops, not 3)
#endif  // j-loop unroll of the full-chunk path
constexpr float kMagic = 8388608.0f;  // 2^23: adding it with round-toward-zero floors into the mantissa

// kBlock16: two block-shared copies of 16-bit counters packed in pairs (a measured alternative for
// fine binning, built with -DACF_U16_HIST=1, exact mode 0 only). kBlockExact: kBlock for exact mode
// 2, whose every group takes the flagging loops, built without the plain ones (measured faster on
// fine bins; the lane-private layout measured slower that way).
enum Layout { kLane = 1, kBlock = 2, kBlock16 = 3, kBlockExact = 4 };
#ifndef ACF_U16_HIST
#define ACF_U16_HIST 0
#endif
enum BinMap { kDirect = 0, kClamp = 1 };
enum Method { kChordPoly = 0, kDotAcos = 1, kDotFastAcos = 2 };

// arccos(x) for x in [0, 1] as sqrt(1 - x) (a0 + a1 x + a2 x^2 + a3 x^3): Abramowitz and Stegun,
// Handbook of Mathematical Functions, formula 4.4.45 (|error| <= 6.7e-5 rad), extended to
// [-1, 0) by arccos(-x) = pi - arccos(x). The approximate mode: fast, not held to the 1e-6 rule.
__device__ __forceinline__ float acos_as4445(float x) {
  const float ax = fabsf(x);
  float r = fmaf(-0.0187293f, ax, 0.0742610f);
  r = fmaf(r, ax, -0.2121144f);
  r = fmaf(r, ax, 1.5707288f);
  r *= sqrtf(1.0f - ax);
  return x < 0.0f ? 3.14159265358979f - r : r;
}

// theta'^2 = q * P(q) for a chord q = |u - v|^2 on [0, 2] (theta' <= 90 degrees), P of degree 7
// fitted by fit_arcsin2.py: absolute theta' error <= 1.8e-8 rad (2.5e-8 after fp32 rounding).
__device__ constexpr float kP0 = 0.99999959294652097f, kP1 = 0.083342611628085594f, kP2 = 0.011049794431887118f,
                           kP3 = 0.0019657095570993176f, kP4 = 4.2347086002697957e-05f,
                           kP5 = 0.00029099553526503564f, kP6 = -9.1427792701640403e-05f,
                           kP7 = 2.3068911858269848e-05f;

// The same on theta' <= 72.4 degrees with degree 5, for groups whose caps keep every theta' below
// 72 degrees: absolute theta' error <= 4.3e-8 rad (5.5e-8 after fp32 rounding).
__device__ constexpr float kS0 = 0.99999908438480867f, kS1 = 0.083350941003199425f, kS2 = 0.011015189062680493f,
                           kS3 = 0.0020057633993448608f, kS4 = 8.1054448294636845e-05f,
                           kS5 = 0.00017064219833417058f;
constexpr float kSmallRad = 1.2566370614359172f;  // 72 degrees

// Between 55 and 125 degrees the dot product d = u.v loses little: theta = pi/2 - asin(d) with
// asin(d) = d * R(d^2). R fitted by fit_asin_mid.py on d^2 <= cos^2(54.5 deg), degree 4: absolute
// theta error <= 1.5e-7 rad (also after fp32 rounding), within the exact mode's window; a higher
// degree would cost one more instruction per pair on nearly half the pairs. Scaled by 1/w on the
// host.
constexpr int kRTerms = 5;
constexpr double kR[kRTerms] = {1.0000027330813104, 0.16651326659029475, 0.077385369858043895,
                                0.0299281303350203, 0.067072790014221492};
constexpr float kMidRad = 0.95993108859688125f;  // groups whose separations all lie in (55, 125) degrees use the dot form

// Every code is the float 2^23 + (histogram entry), entry = floor(theta / w) (direct map, where
// P = pi / w is an integer) or the clamped index (clamp map); the merge clamps entries to nbins - 1.
struct BinParams {
  float magic_far;    // direct: 2^23 + P, the far-side (theta > 90 deg) constant of the chord form
  float magic_mid;    // direct, P even: 2^23 + P/2, the constant of the dot form
  // Exact mode: each form has its own S, so that its window (2^-S bins) covers its own error bound:
  // S (full-range and general chord, clamp map, masked units), S_small (short chord), S_mid (dot).
  float inv_w_f;      // exact mode: 2^S / w (fine code with S fractional bits)
  float inv_w_fs;     // exact mode: 2^S_small / w
  float magic_far_fs; // exact mode: 2^23 + P 2^S_small + 1
  float clamp_fs;     // exact mode: (clamp_c + 0.5) * 2^S_small (clamp map)
  // The fine code is biased by one fine unit (every fine constant carries + 1), so a pair lies
  // within one fine unit of an edge exactly when its low S bits are 0 or 1.
  float magic_f;      // exact mode: 2^23 + 1
  float magic_far_f;  // exact mode: 2^23 + P 2^S + 1
  float magic_mid_f;  // exact mode: 2^23 + (P/2) 2^S_mid + 1
  float clamp_f;      // exact mode: (clamp_c + 0.5) * 2^S (clamp map)
  float rc[kRTerms];   // dot form: kR[k] / w
  float rc_f[kRTerms]; // exact mode: kR[k] 2^S_mid / w
  int mid;            // 1: groups between 55 and 125 degrees use the dot form
  int small;          // 1: groups whose theta' stays below 72 degrees use the degree-5 chord polynomial
  int fine_shift;     // exact mode: S
  int fine_shift_small;  // exact mode: S_small
  int fine_shift_mid;    // exact mode: S_mid
  int kmax;           // exact mode: highest bin a separation <= 180 degrees can reach
  unsigned int zone0, span0, zone1, span1;  // exact mode: entries e with e - zone <= span (unsigned) are re-decided
  float clamp_c;      // largest index (clamp map)
  float inv_w;        // 1 / w in radians
  int nbins;
  int entries;        // histogram entries in shared memory
};

// Exact mode with a block-shared histogram (dense flags): the flags of one lane over one j-group,
// 32 bytes. Word k holds, in bit b, the flag of the pair (i = kJT r + islot(k, lane), j = j + b);
// pc is the group's path code.
struct __align__(32) GroupRecord {
  uint32_t w[4];
  uint32_t r, j, pc, pad;
};

struct PairParams {
  const float4* __restrict__ vi;
  const float4* __restrict__ vj;
  long long ni, nj;
  long long rows;              // i-sets of kJT galaxies: ceil(ni / kJT)
  long long cols;              // j-chunks of kJT galaxies: ceil(nj / kJT)
  long long unit_begin;        // this launch handles units [unit_begin, unit_end)
  long long unit_end;
  int sym;                     // 1: pairs j > i of one catalog, counted twice
  int accumulate;              // 0: zero the partial rows first; 1: add to them (later launches)
  unsigned int inc;            // 2 (sym) or 1 (cross)
  unsigned long long* partial; // [gridDim.x][nbins]
  unsigned int* ticket;        // unit dispenser; zero before the launch
  const float4* __restrict__ icap32;   // caps of 32-galaxy groups of the i catalog (sorted order)
  const float4* __restrict__ jcap32;   // caps of 32-galaxy groups of the j catalog
  long long igroups;                   // number of 32-galaxy groups of the i catalog
  int exact_mode;                      // 0 off, 1 groups that may hold separations < theta_lo or > 180 - theta_lo, 2 all
  float exact_lo;                      // theta_lo in radians
  // exact mode: the queue of flag records, one per (warp i-set, j) holding a flagged pair (see
  // push_record): warp w of block b (region g = b * warps + w) owns slots [g qbatch, (g + 1) qbatch),
  // then a shared spill region follows all regions
  uint2* qhdr;                         // (sorted j, i-set row | path code << 24)
  uint4* qmask;                        // per i-vector slot k of the lanes: the ballot of flagged lanes
  unsigned int* qspill;                // spill slots handed out
  unsigned int* qused;                 // per region: records the warp wrote (its own slots, then spill)
  unsigned int* qflagged;              // pairs flagged (for reporting)
  unsigned int* qoverflow;             // flagged pairs whose record found no slot (kept their fp32 bin)
  unsigned int qcap;                   // queue slots
  unsigned int qbatch;                 // slots a warp owns
  // exact mode with the block-shared histogram: group records instead (no queue, no overflow). Unit
  // u of the launch, j-group g: gi = (u - unit_begin) * 4 + g; gbal[gi] = the ballot of the lanes
  // whose record grec[gi * 32 + lane] holds a flag (the others are not written)
  unsigned int* gbal;
  GroupRecord* grec;
  unsigned long long* path_pairs;      // pairs evaluated per path: chord fixed, chord general,
                                       // chord fixed+flag, chord general+flag, masked/ragged units,
                                       // dot form, dot form+flag, short chord, short chord+flag
                                       // (all pairs computed)
  BinParams bp;
};

// ------------------------------------------------------------------ bounds-check build

// With -DACF_DEBUG_BOUNDS every shared-memory histogram index, tile index and global row index is
// checked; the first violation is recorded here (no trap) and the access is skipped.
struct DebugRecord {
  unsigned int count;
  int kind;  // 1 histogram entry, 2 tile index, 3 partial row index, 4 i-vector index
  long long a, b;
  float f[8];
};
#ifdef ACF_DEBUG_BOUNDS
__device__ DebugRecord g_debug;
__device__ __noinline__ void debug_note(int kind, long long a, long long b, float f0 = 0, float f1 = 0, float f2 = 0,
                                        float f3 = 0, float f4 = 0, float f5 = 0, float f6 = 0, float f7 = 0) {
  if (atomicAdd(&g_debug.count, 1u) == 0u) {
    g_debug.kind = kind;
    g_debug.a = a;
    g_debug.b = b;
    float v[8] = {f0, f1, f2, f3, f4, f5, f6, f7};
    for (int k = 0; k < 8; ++k) g_debug.f[k] = v[k];
  }
}
#define ACF_CHECK(cond, ...) (((cond)) ? true : (debug_note(__VA_ARGS__), false))
#else
#define ACF_CHECK(cond, ...) true
#endif

// ------------------------------------------------------------------ small PTX helpers

// Callers pass arguments >= 1e-26 (never subnormal), so flushing subnormals changes nothing and
// spares the input range check that the non-ftz form carries.
__device__ __forceinline__ float sqrt_approx(float x) {
  float y;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// round-toward-zero add and fma as compiler intrinsics (not inline asm), so that a constant operand
// can come straight from the constant bank instead of a register
__device__ __forceinline__ float add_rz(float a, float b) { return __fadd_rz(a, b); }

// three-input logic op; lut is the truth table over (a=0xF0, b=0xCC, c=0xAA)
template <int LUT>
__device__ __forceinline__ uint32_t lop3(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t y;
  asm("lop3.b32 %0, %1, %2, %3, %4;" : "=r"(y) : "r"(a), "r"(b), "r"(c), "n"(LUT));
  return y;
}

// a * b + c with one rounding, toward zero
__device__ __forceinline__ float fma_rz(float a, float b, float c) { return __fmaf_rz(a, b, c); }

__device__ __forceinline__ void red_shared_add(uint32_t addr, uint32_t v) {
  asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// ACF_MATCH_AGG=1 builds (a measured alternative for the block-shared histogram): lanes of a warp
// that add to the same counter are grouped by __match_any_sync and the group's lowest lane adds the
// group's total, so a warp issues one red per distinct counter instead of one per lane.
#ifndef ACF_MATCH_AGG
#define ACF_MATCH_AGG 0
#endif
// Add v (the same in every lane) to the shared counter at byte address a; `aggregate` selects the
// warp aggregation (block-shared layouts, in ACF_MATCH_AGG builds).
__device__ __forceinline__ void hist_add(uint32_t a, uint32_t v, bool aggregate) {
#if ACF_MATCH_AGG
  if (aggregate) {
    const uint32_t peers = __match_any_sync(__activemask(), a);
    if ((int)(threadIdx.x & 31) == __ffs(peers) - 1) red_shared_add(a, v * (uint32_t)__popc(peers));
    return;
  }
#else
  (void)aggregate;
#endif
  red_shared_add(a, v);
}

// Add v to the 16-bit counter at shared byte address a16 (two counters per 32-bit word, so the add
// goes to the word). The thread whose add takes the counter from below 0x8000 to 0x8000 or more
// takes 0x8000 back out and returns true: its caller adds 0x8000 to the counter's bin elsewhere.
// Adds in flight meanwhile only raise the counter further, and stay far below 0x8000 in total, so
// the counter never carries into its neighbour.
__device__ __forceinline__ bool add_u16(uint32_t a16, uint32_t v) {
  const uint32_t word = a16 & ~3u, sh = (a16 & 2u) * 8u;
  uint32_t old;
  asm volatile("atom.shared.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(word), "r"(v << sh) : "memory");
  const uint32_t h = (old >> sh) & 0xFFFFu;
  if (h < 0x8000u && h + v >= 0x8000u) {
    red_shared_add(word, 0u - (0x8000u << sh));
    return true;
  }
  return false;
}

__device__ __forceinline__ void cp_async16(uint32_t smem_addr, const void* gptr) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr), "l"(gptr) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ catalog conversion

// (RA, Dec) in arcminutes -> unit vector (cos d cos a, cos d sin a, sin d), computed in fp64 and
// rounded to fp32. Non-finite inputs become (0, 0) so that every vector has unit length.
__device__ __forceinline__ float4 radec_to_unit(float ra_arcmin, float dec_arcmin) {
  const double k = 3.14159265358979323846 / 10800.0;
  double a = (double)ra_arcmin * k;
  double d = (double)dec_arcmin * k;
  if (!isfinite(a) || !isfinite(d)) { a = 0.0; d = 0.0; }
  double sa, ca, sd, cd;
  sincos(a, &sa, &ca);
  sincos(d, &sd, &cd);
  return make_float4((float)(cd * ca), (float)(cd * sa), (float)sd, 0.0f);
}

// ------------------------------------------------------------------ spatial order and caps
//
// Catalogs are put in a spatial order before pairing: galaxies sorted by cell of a cube map
// (6 faces x 64 x 64 cells, Hilbert order within a face). A warp's i-galaxies and a j-chunk then
// each cover a small patch of sky, bounded by a "cap" (centre, angular radius). From two caps
// the kernel knows when every pair of a (warp, chunk) is surely below or surely above 90
// degrees, and drops the per-pair sign decision there, and when every pair lies between 55 and
// 125 degrees, where it uses the dot form. The chord loops compute every pair's code with the same
// arithmetic whichever of them evaluates it; the dot form computes a different (equally valid)
// approximation, so a mid-range pair within ~4e-7 rad of an edge may bin by its grouping.

constexpr int kFaceBits = 6;
constexpr int kFaceCells = 1 << kFaceBits;
constexpr int kCells = 6 * kFaceCells * kFaceCells;

// Position of cell (x, y) along the Hilbert curve through a 2^kFaceBits square: consecutive
// positions are adjacent cells, so runs of sorted galaxies stay compact (no Morton jumps).
__device__ __forceinline__ unsigned int hilbert_index(unsigned int x, unsigned int y) {
  unsigned int d = 0;
  for (unsigned int s = kFaceCells / 2; s > 0; s >>= 1) {
    const unsigned int rx = (x & s) ? 1u : 0u, ry = (y & s) ? 1u : 0u;
    d += s * s * ((3u * rx) ^ ry);
    if (ry == 0) {
      if (rx == 1) {
        x = s - 1 - (x & (s - 1)) + (x & ~(s - 1));
        y = s - 1 - (y & (s - 1)) + (y & ~(s - 1));
      }
      const unsigned int t = x;
      x = y;
      y = t;
    }
  }
  return d;
}

__device__ __forceinline__ unsigned int cell_of(double x, double y, double z) {
  const double ax = fabs(x), ay = fabs(y), az = fabs(z);
  int face;
  double u, v, m;
  if (ax >= ay && ax >= az) { face = x >= 0 ? 0 : 1; m = ax; u = y; v = z; }
  else if (ay >= az) { face = y >= 0 ? 2 : 3; m = ay; u = x; v = z; }
  else { face = z >= 0 ? 4 : 5; m = az; u = x; v = y; }
  int iu = (int)((u / m + 1.0) * 0.5 * kFaceCells);
  int iv = (int)((v / m + 1.0) * 0.5 * kFaceCells);
  iu = iu < 0 ? 0 : (iu >= kFaceCells ? kFaceCells - 1 : iu);
  iv = iv < 0 ? 0 : (iv >= kFaceCells ? kFaceCells - 1 : iv);
  return (unsigned int)face * (kFaceCells * kFaceCells) + hilbert_index((unsigned)iu, (unsigned)iv);
}

// Sort key of a galaxy: its cell, from fp32 arithmetic (the key only has to be a deterministic
// function of the input; vectors near a cell border may fall on either side).
__device__ __forceinline__ unsigned int cell_key(float ra_arcmin, float dec_arcmin) {
  const float k = 3.14159265358979323846f / 10800.0f;
  float a = ra_arcmin * k, d = dec_arcmin * k;
  if (!isfinite(a) || !isfinite(d)) { a = 0.0f; d = 0.0f; }
  float sa, ca, sd, cd;
  sincosf(a, &sa, &ca);
  sincosf(d, &sd, &cd);
  return cell_of((double)(cd * ca), (double)(cd * sa), (double)sd);
}

// (RA, Dec) arcminutes -> fp64 unit vector; non-finite inputs become (0, 0).
__device__ __forceinline__ void unit64(float ra_arcmin, float dec_arcmin, double& x, double& y, double& z) {
  const double k = 3.14159265358979323846 / 10800.0;
  double a = (double)ra_arcmin * k, d = (double)dec_arcmin * k;
  if (!isfinite(a) || !isfinite(d)) { a = 0.0; d = 0.0; }
  double sa, ca, sd, cd;
  sincos(a, &sa, &ca);
  sincos(d, &sd, &cd);
  x = cd * ca;
  y = cd * sa;
  z = sd;
}

// The sort is a stable two-pass LSD radix sort on the cell key (15 bits: 8, then 7), so galaxies
// of one cell keep their input order and the spatial order, the groups and their caps depend on
// the input alone. Each pass: per-tile digit counts, one exclusive scan over (digit, tile), and a
// stable scatter in which every tile ranks its elements round by round (warp match + warp totals).
constexpr int kSortThreads = 256;
constexpr int kSortRounds = 8;
constexpr int kSortTile = kSortThreads * kSortRounds;  // elements per tile (one block)
constexpr int kSortDigits = 256;

// One catalog's preparation: its input, its sort scratch and its outputs. The preparation kernels
// take up to two catalogs at once (PrepBatch, blockIdx.y selects the catalog), so that both catalogs
// of a cross-correlation are sorted and converted by the same launches.
// A unit vector as double-single components, 32 bytes (one sector): h = (hx, hy, hz, lx), l = (ly,
// lz, 0, 0); hx = the fp32 rounding of the fp64 x, lx = the fp32 rounding of what it leaves.
struct __align__(32) DsVec {
  float4 h, l;
};

// One 256-bit load of a DsVec, as the hi (x, y, z) and lo (x, y, z) parts (w = 0).
__device__ __forceinline__ void load_ds(const DsVec* p, float4& hi, float4& lo) {
  float lx;
  asm("ld.global.nc.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=f"(hi.x), "=f"(hi.y), "=f"(hi.z), "=f"(lx), "=f"(lo.y), "=f"(lo.z), "=f"(hi.w), "=f"(lo.w)
      : "l"(p));
  lo.x = lx;
}

// One 256-bit store of a group record (its lane's flags, the i-set row, the group's first j, path).
__device__ __forceinline__ void store_group_record(GroupRecord* p, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                                   uint32_t r, uint32_t j, uint32_t pc) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w0), "r"(w1), "r"(w2), "r"(w3),
               "r"(r), "r"(j), "r"(pc), "r"(0u)
               : "memory");
}

// One 256-bit load of a group record: the flag words (m) and (r, j, pc, 0) (h).
__device__ __forceinline__ void load_group_record(const GroupRecord* p, uint4& m, uint4& h) {
  asm("ld.global.nc.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(m.x), "=r"(m.y), "=r"(m.z), "=r"(m.w), "=r"(h.x), "=r"(h.y), "=r"(h.z), "=r"(h.w)
      : "l"(p));
}

struct PrepCat {
  const float* ra;        // input, arcminutes
  const float* dec;
  long long n;
  int tiles;              // sort tiles of kSortTile galaxies
  unsigned int* key0;     // sort: cell keys in input order; at the end the order (position -> input index)
  unsigned int* key1;     // sort: keys after the first pass
  unsigned int* idx1;     // sort: input indices after the first pass
  unsigned int* counts;   // sort: digit counts per tile, then their offsets
  float4* v;              // outputs: fp32 vectors, the double-single vectors, fp64 vectors, caps
  DsVec* ds;
  double4_32a* v64;
  float4* cap32;
  float4* cap128;
};
struct PrepBatch {
  PrepCat c[2];
};

// Digit counts of one tile. Pass 1 (PASS1) also computes every galaxy's cell key. Digits at bit
// `shift`.
template <bool PASS1>
__global__ void __launch_bounds__(kSortThreads) sort_count_kernel(const PrepBatch b, int shift) {
  const PrepCat& C = b.c[blockIdx.y];
  if ((int)blockIdx.x >= C.tiles) return;
  __shared__ unsigned int h[kSortDigits];
  for (int d = threadIdx.x; d < kSortDigits; d += kSortThreads) h[d] = 0u;
  __syncthreads();
  const long long base = (long long)blockIdx.x * kSortTile;
  for (int r = 0; r < kSortRounds; ++r) {
    const long long i = base + r * kSortThreads + threadIdx.x;
    if (i < C.n) {
      unsigned int k;
      if (PASS1) {
        k = cell_key(C.ra[i], C.dec[i]);
        C.key0[i] = k;
      } else {
        k = C.key1[i];
      }
      atomicAdd(&h[(k >> shift) & (kSortDigits - 1)], 1u);
    }
  }
  __syncthreads();
  for (int d = threadIdx.x; d < kSortDigits; d += kSortThreads) C.counts[(size_t)d * C.tiles + blockIdx.x] = h[d];
}

// In-place exclusive prefix sum of a catalog's tiles * kSortDigits counts, one block of 1024 threads
// per catalog: rounds of 1024 consecutive values (coalesced loads), each scanned with warp shuffles
// and the 32 warp totals, plus the carry.
__global__ void __launch_bounds__(1024) scan_kernel(const PrepBatch b) {
  const PrepCat& C = b.c[blockIdx.y];
  unsigned int* __restrict__ v = C.counts;
  const long long m = (long long)C.tiles * kSortDigits;
  __shared__ unsigned int warp_sum[32];
  __shared__ unsigned int carry;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  if (t == 0) carry = 0u;
  __syncthreads();
  for (long long base = 0; base < m; base += 1024) {
    const long long c = base + t;
    const unsigned int x = c < m ? v[c] : 0u;
    unsigned int s = x;  // inclusive scan within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane == 31) warp_sum[warp] = s;
    __syncthreads();
    if (warp == 0) {  // scan the warp totals
      unsigned int w = warp_sum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_sum[lane] = w;  // inclusive
    }
    __syncthreads();
    const unsigned int before = carry + (warp > 0 ? warp_sum[warp - 1] : 0u) + s - x;
    if (c < m) v[c] = before;
    __syncthreads();
    if (t == 1023) carry = before + x;
    __syncthreads();
  }
}

// Stable scatter of one tile. Element i of the tile goes to offset(digit, tile) + the number of
// earlier elements of the tile with the same digit: rounds of 256 in input order; within a round a
// warp ranks its lanes with __match_any_sync, and the warps' per-digit totals rank the warps.
// Pass 1 (FINAL = false) moves (key, input index) from key0 to key1/idx1; pass 2 moves only the
// input index, from idx1 into key0 (the order; pass 2 no longer reads key0).
template <bool FINAL>
__global__ void __launch_bounds__(kSortThreads) sort_scatter_kernel(const PrepBatch b, int shift) {
  const PrepCat& C = b.c[blockIdx.y];
  if ((int)blockIdx.x >= C.tiles) return;
  const unsigned int* __restrict__ keys_in = FINAL ? C.key1 : C.key0;
  const long long n = C.n;
  constexpr int W = kSortThreads / 32;
  __shared__ unsigned int running[kSortDigits];      // elements of each digit placed by earlier rounds
  __shared__ unsigned int wcount[W][kSortDigits];    // this round: elements of each digit per warp
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  for (int d = t; d < kSortDigits; d += kSortThreads) running[d] = C.counts[(size_t)d * C.tiles + blockIdx.x];
  const long long base = (long long)blockIdx.x * kSortTile;
  const unsigned int lt = (1u << lane) - 1u;
  for (int r = 0; r < kSortRounds; ++r) {
    for (int k = t; k < W * kSortDigits; k += kSortThreads) (&wcount[0][0])[k] = 0u;
    __syncthreads();
    const long long i = base + r * kSortThreads + t;
    const bool ok = i < n;
    const unsigned int key = ok ? keys_in[i] : 0u;
    const unsigned int dig = ok ? (key >> shift) & (kSortDigits - 1) : kSortDigits;  // kSortDigits: no element
    const unsigned int peers = __match_any_sync(0xffffffffu, dig);
    const unsigned int rank = __popc(peers & lt);
    if (ok && rank == 0) wcount[warp][dig] = __popc(peers);
    __syncthreads();
    if (ok) {
      unsigned int pos = running[dig] + rank;
      for (int w = 0; w < warp; ++w) pos += wcount[w][dig];
      if (ACF_CHECK(pos < (unsigned long long)n, 5, i, pos)) {
        if (FINAL) {
          C.key0[pos] = C.idx1[i];
        } else {
          C.idx1[pos] = (unsigned int)i;
          C.key1[pos] = key;
        }
      }
    }
    __syncthreads();
    for (int d = t; d < kSortDigits; d += kSortThreads) {
      unsigned int tot = 0u;
#pragma unroll
      for (int w = 0; w < W; ++w) tot += wcount[w][d];
      running[d] += tot;
    }
    __syncthreads();
  }
}

// Unit vectors in sorted order, as fp32 (pair kernel) and fp64 (exact re-decision of flagged
// pairs): position p holds input galaxy order[p] (key0 after the sort).
// v is the fp32 rounding of each fp64 component and lo the fp32 rounding of what remains
// (|x - hi - lo| <= 2^-48 |x|): together a double-single copy for the fix-up.
__global__ void vectors_kernel(const PrepBatch b) {
  const PrepCat& C = b.c[blockIdx.y];
  for (long long p = blockIdx.x * (long long)blockDim.x + threadIdx.x; p < C.n; p += (long long)gridDim.x * blockDim.x) {
    const unsigned int src = C.key0[p];
    if (ACF_CHECK(src < (unsigned long long)C.n, 5, p, src)) {
      double x, y, z;
      unit64(C.ra[src], C.dec[src], x, y, z);
      const float hx = (float)x, hy = (float)y, hz = (float)z;
      C.v[p] = make_float4(hx, hy, hz, 0.0f);
      DsVec d;
      d.h = make_float4(hx, hy, hz, (float)(x - (double)hx));
      d.l = make_float4((float)(y - (double)hy), (float)(z - (double)hz), 0.0f, 0.0f);
      C.ds[p] = d;
      C.v64[p] = make_double4_32a(x, y, z, 0.0);
    }
  }
}

// Angular radius, with a small safety margin, of the chord-distance sq = |c - v|^2.
__device__ __forceinline__ float chord_to_angle(float sq) { return 2.0f * asinf(fminf(sqrtf(sq) * 0.5f, 1.0f)); }
constexpr float kCapMargin = 2e-5f;

// One warp per 128 sorted galaxies: the cap of each 32-galaxy group and of the whole chunk.
// Empty groups get radius 4 (> pi), which no decision can use.
__global__ void caps_kernel(const PrepBatch b) {
  const PrepCat& C = b.c[blockIdx.y];
  const float4* __restrict__ v = C.v;
  const long long n = C.n;
  float4* __restrict__ cap32 = C.cap32;
  float4* __restrict__ cap128 = C.cap128;
  const int lane = threadIdx.x & 31;
  const long long chunk = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nchunks = (n + 127) / 128;
  if (chunk >= nchunks) return;
  float4 m[4];
  bool ok[4];
  float tx = 0.f, ty = 0.f, tz = 0.f;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const long long i = chunk * 128 + g * 32 + lane;
    ok[g] = i < n;
    m[g] = ok[g] ? v[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    tx += m[g].x; ty += m[g].y; tz += m[g].z;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tx += __shfl_xor_sync(0xffffffffu, tx, o);
    ty += __shfl_xor_sync(0xffffffffu, ty, o);
    tz += __shfl_xor_sync(0xffffffffu, tz, o);
  }
  const float tn = rsqrtf(fmaxf(tx * tx + ty * ty + tz * tz, 1e-30f));
  tx *= tn; ty *= tn; tz *= tn;
  float tmax = 0.f;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    float gx = m[g].x, gy = m[g].y, gz = m[g].z;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      gx += __shfl_xor_sync(0xffffffffu, gx, o);
      gy += __shfl_xor_sync(0xffffffffu, gy, o);
      gz += __shfl_xor_sync(0xffffffffu, gz, o);
    }
    const float gn = rsqrtf(fmaxf(gx * gx + gy * gy + gz * gz, 1e-30f));
    gx *= gn; gy *= gn; gz *= gn;
    float dx = gx - m[g].x, dy = gy - m[g].y, dz = gz - m[g].z;
    float sq = ok[g] ? dx * dx + dy * dy + dz * dz : 0.f;
    dx = tx - m[g].x; dy = ty - m[g].y; dz = tz - m[g].z;
    tmax = fmaxf(tmax, ok[g] ? dx * dx + dy * dy + dz * dz : 0.f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq = fmaxf(sq, __shfl_xor_sync(0xffffffffu, sq, o));
    const bool any = __any_sync(0xffffffffu, ok[g]);
    if (lane == 0) cap32[chunk * 4 + g] = make_float4(gx, gy, gz, any ? chord_to_angle(sq) + kCapMargin : 4.0f);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
  if (lane == 0) cap128[chunk] = make_float4(tx, ty, tz, chord_to_angle(tmax) + kCapMargin);
}

// ------------------------------------------------------------------ bin index of one pair

// The float 2^23 + (histogram entry), whose bit pattern is bits(2^23) + entry. Symmetric in (u, v) bit for bit:
// the products commute and u - s v = -(v - s u) rounds to the same magnitude.
template <int MAP, int METHOD, bool FINE = false>
__device__ __forceinline__ float pair_code(float xi, float yi, float zi, float xj, float yj, float zj,
                                           const BinParams& bp) {
  const float d = fmaf(zi, zj, fmaf(yi, yj, xi * xj));
  if (METHOD == kDotAcos || METHOD == kDotFastAcos) {
    // the page's route: arccos of the (clamped) cosine, scaled by 1/w and truncated; acosf, or the
    // polynomial of the approximate mode
    const float c = fminf(fmaxf(d, -1.0f), 1.0f);
    const float t = (METHOD == kDotAcos ? acosf(c) : acos_as4445(c)) * bp.inv_w;
    return add_rz(fminf(t, bp.clamp_c), kMagic);
  } else {
    const uint32_t db = __float_as_uint(d);
    // ns = -sign(d) as +-1.0: (d & signmask) ^ bits(-1.0), one logic op
#if ACF_ASM_LOP3
    const float ns = __uint_as_float(lop3<0x6A>(db, 0x80000000u, 0xbf800000u));
#else
    const float ns = __uint_as_float((db & 0x80000000u) ^ 0xbf800000u);
#endif
    const float dx = fmaf(ns, xj, xi);
    const float dy = fmaf(ns, yj, yi);
    const float dz = fmaf(ns, zj, zi);
    // 1e-30 keeps t' > 0 for identical or exactly antipodal vectors (see the mirror map)
    const float q = fmaf(dz, dz, fmaf(dy, dy, fmaf(dx, dx, 1e-30f)));
    float p = fmaf(kP7, q, kP6);
    p = fmaf(p, q, kP5);
    p = fmaf(p, q, kP4);
    p = fmaf(p, q, kP3);
    p = fmaf(p, q, kP2);
    p = fmaf(p, q, kP1);
    p = fmaf(p, q, kP0);
    const float th = sqrt_approx(p * q);  // theta' in radians
    if (MAP == kDirect) {
      // near side (s = +1): floor(theta'/w) exactly, by one fma rounded toward zero onto 2^23;
      // far side: the same fma of -theta' onto 2^23 + P gives P - ceil(theta'/w), which is exactly
      // floor((pi - theta')/w) = floor(theta/w) when P = pi/w is an integer.
      // theta' carrying the sign of d: th | (d & signmask), one logic op
      const float m = (int)db < 0 ? (FINE ? bp.magic_far_f : bp.magic_far) : (FINE ? bp.magic_f : kMagic);
#if ACF_ASM_LOP3
      return fma_rz(__uint_as_float(lop3<0xF8>(__float_as_uint(th), db, 0x80000000u)), FINE ? bp.inv_w_f : bp.inv_w, m);
#else
      return fma_rz(__uint_as_float(__float_as_uint(th) | (db & 0x80000000u)), FINE ? bp.inv_w_f : bp.inv_w, m);
#endif
    } else {
      const float h = fmaf(ns, 1.57079632679489662f, 1.57079632679489662f);  // 0 or pi
      const float tr = fmaf(-ns, th, h);                                       // theta
      return FINE ? add_rz(fminf(tr * bp.inv_w_f, bp.clamp_f), bp.magic_f) : add_rz(fminf(tr * bp.inv_w, bp.clamp_c), kMagic);
    }
  }
}

// histogram entry -> bin (both maps index entries by bin; entries past the last bin clamp to it)
template <int MAP>
__device__ __forceinline__ int entry_to_bin(int e, const BinParams& bp) {
  const int k = e < 0 ? 0 : e;
  return k > bp.nbins - 1 ? bp.nbins - 1 : k;
}

// The same code as pair_code<MAP, kChordPoly> for a pair whose sign(u.v) is known in advance
// (the caps of its warp and j-group put every separation below 90 degrees, or every one above):
// ns = -sign as +-1.0, iws = sign / w (or sign * 2^S / w for the fine code) and h (direct map:
// 2^23 or the far-side constant; clamp map: 0 or pi / w) are registers chosen per j-group. Bit for
// bit the general code takes these steps for such a pair: fma(ns, v, u) is the same difference or
// sum, and the far-side code fma_rz(-theta', 1/w, m) is fma_rz(theta', -1/w, m). Only the dot
// product, the sign-bit operation and the choice of constant are dropped.
// SMALL: the degree-5 polynomial, for groups whose caps keep every theta' below 72 degrees.
template <int MAP, bool FINE = false, bool SMALL = false>
__device__ __forceinline__ float pair_code_fixed(float xi, float yi, float zi, float xj, float yj, float zj, float ns,
                                                 float iws, float h, const BinParams& bp) {
  const float dx = fmaf(ns, xj, xi);
  const float dy = fmaf(ns, yj, yi);
  const float dz = fmaf(ns, zj, zi);
  const float q = fmaf(dz, dz, fmaf(dy, dy, fmaf(dx, dx, 1e-30f)));
  float p;
  if (SMALL) {
    p = fmaf(kS5, q, kS4);
    p = fmaf(p, q, kS3);
    p = fmaf(p, q, kS2);
    p = fmaf(p, q, kS1);
    p = fmaf(p, q, kS0);
  } else {
    p = fmaf(kP7, q, kP6);
    p = fmaf(p, q, kP5);
    p = fmaf(p, q, kP4);
    p = fmaf(p, q, kP3);
    p = fmaf(p, q, kP2);
    p = fmaf(p, q, kP1);
    p = fmaf(p, q, kP0);
  }
  const float th = sqrt_approx(p * q);
  if (MAP == kDirect) {
    return fma_rz(th, iws, h);
  } else {
    // theta / w = th * iws + h with h = 0 (near side) or pi / w (far side); iws = -1/w there; the
    // fine clamp is in units of the form's own window (S_small fine bits for the short chord)
    const float t = fmaf(th, iws, h);
    return add_rz(fminf(t, FINE ? (SMALL ? bp.clamp_fs : bp.clamp_f) : bp.clamp_c), FINE ? bp.magic_f : kMagic);
  }
}

// Exact mode, fixed sign: the fine code (returned) and the plain code of the same pair (coarse),
// from one theta'. The fine constants are the plain ones times 2^S exactly (plus the bias), so
// both floor the same real number: their entries agree unless the fine code flags the pair.
template <int MAP, bool SMALL>
__device__ __forceinline__ float pair_code_fixed2(float xi, float yi, float zi, float xj, float yj, float zj,
                                                  float ns, float iws_f, float h_f, float iws, float h,
                                                  const BinParams& bp, uint32_t& coarse) {
  const float dx = fmaf(ns, xj, xi);
  const float dy = fmaf(ns, yj, yi);
  const float dz = fmaf(ns, zj, zi);
  const float q = fmaf(dz, dz, fmaf(dy, dy, fmaf(dx, dx, 1e-30f)));
  float p;
  if (SMALL) {
    p = fmaf(kS5, q, kS4);
    p = fmaf(p, q, kS3);
    p = fmaf(p, q, kS2);
    p = fmaf(p, q, kS1);
    p = fmaf(p, q, kS0);
  } else {
    p = fmaf(kP7, q, kP6);
    p = fmaf(p, q, kP5);
    p = fmaf(p, q, kP4);
    p = fmaf(p, q, kP3);
    p = fmaf(p, q, kP2);
    p = fmaf(p, q, kP1);
    p = fmaf(p, q, kP0);
  }
  const float th = sqrt_approx(p * q);
  if (MAP == kDirect) {
    coarse = __float_as_uint(fma_rz(th, iws, h));
    return fma_rz(th, iws_f, h_f);
  } else {
    const float t = fmaf(th, iws, h);
    const float tf = fmaf(th, iws_f, h_f);
    coarse = __float_as_uint(add_rz(fminf(t, bp.clamp_c), kMagic));
    return add_rz(fminf(tf, SMALL ? bp.clamp_fs : bp.clamp_f), bp.magic_f);
  }
}

// The dot form, for pairs whose caps put theta in (55, 125) degrees (direct map, P even):
// theta / w = P/2 - d R(d^2) / w, floored exactly by one fma rounded toward zero onto 2^23 + P/2
// (the product of the two fp32 operands enters unrounded). Worst-case theta error: d carries
// <= 2.1e-7 from the fp32 vectors and the dot product, i.e. <= 2.6e-7 rad where sin theta >=
// sin 55 deg, plus <= 3.2e-7 from the polynomial (fit 1.6e-7, Horner 1e-7) and its scaling
// (5.7e-8): <= 6e-7 in all.
template <bool FINE = false>
__device__ __forceinline__ float pair_code_mid(float xi, float yi, float zi, float xj, float yj, float zj,
                                               const BinParams& bp) {
#define ACF_RC(k) (FINE ? bp.rc_f[k] : bp.rc[k])
  const float d = fmaf(zi, zj, fmaf(yi, yj, xi * xj));
  const float t = d * d;
  float p = fmaf(ACF_RC(4), t, ACF_RC(3));
  p = fmaf(p, t, ACF_RC(2));
  p = fmaf(p, t, ACF_RC(1));
  p = fmaf(p, t, ACF_RC(0));
#undef ACF_RC
  return fma_rz(-d, p, FINE ? bp.magic_mid_f : bp.magic_mid);
}

// Cap of K consecutive 32-galaxy groups: centre = normalised sum of the group centres, radius =
// the largest (distance to a group centre + that group's radius). Empty groups are skipped.
template <int K>
__device__ __forceinline__ float4 union_caps(const float4* __restrict__ cap32, long long g0, long long ngroups) {
  float cx = 0.f, cy = 0.f, cz = 0.f;
  float4 c[K];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    c[k] = (g0 + k < ngroups) ? __ldg(cap32 + g0 + k) : make_float4(1.f, 0.f, 0.f, 4.0f);
    if (c[k].w <= 3.2f) { cx += c[k].x; cy += c[k].y; cz += c[k].z; }
  }
  const float nn = rsqrtf(fmaxf(cx * cx + cy * cy + cz * cz, 1e-30f));
  cx *= nn; cy *= nn; cz *= nn;
  float r = 0.f;
  bool any = false;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    if (c[k].w <= 3.2f) {
      const float dx = cx - c[k].x, dy = cy - c[k].y, dz = cz - c[k].z;
      r = fmaxf(r, chord_to_angle(dx * dx + dy * dy + dz * dz) + c[k].w);
      any = true;
    }
  }
  return make_float4(cx, cy, cz, any ? r + kCapMargin : 4.0f);
}

enum Path { kGeneral = 0, kBelow90 = 1, kAbove90 = 2 };
template <int P>
struct PathTag {
  static constexpr int value = P;
};

// Which loop a (warp, j-group) may use: every pair surely below 90 degrees, surely above, or
// mixed. Two caps at centre angle tc and radii ra, rb hold only separations in
// [tc - ra - rb, tc + ra + rb]; all are below 90 degrees iff cos tc > sin(ra + rb) and all above
// iff cos tc < -sin(ra + rb). __sinf/__cosf are accurate to ~1e-6 here and the margins cover it.
// kExactBit is added when the exact mode must check this group: mode 2 always, mode 1 when some
// separation may be below lo or above pi - lo (cos tc > cos(lo + r) or < -cos(lo + r)).
// kMidBit is added when every separation lies in (55, 125) degrees (|cos tc| < cos(55 deg + r))
// and the dot form is on; in mode 1 never for a group the exact mode checks, so every pair the
// exact mode may re-decide is binned by a chord form. Otherwise kSmallBit is added when every
// theta' lies below 72 degrees on one side of 90 (|cos tc| > cos(72 deg - r)).
constexpr int kExactBit = 4;
constexpr int kMidBit = 8;
constexpr int kSmallBit = 16;
__device__ __forceinline__ int choose_path(float4 a, float4 b, int mode, float lo, int mid, int small) {
  const float dot = a.x * b.x + a.y * b.y + a.z * b.z;
  const float r = a.w + b.w + 1e-4f;
  int path = kGeneral;
  if (r < 1.5f) {
    const float sr = __sinf(r) + 1e-5f;
    if (dot > sr) path = kBelow90;
    else if (dot < -sr) path = kAbove90;
  }
  if (mid && r < 0.75f) {
    const float cm = __cosf(kMidRad + r) - 1e-5f;
    if (fabsf(dot) < cm) path |= kMidBit;
  }
  if (small && !(path & kMidBit) && r < kSmallRad) {
    const float cs = __cosf(kSmallRad - r) + 1e-5f;
    if (fabsf(dot) > cs) path |= kSmallBit;  // implies a fixed sign
  }
  if (mode == 2) return path | kExactBit;
  if (mode == 1) {
    const float x = lo + r;
    if (x >= 3.0f) return (path & ~kMidBit) | kExactBit;
    const float cl = __cosf(x) - 1e-5f;
    if (dot > cl || dot < -cl) return (path & ~kMidBit) | kExactBit;
  }
  return path;
}

// The registers of a fixed-sign chord loop (see pair_code_fixed) for a group of path code pc: ns =
// -sign of u.v, the scale and constant of the plain code (iws_c, h_c) and of the code the loop
// bins or flags with (iws, h: the fine ones when `fine`, S_small bits for a short-chord group).
// The pair kernel and the exact re-decision derive them here alike, so that the re-decision
// recomputes a flagged pair's codes bit for bit.
struct ChordConsts {
  float ns, iws, h, iws_c, h_c;
};
template <int MAP>
__device__ __forceinline__ ChordConsts chord_consts(int pc, bool fine, const BinParams& bp) {
  const bool below = (pc & 3) == kBelow90;
  ChordConsts c;
  c.ns = below ? -1.0f : 1.0f;
  c.iws_c = below ? bp.inv_w : -bp.inv_w;
  if (MAP == kDirect) c.h_c = below ? kMagic : bp.magic_far;
  else c.h_c = below ? 0.0f : 3.14159265358979323846f * bp.inv_w;
  c.iws = c.iws_c;
  c.h = c.h_c;
  if (fine) {
    const bool sm = (pc & kSmallBit) != 0;
    const float iwf = sm ? bp.inv_w_fs : bp.inv_w_f;
    c.iws = below ? iwf : -iwf;
    if (MAP == kDirect) c.h = below ? bp.magic_f : (sm ? bp.magic_far_fs : bp.magic_far_f);
    else c.h = below ? 0.0f : 3.14159265358979323846f * iwf;
  }
  return c;
}

template <bool F>
struct FineTag {
  static constexpr bool value = F;
};
template <int X>
struct FormTag {
  static constexpr int value = X;
};

// Add one pair to the shared histogram. With F (exact mode) the code carries fine_shift extra
// fractional bits, biased by one unit: the entry is the code's integer part. Returns whether the
// pair lies within one fine unit of an edge (biased fraction 0 or 1); such pairs are recorded
// (push_record).
// A pair at one fine unit below an edge is counted one entry up; the exact re-decision moves it.
// shift 1 is the kBlock16 layout: 16-bit counters, whose overflow goes to the block's row.
template <bool F, int MAP>
__device__ __forceinline__ bool add_pair(const PairParams& p, uint32_t cb, uint32_t base, uint32_t base_f, int shift,
                                         int S, uint32_t magic_bits, int i, int j, float xi, float yi, float zi,
                                         float4 v, uint32_t inc) {
  if (!F) {
    if (ACF_CHECK(cb - magic_bits < (uint32_t)p.bp.entries, 1, (long long)(cb - magic_bits), i,
                  __uint_as_float(cb), xi, yi, zi, v.x, v.y, v.z, (float)j)) {
      if (shift == 1) {
        if (add_u16((cb << 1) + base, inc))
          atomicAdd(p.partial + (size_t)blockIdx.x * p.bp.nbins + entry_to_bin<MAP>((int)(cb - magic_bits), p.bp),
                    0x8000ull);
      } else {
        hist_add((cb << shift) + base, inc, shift == 2);
      }
    }
    return false;
  } else {
    if (ACF_CHECK(((cb - magic_bits) >> S) < (uint32_t)p.bp.entries, 6, (long long)((cb - magic_bits) >> S), i,
                  __uint_as_float(cb), xi, yi, zi, v.x, v.y, v.z, (float)j))
      hist_add(((cb >> S) << shift) + base_f, inc, shift == 2);
    return (cb & ((1u << S) - 1u)) <= 1u;
  }
}

// Exact mode: record, for the re-decision, a j whose pairs with the warp's i-set hold at least one
// flagged pair (a fine code within one fine unit of an edge). One record per warp and j: the header
// (j, the i-set row r, the group's path code pc) and for each i-vector slot k the ballot of the lanes
// whose pair (i = kJT r + islot(k, lane), j) is flagged. The re-decision recomputes each such pair's
// codes from the same vectors with the same device code (the path code fixes the form), so that
// the record need not carry them. The warp's records go to its own region of the queue at its
// cursor `cur` (the same value in every lane; no atomic), and past the region's end to slots of the
// spill region (one global counter). Called by every lane. Returns whether the record found a slot;
// if not, its pairs keep their fp32 bins and are counted as flagged and as overflow. (These per-j
// records serve the kernels whose flags are rare; the block-shared exact kernel, whose flags are
// dense, keeps group records instead: see GroupRecord.)
static_assert(kJT == 128, "a flag record holds four 32-lane ballots");
__device__ __forceinline__ bool push_record(const PairParams& p, unsigned int region, unsigned int& cur, int r, int j, int pc,
                                            uint32_t m0, uint32_t m1, uint32_t m2, uint32_t m3) {
  const bool lead = (threadIdx.x & 31) == 0;
  const uint2 hdr = make_uint2((unsigned)j, (unsigned)r | ((unsigned)pc << 24));
  if (cur < p.qbatch) {
    if (lead) {
      const size_t slot = (size_t)region * p.qbatch + cur;
      p.qhdr[slot] = hdr;
      p.qmask[slot] = make_uint4(m0, m1, m2, m3);
    }
    ++cur;
    return true;
  }
  ++cur;
  bool ok = false;
  if (lead) {
    // spill slots start after every warp's region
    const unsigned int regions = gridDim.x * (blockDim.x >> 5);
    const unsigned long long slot = (unsigned long long)regions * p.qbatch + atomicAdd(p.qspill, 1u);
    if (slot < p.qcap) {
      p.qhdr[slot] = hdr;
      p.qmask[slot] = make_uint4(m0, m1, m2, m3);
      ok = true;
    } else {
      const unsigned int n = __popc(m0) + __popc(m1) + __popc(m2) + __popc(m3);
      atomicAdd(p.qoverflow, n);
      atomicAdd(p.qflagged, n);
    }
  }
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// A flagged pair of a single-code loop that is not re-decided keeps its fp32 bin: if the one-unit
// bias carried it into the next entry (biased fraction 0), its count moves back. cb is its fine code
// (S fractional bits), base_f/shift the histogram addressing of the loop.
__device__ __forceinline__ void carry_back(uint32_t cb, int S, uint32_t base_f, int shift, uint32_t inc) {
  if ((cb & ((1u << S) - 1u)) == 0u) {
    const uint32_t a = ((cb >> S) << shift) + base_f;
    red_shared_add(a, 0u - inc);
    red_shared_add(a - (1u << shift), inc);
  }
}

// ------------------------------------------------------------------ pair kernel

// Which galaxy of a warp's i-set (kJT = 32 K consecutive sorted galaxies) lane `lane` holds in its
// slot k. ACF_ISPREAD 1: lane l holds galaxies K l .. K l + K - 1, so that the 32 lanes of one slot
// spread over the whole i-set and their separations to one j over more bins (fewer lanes adding to
// the same counter of a block-shared histogram at once); 0: lane l holds l, l + 32, ... The pairs, the
// caps and the forms are the same either way.
#ifndef ACF_ISPREAD
#define ACF_ISPREAD 1
#endif
template <int K>
__device__ __forceinline__ int islot(int k, int lane) {
  return ACF_ISPREAD ? lane * K + k : k * 32 + lane;
}

// Map unit u to (i-set row r, j-chunk column c). For DD/RR row r holds columns r .. cols-1 and
// starts at S(r) = r*cols - r*(r-1)/2.
__device__ __forceinline__ void unit_coords(const PairParams& p, long long u, int& r, int& c) {
  const long long cj = p.cols;
  if (!p.sym) {
    r = (int)(u / cj);
    c = (int)(u - (long long)r * cj);
    return;
  }
  long long lo = 0, hi = p.rows - 1;
  while (lo < hi) {
    const long long mid = (lo + hi + 1) >> 1;
    if (mid * cj - mid * (mid - 1) / 2 <= u) lo = mid;
    else hi = mid - 1;
  }
  r = (int)lo;
  c = (int)(lo + (u - (lo * cj - lo * (lo - 1) / 2)));
}

template <int K, int THREADS, int LAYOUT, int MAP, int METHOD>
__device__ __forceinline__ void flush_hist(const PairParams& p, uint32_t* hist, bool zero) {
  unsigned long long* row = p.partial + (size_t)blockIdx.x * p.bp.nbins;
  if (LAYOUT == kLane) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int e = warp; e < p.bp.entries; e += THREADS / 32) {
      unsigned long long v = hist[e * 32 + lane];
      if (zero) hist[e * 32 + lane] = 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && v && ACF_CHECK(entry_to_bin<MAP>(e, p.bp) < p.bp.nbins, 3, e, entry_to_bin<MAP>(e, p.bp)))
        atomicAdd(row + entry_to_bin<MAP>(e, p.bp), v);
    }
  } else if (LAYOUT == kBlock16) {
    const int words = (p.bp.entries + 1) / 2;  // per copy
    for (int e = threadIdx.x; e < p.bp.entries; e += THREADS) {
      const int sh = (e & 1) * 16;
      const unsigned long long v = ((hist[e >> 1] >> sh) & 0xFFFFu) + ((hist[words + (e >> 1)] >> sh) & 0xFFFFu);
      if (v && ACF_CHECK(entry_to_bin<MAP>(e, p.bp) < p.bp.nbins, 3, e, entry_to_bin<MAP>(e, p.bp)))
        atomicAdd(row + entry_to_bin<MAP>(e, p.bp), v);
    }
    if (zero) {
      __syncthreads();
      for (int w = threadIdx.x; w < 2 * words; w += THREADS) hist[w] = 0;
    }
  } else {
    for (int e = threadIdx.x; e < p.bp.entries; e += THREADS) {
      const unsigned long long v = hist[e];
      if (zero) hist[e] = 0;
      if (v && ACF_CHECK(entry_to_bin<MAP>(e, p.bp) < p.bp.nbins, 3, e, entry_to_bin<MAP>(e, p.bp)))
        atomicAdd(row + entry_to_bin<MAP>(e, p.bp), v);
    }
  }
}

// Work unit = one warp's i-set (kJT = 32*K spatially consecutive i-galaxies, K per lane, in
// registers) against one j-chunk of kJT galaxies (in the warp's own shared-memory tile). Warps
// take units from a global ticket independently and never wait for each other inside the loop:
// each streams its own double-buffered j-tiles with cp.async and synchronises only with
// __syncwarp. All warps of the block add into one shared histogram (lane-private copies).
// GROUPS 1 (small problems): a unit is one 32-galaxy j-group of such a pair of chunks, four units
// per chunk pair, so that few galaxies still spread over many warps.
template <int K, int THREADS, int LAYOUT, int MAP, int METHOD, int GROUPS = 4>
__global__ void __launch_bounds__(THREADS, 1) pair_kernel(const PairParams p) {
  static_assert(32 * K == kJT, "an i-set and a j-chunk have the same size");
  constexpr int WARPS = THREADS / 32;
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float4* my_tiles = reinterpret_cast<float4*>(smem) + warp * 2 * kJT;  // [2][kJT] per warp
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + WARPS * 2 * kJT * sizeof(float4));

  // per warp: j-groups run on each path (see path_pairs), and the cap of the warp's current i-set
  // (kept here, not in registers, to leave the hot loops all the registers)
  __shared__ unsigned int s_paths[WARPS][9];
  __shared__ float4 s_icap[WARPS];
  const int words = (LAYOUT == kLane) ? p.bp.entries * 32 : (LAYOUT == kBlock16 ? 2 * ((p.bp.entries + 1) / 2) : p.bp.entries);
  for (int w = tid; w < words; w += THREADS) hist[w] = 0;
  unsigned long long* row = p.partial + (size_t)blockIdx.x * p.bp.nbins;
  if (!p.accumulate)
    for (int k = tid; k < p.bp.nbins; k += THREADS) row[k] = 0ull;
  __syncthreads();

  const uint32_t hist_addr = (uint32_t)__cvta_generic_to_shared(hist);
  const uint32_t tiles_addr = (uint32_t)__cvta_generic_to_shared(my_tiles);
  // every code is the float 2^23 + entry (the mirror offset is already inside the code)
  const uint32_t magic_bits = __float_as_uint(kMagic);
  // address of entry e in this lane's copy = (code bits << shift) + base
  // kBlock16: the first half of the warps adds to copy 0, the second half to copy 1 (2 bytes a counter)
  const uint32_t copy16 = (LAYOUT == kBlock16 && warp >= WARPS / 2) ? (uint32_t)((p.bp.entries + 1) / 2) * 4u : 0u;
  const uint32_t base = (LAYOUT == kLane)     ? hist_addr + lane * 4u - (magic_bits << 7)
                        : (LAYOUT == kBlock16) ? hist_addr + copy16 - (magic_bits << 1)
                                               : hist_addr - (magic_bits << 2);
  constexpr int SHIFT = (LAYOUT == kLane) ? 7 : (LAYOUT == kBlock16 ? 1 : 2);
  // exact mode: the fine code is 2^23 + (entry << S) + fraction; entry = (bits >> S) - (bits(2^23) >> S)
  const uint32_t base_f = (LAYOUT == kLane) ? hist_addr + lane * 4u - ((magic_bits >> p.bp.fine_shift) << 7)
                                            : hist_addr - ((magic_bits >> p.bp.fine_shift) << 2);
  const uint32_t base_fm = (LAYOUT == kLane) ? hist_addr + lane * 4u - ((magic_bits >> p.bp.fine_shift_mid) << 7)
                                             : hist_addr - ((magic_bits >> p.bp.fine_shift_mid) << 2);
  const int ni = (int)p.ni, nj = (int)p.nj;
  const uint32_t inc = p.inc;  // the histogram increment: 2 for DD/RR pairs i < j, 1 for DR
  // exact mode: this warp's region of the flag-record queue and its cursor there (warp-uniform)
  const unsigned int region = blockIdx.x * WARPS + warp;
  unsigned int cur = 0u;

  // tickets: the unit being computed (u), the one whose tile is in flight (un), and one fetched
  // ahead by lane 0 while computing (its latency hides behind the unit)
  unsigned int t = 0, tn = 0;
  if (lane == 0) {
    t = atomicAdd(p.ticket, 1u);
    tn = atomicAdd(p.ticket, 1u);
  }
  long long u = p.unit_begin + __shfl_sync(0xffffffffu, t, 0);
  long long un = p.unit_begin + __shfl_sync(0xffffffffu, tn, 0);
  auto load_tile = [&](int c, int b) {
    const int j0 = c * kJT;
#pragma unroll
    for (int m = 0; m < kJT / 32; ++m) {
      const int jj = m * 32 + lane;
      if (j0 + jj < nj) cp_async16(tiles_addr + (uint32_t)(b * kJT + jj) * 16u, p.vj + j0 + jj);
    }
    cp_async_commit();
  };
  if (u < p.unit_end) {
    // unit -> (i-set row, j-chunk column, j-group when a unit is one group)
    auto unit_of = [&](long long uu, int& r_, int& c_, int& g_) {
      if constexpr (GROUPS == 1) {
        unit_coords(p, uu >> 2, r_, c_);
        g_ = (int)(uu & 3);
      } else {
        unit_coords(p, uu, r_, c_);
        g_ = 0;
      }
    };
    int r, c, gs;
    unit_of(u, r, c, gs);
    load_tile(c, 0);
    float xi[K], yi[K], zi[K];
    if (lane < 9) s_paths[warp][lane] = 0u;
    int cur_r = -1, buf = 0;
    // j-groups per path (x 32*kJT pairs): chord fixed, chord general, the same with flags, dot form,
    // dot form with flags
    // path slots: 0 chord fixed, 1 chord general, 2 and 3 the same with flags, 4 masked units (in
    // units of kJT pairs), 5 dot form, 6 dot form with flags, 7 short chord, 8 short chord with flags
    auto count_path = [&](int slot, unsigned int n) {
      if (lane == 0) s_paths[warp][slot] += n;
    };
    while (true) {
      int rn = 0, cn = 0, gsn = 0;
      if (un < p.unit_end) {
        unit_of(un, rn, cn, gsn);
        load_tile(cn, buf ^ 1);
      } else {
        cp_async_commit();
      }
      unsigned int ta = 0;
      if (lane == 0) ta = atomicAdd(p.ticket, 1u);
      const int i0 = r * kJT;
      if (r != cur_r) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
          int i = i0 + islot<K>(k, lane);
          i = i < ni ? i : ni - 1;
          const float4 v = __ldg(p.vi + i);
          xi[k] = v.x;
          yi[k] = v.y;
          zi[k] = v.z;
          (void)ACF_CHECK(fabsf(v.x * v.x + v.y * v.y + v.z * v.z - 1.0f) < 1e-3f, 4, i, r, v.x, v.y, v.z);
        }
        if (METHOD == kChordPoly) {
          const float4 icap = union_caps<K>(p.icap32, (long long)i0 / 32, p.igroups);
          if (lane == 0) s_icap[warp] = icap;
          __syncwarp();
        }
        cur_r = r;
      }
      cp_async_wait<1>();
      __syncwarp();  // this unit's tile, copied by all lanes, is visible to all lanes

      const float4* tile = my_tiles + buf * kJT;
      const int j0 = c * kJT;
      const int jn = min(kJT, nj - j0);
      const bool full = (jn == kJT) && (i0 + kJT <= ni) && (!p.sym || c > r);
#ifdef ACF_DEBUG_BOUNDS
      for (int jj = 0; jj < jn; ++jj) {
        const float4 v = tile[jj];
        (void)ACF_CHECK(fabsf(v.x * v.x + v.y * v.y + v.z * v.z - 1.0f) < 1e-3f, 2, j0 + jj, u, v.x, v.y, v.z, (float)buf);
      }
#endif
      // group records (block-shared exact kernel): after each j-group, every lane with a flag writes
      // its record and lane 0 the ballot of those lanes (for every group of every unit, so that the
      // fix-up reads no stale ballot)
      auto group_flush = [&](const uint32_t(&fw)[K], int g, int pc) {
        static_assert(K == 4, "four flag words per record");
        const bool any = (fw[0] | fw[1] | fw[2] | fw[3]) != 0u;
        const unsigned int bal = __ballot_sync(0xffffffffu, any);
        const size_t gi = (size_t)(u - p.unit_begin) * 4 + g;
        if (any) store_group_record(p.grec + gi * 32 + lane, fw[0], fw[1], fw[2], fw[3], (uint32_t)r, (uint32_t)(j0 + g * 32),
                                    (uint32_t)pc);
        if (lane == 0) p.gbal[gi] = bal;
      };
      if (full) {
        // one loop per (32-galaxy j-group, path); the path is uniform across the warp. The fixed
        // chord loops take the sign in registers (ns, iws, h); the dot-form loop needs no sign; the
        // fine (exact) loops are rare and kept rolled so that all live loop bodies fit the
        // instruction cache.
        // (ns, iws, h): sign, scale and constant of a fixed-sign chord loop (fine ones when F);
        // (iws_c, h_c): the plain scale and constant, for the two-code fine loops
        auto run = [&](auto form, auto fine, int jbeg, int pc, float ns, float iws, float h, float iws_c, float h_c) {
          constexpr int X = decltype(form)::value;  // 0 chord general, 1 chord fixed sign, 2 dot form,
                                                    // 3 short chord (fixed sign)
          constexpr bool F = decltype(fine)::value;
          // the general and the full-range fixed chord loops are rare once the caps pick the dot form
          // across 90 degrees and the short chord below 72: rolled
          constexpr int U = (F || X == 0 || X == 1) ? kJJUnrollFine : kJJUnroll;
          // j-vector jj of this group: a shared-memory broadcast, or (measured alternative) one
          // vector per lane held in registers and broadcast by three shuffles
#if ACF_J_SHUFFLE
          const float4 vl = tile[jbeg + lane];
          auto jvec = [&](int jj) -> float4 {
            const int src = jj - jbeg;
            return make_float4(__shfl_sync(0xffffffffu, vl.x, src), __shfl_sync(0xffffffffu, vl.y, src),
                               __shfl_sync(0xffffffffu, vl.z, src), 0.0f);
          };
#else
          auto jvec = [&](int jj) -> float4 { return tile[jj]; };
#endif
          auto code_of = [&](int k, float4 v) -> uint32_t {
            return __float_as_uint(
                X == 2   ? pair_code_mid<F>(xi[k], yi[k], zi[k], v.x, v.y, v.z, p.bp)
                : X == 3 ? pair_code_fixed<MAP, F, true>(xi[k], yi[k], zi[k], v.x, v.y, v.z, ns, iws, h, p.bp)
                : X == 1 ? pair_code_fixed<MAP, F>(xi[k], yi[k], zi[k], v.x, v.y, v.z, ns, iws, h, p.bp)
                         : pair_code<MAP, METHOD, F>(xi[k], yi[k], zi[k], v.x, v.y, v.z, p.bp));
          };
          // this form's fine shift, and the histogram base of its fine code (single-code loops)
          const int SF = X == 2 ? p.bp.fine_shift_mid : (X == 3 ? p.bp.fine_shift_small : p.bp.fine_shift);
          const uint32_t bf = X == 2 ? base_fm : base_f;
          const uint32_t fmask = (1u << SF) - 1u;
          if constexpr (!F && U > 1 && kJJBatch > 1) {
            // plain loops: load kJJBatch j-vectors, then every code, then every atomic
            constexpr int B = kJJBatch;
#pragma unroll 1
            for (int jj = jbeg; jj < jbeg + 32; jj += B) {
              float4 vv[B];
#pragma unroll
              for (int u = 0; u < B; ++u) vv[u] = jvec(jj + u);
              uint32_t cb[B * K];
#pragma unroll
              for (int u = 0; u < B; ++u)
#pragma unroll
                for (int k = 0; k < K; ++k) cb[u * K + k] = code_of(k, vv[u]);
#pragma unroll
              for (int u = 0; u < B; ++u)
#pragma unroll
                for (int k = 0; k < K; ++k)
                  add_pair<false, MAP>(p, cb[u * K + k], base, bf, SHIFT, SF, magic_bits, i0 + islot<K>(k, lane), j0 + jj + u,
                                  xi[k], yi[k], zi[k], vv[u], inc);
            }
          } else if constexpr (F && (X == 1 || X == 3)) {
            // fixed-sign chord with flags: the plain code addresses the histogram (as without flags),
            // the fine code, from the same theta', only decides the flag
            [[maybe_unused]] uint32_t fw[K] = {};  // group records: this lane's flag words over the group
            [[maybe_unused]] uint32_t jbit = 1u;
#pragma unroll kJJUnrollFine2
            for (int jj = jbeg; jj < jbeg + 32; ++jj) {
              const float4 v = jvec(jj);
              uint32_t cfs[K], ccs[K];
              [[maybe_unused]] uint32_t low = 0xFFFFFFFFu;
              [[maybe_unused]] bool fl = false;
#pragma unroll
              for (int k = 0; k < K; ++k) {
                cfs[k] = __float_as_uint(pair_code_fixed2<MAP, X == 3>(xi[k], yi[k], zi[k], v.x, v.y, v.z, ns, iws, h,
                                                                        iws_c, h_c, p.bp, ccs[k]));
                add_pair<false, MAP>(p, ccs[k], base, bf, SHIFT, SF, magic_bits, i0 + islot<K>(k, lane), j0 + jj, xi[k], yi[k],
                                zi[k], v, inc);
                if constexpr (LAYOUT == kBlockExact) {
                  fw[k] |= (cfs[k] & (fmask & ~1u)) == 0u ? jbit : 0u;
                } else {
#if ACF_FLAG_PRED
                  fl |= (cfs[k] & (fmask & ~1u)) == 0u;
#else
                  low = min(low, cfs[k] & fmask);
#endif
                }
              }
              if constexpr (LAYOUT == kBlockExact) {
                jbit <<= 1;
              } else if (__any_sync(0xffffffffu, ACF_FLAG_PRED ? fl : low <= 1u)) {
                // the count went to the plain code's entry: nothing to move back without a record
                (void)push_record(p, region, cur, r, j0 + jj, pc, __ballot_sync(0xffffffffu, (cfs[0] & fmask) <= 1u),
                                  __ballot_sync(0xffffffffu, (cfs[1] & fmask) <= 1u),
                                  __ballot_sync(0xffffffffu, (cfs[2] & fmask) <= 1u),
                                  __ballot_sync(0xffffffffu, (cfs[3] & fmask) <= 1u));
              }
            }
            if constexpr (LAYOUT == kBlockExact) group_flush(fw, jbeg / 32, pc);
          } else {
            [[maybe_unused]] uint32_t fw[K] = {};  // group records (F): this lane's flag words over the group
            [[maybe_unused]] uint32_t jbit = 1u;
#pragma unroll U
            for (int jj = jbeg; jj < jbeg + 32; ++jj) {
              const float4 v = jvec(jj);
              uint32_t cbs[K];
              [[maybe_unused]] uint32_t low = 0xFFFFFFFFu;  // exact mode: smallest biased fraction of this j's pairs
              [[maybe_unused]] bool fl = false;
#pragma unroll
              for (int k = 0; k < K; ++k) {
                cbs[k] = code_of(k, v);
                add_pair<F, MAP>(p, cbs[k], base, bf, SHIFT, SF, magic_bits, i0 + islot<K>(k, lane), j0 + jj, xi[k], yi[k], zi[k],
                            v, inc);
                if constexpr (F && LAYOUT == kBlockExact) {
                  fw[k] |= (cbs[k] & (fmask & ~1u)) == 0u ? jbit : 0u;
                } else {
#if ACF_FLAG_PRED
                  if (F) fl |= (cbs[k] & (fmask & ~1u)) == 0u;
#else
                  if (F) low = min(low, cbs[k] & fmask);
#endif
                }
              }
              if constexpr (F && LAYOUT == kBlockExact) {
                jbit <<= 1;
              } else if (F && __any_sync(0xffffffffu, ACF_FLAG_PRED ? fl : low <= 1u)) {
                // near-edge pairs are rare: one warp vote per j, then the queue for the lanes that need it
                if (!push_record(p, region, cur, r, j0 + jj, pc, __ballot_sync(0xffffffffu, (cbs[0] & fmask) <= 1u),
                                 __ballot_sync(0xffffffffu, (cbs[1] & fmask) <= 1u),
                                 __ballot_sync(0xffffffffu, (cbs[2] & fmask) <= 1u),
                                 __ballot_sync(0xffffffffu, (cbs[3] & fmask) <= 1u))) {
#pragma unroll
                  for (int k = 0; k < K; ++k) carry_back(cbs[k], SF, bf, SHIFT, inc);
                }
              }
            }
            if constexpr (F && LAYOUT == kBlockExact) group_flush(fw, jbeg / 32, pc);
          }
        };
        // the four j-groups' paths, one per lane of lanes 0..3 (one pass of the decision per unit)
        int pc_lane = kGeneral;
        if (METHOD == kChordPoly && lane < kJT / 32)
          pc_lane = choose_path(s_icap[warp], __ldg(p.jcap32 + c * (kJT / 32) + lane), p.exact_mode, p.exact_lo,
                                MAP == kDirect ? p.bp.mid : 0, p.bp.small);
#pragma unroll 1
        for (int g = GROUPS == 1 ? gs : 0; g < (GROUPS == 1 ? gs + 1 : kJT / 32); ++g) {
          const int pc = __shfl_sync(0xffffffffu, pc_lane, g);
          const int path = pc & 3;
          const bool fine = LAYOUT == kBlockExact || (pc & kExactBit) != 0;
          if (pc & kMidBit) {
            count_path(fine ? 6 : 5, 1u);
            if (LAYOUT == kBlockExact || fine) run(FormTag<2>(), FineTag<true>(), g * 32, pc, 0.f, 0.f, 0.f, 0.f, 0.f);
            else run(FormTag<2>(), FineTag<false>(), g * 32, pc, 0.f, 0.f, 0.f, 0.f, 0.f);
            continue;
          }
          const ChordConsts cc = chord_consts<MAP>(pc, fine, p.bp);
          const float ns = cc.ns, iws = cc.iws, h = cc.h, iws_c = cc.iws_c, h_c = cc.h_c;
          if (pc & kSmallBit) {
            count_path(fine ? 8 : 7, 1u);
            if (LAYOUT == kBlockExact || fine) run(FormTag<3>(), FineTag<true>(), g * 32, pc, ns, iws, h, iws_c, h_c);
            else run(FormTag<3>(), FineTag<false>(), g * 32, pc, ns, iws, h, iws_c, h_c);
            continue;
          }
          count_path(path == kGeneral ? (fine ? 3 : 1) : (fine ? 2 : 0), 1u);
          if (path == kGeneral) {
            if (LAYOUT == kBlockExact || fine) run(FormTag<0>(), FineTag<true>(), g * 32, pc, ns, iws, h, iws_c, h_c);
            else run(FormTag<0>(), FineTag<false>(), g * 32, pc, ns, iws, h, iws_c, h_c);
          } else {
            if (LAYOUT == kBlockExact || fine) run(FormTag<1>(), FineTag<true>(), g * 32, pc, ns, iws, h, iws_c, h_c);
            else run(FormTag<1>(), FineTag<false>(), g * 32, pc, ns, iws, h, iws_c, h_c);
          }
        }
      } else {
        // pair (i, j) counts iff jj > thr[k]: thr = -1 for every j, a diagonal offset when only
        // j > i counts (DD/RR), INT_MAX for an i beyond the catalog
        int thr[K];
#pragma unroll
        for (int k = 0; k < K; ++k) {
          const int i = i0 + islot<K>(k, lane);
          const int tt = p.sym ? i - j0 : -1;
          thr[k] = (i >= ni) ? 0x7fffffff : max(-1, min(tt, kJT));
        }
        // (flagged pairs are recorded with the general chord's path code, kGeneral: the form this loop uses)
        auto edge = [&](auto fine) {
          constexpr bool F = decltype(fine)::value;
#pragma unroll 1
          for (int jj = GROUPS == 1 ? gs * 32 : 0; jj < (GROUPS == 1 ? min(jn, gs * 32 + 32) : jn); ++jj) {
            const float4 v = tile[jj];
            uint32_t cbs[K];
            bool fk[K];
#pragma unroll
            for (int k = 0; k < K; ++k) {
              cbs[k] = __float_as_uint(pair_code<MAP, METHOD, F>(xi[k], yi[k], zi[k], v.x, v.y, v.z, p.bp));
              fk[k] = jj > thr[k] &&
                      add_pair<F, MAP>(p, cbs[k], base, base_f, SHIFT, p.bp.fine_shift, magic_bits, i0 + islot<K>(k, lane),
                                       j0 + jj, xi[k], yi[k], zi[k], v, inc);
            }
            if (F && __any_sync(0xffffffffu, fk[0] || fk[1] || fk[2] || fk[3])) {
              if (!push_record(p, region, cur, r, j0 + jj, kGeneral, __ballot_sync(0xffffffffu, fk[0]),
                               __ballot_sync(0xffffffffu, fk[1]), __ballot_sync(0xffffffffu, fk[2]),
                               __ballot_sync(0xffffffffu, fk[3]))) {
#pragma unroll
                for (int k = 0; k < K; ++k)
                  if (fk[k]) carry_back(cbs[k], p.bp.fine_shift, base_f, SHIFT, inc);
              }
            }
          }
        };
        if constexpr (LAYOUT == kBlockExact) {
          // the same with group records: every group of the unit is flushed, the empty ones too
#pragma unroll 1
          for (int g = 0; g < kJT / 32; ++g) {
            uint32_t fw[K] = {};
#pragma unroll 1
            for (int jj = g * 32; jj < min(jn, g * 32 + 32); ++jj) {
              const float4 v = tile[jj];
#pragma unroll
              for (int k = 0; k < K; ++k) {
                const uint32_t cb = __float_as_uint(pair_code<MAP, METHOD, true>(xi[k], yi[k], zi[k], v.x, v.y, v.z, p.bp));
                if (jj > thr[k] && add_pair<true, MAP>(p, cb, base, base_f, SHIFT, p.bp.fine_shift, magic_bits,
                                                       i0 + islot<K>(k, lane), j0 + jj, xi[k], yi[k], zi[k], v, inc))
                  fw[k] |= 1u << (jj - g * 32);
              }
            }
            group_flush(fw, g, kGeneral);
          }
        } else if (p.exact_mode && METHOD == kChordPoly) {
          edge(FineTag<true>());
        } else {
          edge(FineTag<false>());
        }
        count_path(4, GROUPS == 1 ? (unsigned int)max(0, min(jn, gs * 32 + 32) - gs * 32) : (unsigned int)jn);
      }
      __syncwarp();  // every lane is done with this buffer before the next prefetch refills it
      if (un >= p.unit_end) break;
      u = un;
      r = rn;
      c = cn;
      gs = gsn;
      un = p.unit_begin + __shfl_sync(0xffffffffu, ta, 0);
      buf ^= 1;
    }
    cp_async_wait<0>();
    if (lane == 0) {
      constexpr unsigned long long G = 32 * kJT;
#pragma unroll 1
      for (int k = 0; k < 9; ++k) {
        const unsigned long long n = (unsigned long long)s_paths[warp][k] * (k == 4 ? (unsigned long long)kJT : G);
        if (n) atomicAdd(p.path_pairs + k, n);
      }
    }
  }
  // the records of this warp's own region (the fix-up reads that many)
  if (LAYOUT != kBlockExact && p.exact_mode && lane == 0) p.qused[region] = min(cur, p.qbatch);
  __syncthreads();
  flush_hist<K, THREADS, LAYOUT, MAP, METHOD>(p, hist, false);
}

// ------------------------------------------------------------------ merge, omega, diagnostics

// out[k] = sum over blocks of partial[b][k]; auto-correlations add the n self-pairs to bin 0.
// A block owns 32 consecutive bins (one per lane, coalesced reads); its 8 warps split the rows
// and combine their sums in shared memory.
constexpr int kMergeWarps = 8;
__global__ void __launch_bounds__(32 * kMergeWarps) merge_kernel(const unsigned long long* __restrict__ partial,
                                                                int rows, int nbins, unsigned long long self_pairs,
                                                                const unsigned long long* __restrict__ delta,
                                                                unsigned long long* __restrict__ out) {
  __shared__ unsigned long long acc[kMergeWarps][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int k = blockIdx.x * 32 + lane;
  unsigned long long s = 0ull;
  if (k < nbins) {
#pragma unroll 4
    for (int r = warp; r < rows; r += kMergeWarps) s += partial[(size_t)r * nbins + k];
  }
  acc[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && k < nbins) {
    unsigned long long t = (k == 0) ? self_pairs : 0ull;
    if (delta) t += delta[k];  // exact mode: counts moved by the exact re-decision (two's complement)
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) t += acc[w][lane];
    out[k] = t;
  }
}

__global__ void omega_kernel(const unsigned long long* __restrict__ dd, const unsigned long long* __restrict__ dr,
                             const unsigned long long* __restrict__ rr, int nbins, double f_dd, double f_dr,
                             double* __restrict__ omega) {
  for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < nbins; k += gridDim.x * blockDim.x) {
    const unsigned long long r = rr[k];
    if (r == 0ull) {
      omega[k] = __longlong_as_double(0x7ff8000000000000ll);  // NaN
    } else {
      const double num = (double)dd[k] * f_dd - 2.0 * (double)dr[k] * f_dr + (double)r;
      omega[k] = num / (double)r;
    }
  }
}

// Edge thresholds of the exact re-decision, in fp64: bin k starts where the difference chord
// reaches T[k] = 4 sin^2(k w / 2), or, for pairs past 90 degrees, where the sum chord falls to
// U[k] = 4 cos^2(k w / 2). The re-decision of a pair counted in bin k takes the difference chord
// while the fp32 rounding of T[k] is at most 2; T rises with k up to kmax (k w <= 180 degrees), so
// those bins are 0 .. kd, and kd is written too.
__global__ void edge_table_kernel(double w_rad, int nbins, int kmax, double* __restrict__ T, double* __restrict__ U,
                                  float2* __restrict__ Tds, float2* __restrict__ Uds, int* __restrict__ kd) {
  for (int k = blockIdx.x * blockDim.x + threadIdx.x; k <= nbins; k += gridDim.x * blockDim.x) {
    double sh, ch;
    sincos(0.5 * w_rad * k, &sh, &ch);
    const double t = 4.0 * sh * sh, u = 4.0 * ch * ch;
    T[k] = t;
    U[k] = u;
    // double-single copies: hi = fp32 rounding, lo = fp32 rounding of the rest
    const float th = (float)t, uh = (float)u;
    Tds[k] = make_float2(th, (float)(t - (double)th));
    Uds[k] = make_float2(uh, (float)(u - (double)uh));
    if (k <= kmax && th <= 2.0f) {
      bool last = k == kmax;
      if (!last) {
        double sh1, ch1;
        sincos(0.5 * w_rad * (k + 1), &sh1, &ch1);  // T[k + 1], as the thread of k + 1 computes it
        last = (float)(4.0 * sh1 * sh1) > 2.0f;
      }
      if (last) *kd = k;
    }
  }
}

// ------------------------------------------------------------------ exact re-decision

// Knuth's TwoSum: s + t == a + b exactly (round-to-nearest; the _rn intrinsics keep the compiler from
// contracting or reordering these operations).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& t) {
  s = __fadd_rn(a, b);
  const float bv = __fsub_rn(s, a);
  const float av = __fsub_rn(s, bv);
  t = __fadd_rn(__fsub_rn(a, av), __fsub_rn(b, bv));
}

// The dot product of two double-single unit vectors (hi + lo), returned as dh + dl. Error against
// the dot product of the fp64 vectors that hi + lo round (|a|, |b| = 1):
//  - representation: |hi + lo - x| <= 2^-48 |x| per component, so <= 2^-47 on the dot product;
//  - products: hi hi' as the fp32 product plus its exact fma remainder; the three cross terms (and
//    lo lo') added to that remainder by fma, each rounding <= 2^-24 of a remainder below 3 2^-24 of
//    the component's product: <= 9 2^-48 over the three components; the remainders' two fp32 sums
//    <= 6 2^-48;
//  - the sum: two exact TwoSums, then two fp32 adds of their remainders and the products'
//    (below 8 2^-24 in all): <= 13 2^-48; the final TwoSum is exact.
// In all <= 30 2^-48 = 1.07e-13.
constexpr float kDotErr = 1.07e-13f;
__device__ __forceinline__ void ds_dot(float4 ah, float4 al, float4 bh, float4 bl, float& dh, float& dl) {
  const float a_h[3] = {ah.x, ah.y, ah.z}, a_l[3] = {al.x, al.y, al.z};
  const float b_h[3] = {bh.x, bh.y, bh.z}, b_l[3] = {bl.x, bl.y, bl.z};
  float p[3], r = 0.0f;
#pragma unroll
  for (int c = 0; c < 3; ++c) {
    p[c] = __fmul_rn(a_h[c], b_h[c]);
    float e = __fmaf_rn(a_h[c], b_h[c], -p[c]);  // exact
    e = __fmaf_rn(a_h[c], b_l[c], e);
    e = __fmaf_rn(a_l[c], b_h[c], e);
    e = __fmaf_rn(a_l[c], b_l[c], e);
    r = c == 0 ? e : __fadd_rn(r, e);
  }
  float s1, t1, s2, t2;
  two_sum(p[0], p[1], s1, t1);
  two_sum(s1, p[2], s2, t2);
  two_sum(s2, __fadd_rn(r, __fadd_rn(t1, t2)), dh, dl);
}

// The chord q = |a + sg b|^2 = 2 + 2 sg (a.b) of two unit vectors (sg = -1: the difference chord,
// +1: the sum chord) from their double-single dot product, as qh + ql. 2 + 2 sg dh is split exactly
// by TwoSum; the one rounding of its remainder plus 2 sg dl is below 2^-24 of 6 2^-24. With the dot
// product's error: |q - exact| <= 2 kDotErr + 2.2e-14.
__device__ __forceinline__ void ds_chord_from_dot(float dh, float dl, float sg, float& qh, float& ql) {
  float t;
  two_sum(2.0f, 2.0f * sg * dh, qh, t);
  ql = __fadd_rn(t, 2.0f * sg * dl);
}

// Side of q = qh + ql against a double-single table value: +1 above, -1 below, 0 within eps (then
// only the fp64 re-decision can tell). qh - th is exact when the two are within a factor of 2.
__device__ __forceinline__ int ds_side(float qh, float ql, float2 t, float eps) {
  const float d = __fadd_rn(__fsub_rn(qh, t.x), __fsub_rn(ql, t.y));
  return d > eps ? 1 : (d < -eps ? -1 : 0);
}

// The codes a pair-kernel loop computed for a recorded pair (a = its i-vector, b = its j-vector, fp32
// as the kernel read them), from the record's path code: the fine code cb with its S fractional bits,
// the entry e_cnt its count went to, and whether the loop was a single-code one (whose entry is the
// fine code's integer part, which the one-unit bias may have carried one entry up). The same device
// functions as the loops, with the same constants, so every value is bit for bit the kernel's.
template <int MAP>
__device__ __forceinline__ void recorded_codes(int pc, float4 a, float4 b, const BinParams& bp, uint32_t& cb,
                                               uint32_t& e_cnt, bool& single, int& S) {
  const uint32_t magic_bits = __float_as_uint(kMagic);
  if (pc & kMidBit) {
    cb = __float_as_uint(pair_code_mid<true>(a.x, a.y, a.z, b.x, b.y, b.z, bp));
    S = bp.fine_shift_mid;
    e_cnt = (cb - magic_bits) >> S;
    single = true;
  } else if ((pc & 3) == kGeneral) {
    cb = __float_as_uint(pair_code<MAP, kChordPoly, true>(a.x, a.y, a.z, b.x, b.y, b.z, bp));
    S = bp.fine_shift;
    e_cnt = (cb - magic_bits) >> S;
    single = true;
  } else {
    const ChordConsts c = chord_consts<MAP>(pc, true, bp);
    uint32_t coarse;
    if (pc & kSmallBit) {
      cb = __float_as_uint(
          pair_code_fixed2<MAP, true>(a.x, a.y, a.z, b.x, b.y, b.z, c.ns, c.iws, c.h, c.iws_c, c.h_c, bp, coarse));
      S = bp.fine_shift_small;
    } else {
      cb = __float_as_uint(
          pair_code_fixed2<MAP, false>(a.x, a.y, a.z, b.x, b.y, b.z, c.ns, c.iws, c.h, c.iws_c, c.h_c, bp, coarse));
      S = bp.fine_shift;
    }
    e_cnt = coarse - magic_bits;
    single = false;
  }
}

struct FixupParams {
  const uint2* qhdr;                  // flag records (see push_record)
  const uint4* qmask;
  const unsigned int* qused;          // per pair-kernel warp: records of its region
  const unsigned int* qspill;         // spill records handed out
  unsigned int regions;               // pair-kernel warps (regions)
  unsigned int qbatch, qcap;          // records per region, records in all
  const DsVec *ds_i, *ds_j;           // double-single vectors (hi: the fp32 vectors the pair kernel read)
  const double4_32a *vi, *vj;         // fp64 vectors
  const double *T, *U;                // fp64 edge tables
  const float2 *Tds, *Uds;            // the same as double-single pairs
  const int* kd;                      // the last bin whose lower edge the difference chord decides
  // group records (GROUPED): the pair kernel's ballots and records, groups in all, batch dispenser
  const unsigned int* gbal;
  const GroupRecord* grec;
  unsigned long long ngroups;
  unsigned int* gticket;
  BinParams bp;
  unsigned int inc;                   // histogram increment of the pair kernel's launch
  unsigned long long* delta;          // per-bin moves (two's complement)
  unsigned int* moved;                // pairs moved
  unsigned int* redone;               // pairs decided again in fp64
  unsigned int* flagged;              // pairs re-decided (flagged and recorded)
};

// Re-decide every flagged pair of the records a pair-kernel launch wrote, exactly, and record the
// move of its count if the fast code put it in a neighbouring bin. Runs after every pair-kernel
// launch (the queue then starts empty again); the merge adds delta[] to the counts.
// The decision is the fp64 one: the chord q of the fp64 unit vectors against the fp64 edge tables
// T[k] = 4 sin^2(k w / 2) (bins whose lower edge is up to 90 degrees, difference chord) or
// U[k] = 4 cos^2(k w / 2) (the others, sum chord), each exact enough where the other loses relative
// precision. A double-single pass (fp32 hi + lo, about 48 bits) takes it first: where it lies farther
// than its error bound from a table value it decides as the fp64 comparison would; within that bound
// (about 1e-13 relative, against a flagged pair's 1e-6 rad window) the pair is redone in fp64.
// Pairs outside the exact zone (mode 1) keep their fp32 bin; a single-code loop's count that the bias
// carried one entry up moves back.
// Per-j records (GROUPED 0): the queue holds one region of qbatch records per pair-kernel warp
// (region g: qused[g] in use), then spill records. Fix-up warp g takes region g, whose records came
// from one pair-kernel warp in order (consecutive records share an i-set, and mostly a path code),
// and a share of the spill records. Group records (GROUPED > 0): warps take batches of GROUPED groups
// from a ticket.
// SMEM 2: the double-single tables and per-bin moves in shared memory; 1: the moves only; 0: neither.
// Shared moves reach delta[] once per block.
constexpr int kFixupThreads = 256;
// Fix-up: pairs a lane decides per round (their vector loads all in flight together): 2 measured
// 0.54 against 0.63 ms per fine-binning fix-up launch (19 against 16 threads per instruction); with
// group records 3 and 4 spill and are slower (fine-binning steps 70.6 and 76.3 against 65.2 ms, and
// 67.2 / 74.9 ms with 3 blocks per SM)
#ifndef ACF_FIXUP_PAIRS
#define ACF_FIXUP_PAIRS 2
#endif
constexpr int kFixupPairs = ACF_FIXUP_PAIRS;
// Fix-up of group records: groups per ticket where nearly every lane holds a record (a batch ends
// with the warp's last record of it, so smaller batches shorten the launch's tail; measured on fine
// bins: 4 and 16 groups slower than 8); where records are sparse, batches of 32 groups (so that warps
// do not spend their time taking tickets for nearly empty batches)
#ifndef ACF_FIXUP_BATCH
#define ACF_FIXUP_BATCH 8
#endif
constexpr int kFixupBatch = ACF_FIXUP_BATCH;
template <int MAP, int SMEM, int GROUPED>
__global__ void __launch_bounds__(kFixupThreads, ACF_FIXUP_MINB) fixup_kernel(const FixupParams f) {
  constexpr int WARPS = kFixupThreads / 32;
  extern __shared__ __align__(16) unsigned char fsm[];
  __shared__ unsigned int s_moved, s_redone, s_flagged;
  __shared__ uint4 s_list[WARPS][32 * kFixupPairs];  // per warp: (i, j, path code, 0) of the pairs of one round
  const BinParams& bp = f.bp;
  const int nb = bp.nbins;
  const float2* tT = f.Tds;
  const float2* tU = f.Uds;
  const int kd = *f.kd;
  int* sd = nullptr;
  if (SMEM >= 1) {
    sd = reinterpret_cast<int*>(fsm);
    for (int k = threadIdx.x; k < nb; k += blockDim.x) sd[k] = 0;
  }
  if (SMEM == 2) {
    float2* sT = reinterpret_cast<float2*>(fsm + (((size_t)nb * 4 + 15) & ~(size_t)15));
    float2* sU = sT + (nb + 1);
    for (int k = threadIdx.x; k <= nb; k += blockDim.x) {
      sT[k] = f.Tds[k];
      sU[k] = f.Uds[k];
    }
    tT = sT;
    tU = sU;
  }
  if (threadIdx.x == 0) s_moved = s_redone = s_flagged = 0u;
  __syncthreads();
  unsigned int my_moved = 0u, my_redone = 0u, my_flagged = 0u;
  // move one count between bins (k_from -> k_to)
  auto move = [&](int k_from, int k_to) {
    if (k_from == k_to) return;
    if (SMEM >= 1) {
      atomicAdd(sd + k_from, -(int)f.inc);
      atomicAdd(sd + k_to, (int)f.inc);
    } else {
      atomicAdd(f.delta + k_from, (unsigned long long)(-(long long)f.inc));
      atomicAdd(f.delta + k_to, (unsigned long long)f.inc);
    }
    ++my_moved;
  };
  // The bin of a flagged pair (i, j) whose count went to bin kf, from the double-single dot product
  // of its vectors (dh + dl): k0 = kf (at most kmax) and the walk across the edges the pair lies
  // beyond, starting from the table values at k0 and k0 + 1 (loaded before, together with the other
  // pairs' of the round). The difference chord and T[] below 90 degrees (the side the table at k0
  // gives), the sum chord and U[] above; on both sides the pair lies below edge k when
  // sg (q - t_k) < 0 (sg = 1 with T, -1 with U: the sum chord falls as the separation grows).
  auto decide = [&](int i, int j, int k0, float dh, float dl, float2 e_lo, float2 e_hi) {
    const bool diff = k0 <= kd;
    const float2* tb = diff ? tT : tU;
    const int sg = diff ? 1 : -1;
    float qh, ql;
    ds_chord_from_dot(dh, dl, diff ? -1.0f : 1.0f, qh, ql);
    // the bound on q's error (2 kDotErr + 2.2e-14), plus the double-single tables' 2^-48 relative
    // (T, U <= 4), the fp64 computation's own rounding (<= 2.2e-15) and the rounding of the side
    // test's remainder difference (<= 2.9e-14): 2.8e-13, with some margin
    const float eps = 4e-13f;
    int k = k0;
    bool sure = true;
    int c = k > 0 ? sg * ds_side(qh, ql, e_lo, eps) : 1;
    if (c <= 0) {
      // below the lower edge (or too close to it to tell)
      if (c == 0) sure = false;
      else
        for (--k; k > 0 && (c = sg * ds_side(qh, ql, tb[k], eps)) <= 0; --k) if (!c) { sure = false; break; }
    } else if (k < bp.kmax) {
      c = sg * ds_side(qh, ql, e_hi, eps);
      if (c >= 0) {
        // at or above the upper edge
        if (c == 0) sure = false;
        else
          for (++k; k < bp.kmax && (c = sg * ds_side(qh, ql, tb[k + 1], eps)) >= 0; ++k) if (!c) { sure = false; break; }
      }
    }
    if (!sure) {
      // too close to an edge for the double-single bound: the same comparisons in fp64
      ++my_redone;
      const double4_32a a = f.vi[i], b = f.vj[j];
      k = k0;
      if (diff) {
        const double dx = a.x - b.x, dy = a.y - b.y, dz = a.z - b.z;
        const double q = dx * dx + dy * dy + dz * dz;
        while (k > 0 && q < f.T[k]) --k;
        while (k < bp.kmax && q >= f.T[k + 1]) ++k;
      } else {
        const double dx = a.x + b.x, dy = a.y + b.y, dz = a.z + b.z;
        const double q = dx * dx + dy * dy + dz * dz;
        while (k > 0 && q > f.U[k]) --k;
        while (k < bp.kmax && q <= f.U[k + 1]) ++k;
      }
    }
    return k;
  };
  // one flagged pair (i, j, path code pc of the group that computed it) and its vectors: the codes
  // the pair kernel computed; in the exact zone the pair is decided again (its first two edge values
  // load while the dot product is summed), outside it (mode 1) the fp32 bin stands, less the carry
  // of a single-code loop's bias
  auto pair = [&](int i, int j, int pc, float4 ah, float4 al, float4 bh, float4 bl) {
    ++my_flagged;
    uint32_t cb, en;
    bool single;
    int S;
    recorded_codes<MAP>(pc, ah, bh, bp, cb, en, single, S);
    const int ec = (int)en < 0 ? 0 : ((int)en >= bp.entries ? bp.entries - 1 : (int)en);
    const int kf = entry_to_bin<MAP>(ec, bp);
    if (en - bp.zone0 <= bp.span0 || en - bp.zone1 <= bp.span1) {
      const int k0 = kf > bp.kmax ? bp.kmax : kf;
      const float2* tb = k0 <= kd ? tT : tU;
      const float2 e_lo = tb[k0], e_hi = tb[k0 + 1];
      float dh, dl;
      ds_dot(ah, al, bh, bl, dh, dl);
      move(kf, decide(i, j, k0, dh, dl, e_lo, e_hi));
    } else if (single && (cb & ((1u << S) - 1u)) == 0u) {
      move(kf, entry_to_bin<MAP>(ec > 0 ? ec - 1 : 0, bp));
    }
  };
  // Each lane walks its own sequence of records, holding the flagged pairs of one record that are
  // still to do (the next record already loading; next(h, m) loads it as h = (i-set row, j, path
  // code) and m = the four flag words, or returns false). Per round the warp packs up to
  // 32 kFixupPairs of those pairs into its list (a warp scan of the lanes' counts gives each lane its
  // slots), and then every lane decides the pairs at slots lane, lane + 32, ..., their vectors all
  // loading before the first is decided: the lanes stay converged however the pairs spread over the
  // records. Pairs of the dot form fill the list from the front, the chord forms' from the back, so
  // that most 32-slot groups hold one form only (the two recompute their codes differently).
  // Bit b of flag word k: per-j records, the pair (i = kJT row + islot(k, b), j); group records, the
  // pair (i = kJT row + islot(k, lane), j + b) (the record of this lane of its group).
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint4* list = s_list[warp];
  auto rounds = [&](auto next) {
    uint4 hn = make_uint4(0u, 0u, 0u, 0u), h = hn, mn = hn;
    uint32_t m[4] = {0u, 0u, 0u, 0u};  // pairs of the current record still to do
    bool has_next = next(hn, mn);
    while (true) {
      if ((m[0] | m[1] | m[2] | m[3]) == 0u && has_next) {
        h = hn;
        m[0] = mn.x; m[1] = mn.y; m[2] = mn.z; m[3] = mn.w;
        has_next = next(hn, mn);
      }
      const unsigned int pc = h.z;
      const bool back = !(pc & kMidBit);
      const unsigned int cnt = __popc(m[0]) + __popc(m[1]) + __popc(m[2]) + __popc(m[3]);  // <= 128
      // dot-form counts in the low half, chord-form counts in the high half (totals <= 4096)
      const unsigned int own = back ? cnt << 16 : cnt;
      unsigned int incl = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned int tot = __shfl_sync(0xffffffffu, incl, 31);
      if (tot == 0u) break;  // a lane with a record left always has a pair to do
      constexpr unsigned int L = 32u * kFixupPairs;  // list length
      const unsigned int nfront = min(tot & 0xFFFFu, L), nback = min(tot >> 16, L - nfront);
      {
        const unsigned int ex = incl - own;
        unsigned int r = back ? ex >> 16 : ex & 0xFFFFu;  // this lane's first pair among its form's
        const unsigned int lim = back ? nback : nfront;
        const unsigned int row = h.x, jr = h.y;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          while (m[k] && r < lim) {
            const int b = __ffs(m[k]) - 1;
            m[k] &= m[k] - 1u;
            const unsigned int i = row * kJT + islot<kJT / 32>(k, GROUPED ? lane : b);
            list[back ? L - 1u - r : r] = make_uint4(i, GROUPED ? jr + b : jr, pc, 0u);
            ++r;
          }
        }
      }
      __syncwarp();
      uint4 e[kFixupPairs];
      float4 ah[kFixupPairs], al[kFixupPairs], bh[kFixupPairs], bl[kFixupPairs];
#pragma unroll
      for (int u = 0; u < kFixupPairs; ++u) {
        const unsigned int s = lane + 32u * u;
        const bool ok = s < nfront || s >= L - nback;
        e[u] = ok ? list[s] : make_uint4(0u, 0u, 0u, 0xFFFFFFFFu);
        if (ok) {
          load_ds(f.ds_i + e[u].x, ah[u], al[u]);
          load_ds(f.ds_j + e[u].y, bh[u], bl[u]);
        }
      }
      __syncwarp();
#pragma unroll
      for (int u = 0; u < kFixupPairs; ++u)
        if (e[u].w == 0u) pair((int)e[u].x, (int)e[u].y, (int)e[u].z, ah[u], al[u], bh[u], bl[u]);
    }
  };
  if constexpr (GROUPED != 0) {
    // batches of GROUPED groups from a ticket (the next ticket fetched while a batch is done);
    // in each, lane l takes the records of lane l of the groups whose ballot holds l
    unsigned int bt = 0u;
    if (lane == 0) bt = atomicAdd(f.gticket, 1u);
    bt = __shfl_sync(0xffffffffu, bt, 0);
    while (true) {
      const unsigned long long g0 = (unsigned long long)GROUPED * bt;
      if (g0 >= f.ngroups) break;
      unsigned int bn = 0u;
      if (lane == 0) bn = atomicAdd(f.gticket, 1u);
      const unsigned int bal = lane < GROUPED && g0 + lane < f.ngroups ? f.gbal[g0 + lane] : 0u;
      unsigned int mine = 0u;  // bit q: group g0 + q holds a record of this lane
#pragma unroll
      for (int q = 0; q < GROUPED; ++q) mine |= ((__shfl_sync(0xffffffffu, bal, q) >> lane) & 1u) << q;
      bt = __shfl_sync(0xffffffffu, bn, 0);
      rounds([&](uint4& hn, uint4& mn) {
        if (!mine) return false;
        const int q = __ffs(mine) - 1;
        mine &= mine - 1u;
        load_group_record(f.grec + (g0 + (unsigned)q) * 32 + lane, mn, hn);
        return true;
      });
    }
  } else {
    // this warp's region, then its share of the spill records
    const unsigned long long nbatch = (unsigned long long)f.regions * f.qbatch;
    const unsigned int nspill = nbatch < f.qcap ? (unsigned int)min((unsigned long long)*f.qspill, f.qcap - nbatch) : 0u;
    const unsigned int gw = blockIdx.x * WARPS + warp, nw = gridDim.x * WARPS;
    const unsigned int nmine = gw < f.regions ? min(f.qused[gw], f.qbatch) : 0u;
    auto records = [&](unsigned long long base, unsigned int n, unsigned int t, unsigned int stride) {
      rounds([&](uint4& hn, uint4& mn) {
        if (t >= n) return false;
        const uint2 q = f.qhdr[base + t];
        mn = f.qmask[base + t];
        hn = make_uint4(q.y & 0xFFFFFFu, q.x, q.y >> 24, 0u);
        t += stride;
        return true;
      });
    };
    records((unsigned long long)gw * f.qbatch, nmine, lane, 32);
    records(nbatch, nspill, gw * 32 + lane, nw * 32);
  }
  for (int o = 16; o > 0; o >>= 1) {
    my_moved += __shfl_xor_sync(0xffffffffu, my_moved, o);
    my_redone += __shfl_xor_sync(0xffffffffu, my_redone, o);
    my_flagged += __shfl_xor_sync(0xffffffffu, my_flagged, o);
  }
  if (lane == 0 && my_moved) atomicAdd(&s_moved, my_moved);
  if (lane == 0 && my_redone) atomicAdd(&s_redone, my_redone);
  if (lane == 0 && my_flagged) atomicAdd(&s_flagged, my_flagged);
  __syncthreads();
  if (threadIdx.x == 0 && s_moved) atomicAdd(f.moved, s_moved);
  if (threadIdx.x == 0 && s_redone) atomicAdd(f.redone, s_redone);
  if (threadIdx.x == 0 && s_flagged) atomicAdd(f.flagged, s_flagged);
  if (SMEM >= 1) {
    for (int k = threadIdx.x; k < nb; k += blockDim.x)
      if (sd[k]) atomicAdd(f.delta + k, (unsigned long long)(long long)sd[k]);
  }
}

// form 1: what a group the caps bound tightly computes: pairs with |u.v| < cos(55 deg) take the
// dot form, pairs with |u.v| > cos(72 deg) the short chord, the others the full-range chord form;
// form 0: the full-range chord form for every pair.
template <int MAP, int METHOD>
__global__ void pair_bins_kernel(const float* __restrict__ ra1, const float* __restrict__ dec1,
                                 const float* __restrict__ ra2, const float* __restrict__ dec2, long long n,
                                 BinParams bp, int form, int* __restrict__ bins) {
  const uint32_t magic_bits = __float_as_uint(kMagic);  // code = 2^23 + entry
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const float4 u = radec_to_unit(ra1[i], dec1[i]);
    const float4 v = radec_to_unit(ra2[i], dec2[i]);
    const float d = fmaf(u.z, v.z, fmaf(u.y, v.y, u.x * v.x));
    const bool mid = form == 1 && MAP == kDirect && METHOD == kChordPoly && bp.mid && fabsf(d) < 0.57357644f;
    const bool small = form == 1 && METHOD == kChordPoly && bp.small && fabsf(d) > 0.30901699f;  // cos 72 deg
    float code;
    if (mid) {
      code = pair_code_mid<false>(u.x, u.y, u.z, v.x, v.y, v.z, bp);
    } else if (small) {
      const bool near = !(__float_as_uint(d) >> 31);
      const float h = MAP == kDirect ? (near ? kMagic : bp.magic_far) : (near ? 0.0f : 3.14159265358979323846f * bp.inv_w);
      code = pair_code_fixed<MAP, false, true>(u.x, u.y, u.z, v.x, v.y, v.z, near ? -1.0f : 1.0f,
                                               near ? bp.inv_w : -bp.inv_w, h, bp);
    } else {
      code = pair_code<MAP, METHOD>(u.x, u.y, u.z, v.x, v.y, v.z, bp);
    }
    int e = (int)(__float_as_uint(code) - magic_bits);
    e = e < 0 ? 0 : (e >= bp.entries ? bp.entries - 1 : e);
    bins[i] = entry_to_bin<MAP>(e, bp);
  }
}

// ------------------------------------------------------------------ FP32 issue ceiling

// Independent FMA chains (kFmaChains per thread) for a runtime iteration count: the FP32 issue rate
// the hardware sustains, measured the way a roofline ceiling is (one instruction class, enough
// independent work to cover its latency). Every thread writes the sum of its chains so nothing is
// dead code; the host replays thread 0 to check the kernel really ran.
constexpr int kFmaChains = 8;
__global__ void __launch_bounds__(1024) fma_peak_kernel(float a, float b, long long iters, float* __restrict__ out) {
  float x[kFmaChains];
#pragma unroll
  for (int c = 0; c < kFmaChains; ++c) x[c] = (float)threadIdx.x * 1e-3f + (float)c;
#pragma unroll 16
  for (long long it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < kFmaChains; ++c) x[c] = fmaf(x[c], a, b);
  }
  float s = 0.0f;
#pragma unroll
  for (int c = 0; c < kFmaChains; ++c) s += x[c];
  out[blockIdx.x * (long long)blockDim.x + threadIdx.x] = s;
}

}  // namespace acf
