// Device code of the GB300 angular-correlation library (sm_103a, CUDA cores).
//
// The method is that of "CUDA Deep Dive: 10B Galaxy Pairs on an RTX 5080": bin the angular
// separation theta of every ordered pair of two galaxy catalogs (section "The problem"), using
// DD/RR symmetry (section "L1"), per-galaxy precomputation (section "L2"), a register i-tile
// against a shared-memory j-tile (section "L3") and whole-tile diagonal skipping (section "L5").
// What differs from the page, and why:
//   * each galaxy becomes an fp32 unit vector once (built in fp64), so a pair costs a dot product
//     instead of a cosine of the RA difference;
//   * the separation is taken from the CHORD, not from arccos of the dot product: with
//     s = sign(u.v), q = |u - s v|^2 = 4 sin^2(theta'/2), theta' = theta (s = +1) or
//     pi - theta (s = -1), theta' <= 90 deg. q keeps full relative precision at small and near-
//     antipodal separations, where arccos of an fp32 dot product loses up to ~3e-4 rad;
//   * theta'^2 / w^2 = q * P(q) with a degree-7 polynomial P (absolute theta' error <= 2.5e-8 rad),
//     one sqrt.approx gives t' = theta'/w, and the bin index comes from t' by exact float
//     rounding tricks instead of acos, multiply and float-to-int conversion;
//   * each histogram lives in shared memory as 32 lane-private copies (word = bin*32 + lane), so a
//     warp's 32 increments always hit 32 different banks and the shared-memory atomic unit
//     retires one warp instruction per clock; very fine binnings fall back to one block-shared
//     copy;
//   * persistent blocks walk a precomputed chunk list (only the upper triangle for DD/RR), and
//     per-block counts go to per-block uint64 rows that a final kernel reduces.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace acf {

constexpr int kJT = 128;  // j-galaxies per shared-memory chunk
#ifndef ACF_JJ_UNROLL
#define ACF_JJ_UNROLL 4
#endif
constexpr int kJJUnroll = ACF_JJ_UNROLL;
#ifndef ACF_ASM_LOP3
#define ACF_ASM_LOP3 1  // write the two sign-bit logic ops as explicit lop3 (2 ops, not 3)
#endif  // j-loop unroll of the full-chunk path
constexpr float kMagic = 8388608.0f;  // 2^23: adding it with round-toward-zero floors into the mantissa

enum Layout { kLane = 1, kBlock = 2 };
enum BinMap { kMirror = 0, kClamp = 1 };
enum Method { kChordPoly = 0, kDotAcos = 1 };

// theta'^2 = q * P(q) for a chord q = |u - v|^2 on [0, 2] (theta' <= 90 degrees), P of degree 7
// fitted by fit_arcsin2.py: absolute theta' error <= 1.8e-8 rad (2.5e-8 after fp32 rounding).
__device__ constexpr float kP0 = 0.99999959294652097f, kP1 = 0.083342611628085594f, kP2 = 0.011049794431887118f,
                           kP3 = 0.0019657095570993176f, kP4 = 4.2347086002697957e-05f,
                           kP5 = 0.00029099553526503564f, kP6 = -9.1427792701640403e-05f,
                           kP7 = 2.3068911858269848e-05f;

struct BinParams {
  float magic;     // 2^23 + off (mirror) or 2^23 (clamp)
  float clamp_c;   // largest index (clamp map)
  float inv_w;     // 1 / w in radians (acos method)
  int off;         // mirror: index of theta' = 0 on the near side
  int p_int;       // mirror: P as an integer
  int nbins;
  int entries;     // histogram entries in shared memory
};

struct PairParams {
  const float4* __restrict__ vi;
  const float4* __restrict__ vj;
  long long ni, nj;
  long long total_chunks;
  long long chunks_per_row;    // CJ = ceil(nj / kJT)
  long long rows;              // TI = ceil(ni / BI)
  int sym;                     // 1: pairs j > i of one catalog, counted twice
  int row_step;                // BI / kJT (sym rows start at ib * row_step)
  unsigned int inc;            // 2 (sym) or 1 (cross)
  unsigned int flush_every;    // chunks between flushes of the 32-bit shared counters
  unsigned long long* partial; // [gridDim.x][nbins]
  unsigned int* ticket;        // chunk dispenser; zero before the launch
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

__device__ __forceinline__ float add_rz(float a, float b) {
  float y;
  asm("add.rz.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
  return y;
}

// three-input logic op; lut is the truth table over (a=0xF0, b=0xCC, c=0xAA)
template <int LUT>
__device__ __forceinline__ uint32_t lop3(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t y;
  asm("lop3.b32 %0, %1, %2, %3, %4;" : "=r"(y) : "r"(a), "r"(b), "r"(c), "n"(LUT));
  return y;
}

// a * b + c with one rounding, toward zero
__device__ __forceinline__ float fma_rz(float a, float b, float c) {
  float y;
  asm("fma.rz.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

__device__ __forceinline__ void red_shared_add(uint32_t addr, uint32_t v) {
  asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
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

// Also zeroes the pair kernel's chunk dispenser, which the next pair launch on the stream uses.
__global__ void convert_kernel(const float* __restrict__ ra, const float* __restrict__ dec, long long n,
                               float4* __restrict__ v, unsigned int* __restrict__ ticket) {
  if (blockIdx.x == 0 && threadIdx.x == 0 && ticket) *ticket = 0u;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    v[i] = radec_to_unit(ra[i], dec[i]);
}

// ------------------------------------------------------------------ bin index of one pair

// The float 2^23 + (histogram entry), whose bit pattern is bits(2^23) + entry. Symmetric in (u, v) bit for bit:
// the products commute and u - s v = -(v - s u) rounds to the same magnitude.
template <int MAP, int METHOD>
__device__ __forceinline__ float pair_code(float xi, float yi, float zi, float xj, float yj, float zj,
                                           const BinParams& bp) {
  const float d = fmaf(zi, zj, fmaf(yi, yj, xi * xj));
  if (METHOD == kDotAcos) {
    // the page's route: arccos of the (clamped) cosine, scaled by 1/w and truncated
    const float t = acosf(fminf(fmaxf(d, -1.0f), 1.0f)) * bp.inv_w;
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
    if (MAP == kMirror) {
      // near side (s = +1): floor(theta'/w) exactly, by one fma rounded toward zero onto 2^23 + off;
      // far side: the same fma of -theta' gives off - ceil(theta'/w), and bin P - ceil(theta'/w)
      // is exactly floor((pi - theta')/w) when P = pi/w is an integer.
      // theta' carrying the sign of d: th | (d & signmask), one logic op
#if ACF_ASM_LOP3
      return fma_rz(__uint_as_float(lop3<0xF8>(__float_as_uint(th), db, 0x80000000u)), bp.inv_w, bp.magic);
#else
      return fma_rz(__uint_as_float(__float_as_uint(th) | (db & 0x80000000u)), bp.inv_w, bp.magic);
#endif
    } else {
      const float h = fmaf(ns, 1.57079632679489662f, 1.57079632679489662f);  // 0 or pi
      const float t = fmaf(-ns, th, h) * bp.inv_w;                             // theta / w
      return add_rz(fminf(t, bp.clamp_c), kMagic);
    }
  }
}

// histogram entry -> bin
template <int MAP>
__device__ __forceinline__ int entry_to_bin(int e, const BinParams& bp) {
  int k = e;
  if (MAP == kMirror) k = (e >= bp.off) ? e - bp.off : e + bp.p_int - bp.off;
  k = k < 0 ? 0 : k;
  return k > bp.nbins - 1 ? bp.nbins - 1 : k;
}

// ------------------------------------------------------------------ pair kernel

// Map chunk q to (row ib, chunk column jc). The host guarantees chunk counts below 2^32 and
// catalogs below 2^31 galaxies, so 32-bit indices suffice.
__device__ __forceinline__ void chunk_coords(const PairParams& p, unsigned int q, int& ib, int& jc) {
  const long long cj = p.chunks_per_row;
  if (!p.sym) {
    ib = (int)(q / (unsigned long long)cj);
    jc = (int)(q - (unsigned long long)ib * cj);
    return;
  }
  // row r starts at S(r) = r*CJ - R*r*(r-1)/2; largest r with S(r) <= q
  long long lo = 0, hi = p.rows - 1;
  while (lo < hi) {
    const long long mid = (lo + hi + 1) >> 1;
    const long long s = mid * cj - (long long)p.row_step * mid * (mid - 1) / 2;
    if (s <= (long long)q) lo = mid;
    else hi = mid - 1;
  }
  ib = (int)lo;
  jc = (int)(lo * p.row_step + ((long long)q - (lo * cj - (long long)p.row_step * lo * (lo - 1) / 2)));
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
  } else {
    for (int e = threadIdx.x; e < p.bp.entries; e += THREADS) {
      const unsigned long long v = hist[e];
      if (zero) hist[e] = 0;
      if (v && ACF_CHECK(entry_to_bin<MAP>(e, p.bp) < p.bp.nbins, 3, e, entry_to_bin<MAP>(e, p.bp)))
        atomicAdd(row + entry_to_bin<MAP>(e, p.bp), v);
    }
  }
}

// One chunk = the block's BI = THREADS*K i-galaxies (K per thread, in registers) against kJT
// j-galaxies (in shared memory). Chunks are handed out by an atomic ticket so that uneven chunk
// costs (ragged tails, diagonal chunks of DD/RR) spread over all blocks; the ticket two chunks
// ahead is fetched while the current chunk is computed.
template <int K, int THREADS, int LAYOUT, int MAP, int METHOD>
__global__ void __launch_bounds__(THREADS, 65536 / (THREADS * 64)) pair_kernel(const PairParams p) {
  constexpr int BI = THREADS * K;
  extern __shared__ __align__(16) unsigned char smem[];
  float4* tiles = reinterpret_cast<float4*>(smem);                    // [2][kJT]
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + 2 * kJT * sizeof(float4));
  __shared__ unsigned int s_ticket[2];
  const int tid = threadIdx.x, lane = tid & 31;

  // zero this block's histogram and its partial row
  const int words = (LAYOUT == kLane) ? p.bp.entries * 32 : p.bp.entries;
  for (int w = tid; w < words; w += THREADS) hist[w] = 0;
  unsigned long long* row = p.partial + (size_t)blockIdx.x * p.bp.nbins;
  for (int k = tid; k < p.bp.nbins; k += THREADS) row[k] = 0ull;
  if (tid == 0) {
    s_ticket[0] = atomicAdd(p.ticket, 1u);
    s_ticket[1] = atomicAdd(p.ticket, 1u);
  }

  const uint32_t hist_addr = (uint32_t)__cvta_generic_to_shared(hist);
  const uint32_t tiles_addr = (uint32_t)__cvta_generic_to_shared(tiles);
  // every code is the float 2^23 + entry (the mirror offset is already inside the code)
  const uint32_t magic_bits = __float_as_uint(kMagic);
  // address of entry e in this lane's copy = (code bits << shift) + base
  const uint32_t base = (LAYOUT == kLane) ? hist_addr + lane * 4u - (magic_bits << 7) : hist_addr - (magic_bits << 2);
  constexpr int SHIFT = (LAYOUT == kLane) ? 7 : 2;
  const unsigned long long C = (unsigned long long)p.total_chunks;

  __syncthreads();
  const unsigned int C32 = (unsigned int)C;
  unsigned int q = s_ticket[0], qn = s_ticket[1];
  if (q < C32) {
    const int ni = (int)p.ni, nj = (int)p.nj;
    int ib, jc;
    chunk_coords(p, q, ib, jc);
    {
      const int j0 = jc * kJT;
      const int jn = min(kJT, nj - j0);
      if (tid < jn) cp_async16(tiles_addr + tid * 16u, p.vj + j0 + tid);
    }
    cp_async_commit();
    float xi[K], yi[K], zi[K];
    int cur_ib = -1;
    unsigned int since_flush = 0;
    int it = 0;  // iteration count: tile buffer it & 1, ticket mailbox slot it & 1
    while (true) {
      const int buf = it & 1;
      const int i0 = ib * BI;
      if (ib != cur_ib) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
          int i = i0 + k * THREADS + tid;
          i = i < ni ? i : ni - 1;
          const float4 v = __ldg(p.vi + i);
          xi[k] = v.x;
          yi[k] = v.y;
          zi[k] = v.z;
          (void)ACF_CHECK(fabsf(v.x * v.x + v.y * v.y + v.z * v.z - 1.0f) < 1e-3f, 4, i, ib, v.x, v.y, v.z);
        }
        cur_ib = ib;
      }
      // One barrier per chunk: after it this chunk's tile is visible, every warp has finished the
      // previous chunk (so the other buffer may be refilled) and the ticket that thread 0 posted
      // in the previous iteration is readable.
      cp_async_wait<0>();
      __syncthreads();
      if (it > 0) qn = s_ticket[(it - 1) & 1];
      int nib = 0, njc = 0;
      if (qn < C32) {
        chunk_coords(p, qn, nib, njc);
        const int j0 = njc * kJT;
        const int jn = min(kJT, nj - j0);
        if (tid < jn) cp_async16(tiles_addr + (uint32_t)((buf ^ 1) * kJT + tid) * 16u, p.vj + j0 + tid);
      }
      cp_async_commit();
      unsigned int t_after = 0;
      if (tid == 0) t_after = atomicAdd(p.ticket, 1u);  // the chunk after qn; posted below

      const float4* tile = tiles + buf * kJT;
      const int j0 = jc * kJT;
      const int jn = min(kJT, nj - j0);
      const bool full = (jn == kJT) && (i0 + BI <= ni) && (!p.sym || j0 >= i0 + BI);
#ifdef ACF_DEBUG_BOUNDS
      for (int jj = 0; jj < jn; ++jj) {
        const float4 v = tile[jj];
        (void)ACF_CHECK(fabsf(v.x * v.x + v.y * v.y + v.z * v.z - 1.0f) < 1e-3f, 2, j0 + jj, q, v.x, v.y, v.z, (float)buf);
      }
#endif
      if (full) {
#pragma unroll kJJUnroll
        for (int jj = 0; jj < kJT; ++jj) {
          const float4 v = tile[jj];
#pragma unroll
          for (int k = 0; k < K; ++k) {
            const float code = pair_code<MAP, METHOD>(xi[k], yi[k], zi[k], v.x, v.y, v.z, p.bp);
            if (ACF_CHECK(__float_as_uint(code) - magic_bits < (uint32_t)p.bp.entries, 1,
                          (long long)(__float_as_uint(code) - magic_bits), i0 + k * THREADS + tid, code, xi[k], yi[k],
                          zi[k], v.x, v.y, v.z, (float)jj))
              red_shared_add((__float_as_uint(code) << SHIFT) + base, p.inc);
          }
        }
      } else {
        // pair (i, j) counts iff jj > thr[k]: thr = -1 for every j, a diagonal offset when only
        // j > i counts (DD/RR), INT_MAX for an i beyond the catalog
        int thr[K];
#pragma unroll
        for (int k = 0; k < K; ++k) {
          const int i = i0 + k * THREADS + tid;
          const int t = p.sym ? i - j0 : -1;
          thr[k] = (i >= ni) ? 0x7fffffff : max(-1, min(t, kJT));
        }
        for (int jj = 0; jj < jn; ++jj) {
          const float4 v = tile[jj];
#pragma unroll
          for (int k = 0; k < K; ++k) {
            const float code = pair_code<MAP, METHOD>(xi[k], yi[k], zi[k], v.x, v.y, v.z, p.bp);
            if (jj > thr[k] &&
                ACF_CHECK(__float_as_uint(code) - magic_bits < (uint32_t)p.bp.entries, 1,
                          (long long)(__float_as_uint(code) - magic_bits), i0 + k * THREADS + tid, code, xi[k], yi[k],
                          zi[k], v.x, v.y, v.z, (float)jj))
              red_shared_add((__float_as_uint(code) << SHIFT) + base, p.inc);
          }
        }
      }
      // Slot it&1 is next written two iterations later, after a barrier every thread passes only
      // once it has read this value, so one barrier per chunk is enough.
      if (tid == 0) s_ticket[it & 1] = t_after;
      if (++since_flush == p.flush_every) {
        __syncthreads();
        flush_hist<K, THREADS, LAYOUT, MAP, METHOD>(p, hist, true);
        __syncthreads();
        since_flush = 0;
      }
      if (qn >= C32) break;
      q = qn;
      ib = nib;
      jc = njc;
      ++it;
    }
    cp_async_wait<0>();
  }
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

template <int MAP, int METHOD>
__global__ void pair_bins_kernel(const float* __restrict__ ra1, const float* __restrict__ dec1,
                                 const float* __restrict__ ra2, const float* __restrict__ dec2, long long n,
                                 BinParams bp, int* __restrict__ bins) {
  const uint32_t magic_bits = __float_as_uint(kMagic);  // code = 2^23 + entry
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const float4 u = radec_to_unit(ra1[i], dec1[i]);
    const float4 v = radec_to_unit(ra2[i], dec2[i]);
    const float code = pair_code<MAP, METHOD>(u.x, u.y, u.z, v.x, v.y, v.z, bp);
    int e = (int)(__float_as_uint(code) - magic_bits);
    e = e < 0 ? 0 : (e >= bp.entries ? bp.entries - 1 : e);
    bins[i] = entry_to_bin<MAP>(e, bp);
  }
}

}  // namespace acf
