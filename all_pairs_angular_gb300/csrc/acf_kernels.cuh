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
constexpr float kMagic = 8388608.0f;  // 2^23: adding it with round-toward-zero floors into the mantissa

enum Layout { kLane = 1, kBlock = 2 };
enum BinMap { kMirror = 0, kClamp = 1 };
enum Method { kChordPoly = 0, kDotAcos = 1 };

struct BinParams {
  float c[8];      // coefficients of q * P(q) = (theta'/w)^2, lowest degree first
  float magic;     // 2^23 + off (mirror) or 2^23 (clamp)
  float half_p;    // P/2 with P = pi / w (clamp map)
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

__device__ __forceinline__ float sqrt_approx(float x) {
  float y;
  asm("sqrt.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float add_rz(float a, float b) {
  float y;
  asm("add.rz.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
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

__global__ void convert_kernel(const float* __restrict__ ra, const float* __restrict__ dec, long long n,
                               float4* __restrict__ v) {
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
    const uint32_t sbit = __float_as_uint(d) & 0x80000000u;
    const float s = __uint_as_float(sbit | 0x3f800000u);  // +1 or -1
    const float dx = fmaf(-s, xj, xi);
    const float dy = fmaf(-s, yj, yi);
    const float dz = fmaf(-s, zj, zi);
    // 1e-30 keeps t' > 0 for identical or exactly antipodal vectors (see the mirror map)
    const float q = fmaf(dz, dz, fmaf(dy, dy, fmaf(dx, dx, 1e-30f)));
    float p = bp.c[7];
    p = fmaf(p, q, bp.c[6]);
    p = fmaf(p, q, bp.c[5]);
    p = fmaf(p, q, bp.c[4]);
    p = fmaf(p, q, bp.c[3]);
    p = fmaf(p, q, bp.c[2]);
    p = fmaf(p, q, bp.c[1]);
    p = fmaf(p, q, bp.c[0]);
    const float tp = sqrt_approx(p * q);  // theta' / w
    if (MAP == kMirror) {
      // near side (s = +1): index off + floor(t'); far side: round-toward-zero of (2^23 + off - t')
      // gives off - ceil(t'), and bin P - ceil(t') is exactly floor(P - t') when P is an integer.
      return add_rz(__uint_as_float(__float_as_uint(tp) | sbit), bp.magic);
    } else {
      const float h = fmaf(s, -bp.half_p, bp.half_p);  // 0 or P
      const float t = fmaf(s, tp, h);                   // t' or P - t'
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

// Map chunk q to (row ib, chunk column jc).
__device__ __forceinline__ void chunk_coords(const PairParams& p, long long q, long long& ib, long long& jc) {
  if (!p.sym) {
    ib = q / p.chunks_per_row;
    jc = q - ib * p.chunks_per_row;
    return;
  }
  // row r starts at S(r) = r*CJ - R*r*(r-1)/2; largest r with S(r) <= q
  long long lo = 0, hi = p.rows - 1;
  while (lo < hi) {
    const long long mid = (lo + hi + 1) >> 1;
    const long long s = mid * p.chunks_per_row - (long long)p.row_step * mid * (mid - 1) / 2;
    if (s <= q) lo = mid;
    else hi = mid - 1;
  }
  ib = lo;
  jc = ib * p.row_step + (q - (ib * p.chunks_per_row - (long long)p.row_step * ib * (ib - 1) / 2));
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

template <int K, int THREADS, int LAYOUT, int MAP, int METHOD>
__global__ void __launch_bounds__(THREADS) pair_kernel(const PairParams p) {
  constexpr int BI = THREADS * K;
  extern __shared__ __align__(16) unsigned char smem[];
  float4* tiles = reinterpret_cast<float4*>(smem);                    // [2][kJT]
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + 2 * kJT * sizeof(float4));
  const int tid = threadIdx.x, lane = tid & 31;

  // zero this block's histogram and its partial row
  const int words = (LAYOUT == kLane) ? p.bp.entries * 32 : p.bp.entries;
  for (int w = tid; w < words; w += THREADS) hist[w] = 0;
  unsigned long long* row = p.partial + (size_t)blockIdx.x * p.bp.nbins;
  for (int k = tid; k < p.bp.nbins; k += THREADS) row[k] = 0ull;

  const uint32_t hist_addr = (uint32_t)__cvta_generic_to_shared(hist);
  const uint32_t tiles_addr = (uint32_t)__cvta_generic_to_shared(tiles);
  // every code is the float 2^23 + entry (the mirror offset is already inside the code)
  const uint32_t magic_bits = __float_as_uint(kMagic);
  // address of entry e in this lane's copy = (code bits << shift) + base
  const uint32_t base = (LAYOUT == kLane) ? hist_addr + lane * 4u - (magic_bits << 7) : hist_addr - (magic_bits << 2);
  constexpr int SHIFT = (LAYOUT == kLane) ? 7 : 2;

  const long long C = p.total_chunks, G = gridDim.x;
  const long long q0 = (long long)blockIdx.x * C / G, q1 = ((long long)blockIdx.x + 1) * C / G;

  __syncthreads();
  if (q0 < q1) {
    long long ib, jc;
    chunk_coords(p, q0, ib, jc);
    // first j-chunk
    {
      const long long j0 = jc * kJT;
      const long long jn = min((long long)kJT, p.nj - j0);
      if (tid < jn) cp_async16(tiles_addr + tid * 16u, p.vj + j0 + tid);
      cp_async_commit();
    }
    float xi[K], yi[K], zi[K];
    long long cur_ib = -1;
    unsigned int since_flush = 0;
    for (long long q = q0; q < q1; ++q) {
      const int buf = (int)((q - q0) & 1);
      // prefetch the next chunk into the other buffer
      long long nib = ib, njc = jc + 1;
      if (njc == p.chunks_per_row) {
        nib = ib + 1;
        njc = p.sym ? nib * p.row_step : 0;
      }
      if (q + 1 < q1) {
        const long long j0 = njc * kJT;
        const long long jn = min((long long)kJT, p.nj - j0);
        if (tid < jn) cp_async16(tiles_addr + (uint32_t)((buf ^ 1) * kJT + tid) * 16u, p.vj + j0 + tid);
      }
      cp_async_commit();
      // i-vectors of this row
      const long long i0 = ib * BI;
      if (ib != cur_ib) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
          long long i = i0 + k * THREADS + tid;
          i = i < p.ni ? i : p.ni - 1;
          const float4 v = __ldg(p.vi + i);
          xi[k] = v.x;
          yi[k] = v.y;
          zi[k] = v.z;
          ACF_CHECK(fabsf(v.x * v.x + v.y * v.y + v.z * v.z - 1.0f) < 1e-3f, 4, i, ib, v.x, v.y, v.z);
        }
        cur_ib = ib;
      }
      cp_async_wait<1>();
      __syncthreads();

      const float4* tile = tiles + buf * kJT;
      const long long j0 = jc * kJT;
      const int jn = (int)min((long long)kJT, p.nj - j0);
      const bool full = (jn == kJT) && (i0 + BI <= p.ni) && (!p.sym || j0 >= i0 + BI);
#ifdef ACF_DEBUG_BOUNDS
      for (int jj = 0; jj < jn; ++jj) {
        const float4 v = tile[jj];
        ACF_CHECK(fabsf(v.x * v.x + v.y * v.y + v.z * v.z - 1.0f) < 1e-3f, 2, j0 + jj, q, v.x, v.y, v.z, (float)buf);
      }
#endif
      if (full) {
#pragma unroll 2
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
        for (int jj = 0; jj < jn; ++jj) {
          const float4 v = tile[jj];
          const long long j = j0 + jj;
#pragma unroll
          for (int k = 0; k < K; ++k) {
            const long long i = i0 + k * THREADS + tid;
            const bool ok = (i < p.ni) && (!p.sym || j > i);
            const float code = pair_code<MAP, METHOD>(xi[k], yi[k], zi[k], v.x, v.y, v.z, p.bp);
            if (ok && ACF_CHECK(__float_as_uint(code) - magic_bits < (uint32_t)p.bp.entries, 1,
                                (long long)(__float_as_uint(code) - magic_bits), i, code, xi[k], yi[k], zi[k], v.x,
                                v.y, v.z, (float)jj))
              red_shared_add((__float_as_uint(code) << SHIFT) + base, p.inc);
          }
        }
      }
      __syncthreads();  // the buffer just read is refilled two chunks from now
      if (++since_flush == p.flush_every) {
        flush_hist<K, THREADS, LAYOUT, MAP, METHOD>(p, hist, true);
        __syncthreads();
        since_flush = 0;
      }
      ib = nib;
      jc = njc;
    }
    cp_async_wait<0>();
  }
  __syncthreads();
  flush_hist<K, THREADS, LAYOUT, MAP, METHOD>(p, hist, false);
}

// ------------------------------------------------------------------ merge, omega, diagnostics

// out[k] = sum over blocks of partial[b][k]; auto-correlations add the n self-pairs to bin 0.
__global__ void merge_kernel(const unsigned long long* __restrict__ partial, int rows, int nbins,
                             unsigned long long self_pairs, unsigned long long* __restrict__ out) {
  for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < nbins; k += gridDim.x * blockDim.x) {
    unsigned long long s = (k == 0) ? self_pairs : 0ull;
    for (int r = 0; r < rows; ++r) s += partial[(size_t)r * nbins + k];
    out[k] = s;
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
