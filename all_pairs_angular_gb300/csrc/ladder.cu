// The optimisation ladder of "CUDA Deep Dive: 10B Galaxy Pairs on an RTX 5080" (section "The
// ladder", levels L0 to L5), rebuilt as GB300 kernels for like-for-like measurement. Each level
// adds one change to the previous one, as on the page; all three histogram families (DD, DR, RR)
// are computed by one kernel launch, with per-block shared-memory histograms flushed to global
// uint64 counts, and the pair formula is the page's: theta = arccos(sin d1 sin d2 +
// cos d1 cos d2 cos(a1 - a2)) in fp32 radians, bin = truncated theta / w clamped to the last bin.
// The page builds with --use_fast_math, so the sines and cosines here are the fast intrinsics.
//
//   L0  one thread per (i, j), 32 x 32 blocks, per-pair sin/cos, acosf, no symmetry
//   L1  + DD/RR symmetry: only j >= i, off-diagonal pairs counted twice
//   L2  + sin/cos of the declinations computed once per galaxy (here by a small kernel)
//   L3  + tiling: one i per thread in registers, a TILE-wide j-tile staged in shared memory
//   L4  + arccos polynomial (Abramowitz and Stegun 4.4.45) instead of acosf
//   L5  + unrolled inner loop, launch bounds, whole-block skip of DD/RR below the diagonal
//
// This is a measurement ladder, not the library's path: its fp32 arithmetic misbins pairs near
// edges (L4 by design); every level keeps the totals exact. L0-L3 give bit-identical histograms,
// as do L4 and L5, because every level evaluates a pair with the same expression.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/acf.h"

namespace {

constexpr int kLadderTile = 512;

struct LadderArgs {
  const float* ra_d;   // radians
  const float* ra_r;
  const float* sd_d;   // sin/cos of the declinations (L2 and up) or the declinations themselves
  const float* cd_d;
  const float* sd_r;
  const float* cd_r;
  int n;
  int nbins;
  float inv_w;         // 1 / w in radians
  unsigned long long* dd;
  unsigned long long* dr;
  unsigned long long* rr;
};

// One pair, the same expression at every level (products commute, so it is symmetric in i, j).
template <bool FAST>
__device__ __forceinline__ int ladder_bin(float si, float ci, float ai, float sj, float cj, float aj, const LadderArgs& a) {
  float c = fmaf(si, sj, ci * cj * __cosf(ai - aj));
  c = fminf(fmaxf(c, -1.0f), 1.0f);
  float th;
  if (FAST) {
    const float x = fabsf(c);
    float r = fmaf(-0.0187293f, x, 0.0742610f);
    r = fmaf(r, x, -0.2121144f);
    r = fmaf(r, x, 1.5707288f);
    r *= sqrtf(1.0f - x);
    th = c < 0.0f ? 3.14159265358979f - r : r;
  } else {
    th = acosf(c);
  }
  const int k = (int)(th * a.inv_w);
  return k < a.nbins - 1 ? k : a.nbins - 1;
}

__device__ __forceinline__ void zero_hist(unsigned int* h, int words) {
  for (int k = threadIdx.x + threadIdx.y * blockDim.x; k < words; k += blockDim.x * blockDim.y) h[k] = 0u;
}

__device__ __forceinline__ void flush_hists(const unsigned int* h, const LadderArgs& a) {
  const int t = threadIdx.x + threadIdx.y * blockDim.x, nt = blockDim.x * blockDim.y;
  for (int k = t; k < 3 * a.nbins; k += nt) {
    const unsigned int v = h[k];
    if (!v) continue;
    unsigned long long* out = k < a.nbins ? a.dd : (k < 2 * a.nbins ? a.dr : a.rr);
    atomicAdd(out + (k % a.nbins), (unsigned long long)v);
  }
}

// L0 - L2: one thread per (i, j) in 32 x 32 blocks.
template <int LEVEL>
__global__ void ladder_pair_kernel(LadderArgs a) {
  extern __shared__ unsigned int h[];  // DD, DR, RR: 3 x nbins
  zero_hist(h, 3 * a.nbins);
  __syncthreads();
  const int i = blockIdx.y * 32 + threadIdx.y;
  const int j = blockIdx.x * 32 + threadIdx.x;
  if (i < a.n && j < a.n) {
    float sdi, cdi, sdj, cdj, sri, cri, srj, crj;
    if (LEVEL >= 2) {
      sdi = a.sd_d[i]; cdi = a.cd_d[i]; sdj = a.sd_d[j]; cdj = a.cd_d[j];
      sri = a.sd_r[i]; cri = a.cd_r[i]; srj = a.sd_r[j]; crj = a.cd_r[j];
    } else {
      __sincosf(a.sd_d[i], &sdi, &cdi);
      __sincosf(a.sd_d[j], &sdj, &cdj);
      __sincosf(a.sd_r[i], &sri, &cri);
      __sincosf(a.sd_r[j], &srj, &crj);
    }
    const float adi = a.ra_d[i], adj = a.ra_d[j], ari = a.ra_r[i], arj = a.ra_r[j];
    atomicAdd(&h[a.nbins + ladder_bin<false>(sdi, cdi, adi, srj, crj, arj, a)], 1u);
    if (LEVEL == 0) {
      atomicAdd(&h[ladder_bin<false>(sdi, cdi, adi, sdj, cdj, adj, a)], 1u);
      atomicAdd(&h[2 * a.nbins + ladder_bin<false>(sri, cri, ari, srj, crj, arj, a)], 1u);
    } else if (j >= i) {
      const unsigned int inc = 1u + (unsigned int)(j != i);
      atomicAdd(&h[ladder_bin<false>(sdi, cdi, adi, sdj, cdj, adj, a)], inc);
      atomicAdd(&h[2 * a.nbins + ladder_bin<false>(sri, cri, ari, srj, crj, arj, a)], inc);
    }
  }
  __syncthreads();
  flush_hists(h, a);
}

// L3 - L5: one i per thread, TILE-wide j-tiles in shared memory.
template <int LEVEL>
__global__ void __launch_bounds__(kLadderTile) ladder_tile_kernel(LadderArgs a) {
  extern __shared__ unsigned int h[];  // 3 x nbins, then the j-tile
  float* tj = reinterpret_cast<float*>(h + 3 * a.nbins);  // 6 x TILE: sin/cos/ra of D, then of R
  zero_hist(h, 3 * a.nbins);
  const int tid = threadIdx.x;
  const int i_base = blockIdx.y * kLadderTile, j_base = blockIdx.x * kLadderTile;
  const int i = i_base + tid;
  const int j_count = min(kLadderTile, a.n - j_base);
  if (tid < j_count) {
    const int j = j_base + tid;
    tj[tid] = a.sd_d[j];
    tj[kLadderTile + tid] = a.cd_d[j];
    tj[2 * kLadderTile + tid] = a.ra_d[j];
    tj[3 * kLadderTile + tid] = a.sd_r[j];
    tj[4 * kLadderTile + tid] = a.cd_r[j];
    tj[5 * kLadderTile + tid] = a.ra_r[j];
  }
  __syncthreads();
  // L5: a block wholly below the diagonal holds no j >= i: skip DD and RR there
  const bool do_sym = LEVEL < 5 || (j_base + j_count - 1) >= i_base;
  if (i < a.n) {
    const float sdi = a.sd_d[i], cdi = a.cd_d[i], adi = a.ra_d[i];
    const float sri = a.sd_r[i], cri = a.cd_r[i], ari = a.ra_r[i];
    constexpr bool FAST = LEVEL >= 4;
    constexpr int kUnroll = LEVEL >= 5 ? 8 : 1;
#pragma unroll kUnroll
    for (int jj = 0; jj < j_count; ++jj) {
      atomicAdd(&h[a.nbins + ladder_bin<FAST>(sdi, cdi, adi, tj[3 * kLadderTile + jj], tj[4 * kLadderTile + jj],
                                                  tj[5 * kLadderTile + jj], a)], 1u);
      const int j = j_base + jj;
      if (do_sym && j >= i) {
        const unsigned int inc = 1u + (unsigned int)(j != i);
        atomicAdd(&h[ladder_bin<FAST>(sdi, cdi, adi, tj[jj], tj[kLadderTile + jj], tj[2 * kLadderTile + jj], a)], inc);
        atomicAdd(&h[2 * a.nbins + ladder_bin<FAST>(sri, cri, ari, tj[3 * kLadderTile + jj], tj[4 * kLadderTile + jj],
                                                        tj[5 * kLadderTile + jj], a)], inc);
      }
    }
  }
  __syncthreads();
  flush_hists(h, a);
}

// arcmin -> fp32 radians (the page converts in fp32 on the host); with `trig` the sin and cos of
// the declination, else the declination itself (L0, L1 take sin/cos per pair).
__global__ void ladder_prep_kernel(const float* ra, const float* dec, int n, bool trig, float* ra_rad, float* s,
                                   float* c) {
  const float k = 3.14159265358979f / 10800.0f;
  for (int g = blockIdx.x * blockDim.x + threadIdx.x; g < n; g += gridDim.x * blockDim.x) {
    ra_rad[g] = ra[g] * k;
    const float d = dec[g] * k;
    if (trig) {
      __sincosf(d, &s[g], &c[g]);
    } else {
      s[g] = d;
      c[g] = 0.0f;
    }
  }
}

}  // namespace

extern "C" int acf_ladder(int level, const float* ra_d, const float* dec_d, const float* ra_r, const float* dec_r,
                          int64_t n, double bin_width_deg, int32_t nbins, uint64_t* dd, uint64_t* dr, uint64_t* rr,
                          void* stream, float* kernel_ms) {
  if (level < 0 || level > 5 || !ra_d || !dec_d || !ra_r || !dec_r || !dd || !dr || !rr || n <= 0 ||
      !(bin_width_deg > 0.0) || nbins <= 0)
    return ACF_ERR_ARG;
  if (n > (1ll << 30) || nbins > 4000) return ACF_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* buf = nullptr;
  if (cudaMallocAsync(reinterpret_cast<void**>(&buf), sizeof(float) * 6 * (size_t)n, st) != cudaSuccess)
    return ACF_ERR_NOMEM;
  LadderArgs a;
  a.ra_d = buf;
  a.sd_d = buf + n;
  a.cd_d = buf + 2 * n;
  a.ra_r = buf + 3 * n;
  a.sd_r = buf + 4 * n;
  a.cd_r = buf + 5 * n;
  a.n = (int)n;
  a.nbins = nbins;
  a.inv_w = (float)(180.0 / (3.14159265358979323846 * bin_width_deg));
  a.dd = reinterpret_cast<unsigned long long*>(dd);
  a.dr = reinterpret_cast<unsigned long long*>(dr);
  a.rr = reinterpret_cast<unsigned long long*>(rr);
  const int pblocks = (int)std::min<int64_t>((n + 255) / 256, 4096);
  ladder_prep_kernel<<<pblocks, 256, 0, st>>>(ra_d, dec_d, (int)n, level >= 2, buf, buf + n, buf + 2 * n);
  ladder_prep_kernel<<<pblocks, 256, 0, st>>>(ra_r, dec_r, (int)n, level >= 2, buf + 3 * n, buf + 4 * n, buf + 5 * n);
  for (uint64_t* o : {dd, dr, rr}) cudaMemsetAsync(o, 0, sizeof(uint64_t) * (size_t)nbins, st);
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  cudaEventRecord(e0, st);
  const size_t hist = sizeof(unsigned int) * 3 * (size_t)nbins;
  if (level <= 2) {
    const dim3 grid((unsigned)((n + 31) / 32), (unsigned)((n + 31) / 32)), block(32, 32);
    if (level == 0) ladder_pair_kernel<0><<<grid, block, hist, st>>>(a);
    else if (level == 1) ladder_pair_kernel<1><<<grid, block, hist, st>>>(a);
    else ladder_pair_kernel<2><<<grid, block, hist, st>>>(a);
  } else {
    const unsigned t = (unsigned)((n + kLadderTile - 1) / kLadderTile);
    const dim3 grid(t, t);
    const size_t sm = hist + sizeof(float) * 6 * kLadderTile;
    if (level == 3) ladder_tile_kernel<3><<<grid, kLadderTile, sm, st>>>(a);
    else if (level == 4) ladder_tile_kernel<4><<<grid, kLadderTile, sm, st>>>(a);
    else ladder_tile_kernel<5><<<grid, kLadderTile, sm, st>>>(a);
  }
  cudaEventRecord(e1, st);
  cudaError_t e = cudaGetLastError();
  cudaFreeAsync(buf, st);
  if (e == cudaSuccess) e = cudaEventSynchronize(e1);
  float ms = 0.f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (kernel_ms) *kernel_ms = ms;
  return e == cudaSuccess ? ACF_OK : ACF_ERR_CUDA;
}
