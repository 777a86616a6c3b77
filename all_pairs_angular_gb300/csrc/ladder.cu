// The optimisation ladder of "CUDA Deep Dive: 10B Galaxy Pairs on an RTX 5080" (section "The
// ladder", levels L0 to L5), rebuilt as GB300 kernels for like-for-like measurement. Each level
// adds the one change that the page's level table names; all three histogram families (DD, DR, RR)
// come from one kernel launch, with per-block shared-memory histograms added into global uint64
// counts, and a pair is evaluated with the page's formula: theta = arccos(sin d1 sin d2 +
// cos d1 cos d2 cos(a1 - a2)) in fp32 radians, bin = truncated theta / w clamped to the last bin.
// The page builds with fast math, so the sines and cosines here are the fast intrinsics.
//
//   L0  one thread per ordered pair, 32 x 32 threads per block, sin/cos per pair, acosf
//   L1  + DD/RR symmetry: a pair with j > i counts twice, j < i is not evaluated
//   L2  + sin/cos of the declinations once per galaxy (a small kernel here)
//   L3  + tiling: one i per thread in registers, j-tiles of both catalogs in shared memory
//   L4  + the arccos polynomial of Abramowitz and Stegun 4.4.45 instead of acosf
//   L5  + an unrolled j-loop, launch bounds, and no DD/RR work in tiles wholly below the diagonal
//
// How this build expresses them: every galaxy is one 16-byte record (sin d, cos d, ra, 0) of its
// catalog, so a j-tile is staged with one vector load per galaxy and family. Levels 3 and 4 run one
// j-loop that adds the DR pair and, where j >= i, the DD and RR pairs. Level 5 splits it into a DR
// loop over the whole tile and a DD/RR loop that starts at the first j >= i: in a tile below the
// diagonal that loop is empty, and the per-pair test is gone.
//
// This is a measurement ladder, not the library's path: its fp32 arithmetic misbins pairs near
// edges (L4 by design); every level keeps the totals exact. L0-L3 give bit-identical histograms,
// as do L4 and L5, because every level evaluates a pair with the same expression.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/acf.h"

namespace {

constexpr int kLadderTile = 512;                     // i per block and j per tile, levels 3-5
constexpr int kLadderUnroll = 4;                     // level 5's j-loop unroll
constexpr int kLadderMaxBins = 4000;
constexpr size_t kLadderMaxSmem = 227 * 1024;

struct LadderArgs {
  const float4* td;  // per galaxy of D: (sin dec, cos dec, ra, 0) from L2 on, (dec, 0, ra, 0) before
  const float4* tr;  // the same for R
  int n;
  int nbins;
  float inv_w;       // 1 / w in radians
  unsigned long long* dd;
  unsigned long long* dr;
  unsigned long long* rr;
};

// The bin of one pair from the two galaxies' terms (symmetric in the two: products commute).
template <bool POLY>
__device__ __forceinline__ int ladder_bin(float4 g, float4 h, const LadderArgs& a) {
  float c = fmaf(g.x, h.x, g.y * h.y * __cosf(g.z - h.z));
  c = fminf(fmaxf(c, -1.0f), 1.0f);
  float th;
  if (POLY) {
    // A&S 4.4.45 on |c|, reflected for negative cosines
    const float x = fabsf(c);
    const float r = sqrtf(1.0f - x) * fmaf(fmaf(fmaf(-0.0187293f, x, 0.0742610f), x, -0.2121144f), x, 1.5707288f);
    th = c < 0.0f ? 3.14159265358979f - r : r;
  } else {
    th = acosf(c);
  }
  const int k = (int)(th * a.inv_w);
  return min(k, a.nbins - 1);
}

// terms from a declination stored raw (levels 0 and 1 take sin and cos per pair)
__device__ __forceinline__ float4 with_trig(float4 g) {
  float s, c;
  __sincosf(g.x, &s, &c);
  return make_float4(s, c, g.z, 0.0f);
}

// Block histograms: DD in [0, nbins), DR in [nbins, 2 nbins), RR in [2 nbins, 3 nbins).
__device__ __forceinline__ void add_to(unsigned int* h, int family, int bin, unsigned int v, const LadderArgs& a) {
  atomicAdd(h + family * a.nbins + bin, v);
}

__device__ __forceinline__ void clear_block_hists(unsigned int* h, int words, int t, int nt) {
  for (int k = t; k < words; k += nt) h[k] = 0u;
}

__device__ __forceinline__ void add_block_hists(const unsigned int* h, const LadderArgs& a, int t, int nt) {
  unsigned long long* fam[3] = {a.dd, a.dr, a.rr};
  for (int f = 0; f < 3; ++f)
    for (int k = t; k < a.nbins; k += nt) {
      const unsigned int v = h[f * a.nbins + k];
      if (v) atomicAdd(fam[f] + k, (unsigned long long)v);
    }
}

// L0 - L2: one thread per (i, j); threadIdx.y picks i, threadIdx.x picks j.
template <int LEVEL>
__global__ void ladder_pair_kernel(LadderArgs a) {
  extern __shared__ unsigned int h[];
  const int t = threadIdx.y * 32 + threadIdx.x;
  clear_block_hists(h, 3 * a.nbins, t, 1024);
  __syncthreads();
  const int i = blockIdx.y * 32 + threadIdx.y, j = blockIdx.x * 32 + threadIdx.x;
  if (i < a.n && j < a.n) {
    float4 di = a.td[i], dj = a.td[j], ri = a.tr[i], rj = a.tr[j];
    if (LEVEL < 2) {
      di = with_trig(di);
      dj = with_trig(dj);
      ri = with_trig(ri);
      rj = with_trig(rj);
    }
    add_to(h, 1, ladder_bin<false>(di, rj, a), 1u, a);
    // L0 counts every ordered pair; from L1 on only j >= i is evaluated, off-diagonal pairs twice
    const unsigned int w = LEVEL == 0 ? 1u : (j > i ? 2u : (j == i ? 1u : 0u));
    if (w) {
      add_to(h, 0, ladder_bin<false>(di, dj, a), w, a);
      add_to(h, 2, ladder_bin<false>(ri, rj, a), w, a);
    }
  }
  __syncthreads();
  add_block_hists(h, a, t, 1024);
}

// L3 - L5: block (x, y) pairs the i-tile y (one i per thread) with the j-tile x of both catalogs.
template <int LEVEL>
__global__ void __launch_bounds__(LEVEL >= 5 ? kLadderTile : 1024) ladder_tile_kernel(LadderArgs a) {
  constexpr bool POLY = LEVEL >= 4;
  extern __shared__ __align__(16) unsigned char smem[];
  float4* tile = reinterpret_cast<float4*>(smem);  // [0, T): D terms, [T, 2T): R terms
  unsigned int* h = reinterpret_cast<unsigned int*>(smem + 2 * kLadderTile * sizeof(float4));
  const int t = threadIdx.x;
  clear_block_hists(h, 3 * a.nbins, t, kLadderTile);
  const int j0 = blockIdx.x * kLadderTile, i = blockIdx.y * kLadderTile + t;
  const int nt = min(kLadderTile, a.n - j0);  // galaxies in this j-tile
  if (t < nt) {
    tile[t] = a.td[j0 + t];
    tile[kLadderTile + t] = a.tr[j0 + t];
  }
  __syncthreads();
  if (i < a.n) {
    const float4 di = a.td[i], ri = a.tr[i];
    if (LEVEL < 5) {
      for (int k = 0; k < nt; ++k) {
        const float4 dj = tile[k], rj = tile[kLadderTile + k];
        add_to(h, 1, ladder_bin<POLY>(di, rj, a), 1u, a);
        const int j = j0 + k;
        if (j >= i) {
          const unsigned int w = j > i ? 2u : 1u;
          add_to(h, 0, ladder_bin<POLY>(di, dj, a), w, a);
          add_to(h, 2, ladder_bin<POLY>(ri, rj, a), w, a);
        }
      }
    } else {
#pragma unroll kLadderUnroll
      for (int k = 0; k < nt; ++k) add_to(h, 1, ladder_bin<POLY>(di, tile[kLadderTile + k], a), 1u, a);
      // the first j of the tile with j >= i; past the tile's end for a tile below the diagonal
      const int first = max(0, i - j0);
      if (first < nt) {
        // the self-pair (j == i) lies in this tile only on the diagonal, and counts once
        int k = first;
        if (j0 + k == i) {
          add_to(h, 0, ladder_bin<POLY>(di, tile[k], a), 1u, a);
          add_to(h, 2, ladder_bin<POLY>(ri, tile[kLadderTile + k], a), 1u, a);
          ++k;
        }
#pragma unroll kLadderUnroll
        for (; k < nt; ++k) {
          add_to(h, 0, ladder_bin<POLY>(di, tile[k], a), 2u, a);
          add_to(h, 2, ladder_bin<POLY>(ri, tile[kLadderTile + k], a), 2u, a);
        }
      }
    }
  }
  __syncthreads();
  add_block_hists(h, a, t, kLadderTile);
}

// arcmin -> fp32 radians (the page converts in fp32 on the host); with `trig` the record holds the
// sin and cos of the declination, else the declination itself (levels 0 and 1 take them per pair).
__global__ void ladder_prep_kernel(const float* ra, const float* dec, int n, bool trig, float4* terms) {
  const float k = 3.14159265358979f / 10800.0f;
  for (int g = blockIdx.x * blockDim.x + threadIdx.x; g < n; g += gridDim.x * blockDim.x) {
    const float d = dec[g] * k, r = ra[g] * k;
    float s = d, c = 0.0f;
    if (trig) __sincosf(d, &s, &c);
    terms[g] = make_float4(s, c, r, 0.0f);
  }
}

}  // namespace

extern "C" int acf_ladder(int level, const float* ra_d, const float* dec_d, const float* ra_r, const float* dec_r,
                          int64_t n, double bin_width_deg, int32_t nbins, uint64_t* dd, uint64_t* dr, uint64_t* rr,
                          void* stream, float* kernel_ms) {
  if (level < 0 || level > 5 || !ra_d || !dec_d || !ra_r || !dec_r || !dd || !dr || !rr || n <= 0 ||
      !(bin_width_deg > 0.0) || nbins <= 0)
    return ACF_ERR_ARG;
  if (n > (1ll << 30) || nbins > kLadderMaxBins) return ACF_ERR_UNSUPPORTED;
  const size_t hist = sizeof(unsigned int) * 3 * (size_t)nbins;
  const size_t tile_smem = hist + 2 * kLadderTile * sizeof(float4);
  if (level >= 3 && tile_smem > kLadderMaxSmem) return ACF_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float4* buf = nullptr;
  if (cudaMallocAsync(reinterpret_cast<void**>(&buf), sizeof(float4) * 2 * (size_t)n, st) != cudaSuccess)
    return ACF_ERR_NOMEM;
  LadderArgs a;
  a.td = buf;
  a.tr = buf + n;
  a.n = (int)n;
  a.nbins = nbins;
  a.inv_w = (float)(180.0 / (3.14159265358979323846 * bin_width_deg));
  a.dd = reinterpret_cast<unsigned long long*>(dd);
  a.dr = reinterpret_cast<unsigned long long*>(dr);
  a.rr = reinterpret_cast<unsigned long long*>(rr);
  cudaError_t e = cudaSuccess;
  const int pblocks = (int)std::min<int64_t>((n + 255) / 256, 4096);
  ladder_prep_kernel<<<pblocks, 256, 0, st>>>(ra_d, dec_d, (int)n, level >= 2, buf);
  ladder_prep_kernel<<<pblocks, 256, 0, st>>>(ra_r, dec_r, (int)n, level >= 2, buf + n);
  e = cudaGetLastError();
  for (uint64_t* o : {dd, dr, rr})
    if (e == cudaSuccess) e = cudaMemsetAsync(o, 0, sizeof(uint64_t) * (size_t)nbins, st);
  // levels 3-5 may need more than the default 48 KB of dynamic shared memory
  void (*tile_fn)(LadderArgs) = level == 3 ? ladder_tile_kernel<3> : (level == 4 ? ladder_tile_kernel<4> : ladder_tile_kernel<5>);
  if (e == cudaSuccess && level >= 3)
    e = cudaFuncSetAttribute(tile_fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tile_smem);
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (e == cudaSuccess) e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  if (e == cudaSuccess) e = cudaEventRecord(e0, st);
  if (e == cudaSuccess) {
    if (level <= 2) {
      const dim3 grid((unsigned)((n + 31) / 32), (unsigned)((n + 31) / 32)), block(32, 32);
      if (level == 0) ladder_pair_kernel<0><<<grid, block, hist, st>>>(a);
      else if (level == 1) ladder_pair_kernel<1><<<grid, block, hist, st>>>(a);
      else ladder_pair_kernel<2><<<grid, block, hist, st>>>(a);
    } else {
      const unsigned tiles = (unsigned)((n + kLadderTile - 1) / kLadderTile);
      tile_fn<<<dim3(tiles, tiles), kLadderTile, tile_smem, st>>>(a);
    }
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaEventRecord(e1, st);
  cudaFreeAsync(buf, st);
  if (e == cudaSuccess) e = cudaEventSynchronize(e1);
  else cudaStreamSynchronize(st);
  float ms = 0.f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (kernel_ms) *kernel_ms = ms;
  return e == cudaSuccess ? ACF_OK : ACF_ERR_CUDA;
}
