// acf_cli: the whole job from catalog files, the command-line shape of the program on
// "CUDA Deep Dive: 10B Galaxy Pairs on an RTX 5080":
//
//     acf_cli data.txt random.txt omega.out [bin_width_deg [nbins]]     (defaults 0.25 720)
//
// Reads both catalogs (count line, then "ra dec" rows in arcminutes), computes DD, DR, RR and omega
// on GPU 0 through the library's C ABI, checks that every histogram sums to its pair count, and
// writes the table (one row per bin with RR > 0). Exit status 0 on success.
#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "../../include/acf.h"

int main(int argc, char** argv) {
  if (argc < 4 || argc > 6) {
    std::fprintf(stderr, "usage: %s data.txt random.txt omega.out [bin_width_deg [nbins]]\n", argv[0]);
    return 2;
  }
  const double w = argc > 4 ? std::atof(argv[4]) : 0.25;
  const int nbins = argc > 5 ? std::atoi(argv[5]) : 720;
  using clock = std::chrono::steady_clock;
  const auto t0 = clock::now();
  char err[512];
  float *ra_d = nullptr, *dec_d = nullptr, *ra_r = nullptr, *dec_r = nullptr;
  int64_t n_d = 0, n_r = 0;
  if (acf_read_catalog(argv[1], &ra_d, &dec_d, &n_d, err, sizeof err) != ACF_OK ||
      acf_read_catalog(argv[2], &ra_r, &dec_r, &n_r, err, sizeof err) != ACF_OK) {
    std::fprintf(stderr, "acf_cli: %s\n", err);
    return 1;
  }
  const auto t1 = clock::now();
  acf_ctx* ctx = nullptr;
  if (acf_create(&ctx, 0, nullptr) != ACF_OK) {
    std::fprintf(stderr, "acf_cli: no CUDA device\n");
    return 1;
  }
  std::vector<uint64_t> dd(nbins), dr(nbins), rr(nbins);
  std::vector<double> om(nbins);
  int rc = acf_correlate_host(ctx, ra_d, dec_d, n_d, ra_r, dec_r, n_r, w, nbins, dd.data(), dr.data(), rr.data(),
                              om.data());
  if (rc != ACF_OK) {
    std::fprintf(stderr, "acf_cli: %s\n", acf_last_error(ctx));
    return 1;
  }
  const auto t2 = clock::now();
  unsigned long long sdd = 0, sdr = 0, srr = 0;
  for (int k = 0; k < nbins; ++k) {
    sdd += dd[k];
    sdr += dr[k];
    srr += rr[k];
  }
  const bool sums = sdd == (unsigned long long)(n_d * n_d) && sdr == (unsigned long long)(n_d * n_r) &&
                    srr == (unsigned long long)(n_r * n_r);
  if (acf_write_omega(argv[3], dd.data(), dr.data(), rr.data(), om.data(), nbins, w) != ACF_OK) {
    std::fprintf(stderr, "acf_cli: cannot write %s\n", argv[3]);
    return 1;
  }
  const auto t3 = clock::now();
  auto ms = [](clock::time_point a, clock::time_point b) {
    return std::chrono::duration<double, std::milli>(b - a).count();
  };
  std::printf("read %lld + %lld galaxies in %.3f ms; DD, DR, RR, omega in %.3f ms; wrote %s in %.3f ms\n",
              (long long)n_d, (long long)n_r, ms(t0, t1), ms(t1, t2), argv[3], ms(t2, t3));
  std::printf("histogram sums %s: DD %llu DR %llu RR %llu\n", sums ? "correct" : "WRONG", sdd, sdr, srr);
  acf_destroy(ctx);
  acf_free_catalog(ra_d, dec_d);
  acf_free_catalog(ra_r, dec_r);
  return sums ? 0 : 1;
}
