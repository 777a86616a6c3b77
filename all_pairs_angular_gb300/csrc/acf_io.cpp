// Catalog text files and the omega table of the library (host code, part of libacf.so).
//
// The formats are those of the program of "CUDA Deep Dive: 10B Galaxy Pairs on an RTX 5080"
// (sections "mmap + hand-rolled parser vs. fscanf" and the output step of its listing): a catalog
// is ASCII text, a count line and then one "ra dec" row (arcminutes) per galaxy; the result table
// has a header line and one row per bin with RR > 0: bin start in degrees, omega, DD, DR, RR.
// The page's observation that the reader is worth optimising (scanf-style parsing cost more than
// its whole kernel) is followed: the file is mapped and each number goes through std::from_chars,
// which needs no format string and rounds correctly to float.
#include <fcntl.h>
#include <sys/mman.h>
#include <sys/stat.h>
#include <unistd.h>

#include <charconv>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "../../include/acf.h"

namespace {

int io_fail(char* err, int32_t len, int code, const char* fmt, ...) {
  if (err && len > 0) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(err, (size_t)len, fmt, ap);
    va_end(ap);
  }
  return code;
}

const char* skip_space(const char* p, const char* end) {
  while (p < end && (*p == ' ' || *p == '\t' || *p == '\r' || *p == '\n')) ++p;
  return p;
}

// The 1-based line number of position p (for error messages only).
long long line_of(const char* begin, const char* p) {
  long long line = 1;
  for (const char* q = begin; q < p; ++q) line += (*q == '\n');
  return line;
}

}  // namespace

extern "C" int acf_read_catalog(const char* path, float** ra_out, float** dec_out, int64_t* n_out, char* err,
                                int32_t err_len) {
  if (err && err_len > 0) err[0] = '\0';
  if (!path || !ra_out || !dec_out || !n_out) return io_fail(err, err_len, ACF_ERR_ARG, "NULL argument");
  *ra_out = nullptr;
  *dec_out = nullptr;
  *n_out = 0;
  const int fd = open(path, O_RDONLY);
  if (fd < 0) return io_fail(err, err_len, ACF_ERR_ARG, "cannot open %s: %s", path, strerror(errno));
  struct stat st;
  if (fstat(fd, &st) != 0 || st.st_size <= 0) {
    close(fd);
    return io_fail(err, err_len, ACF_ERR_ARG, "%s is empty or unreadable", path);
  }
  const size_t size = (size_t)st.st_size;
  void* map = mmap(nullptr, size, PROT_READ, MAP_PRIVATE, fd, 0);
  close(fd);
  if (map == MAP_FAILED) return io_fail(err, err_len, ACF_ERR_NOMEM, "cannot map %s", path);
  const char* begin = static_cast<const char*>(map);
  const char* end = begin + size;
  int rc = ACF_OK;
  float* ra = nullptr;
  float* dec = nullptr;
  long long n = 0;
  const char* p = skip_space(begin, end);
  auto cnt = std::from_chars(p, end, n);
  if (cnt.ec != std::errc() || n < 0) {
    rc = io_fail(err, err_len, ACF_ERR_ARG, "%s: the first line must hold the galaxy count", path);
  } else {
    p = cnt.ptr;
    ra = static_cast<float*>(malloc(sizeof(float) * (size_t)(n > 0 ? n : 1)));
    dec = static_cast<float*>(malloc(sizeof(float) * (size_t)(n > 0 ? n : 1)));
    if (!ra || !dec) rc = io_fail(err, err_len, ACF_ERR_NOMEM, "cannot allocate %lld galaxies", n);
    for (long long k = 0; rc == ACF_OK && k < n; ++k) {
      p = skip_space(p, end);
      auto a = std::from_chars(p, end, ra[k]);
      const char* q = skip_space(a.ptr, end);
      auto d = a.ec == std::errc() ? std::from_chars(q, end, dec[k]) : a;
      if (a.ec != std::errc() || d.ec != std::errc())
        rc = io_fail(err, err_len, ACF_ERR_ARG, "%s line %lld: expected galaxy %lld of %lld as \"ra dec\"", path,
                     line_of(begin, p), k + 1, n);
      else
        p = d.ptr;
    }
  }
  munmap(map, size);
  if (rc != ACF_OK) {
    free(ra);
    free(dec);
    return rc;
  }
  *ra_out = ra;
  *dec_out = dec;
  *n_out = n;
  return ACF_OK;
}

extern "C" void acf_free_catalog(float* ra, float* dec) {
  free(ra);
  free(dec);
}

extern "C" int acf_write_omega(const char* path, const uint64_t* dd, const uint64_t* dr, const uint64_t* rr,
                               const double* omega, int32_t nbins, double bin_width_deg) {
  if (!path || !dd || !dr || !rr || !omega || nbins <= 0 || !(bin_width_deg > 0.0)) return ACF_ERR_ARG;
  FILE* f = fopen(path, "w");
  if (!f) return ACF_ERR_ARG;
  fprintf(f, "bin start\t\tomega\t        hist_DD\t        hist_DR\t        hist_RR\n");
  for (int32_t k = 0; k < nbins; ++k) {
    if (rr[k] == 0) continue;
    fprintf(f, "%6.3f\t%15f\t%15llu\t%15llu\t%15llu\n", (double)k * bin_width_deg, omega[k],
            (unsigned long long)dd[k], (unsigned long long)dr[k], (unsigned long long)rr[k]);
  }
  const bool ok = ferror(f) == 0;
  return (fclose(f) == 0 && ok) ? ACF_OK : ACF_ERR_ARG;
}
