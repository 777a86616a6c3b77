/*
 * ORACLE — test infrastructure, not part of the library.
 *
 * A plain, slow, fp64 CPU statement of what the galaxy two-point angular correlation computes.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may load it. It shares
 * no code with the CUDA library.
 *
 * Source of the definition: "CUDA Deep Dive: 10B Galaxy Pairs on an RTX 5080"
 *   - section "The problem": the separation of two galaxies at (alpha1, delta1), (alpha2, delta2) is
 *       theta = arccos( sin d1 sin d2 + cos d1 cos d2 cos(a1 - a2) ),
 *     positions are given in arcminutes, the separations are binned in 0.25 degree buckets, there
 *     are three histogram families (DD, DR, RR), every ordered pair is counted (N^2 per family)
 *     and omega = (DD - 2 DR + RR) / RR;
 *   - Appendix A, the bin-index helper: the cosine is clamped to [-1, 1] before arccos, the angle
 *     in degrees times bins-per-degree is truncated to an integer and clamped to the last bin;
 *   - Appendix A, the output writer: omega is formed only where RR > 0.
 *
 * Readings where the page is silent (each stated again in the design notes):
 *   - arithmetic is fp64 throughout; each fp32 arcminute value converts exactly to double and
 *     radians = value * (pi / 10800);
 *   - bin k holds theta_deg in [k w, (k+1) w); theta beyond nbins*w goes to the last bin;
 *   - auto-correlation loops over all n^2 ordered pairs, self-pairs included (they land in bin 0);
 *   - omega with unequal catalog sizes normalises each histogram by its pair total
 *     (n_d^2, n_d n_r, n_r^2); with equal sizes this is exactly the page's expression;
 *     bins with RR = 0 get NaN.
 *
 * Per-galaxy sin/cos of the declination and the right ascension in radians are computed once per
 * galaxy instead of once per pair. They are the same fp64 values either way, so every pair's
 * arithmetic is exactly the formula above.
 *
 * The oracle also counts, for each interior bin edge e_K = K w (K = 1 .. nbins-1), the pairs whose
 * fp64 theta lies within 1e-6 rad below the edge (near_below[K]) or at/above it within 1e-6 rad
 * (near_above[K]). Only those pairs may legitimately land in the neighbouring bin in a faster
 * implementation; the parity checker uses these counts.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_PI 3.14159265358979323846
#define ORACLE_EDGE_TOL_RAD 1e-6

typedef struct {
    double *sin_dec, *cos_dec, *ra_rad;
} galaxies;

static int galaxies_make(galaxies *g, const float *ra_arcmin, const float *dec_arcmin, int64_t n) {
    const size_t bytes = (size_t)(n > 0 ? n : 1) * sizeof(double);
    g->sin_dec = (double *)malloc(bytes);
    g->cos_dec = (double *)malloc(bytes);
    g->ra_rad = (double *)malloc(bytes);
    if (!g->sin_dec || !g->cos_dec || !g->ra_rad) return -1;
    const double arcmin_to_rad = ORACLE_PI / 10800.0;
    for (int64_t i = 0; i < n; ++i) {
        const double a = (double)ra_arcmin[i] * arcmin_to_rad;
        const double d = (double)dec_arcmin[i] * arcmin_to_rad;
        g->ra_rad[i] = a;
        g->sin_dec[i] = sin(d);
        g->cos_dec[i] = cos(d);
    }
    return 0;
}

static void galaxies_free(galaxies *g) {
    free(g->sin_dec);
    free(g->cos_dec);
    free(g->ra_rad);
}

/* The page's separation formula in fp64, with the page's clamp of the cosine to [-1, 1]. */
static double separation_rad(const galaxies *a, int64_t i, const galaxies *b, int64_t j) {
    double c = a->sin_dec[i] * b->sin_dec[j] + a->cos_dec[i] * b->cos_dec[j] * cos(a->ra_rad[i] - b->ra_rad[j]);
    if (c > 1.0) c = 1.0;
    if (c < -1.0) c = -1.0;
    return acos(c);
}

/* Truncate theta / w to a bin and clamp to the last bin. */
static int64_t bin_of(double theta_deg, double w_deg, int32_t nbins) {
    const double kf = floor(theta_deg / w_deg);
    if (kf >= (double)nbins) return nbins - 1;
    if (kf < 0.0) return 0;
    return (int64_t)kf;
}

/* Count one pair into hist and the edge windows. */
static void count_pair(double theta_rad, double w_deg, int32_t nbins, uint64_t *hist, uint64_t *near_below,
                       uint64_t *near_above) {
    const double rad_to_deg = 180.0 / ORACLE_PI;
    const double tol_deg = ORACLE_EDGE_TOL_RAD * rad_to_deg;
    const double theta_deg = theta_rad * rad_to_deg;
    const int64_t k = bin_of(theta_deg, w_deg, nbins);
    hist[k] += 1;
    if (k + 1 <= nbins - 1) {
        const double e = (double)(k + 1) * w_deg; /* the edge above this pair's bin */
        if (e - theta_deg < tol_deg) near_below[k + 1] += 1;
    }
    if (k >= 1) {
        const double e = (double)k * w_deg; /* the edge below */
        if (theta_deg - e < tol_deg) near_above[k] += 1;
    }
}

/*
 * Histogram of the separations of all ordered pairs (i in catalog 1, j in catalog 2).
 * For DD or RR pass the same catalog twice. hist has nbins entries; near_below and near_above
 * have nbins + 1 entries indexed by edge number K (entries 0 and nbins stay 0). Any of the
 * output pointers may be overwritten; all are zeroed first. nthreads <= 0 uses all cores.
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int oracle_histogram(const float *ra1, const float *dec1, int64_t n1, const float *ra2, const float *dec2, int64_t n2,
                     double w_deg, int32_t nbins, int32_t nthreads, uint64_t *hist, uint64_t *near_below,
                     uint64_t *near_above) {
    if (n1 < 0 || n2 < 0 || nbins <= 0 || !(w_deg > 0.0) || !hist || !near_below || !near_above) return -1;
    memset(hist, 0, sizeof(uint64_t) * (size_t)nbins);
    memset(near_below, 0, sizeof(uint64_t) * (size_t)(nbins + 1));
    memset(near_above, 0, sizeof(uint64_t) * (size_t)(nbins + 1));
    if (n1 == 0 || n2 == 0) return 0;
    galaxies a, b;
    if (galaxies_make(&a, ra1, dec1, n1) || galaxies_make(&b, ra2, dec2, n2)) return -1;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        uint64_t *h = (uint64_t *)calloc((size_t)nbins, sizeof(uint64_t));
        uint64_t *lo = (uint64_t *)calloc((size_t)nbins + 1, sizeof(uint64_t));
        uint64_t *hi = (uint64_t *)calloc((size_t)nbins + 1, sizeof(uint64_t));
        if (!h || !lo || !hi) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 16)
#endif
            for (int64_t i = 0; i < n1; ++i)
                for (int64_t j = 0; j < n2; ++j) count_pair(separation_rad(&a, i, &b, j), w_deg, nbins, h, lo, hi);
#ifdef _OPENMP
#pragma omp critical
#endif
            {
                for (int32_t k = 0; k < nbins; ++k) hist[k] += h[k];
                for (int32_t k = 0; k <= nbins; ++k) {
                    near_below[k] += lo[k];
                    near_above[k] += hi[k];
                }
            }
        }
        free(h);
        free(lo);
        free(hi);
    }
    galaxies_free(&a);
    galaxies_free(&b);
    return failed ? -1 : 0;
}

/* theta (radians, fp64) of the n pairs (ra1[k], dec1[k]) - (ra2[k], dec2[k]). */
int oracle_pair_theta(const float *ra1, const float *dec1, const float *ra2, const float *dec2, int64_t n,
                      double *theta_rad) {
    if (n < 0) return -1;
    if (n == 0) return 0;
    galaxies a, b;
    if (galaxies_make(&a, ra1, dec1, n) || galaxies_make(&b, ra2, dec2, n)) return -1;
    for (int64_t k = 0; k < n; ++k) theta_rad[k] = separation_rad(&a, k, &b, k);
    galaxies_free(&a);
    galaxies_free(&b);
    return 0;
}

/* bin of each pair (same rule as oracle_histogram). */
int oracle_pair_bin(const float *ra1, const float *dec1, const float *ra2, const float *dec2, int64_t n, double w_deg,
                    int32_t nbins, int32_t *bins) {
    if (n < 0 || nbins <= 0 || !(w_deg > 0.0)) return -1;
    if (n == 0) return 0;
    galaxies a, b;
    if (galaxies_make(&a, ra1, dec1, n) || galaxies_make(&b, ra2, dec2, n)) return -1;
    const double rad_to_deg = 180.0 / ORACLE_PI;
    for (int64_t k = 0; k < n; ++k) bins[k] = (int32_t)bin_of(separation_rad(&a, k, &b, k) * rad_to_deg, w_deg, nbins);
    galaxies_free(&a);
    galaxies_free(&b);
    return 0;
}

/*
 * Landy-Szalay estimator per bin: omega = (DD/Ndd - 2 DR/Ndr + RR/Nrr) / (RR/Nrr), with the pair
 * totals Ndd = n_d^2, Ndr = n_d n_r, Nrr = n_r^2. Written as (DD f_dd - 2 DR f_dr + RR) / RR with
 * f_dd = Nrr/Ndd and f_dr = Nrr/Ndr, which are exactly 1 when n_d == n_r, so that case is the
 * page's (DD - 2 DR + RR) / RR evaluated in fp64. NaN where RR = 0.
 */
int oracle_omega(const uint64_t *dd, const uint64_t *dr, const uint64_t *rr, int32_t nbins, int64_t n_d, int64_t n_r,
                 double *omega) {
    if (nbins <= 0 || n_d <= 0 || n_r <= 0) return -1;
    const double nd = (double)n_d, nr = (double)n_r;
    const double f_dd = (nr * nr) / (nd * nd);
    const double f_dr = (nr * nr) / (nd * nr);
    for (int32_t k = 0; k < nbins; ++k) {
        if (rr[k] == 0) {
            omega[k] = NAN;
            continue;
        }
        const double num = (double)dd[k] * f_dd - 2.0 * (double)dr[k] * f_dr + (double)rr[k];
        omega[k] = num / (double)rr[k];
    }
    return 0;
}
