/*
 * Seeded synthetic galaxy catalogs (right ascension, declination in arcminutes, fp32).
 *
 * This module only makes inputs. It holds none of the angular-correlation arithmetic
 * (no separations, no binning): both the CUDA path and the CPU oracle are fed from here.
 *
 * Shapes follow the workloads of "CUDA Deep Dive: 10B Galaxy Pairs on an RTX 5080",
 * section "The problem": two catalogs of positions given in arcminutes, one "real"
 * (clustered) and one random. The pages ship no catalogs, so the recipe is ours:
 *   - uniform on the sphere: RA = 21600 u1, Dec = asin(2 u2 - 1) (radians -> arcmin);
 *   - Gaussian clumps: centres uniform on the sphere (or in the patch), members assigned
 *     round-robin, each member offset by (g1, g2) * sigma in the tangent plane (east, north)
 *     of its centre and projected back onto the sphere;
 *   - small field: RA and Dec uniform in [0, patch) arcmin, clump members redrawn until they
 *     land inside the patch.
 * Stream order: R catalog, then D's uniform half, then the clump centres, then the members.
 *
 * Reproducibility across machines: the random stream is splitmix64 -> xoshiro256**, and every
 * floating-point step uses only IEEE-754 +, -, *, / and sqrt, which are correctly rounded on
 * every platform. The few transcendental functions needed (log, sin, cos, atan) are written
 * here from their power series instead of calling libm, whose last-bit results differ between
 * C libraries and CPU architectures. Build with -ffp-contract=off so no compiler fuses a
 * multiply and an add differently on different machines.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

/* ------------------------------------------------------------------ random stream */

typedef struct { uint64_t s[4]; } xs256;

static uint64_t splitmix64(uint64_t *x) {
    uint64_t z = (*x += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static void xs_seed(xs256 *g, uint64_t seed) {
    uint64_t x = seed;
    for (int k = 0; k < 4; ++k) g->s[k] = splitmix64(&x);
}

static inline uint64_t rotl(uint64_t v, int k) { return (v << k) | (v >> (64 - k)); }

static uint64_t xs_next(xs256 *g) {
    uint64_t *s = g->s;
    const uint64_t out = rotl(s[1] * 5, 7) * 9;
    const uint64_t t = s[1] << 17;
    s[2] ^= s[0];
    s[3] ^= s[1];
    s[1] ^= s[2];
    s[0] ^= s[3];
    s[2] ^= t;
    s[3] = rotl(s[3], 45);
    return out;
}

/* uniform double in [0, 1) with 53 random bits */
static double xs_unif(xs256 *g) { return (double)(xs_next(g) >> 11) * 0x1.0p-53; }

/* ------------------------------------------------- portable elementary functions */

static const double K_PI = 3.14159265358979311600e+00;      /* nearest double to pi */
static const double K_PIO2_HI = 1.57079632679489655800e+00; /* pi/2 split for reduction */
static const double K_PIO2_LO = 6.12323399573676603587e-17;
static const double K_LN2_HI = 6.93147180369123816490e-01;
static const double K_LN2_LO = 1.90821492927058770002e-10;

/* natural log for x > 0: x = m 2^e with m in [sqrt(1/2), sqrt(2)), log m = 2 atanh((m-1)/(m+1)) */
static double p_log(double x) {
    int e;
    double m = frexp(x, &e); /* exact: m in [0.5, 1) */
    if (m < 0.70710678118654752440) { m *= 2.0; e -= 1; }
    const double s = (m - 1.0) / (m + 1.0);
    const double s2 = s * s;
    double term = s, sum = 0.0;
    for (int k = 0; k < 16; ++k) { /* |s| <= 0.1716, s^2 <= 0.0295: 16 odd terms reach 1e-24 */
        sum += term / (double)(2 * k + 1);
        term *= s2;
    }
    return 2.0 * sum + (double)e * K_LN2_LO + (double)e * K_LN2_HI;
}

/* sin and cos of r with |r| <= pi/4 (+ tiny) by Taylor series to order 25 */
static void p_sincos_small(double r, double *sn, double *cs) {
    const double r2 = r * r;
    double ts = r, tc = 1.0, ss = 0.0, sc = 0.0;
    for (int k = 0; k < 13; ++k) {
        ss += ts;
        sc += tc;
        ts *= -r2 / (double)((2 * k + 2) * (2 * k + 3));
        tc *= -r2 / (double)((2 * k + 1) * (2 * k + 2));
    }
    *sn = ss;
    *cs = sc;
}

/* sin and cos for |x| <= 8: reduce by the nearest multiple of pi/2 (two-part constant) */
static void p_sincos(double x, double *sn, double *cs) {
    const double q = floor(x / K_PIO2_HI + 0.5);
    const double r = (x - q * K_PIO2_HI) - q * K_PIO2_LO;
    double s, c;
    p_sincos_small(r, &s, &c);
    const int quad = ((int)q) & 3;
    switch (quad) {
    case 0: *sn = s; *cs = c; break;
    case 1: *sn = c; *cs = -s; break;
    case 2: *sn = -s; *cs = -c; break;
    default: *sn = -c; *cs = s; break;
    }
}

/* atan(t) for t >= 0: reduce to |u| <= tan(pi/12) and sum the alternating series */
static double p_atan_pos(double t) {
    int inv = 0;
    if (t > 1.0) { t = 1.0 / t; inv = 1; }
    double base = 0.0;
    const double tan15 = 0.26794919243112270647; /* 2 - sqrt(3) */
    const double sqrt3 = 1.73205080756887729353;
    if (t > tan15) { /* atan t = pi/6 + atan((t sqrt3 - 1)/(t + sqrt3)) */
        t = (t * sqrt3 - 1.0) / (t + sqrt3);
        base = K_PI / 6.0;
    }
    const double u2 = t * t;
    double term = t, sum = 0.0;
    for (int k = 0; k < 20; ++k) { /* |u| <= 0.268: 20 terms reach 1e-25 */
        sum += term / (double)(2 * k + 1);
        term *= -u2;
    }
    double r = base + sum;
    if (inv) r = (K_PIO2_HI - r) + K_PIO2_LO;
    return r;
}

/* atan2 with the usual quadrant convention, result in (-pi, pi] */
static double p_atan2(double y, double x) {
    if (x == 0.0 && y == 0.0) return 0.0;
    const double ay = fabs(y), ax = fabs(x);
    double a = (ax >= ay) ? p_atan_pos(ay / ax) : (K_PIO2_HI - p_atan_pos(ax / ay)) + K_PIO2_LO;
    if (x < 0.0) a = K_PI - a;
    return (y < 0.0) ? -a : a;
}

/* asin via atan2(x, sqrt((1-x)(1+x))) */
static double p_asin(double x) { return p_atan2(x, sqrt((1.0 - x) * (1.0 + x))); }

/* ------------------------------------------------------------- catalog geometry */

static const double ARCMIN_PER_RAD = 10800.0 / 3.14159265358979311600e+00;
static const double RAD_PER_ARCMIN = 3.14159265358979311600e+00 / 10800.0;

static void gauss_pair(xs256 *g, double *g1, double *g2) {
    const double u1 = 1.0 - xs_unif(g); /* (0, 1] */
    const double u2 = xs_unif(g);
    const double r = sqrt(-2.0 * p_log(u1));
    double s, c;
    p_sincos(2.0 * K_PI * u2 - K_PI, &s, &c); /* angle in [-pi, pi): keeps the reduction short */
    *g1 = r * c;
    *g2 = r * s;
}

static void unif_sphere(xs256 *g, float *ra, float *dec) {
    const double u1 = xs_unif(g), u2 = xs_unif(g);
    double r = 21600.0 * u1;
    float fr = (float)r;
    if (fr >= 21600.0f) fr = 0.0f;
    *ra = fr;
    *dec = (float)(p_asin(2.0 * u2 - 1.0) * ARCMIN_PER_RAD);
}

static void unif_patch(xs256 *g, double patch, float *ra, float *dec) {
    const double u1 = xs_unif(g), u2 = xs_unif(g);
    float fr = (float)(patch * u1), fd = (float)(patch * u2);
    if (fr >= (float)patch) fr = 0.0f;
    if (fd >= (float)patch) fd = 0.0f;
    *ra = fr;
    *dec = fd;
}

/* Offset a clump centre (ra_c, dec_c in radians) by (t1 east, t2 north) radians in its tangent
 * plane, project back to the sphere and return arcminutes with RA wrapped into [0, 21600). */
static void tangent_offset(double ra_c, double dec_c, double t1, double t2, float *ra, float *dec) {
    double sa, ca, sd, cd;
    p_sincos(ra_c, &sa, &ca);
    p_sincos(dec_c, &sd, &cd);
    const double cx = cd * ca, cy = cd * sa, cz = sd;
    const double ex = -sa, ey = ca;                       /* east */
    const double nx = -sd * ca, ny = -sd * sa, nz = cd;   /* north */
    const double vx = cx + t1 * ex + t2 * nx;
    const double vy = cy + t1 * ey + t2 * ny;
    const double vz = cz + t2 * nz;
    double a = p_atan2(vy, vx);
    if (a < 0.0) a += 2.0 * K_PI;
    const double d = p_atan2(vz, sqrt(vx * vx + vy * vy));
    double ra_am = a * ARCMIN_PER_RAD;
    float fr = (float)ra_am;
    if (fr >= 21600.0f) fr = 0.0f;
    *ra = fr;
    *dec = (float)(d * ARCMIN_PER_RAD);
}

/*
 * Fill one D/R catalog pair.
 *   patch_arcmin <= 0 : full sky.  > 0 : RA, Dec in [0, patch) arcmin.
 *   D = n_d / 2 uniform + the rest in n_clumps Gaussian clumps of width sigma_arcmin.
 * Returns 0, or -1 on bad arguments, -2 if a confined clump member needed too many redraws.
 */
int synth_catalogs(int64_t n_d, int64_t n_r, int32_t n_clumps, double sigma_arcmin, double patch_arcmin,
                   uint64_t seed, float *ra_d, float *dec_d, float *ra_r, float *dec_r) {
    if (n_d < 0 || n_r < 0 || n_clumps < 0) return -1;
    xs256 g;
    xs_seed(&g, seed);
    const int patch = patch_arcmin > 0.0;
    for (int64_t k = 0; k < n_r; ++k) {
        if (patch) unif_patch(&g, patch_arcmin, &ra_r[k], &dec_r[k]);
        else unif_sphere(&g, &ra_r[k], &dec_r[k]);
    }
    const int64_t n_unif = (n_clumps > 0) ? n_d / 2 : n_d;
    for (int64_t k = 0; k < n_unif; ++k) {
        if (patch) unif_patch(&g, patch_arcmin, &ra_d[k], &dec_d[k]);
        else unif_sphere(&g, &ra_d[k], &dec_d[k]);
    }
    if (n_unif == n_d) return 0;
    /* clump centres, radians */
    enum { MAXC = 4096 };
    if (n_clumps > MAXC) return -1;
    double cra[MAXC], cdec[MAXC];
    for (int c = 0; c < n_clumps; ++c) {
        float fr, fd;
        if (patch) unif_patch(&g, patch_arcmin, &fr, &fd);
        else unif_sphere(&g, &fr, &fd);
        cra[c] = (double)fr * RAD_PER_ARCMIN;
        cdec[c] = (double)fd * RAD_PER_ARCMIN;
    }
    const double sig = sigma_arcmin * RAD_PER_ARCMIN;
    for (int64_t k = n_unif; k < n_d; ++k) {
        const int c = (int)((k - n_unif) % n_clumps);
        int tries = 0;
        for (;;) {
            double g1, g2;
            gauss_pair(&g, &g1, &g2);
            float fr, fd;
            tangent_offset(cra[c], cdec[c], g1 * sig, g2 * sig, &fr, &fd);
            if (!patch || (fr >= 0.0f && fr < (float)patch_arcmin && fd >= 0.0f && fd < (float)patch_arcmin)) {
                ra_d[k] = fr;
                dec_d[k] = fd;
                break;
            }
            if (++tries > 100000) return -2;
        }
    }
    return 0;
}

/* k distinct indices from [0, n), sorted ascending (Floyd's sampling + insertion into a bitmap). */
int synth_sample_rows(int64_t n, int64_t k, uint64_t seed, int64_t *out, uint8_t *scratch_bitmap /* n bytes */) {
    if (n < 0 || k < 0 || k > n) return -1;
    xs256 g;
    xs_seed(&g, seed ^ 0x5A17E5A17E5A17E5ull);
    memset(scratch_bitmap, 0, (size_t)n);
    for (int64_t j = n - k; j < n; ++j) {
        const int64_t t = (int64_t)(xs_unif(&g) * (double)(j + 1)); /* 0..j */
        const int64_t pick = (t > j) ? j : t;
        if (scratch_bitmap[pick]) scratch_bitmap[j] = 1;
        else scratch_bitmap[pick] = 1;
    }
    int64_t m = 0;
    for (int64_t i = 0; i < n; ++i)
        if (scratch_bitmap[i]) out[m++] = i;
    return (m == k) ? 0 : -3;
}

/* exported so tests can pin the portable elementary functions against libm */
double synth_p_log(double x) { return p_log(x); }
double synth_p_sin(double x) { double s, c; p_sincos(x, &s, &c); return s; }
double synth_p_cos(double x) { double s, c; p_sincos(x, &s, &c); return c; }
double synth_p_atan2(double y, double x) { return p_atan2(y, x); }
double synth_p_asin(double x) { return p_asin(x); }
