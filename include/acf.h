/*
 * acf.h — C ABI of the GB300 angular-correlation library (libacf.so).
 *
 * What it computes ("CUDA Deep Dive: 10B Galaxy Pairs on an RTX 5080", section "The problem"):
 * for galaxies given by right ascension alpha and declination delta in ARCMINUTES, the angular
 * separation of a pair is
 *     theta = arccos( sin d1 sin d2 + cos d1 cos d2 cos(a1 - a2) ),
 * every ordered pair of two catalogs is binned by theta into bins of equal width, giving the
 * histograms DD (real-real), DR (real-random) and RR (random-random), and the Landy-Szalay
 * estimator is omega = (DD - 2 DR + RR) / RR.
 *
 * Binning (Appendix A of the same page, the bin-index helper): bin k holds theta in
 * [k w, (k+1) w); separations beyond nbins * w are clamped into the last bin, so every pair is
 * counted and a histogram always sums to n1 * n2.
 *
 * Precision: the kernels work in fp32 on unit vectors built in fp64. In the default exact mode 2
 * every pair whose fp32 separation falls within its form's worst-case error of a bin edge is
 * re-decided as fp64 would decide it from the same unit vectors (a double-single pass settles all
 * but those within ~1e-13 relative of the edge, which are redone in fp64), so every bin is the one
 * the fp64 formula gives (up to ~1e-15 relative): the histograms equal those of the fp64 definition. Without it (exact
 * modes 0 and 1), a pair can land in a neighbouring bin only if its fp64 theta lies near that edge:
 * the worst-case error (every rounding aligned) is 6e-7 rad for the dot form used between 55 and
 * 125 degrees, 1.05e-6 for the chord form below 72 degrees and 1.25e-6 near 90 degrees for the
 * full-range chord form; the largest measured on millions of test pairs is 2.4e-7.
 *
 * Conventions for every entry point:
 *   - Array arguments marked "device" are caller-owned CUDA device pointers on the context's
 *     device. The library never frees them and never keeps them after the call returns.
 *   - Work is enqueued on the context's stream and is asynchronous unless stated otherwise;
 *     synchronise that stream before reading outputs. Calls on one context must be ordered on
 *     that stream (the context owns one workspace that consecutive calls reuse).
 *   - Every function returns ACF_OK (0) or a negative ACF_ERR_* code and never exits the
 *     process. acf_last_error() gives a message for the last failure on that context.
 *     Launch errors are detected at once; faults inside a kernel surface on a later call or sync.
 *   - Non-finite RA/Dec inputs are treated as (0, 0) so no kernel can index out of bounds; their
 *     pairs are therefore binned as if the galaxy sat at RA = Dec = 0.
 */
#ifndef ACF_H
#define ACF_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ACF_OK 0
#define ACF_ERR_ARG (-1)         /* NULL pointer where data is required, n < 0, nbins <= 0, bad width */
#define ACF_ERR_UNSUPPORTED (-2) /* histogram too large for the shared-memory plan (see acf_histogram) */
#define ACF_ERR_NOMEM (-3)       /* device or pinned host allocation failed */
#define ACF_ERR_CUDA (-4)        /* a CUDA runtime call or kernel launch failed */

typedef struct acf_ctx acf_ctx;

/* Library version string, e.g. "acf 0.1 sm_103a". Static storage. */
const char *acf_version(void);

/*
 * Create a context on CUDA device `device` that enqueues work on `cuda_stream` (a cudaStream_t;
 * NULL means the legacy default stream). The context owns a device workspace that grows on
 * demand and is freed by acf_destroy. *out receives the handle (NULL on failure).
 */
int acf_create(acf_ctx **out, int device, void *cuda_stream);

/* Free the context and its workspace (synchronises its stream first). NULL is a no-op. */
void acf_destroy(acf_ctx *ctx);

/* Message describing the last failure on this context ("" if none). Valid until the next call. */
const char *acf_last_error(const acf_ctx *ctx);

/* Switch the context to another stream. Synchronises the old stream first. */
int acf_set_stream(acf_ctx *ctx, void *cuda_stream);

/*
 * One histogram of angular separations (the DD, DR or RR of section "The problem").
 *
 *   ra, dec      device float[n]  first catalog, arcminutes
 *   ra2, dec2    device float[n2] second catalog, arcminutes; pass NULL/NULL (n2 ignored), or the
 *                same pointers and n2 == n, for an auto-correlation (DD or RR)
 *   bin_width_deg  bin width w in degrees, finite and > 0
 *   nbins        number of bins, > 0
 *   out          device uint64[nbins], OVERWRITTEN with the counts
 *
 * Cross-correlation counts all n * n2 ordered pairs. Auto-correlation counts all n^2 ordered
 * pairs: each unordered pair i != j is evaluated once and counted twice, and the n self-pairs
 * (theta = 0) are added to bin 0, as in the symmetric scheme of the page's section "L1: DD/RR
 * symmetry". Either way sum(out) == n * n2 exactly.
 * n == 0 or n2 == 0 gives an all-zero histogram. Returns ACF_ERR_UNSUPPORTED when the
 * per-block shared-memory histogram does not fit: that needs min(nbins, 180/w + 1) <= 49152
 * (or, when 180/w is an integer, 180/w + 2 <= 49152).
 */
int acf_histogram(acf_ctx *ctx, const float *ra, const float *dec, int64_t n, const float *ra2, const float *dec2,
                  int64_t n2, double bin_width_deg, int32_t nbins, uint64_t *out);

/*
 * acf_histogram without any device allocation. The page has no counterpart: this is a service of
 * this library for callers that cannot call cudaMalloc, such as code whose process hands all
 * device memory to another allocator (a framework's caching allocator) or latency-critical code
 * that cannot afford the implicit device synchronisation and driver work of an allocation.
 *
 * Same arguments, semantics and results as acf_histogram, but its scratch (sorted unit vectors,
 * caps, block rows, counters, the exact-mode queue) lives in one file-scope device array of 16 MiB that the library
 * reserves on every GPU that loads it, until the process exits. It calls no cudaMalloc, cudaFree
 * or other allocating routine.
 *   - Limit: about 77 bytes per galaxy of each catalog + ((blocks + 2) * nbins * 8) bytes must fit
 *     in 16 MiB, blocks being the persistent grid (one per SM: 152 on a GB300); larger requests
 *     return ACF_ERR_UNSUPPORTED with the sizes in the message. Two 100k catalogs at 720 bins need
 *     ~16.3 MB. In exact mode the rest of the array holds the queue of pairs to re-decide.
 *     Exact results need a queue that holds one launch's flagged pairs: catalogs of a few tens of
 *     thousands of galaxies at 0.25 degree bins. When the queue overflows (the "exact_overflow"
 *     info key is then > 0; e.g. two 60k catalogs), the pairs that did not fit keep their fp32 bin:
 *     the rule that a pair moves to a neighbouring bin only within 1e-6 rad of its edge is then met
 *     in practice (largest measured error 2.4e-7 rad) but not proven (worst-case bounds up to
 *     1.25e-6 rad), sums stay exact, and because which pairs fit depends on the order in which
 *     blocks fill the queue, such results can differ from run to run.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress);
 *     make that first call before any stream capture. The address is looked up again when the
 *     device's context has changed (e.g. after cudaDeviceReset).
 *   - Every call on a device shares the one array, which keeps the last call's contents; the
 *     kernels re-initialise everything they read. Calls whose work overlaps on the GPU (other
 *     streams, other host threads or contexts) race on it and must be serialised by the caller.
 */
int acf_histogram_noalloc(acf_ctx *ctx, const float *ra, const float *dec, int64_t n, const float *ra2,
                          const float *dec2, int64_t n2, double bin_width_deg, int32_t nbins, uint64_t *out);

/*
 * Landy-Szalay estimator per bin (section "The problem"), computed in fp64 on the device:
 *     omega_k = (DD_k/N_dd - 2 DR_k/N_dr + RR_k/N_rr) / (RR_k/N_rr),
 * N_dd = n_d^2, N_dr = n_d n_r, N_rr = n_r^2 (with n_d == n_r this is (DD - 2DR + RR)/RR).
 * Bins with RR_k = 0 get NaN (the page writes only bins with RR > 0).
 *   dd, dr, rr   device uint64[nbins]
 *   n_d, n_r     catalog sizes, > 0
 *   omega        device double[nbins], overwritten
 */
int acf_omega(acf_ctx *ctx, const uint64_t *dd, const uint64_t *dr, const uint64_t *rr, int32_t nbins, int64_t n_d,
              int64_t n_r, double *omega);

/*
 * The whole job on the device (section "The problem"): DD of the data catalog, DR, RR of the
 * random catalog, and omega. Each catalog is sorted and converted once for the three histograms,
 * so this costs less than three acf_histogram calls plus acf_omega, with the same results.
 *   ra_d, dec_d  device float[n_d];  ra_r, dec_r  device float[n_r]  (arcminutes)
 *   dd, dr, rr   device uint64[nbins], overwritten;  omega  device double[nbins], overwritten
 * Same binning rules as acf_histogram; n_d and n_r must be > 0. Asynchronous on the context's
 * stream. Afterwards the acf_get_info counters describe the last histogram of the three (RR).
 */
int acf_correlate(acf_ctx *ctx, const float *ra_d, const float *dec_d, int64_t n_d, const float *ra_r,
                  const float *dec_r, int64_t n_r, double bin_width_deg, int32_t nbins, uint64_t *dd, uint64_t *dr,
                  uint64_t *rr, double *omega);

/*
 * The whole job from HOST memory: copies the two catalogs to the device, runs acf_correlate,
 * copies the four results back and synchronises the stream before returning.
 *   ra_d, dec_d  host float[n_d];  ra_r, dec_r  host float[n_r]  (arcminutes; pinned memory
 *                gives asynchronous copies, pageable memory works too)
 *   dd, dr, rr   host uint64[nbins], overwritten;  omega  host double[nbins], overwritten
 * Same binning rules as acf_histogram; n_d and n_r must be > 0.
 */
int acf_correlate_host(acf_ctx *ctx, const float *ra_d, const float *dec_d, int64_t n_d, const float *ra_r,
                       const float *dec_r, int64_t n_r, double bin_width_deg, int32_t nbins, uint64_t *dd,
                       uint64_t *dr, uint64_t *rr, double *omega);

/*
 * Diagnostic: the bin that the histogram kernels assign to each of n individual pairs
 * (ra1[k], dec1[k]) - (ra2[k], dec2[k]), computed by the same device code path.
 *   ra1, dec1, ra2, dec2  device float[n];  bins  device int32[n], overwritten
 */
int acf_pair_bins(acf_ctx *ctx, const float *ra1, const float *dec1, const float *ra2, const float *dec2, int64_t n,
                  double bin_width_deg, int32_t nbins, int32_t *bins);

/*
 * Tuning and measurement switches (all optional). Keys:
 *   "threads"        threads per block of the pair kernel: 512 or 1024 (default: 1024 when the
 *                    shared-memory plan allows)
 *   "ctas_per_sm"    resident blocks per SM to launch (default: occupancy maximum)
 *   "bin_method"     0 = chord + arcsin^2 polynomial (default, meets the precision contract);
 *                    1 = dot product + acosf (the page's exact-acos form; measured alternative,
 *                        does NOT meet the precision contract at small or near-180 separations);
 *                    2 = dot product + the arccos polynomial of Abramowitz and Stegun 4.4.45 (the
 *                        approximate mode: error up to 6.7e-5 rad, so many pairs near edges move;
 *                        sums stay exact). Methods 1 and 2 take no exact mode and no range forms.
 *   "layout"         0 = automatic, 1 = lane-private copies, 2 = one block-shared histogram,
 *                    3 = two block-shared copies of 16-bit counters (only in a library built with
 *                        -DACF_U16_HIST=1, and only with "exact" 0; ACF_ERR_UNSUPPORTED otherwise)
 *   "exact"          0 = fp32 bins only (precision contract above);
 *                    1 = re-decide in fp64 the pairs within ~1e-6 rad of an edge whose separation is
 *                        below "exact_below_deg" or above 180 minus it;
 *                    2 = re-decide such pairs at every separation: the histograms then equal those
 *                        of the fp64 formula (default)
 *   "exact_below_deg"  the window of mode 1, whole degrees 0..180 (default 20)
 *   "range_forms"    1 = where the caps of a block of pairs bound its separations, use a cheaper
 *                        form that meets the same precision contract: the dot product with an
 *                        asin polynomial between 55 and 125 degrees (needs 180/w an even integer),
 *                        a degree-5 chord polynomial where theta' stays below 72 degrees (default);
 *                    0 = the full-range chord form for every pair (every pair then gets the same
 *                        code whichever block computes it, so DD of a union splits exactly)
 *   "pair_bins_form" acf_pair_bins: 0 = full-range chord form (default); 1 = the form a tightly
 *                    bounded block would use for that pair's own dot product
 *   "units_per_launch"  cap on work units (128 x 128 pairs) per pair-kernel launch; 0 = automatic
 *                    (large problems are always split so that no 32-bit shared counter can wrap)
 *   "unit_groups"    j-groups of 32 galaxies per work unit: 0 = automatic (default: 1 when the
 *                    problem has fewer than two 128 x 128 chunk pairs per resident warp), 4 = a
 *                    whole chunk pair, 1 = one j-group (lane-private layout, 1024 threads and the
 *                    chord method only; otherwise 4)
 *   "exact_queue"    records of the exact-mode queue (one per warp i-set and j holding a flagged
 *                    pair): 0 = automatic (default: enough for one launch at twice the worst-case flag
 *                    rate), else exactly this many, up to 2^28. A smaller queue can overflow; its
 *                    pairs then keep their fp32 bins (see "exact_overflow"). Plans with one
 *                    block-shared histogram in exact mode 2 keep their flags in group records
 *                    instead (a slot for every lane and j-group of a launch, so they never
 *                    overflow) and ignore this option.
 *   "kernel_timing"  1 = bracket every pair-kernel launch with CUDA events (see acf_kernel_times);
 *                    2 = bracket every exact-mode fix-up launch instead; 0 = off (default)
 *   "graphs"         1 = an acf_correlate or acf_histogram call that repeats an earlier one (the
 *                    same pointers, sizes, binning, options, stream and workspace) replays a CUDA
 *                    graph of its launches: captured the second time the call comes (its kernels
 *                    run from the graph), launched as one graph from then on; the four most
 *                    recent such calls are kept (default). acf_correlate_host does the same, its
 *                    copies included, when every host buffer is page-locked. The results, and
 *                    what acf_get_info reports, are those of the call; the inputs' current
 *                    contents are read.
 *                    With "kernel_timing" on, every launch the graph holds is timed as if it had
 *                    been launched by itself. Calls go launch by launch while
 *                    "inject_launch_error" is set, on the legacy default stream (NULL), and while
 *                    the caller captures the context's stream. 0 = every call launches its
 *                    kernels one by one
 *   "workspace_limit"  bytes the context's device workspaces may grow to; a call that needs more
 *                    returns ACF_ERR_NOMEM and leaves the context usable (0 = no limit, default)
 *   "inject_launch_error"  fault injection for tests, on the host only: the n-th kernel launch from
 *                    now on is reported as failed (ACF_ERR_CUDA, "injected" in the message) and the
 *                    call returns at once; the launch itself ran normally, the device is untouched,
 *                    and the next call works as usual (0 = off, default; it resets after firing)
 * Unknown keys and out-of-range values return ACF_ERR_ARG and leave the option unchanged.
 */
int acf_set_option(acf_ctx *ctx, const char *key, int64_t value);

/*
 * The plan acf_histogram would make for a binning, with default options and the given exact mode
 * (0, 1 or 2), worked out on the host alone: no context, no device, no CUDA call. Writes
 * ACF_PLAN_INFO_FIELDS values to info: [0] bin map (0 direct: 180/w an integer; 1 clamp),
 * [1] histogram entries, [2] layout (1 lane-private copies, 2 one block-shared histogram),
 * [3] pair-kernel threads per block, [4] its dynamic shared memory in bytes, [5] [6] [7] the fine
 * bits S of the exact-mode window for the full-range chord, the short chord and the dot form (0
 * without exact mode), [8] dot form on, [9] short chord on, [10] the last bin index a separation
 * up to 180 degrees reaches, [11] the exact mode the method allows.
 * Returns ACF_ERR_ARG (bad width, nbins <= 0, info NULL, exact outside 0..2) or
 * ACF_ERR_UNSUPPORTED (a histogram larger than the shared memory holds) like acf_histogram.
 */
#define ACF_PLAN_INFO_FIELDS 12
int acf_plan_info(double bin_width_deg, int32_t nbins, int32_t exact, int64_t *info);

/*
 * Read back facts about the last acf_histogram call. Keys: "grid", "threads", "ctas_per_sm",
 * "units", "layout", "bin_map" (0 mirror, 1 clamp), "hist_entries", "smem_bytes",
 * "pairs_evaluated", "launches" (pair-kernel launches the call was split into),
 * "kernel_launches" (kernels this context has launched since acf_create, all entry points; a
 * graph replay counts the kernels in the graph), "graph_replays" (calls served by a graph, see
 * the option "graphs"),
 * "unit_groups" (4: units of a 128 x 128 chunk pair; 1: of one 32-galaxy j-group).
 * These keys synchronise the context's stream and read device counters of the last call:
 *   "pairs_fixed", "pairs_general"  pairs evaluated on the fixed-sign and general loops
 *   "pairs_fixed_exact", "pairs_general_exact"  the same loops with edge flagging (exact mode)
 *   "pairs_masked"                  pairs of diagonal or ragged units (one compare per pair more)
 *   "pairs_mid", "pairs_mid_exact"  the dot form (55..125 degrees), without and with flagging
 *   "pairs_small", "pairs_small_exact"  the degree-5 chord form, without and with flagging
 *   "exact_flagged"  pairs flagged for re-decision;  "exact_moved"  of those, pairs moved a bin;
 *   "exact_overflow"  flagged pairs whose record did not fit in the queue (kept their fp32 bin)
 *   "exact_redone_fp64"  flagged pairs the double-single first pass of the re-decision could not
 *                    settle (within ~1e-13 relative of an edge), decided again in fp64
 * Unknown keys return ACF_ERR_ARG.
 */
int acf_get_info(const acf_ctx *ctx, const char *key, int64_t *value);

/*
 * With "kernel_timing" on: synchronise, write up to `cap` per-launch durations of the pair
 * kernel (option value 1) or of the exact-mode fix-up (value 2) (milliseconds, CUDA events on the
 * context stream) recorded since the last call into ms[], set *count, and clear the record. At
 * most 4096 launches are kept.
 */
int acf_kernel_times(acf_ctx *ctx, float *ms, int32_t cap, int32_t *count);

/*
 * Catalog files and the result table, in the formats of the page's program (sections "mmap +
 * hand-rolled parser vs. fscanf" and its output step). Host code; no context, no GPU needed.
 *
 * acf_read_catalog: read an ASCII catalog (the galaxy count, then that many "ra dec" pairs in
 * arcminutes, separated by any whitespace). On success *ra and *dec receive malloc'ed host arrays
 * of *n floats (free them with acf_free_catalog). Numbers are parsed with correct rounding to
 * float. A missing file, a bad count or fewer pairs than the count give ACF_ERR_ARG with a message
 * (line number) in err[err_len] (nullable); nothing is allocated then.
 */
int acf_read_catalog(const char *path, float **ra, float **dec, int64_t *n, char *err, int32_t err_len);
void acf_free_catalog(float *ra, float *dec);

/*
 * acf_write_omega: write the result table: a header line, then for every bin k with rr[k] > 0 one
 * tab-separated row "bin start (degrees, k * bin_width_deg, %6.3f)  omega (%15f)  DD  DR  RR".
 * Host arrays of nbins values. ACF_ERR_ARG if an argument is invalid or the file cannot be
 * written.
 */
int acf_write_omega(const char *path, const uint64_t *dd, const uint64_t *dr, const uint64_t *rr,
                    const double *omega, int32_t nbins, double bin_width_deg);

/*
 * The optimisation ladder of the page (section "The ladder", levels 0 to 5: one thread per pair;
 * + DD/RR symmetry; + per-galaxy sin/cos; + shared-memory j-tiles; + arccos polynomial; + unroll,
 * launch bounds and whole-block diagonal skip), rebuilt for this GPU as a measurement of each step.
 * Not the library's path: fp32 acos misbins near-edge pairs, level 4 and 5 by design; totals stay
 * exact. Levels 1 to 3 give identical histograms, as do 4 and 5.
 *   level        0..5
 *   ra_d, dec_d, ra_r, dec_r  device float[n] (arcminutes), both catalogs of the same size n
 *   dd, dr, rr   device uint64[nbins], overwritten;  nbins <= 4000
 *   stream       cudaStream_t (NULL: legacy default stream)
 *   kernel_ms    (nullable) host: the histogram kernel's time from CUDA events
 * Synchronous (waits for its stream). Allocates a small scratch buffer (stream-ordered).
 */
int acf_ladder(int level, const float *ra_d, const float *dec_d, const float *ra_r, const float *dec_r, int64_t n,
               double bin_width_deg, int32_t nbins, uint64_t *dd, uint64_t *dr, uint64_t *rr, void *stream,
               float *kernel_ms);

/*
 * Measure the FP32 issue ceiling of this GPU, the denominator of the pair kernel's roofline
 * (independent FMA chains, the method of the "roofline.cu" page's compute ceiling): one timed
 * launch of 2 blocks of 1024 threads per SM, each thread running 8 independent fmaf chains
 * x = x * 0.9999999f + 1e-7f for `iters` iterations from x = tid * 1e-3f + c (c = chain index).
 * Synchronous. *ffma_per_s receives FMA thread-instructions per second; thread0 (nullable, host)
 * receives thread 0's sum of its chains (c = 0..7 in order) so a caller can replay it on the host.
 * Allocates a small device buffer (stream-ordered) for the results.
 */
int acf_fp32_peak(acf_ctx *ctx, int64_t iters, double *ffma_per_s, float *thread0);

#ifdef __cplusplus
}
#endif

#endif /* ACF_H */
