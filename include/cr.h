/*
 * cr.h -- C ABI of the GB300 conditional-simulation library (libcr.so).
 *
 * The library computes the hot path of "Mixed-Precision GPU Acceleration for Confidence
 * Regions of Spatial Excursion Sets" (Zhang, Abdulah, Cao, French, Alomairy, Genton,
 * Keyes): a dense covariance over n locations, a tile Cholesky factor with per-tile
 * FP64/FP32/FP16 precision chosen from a tolerance, the mixed-precision triangular
 * multiply that turns standard-normal draws into correlated fields, the universal-kriging
 * correction, per-location exceedance counts and the calibration of the inner and outer
 * confidence regions.  One process drives one GPU; nothing here is distributed.
 *
 * Conventions (all entry points):
 *  - Every call returns a cr_status; CR_OK = 0.  No exception or abort crosses the ABI.
 *    cr_status_str() names a code, cr_last_error_detail() gives the calling thread's last
 *    message.
 *  - Pointers named d_* are device pointers (allocated and owned by the caller, e.g. by
 *    PyTorch); h_* are host pointers owned by the caller.  The library owns only the
 *    storage behind an opaque cr_tilemat handle (cr_tilemat_create / cr_tilemat_destroy).
 *  - Matrices passed as pointers are column-major with an explicit leading dimension
 *    (LAPACK style) unless stated otherwise.  Sizes are element counts.
 *  - Device work is enqueued on the given stream and is asynchronous, except where a
 *    call returns host values; those calls synchronise the stream and say so.
 *  - Sizes out of range, NULL where a pointer is required, or calls in the wrong order
 *    return CR_ERR_ARG or CR_ERR_STATE without touching the GPU.
 */
#ifndef CR_H
#define CR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* cr_stream;

typedef int cr_status;
enum {
  CR_OK = 0,
  CR_ERR_ARG = 1,             /* invalid argument */
  CR_ERR_CUDA = 2,            /* a CUDA runtime/driver call failed */
  CR_ERR_NOMEM = 3,           /* device allocation inside a tile matrix failed */
  CR_ERR_NOT_SPD = 4,         /* a Cholesky pivot was not positive (see info) */
  CR_ERR_EMPTY_SAMPLE = 5,    /* every simulation left the psi or phi set empty */
  CR_ERR_NONPOS_MSPE = 6,     /* a pointwise MSPE v_i <= 0 */
  CR_ERR_TIMEOUT = 7,         /* a bounded device-side wait gave up */
  CR_ERR_STATE = 8,           /* call made in the wrong order */
  CR_ERR_NOT_IMPLEMENTED = 9,
  CR_ERR_RANGE = 10           /* scaled factor not representable in FP16 */
};

/* Tile precision classes. */
enum { CR_PREC_FP64 = 0, CR_PREC_FP32 = 1, CR_PREC_FP16 = 2 };

/* Covariance families.
 *  CR_COV_MATERN: C(h) = sigma2 2^(1-nu)/Gamma(nu) (h/range)^nu K_nu(h/range), C(0) = sigma2
 *                 (the page's Matern model, Section VI-C; parameterisation as stated here).
 *  CR_COV_POWEXP: C(h) = sigma2 exp(-(h/range)^nu) (Section VI-B.2). */
enum { CR_COV_MATERN = 0, CR_COV_POWEXP = 1 };

typedef struct {
  int family;       /* CR_COV_MATERN or CR_COV_POWEXP */
  double sigma2;    /* marginal variance (theta0) */
  double range;     /* beta > 0 */
  double nu;        /* smoothness > 0 */
  double nugget;    /* added to every diagonal entry (>= 0) */
  int n_pred;       /* rows [0, n_pred) are prediction sites, [n_pred, n) observations */
  double tau2;      /* measurement-error variance, observation diagonal only (Eq.4) */
} cr_cov_params;

/* Result of the precision policy (Section V-D, V-E). */
typedef struct {
  double fixedacc;  /* tolerance used for the final map */
  int iters;        /* maps computed (automatic refinement, Section V-D) */
  int n_fp64, n_fp32, n_fp16;   /* lower tiles per class */
  double R_hp;      /* Eq.10 ratio v_max^HP / v_min^HP (NaN without FP16 tiles) */
  double rho1, rho2;/* Eq.11 ratios */
  int check1, check2;           /* Eq.10 / Eq.11 passed */
  double ell, u_s;  /* Eq.12 bounds */
  double s;         /* applied integer scale (1 = unscaled) */
  int range_ok;     /* ell <= u_s */
} cr_pmap_info;

typedef struct {
  double q_in, q_out;   /* critical values (Section V-C) */
  int n_psi, n_phi;     /* sample sizes after dropping empty-set sentinels */
} cr_calib_info;

typedef struct cr_tilemat_s* cr_tilemat;

/* ---------------------------------------------------------------- housekeeping */
const char* cr_status_str(cr_status code);
const char* cr_last_error_detail(void);
cr_status cr_version(int* major, int* minor);

/* Number of CUDA kernels this library has launched in the process so far (all devices);
 * *count receives the running total.  Host-side counter, no device work. */
cr_status cr_kernel_launches(uint64_t* count);

/* Hands back to the driver the device memory that the library keeps in its stream-ordered
 * scratch pools (one per device).  The conditioning correction takes its scratch from these
 * pools and frees it at the end of each call; the pools keep the freed memory for the next
 * call rather than return it at every synchronisation.  The largest user is the Ozaki
 * product (CR_GEMM_OZAKI): 16 n_o' (n_p + M_b) bytes of slices (n_o' = n_o rounded up to
 * whole chunks of at most 4096 rows, by less than 128 rows per chunk; M_b the columns of one
 * block, all M unless a level's chunk products for all M would exceed 2 GiB), 2 GiB of chunk
 * products at most (one chunk's 4 n_p M_b bytes when that is more), 8 n_p M_b bytes of
 * accumulator, 8 n_o M bytes for R, and S (8 n_p M) in cr_correct_calibrate;
 * cr_krige_correct with CR_GEMM_DF takes 8 n_o (n_p + M) bytes.  Memory still used by work in flight stays in the pool.  No device
 * work; does not synchronise. */
cr_status cr_workspace_trim(void);

/* Device timing of the library's main kernels, for measurement (the paper has no counterpart).
 * While enabled, every launch of a timed kernel is bracketed by two CUDA events recorded on
 * the stream the kernel is launched on, and the durations are accumulated per kernel name:
 *   "k_diag_chol", "k_diag_chol_df"   factor and inverse of one diagonal tile (FP64 / double-float)
 *   "k_split_diag_df"   the double-float executor's results to their storage formats
 *   "k_tc_old", "k_tc_new", "k_tc_trsm", "k_tc_trmm"   tensor-core kernel by mode
 *   "k_cov_stats", "k_cov_stats_refine", "k_generate"   covariance statistics, tile generation
 *   "k_corr", "k_corr_scan"   double-float correction product (plain / fused with the scan)
 *   "k_oz_slice", "oz_gemm", "k_oz_accum"   Ozaki product: operand slicing, the slice GEMMs of
 *                   one level (cuBLAS), the exact accumulation of one level
 *   "k_scan"        calibration scan
 * cr_timing_enable(on) switches recording on (1) or off (0); it does not clear the totals.
 * cr_timing_read(name, &ms, &n) synchronises the device, folds every recorded launch into the
 * totals and returns the total milliseconds and launch count of `name` (0 if never timed).
 * cr_timing_reset() clears all totals.  cr_timing_enable(1) creates a pool of 16384 events
 * (8192 timed launches between two reads); launches beyond the pool are not timed. */
cr_status cr_timing_enable(int on);
cr_status cr_timing_read(const char* kernel, double* total_ms, uint64_t* launches);
cr_status cr_timing_reset(void);

/* Process-wide options (the paper has no counterpart: they control how this library runs
 * the method, not what it computes).  They apply to calls made after the change.
 *  CR_OPT_WAIT_LIMIT_US  wall-clock limit of every bounded device-side wait of the
 *                        factorisation's diagonal executor, in microseconds (default 2000000,
 *                        range [0, 600000000]).  A wait that runs out makes the factorisation
 *                        return CR_ERR_TIMEOUT; the tile matrix stays usable and the next
 *                        cr_potrf_adaptive starts from a clean state.
 *  CR_OPT_DIAG_ARITH     arithmetic of the FP64 diagonal tiles (Section IV-B keeps them FP64):
 *                        CR_DIAG_FP64 on the FP64 units; CR_DIAG_DF as double-float pairs of
 *                        FP32 numbers on the FP32 units (an FP64 emulation with about 48
 *                        significant bits, several times faster on GB300, whose FP64 units
 *                        issue 1/64 of the FP32 lanes per cycle); CR_DIAG_AUTO (default):
 *                        double-float for adaptive factorisations (amp != 0), FP64 for
 *                        all-FP64 ones (amp = 0, including cr_krige's Sigma_y).
 *  CR_OPT_FP64_GEMM      arithmetic of the FP64-class products of the conditioning correction
 *                        (cr_krige_correct, cr_correct_calibrate) and of cr_krige's triangular
 *                        solves with many right-hand sides: CR_GEMM_DF (default) double-float
 *                        on the FP32 units for the correction and FP64 for the solves;
 *                        CR_GEMM_OZAKI the Ozaki scheme on the FP16 tensor cores (Ozaki, Ogita,
 *                        Oishi, Rump, Numer. Algorithms 59, 2012): each operand column cut into
 *                        S slices of 6 bits below a power of two (S = 8 for the correction,
 *                        9 for the solves), the slice products with s + t <= S + 1 computed
 *                        exactly (FP16 inputs, FP32 accumulation over chunks of at most 4096
 *                        rows), one GEMM per level of significance, and summed in double-float.
 *                        With it cr_correct_calibrate writes S to pooled scratch, and cr_krige
 *                        holds two dense n_o x n_o copies of the factor during its solves.
 * cr_set_option returns CR_ERR_ARG for an unknown option or a value out of range. */
enum { CR_OPT_WAIT_LIMIT_US = 1, CR_OPT_DIAG_ARITH = 2, CR_OPT_FP64_GEMM = 4 };
enum { CR_DIAG_AUTO = 0, CR_DIAG_FP64 = 1, CR_DIAG_DF = 2 };
enum { CR_GEMM_DF = 0, CR_GEMM_OZAKI = 1 };
cr_status cr_set_option(int option, long long value);
cr_status cr_get_option(int option, long long* value);

/* Throughput probe of one arithmetic unit, for the roofline denominators of measurements (the
 * paper has no counterpart).  Runs a kernel of iters iterations of independent dependency
 * chains on every SM (8 CTAs of 256 threads per SM), after one warm-up launch, and returns its
 * rate in TFLOP/s (an FMA or MMA multiply-add counts 2 flops per product term):
 *   CR_PEAK_DFMA    FP64 FMA on the FP64 units
 *   CR_PEAK_FFMA    FP32 FMA
 *   CR_PEAK_DF_MAC  the double-float multiply-accumulate of the diagonal executor (an emulated
 *                   FP64 FMA: 2 flops per accumulate, about 12 FP32 instructions)
 *   CR_PEAK_DMMA    FP64 tensor-core MMA (mma.sync m8n8k4)
 * iters in [1, 2^24]; a few thousand give a launch of some milliseconds.  Synchronises. */
enum { CR_PEAK_DFMA = 1, CR_PEAK_FFMA = 2, CR_PEAK_DF_MAC = 3, CR_PEAK_DMMA = 4 };
cr_status cr_peak_probe(int kind, int iters, double* tflops, cr_stream stream);

/* A symmetric n x n matrix stored as its lower tiles (i >= j) of nb x nb entries.
 * NT = ceil(n / nb) tile rows; rows and columns past n are padding and behave like the
 * identity.  nb must be a multiple of 128 with 128 <= nb <= 1024.  The handle owns its
 * device storage (allocated on the current device); destroy frees it. */
cr_status cr_tilemat_create(int n, int nb, cr_tilemat* out);
cr_status cr_tilemat_destroy(cr_tilemat V);
cr_status cr_tilemat_info(cr_tilemat V, int* n, int* nb, int* nt);

/* Spatial ordering of the sites (host only, no device work): h_perm (n int32, caller-owned)
 * receives the permutation that puts the n locations h_xy (row-major pairs (x_i, y_i),
 * FP64, host) in Z-order, so that h_xy[h_perm[0]], h_xy[h_perm[1]], ... are the sorted
 * sites.  The pages do not state an ordering, but their precision maps (Section VI-D,
 * Fig. 5) are banded, which needs nearby sites in nearby tiles: without an ordering,
 * uniformly scattered sites give no FP16-class tile at any tolerance.  Each coordinate is
 * quantised to q = clamp(floor(65536 x), 0, 65535), the key interleaves the bits of q_x
 * (even positions) and q_y (odd positions), and equal keys keep their input order (stable
 * sort).  Callers order the prediction block and the observation block separately, so that
 * the block structure of Eq.4 (prediction sites first) is kept, and pass the permuted sites
 * to cr_cov_build.  Returns CR_ERR_ARG for n < 0, a NULL pointer with n > 0, or a NaN
 * coordinate. */
cr_status cr_morton_order(const double* h_xy, int n, int32_t* h_perm);

/* Joint covariance (Section V Eq.4) of the n locations d_xy (n x 2, row-major pairs
 * (x_i, y_i), device, FP64; copied, so the caller may free it afterwards), prediction sites
 * first.  Computes the per-tile statistics (Frobenius norm, min and max entry over valid
 * entries, Section V-D) in one pass without storing the matrix: the tiles are generated
 * in their precision classes by cr_potrf_adaptive, and cr_tilemat_to_dense / cr_krige
 * evaluate V in FP64 on demand.  For Matern nu in {1/2, 3/2, 5/2} the diagonal tiles'
 * statistics are evaluated in double-float arithmetic (as for cr_tile_stats) and the
 * off-diagonal tiles' in FP32 with a rigorous relative error bound (cr_tile_stats_records);
 * cr_precision_map and cr_tile_stats recompute exactly the records they need.  Other
 * covariances: every tile exact.  Asynchronous. */
cr_status cr_cov_build(cr_tilemat V, const double* d_xy, const cr_cov_params* p, cr_stream stream);

/* Per-tile statistics as NT x NT row-major host arrays (lower part filled), each exact
 * (double-float: about 1e-14 relative, up to ~3e-13 where entries sit at scaled distances
 * near 80, beyond which FP64 takes over): tiles that still hold fast-pass records (below)
 * are recomputed
 * first.  Synchronises the stream used by cr_cov_build.  Any output pointer may be NULL. */
cr_status cr_tile_stats(cr_tilemat V, double* h_frob, double* h_vmin, double* h_vmax);

/* The statistics records as they stand, without recomputing any (same layout as
 * cr_tile_stats), with h_err the relative bound of each record: 0 for an exact one, E > 0
 * for a record of the fast FP32 pass (|record - exact| <= E |exact| for the Frobenius norm,
 * the min and the max; the pass covers the off-diagonal tiles of the closed-form Matern
 * orders, and cr_precision_map recomputes exactly the ones its decisions depend on), or
 * +infinity where no bound holds.  Synchronises like cr_tile_stats. */
cr_status cr_tile_stats_records(cr_tilemat V, double* h_frob, double* h_vmin, double* h_vmax, double* h_err);

/* Tile precision map, FP16 screening checks and covariance scale (Section V-D/E, Alg.2
 * steps 7-10).  amp = 0 keeps every tile FP64 with s = 1.  With auto_mode != 0 the
 * tolerance starts at 1e-4 and shrinks by 0.9 until both checks pass or no FP16 tile is
 * left; otherwise fixedacc is used as given and failed checks are only reported.
 * h_map (NT x NT int8 row-major, lower part written, may be NULL) receives CR_PREC_*.
 * Allocates the per-precision tile storage.  Synchronises. */
cr_status cr_precision_map(cr_tilemat V, int amp, double fixedacc, int auto_mode,
                           int8_t* h_map, cr_pmap_info* info);

/* Adaptive mixed-precision Cholesky (Section IV-B, Alg.2 step 12): scales the tiles by
 * s^2, rounds each to its class, and factors in place, V <- L_s = chol(s^2 V).  FP64
 * tiles run on the FP64 units; FP32/FP16 products on the tensor cores with FP32
 * accumulation.  The diagonal tiles are factored (with their inverses, which turn the
 * off-diagonal triangular solves into products) by an on-device dataflow executor, in FP64
 * or in double-float arithmetic (CR_OPT_DIAG_ARITH).  *info = 0 on success, else the 1-based
 * global column of the first non-positive pivot (LAPACK convention) and CR_ERR_NOT_SPD;
 * CR_ERR_TIMEOUT if a bounded device wait ran out (CR_OPT_WAIT_LIMIT_US).  Synchronises. */
cr_status cr_potrf_adaptive(cr_tilemat V, cr_stream stream, int* info);

/* Copies the tile matrix into a dense n x n column-major FP64 matrix (lower triangle;
 * the strict upper triangle is set to zero).  what = 0: the covariance V built by
 * cr_cov_build; what = 1: the current working tiles as stored in their precision
 * (after cr_potrf_adaptive: the factor L_s); what = 2: first runs the generation step of
 * cr_potrf_adaptive alone (Alg.2 step 12: the tiles of s^2 V written in their precision
 * classes, diagonal tiles as cr_potrf_adaptive would generate them), then copies as for
 * what = 1; it replaces any factor (factor again before cr_trmm_sim) and synchronises.
 * what = 1 and 2 need cr_precision_map first.  Asynchronous for what = 0 and 1. */
cr_status cr_tilemat_to_dense(cr_tilemat V, int what, double* d_out, int ld, cr_stream stream);

/* n x M standard normals (column-major, ldz >= n) from the library's counter-based
 * stream: SplitMix64 on seed + (c+1)*0x9E3779B97F4A7C15, 53-bit uniforms, Box-Muller in
 * FP64; element (i, j) uses pair floor((offset + j n + i) / 2) (Section V-B, Desc_rnorm).
 * Asynchronous. */
cr_status cr_rnorm(double* d_Z, int ldz, int n, int M, uint64_t seed, uint64_t offset,
                   cr_stream stream);

/* Flags of cr_trmm_sim. */
enum {
  CR_TRMM_FP16_DEST = 1,   /* round each output to FP16 before widening (Alg.1 FP16 destination) */
  CR_TRMM_GENERATE = 2,    /* ignore d_Z; draw M_rand from (seed, offset) in FP32 and round */
  CR_TRMM_SPLIT_L = 4,     /* FP32- and FP64-class off-diagonal factor tiles enter as their FP16
                              high/low pair (two MMAs, ~2^-22 relative) instead of the FP16 cast
                              of Alg.1 step 15 (2^-11); FP16-class tiles are exact either way */
  CR_TRMM_FP16_PER_GEMM = 8 /* the FP16 destination of Alg.1 task by task: each block row's
                              products (the diagonal one, then k = i-1 down to 0) are accumulated
                              in FP32 one at a time and the running result is rounded to FP16
                              after each (Y_i = fp16(Y_i + L_ik B_k)); the last rounding is widened
                              into d_Y.  Implies CR_TRMM_FP16_DEST's rounding; allocates an
                              FP16 buffer of n_pad x (M rounded up to 256) on first use */
};

/* Mixed-precision TRMM (Section IV-C Eq.3, Alg.1): Y = L_s B with B = fp16(M_rand / s)
 * when the factor was built with amp != 0, else Y = L M_rand in FP64.  d_Z is the n x M
 * column-major FP64 M_rand (ldz >= n), d_Y the n x M column-major FP64 output
 * (ldy >= n).  With CR_TRMM_GENERATE, M_rand is drawn in FP32 from the stream of
 * cr_rnorm(seed, offset) and d_Z may be NULL.  h_bnorm (may be NULL) receives ||B||_F of
 * the rescaled right-hand side before rounding (Alg.1 step 6); a non-NULL h_bnorm
 * synchronises.  Requires a factored matrix. */
cr_status cr_trmm_sim(cr_tilemat L, const double* d_Z, int ldz, int M, uint64_t seed,
                      uint64_t offset, double* d_Y, int ldy, int flags, double* h_bnorm,
                      cr_stream stream);

/* Universal kriging (Section V-A Eq.5-6, Alg.2 steps 2-6), all in FP64, for the
 * covariance model and locations of V (built by cr_cov_build with n_pred prediction sites
 * first and n_o = n - n_pred observation sites): Sigma_y = V_o + tau2 I is factored as its
 * own FP64 tile matrix, V_op (the n_o x n_p observation/prediction block) is evaluated in
 * FP64.  d_Xo (n_o x 3) and d_Xp (n_p x 3) are column-major trend designs, d_yo the n_o
 * observations.  Outputs: d_W (n_o x n_p column-major, ldw >= n_o) weights, d_zhat (n_p)
 * prediction W^T y_o, d_v (n_p) pointwise MSPE with theta0 = sigma2.  Independent of V's
 * precision map and factor (callable before or after cr_potrf_adaptive).  *info as in
 * cr_potrf_adaptive, for Sigma_y.  Allocates its workspace internally.  Synchronises. */
cr_status cr_krige(cr_tilemat V, const double* d_Xo, const double* d_Xp, const double* d_yo,
                   double* d_W, int ldw, double* d_zhat, double* d_v, cr_stream stream,
                   int* info);

/* Conditioning correction (Section V-B Eq.7): S = M_p + W^T (y_o 1^T - M_o), where the
 * simulations d_Y (n x M column-major, ldy) hold the prediction rows first (M_p = rows
 * [0, n_p), M_o = rows [n_p, n_p + n_o)).  d_S is n_p x M column-major (lds >= n_p).
 * With CR_GEMM_DF (the default, CR_OPT_FP64_GEMM) the product runs in double-float
 * arithmetic on the FP32 units (an FP64 emulation with about 48 significant bits; W and
 * R = y_o 1^T - M_o are rounded to double-float pairs, the sum M_p + W^T R is formed in
 * FP64): |S - S_exact| <= (n_o + 8) 2^-46 (|W|^T |R|)_ij + 2^-52 |S_ij|, with 8 n_o (n_p + M)
 * bytes of pooled scratch (cr_workspace_trim).  With CR_GEMM_OZAKI it is the Ozaki product on
 * the FP16 tensor cores: |S - S_exact| <= n_o 9 2^-48 2^(Ea_i + Eb_j) + 16 2^-47 (|W|^T |R|)_ij
 * + 2^-52 |S_ij| (2^Ea_i, 2^Eb_j the powers of two above the largest magnitudes of column i of
 * W and column j of R); an infinite or NaN entry of W or R makes its row or column of S NaN.
 * Asynchronous. */
cr_status cr_krige_correct(const double* d_W, int ldw, const double* d_yo, const double* d_Y,
                           int ldy, int n_p, int n_o, int M, double* d_S, int lds,
                           cr_stream stream);

/* The correction of cr_krige_correct fused with the calibration of cr_calibrate (or, with
 * negative != 0, of cr_calibrate_negative): each 64 x 64 block of S is computed by the same
 * double-float product and handed straight to the scan's decisions, so S is never written
 * (n_p x M doubles of HBM traffic saved).  Arguments as in those two calls; the results are
 * identical to cr_calibrate(cr_krige_correct(...)) on the same inputs.  Library-managed
 * scratch, 8 n_o (n_p + M) + 8 n_p + 16 M + 16 ceil(n_p / 64) M bytes, grown on demand and
 * shared by all calls: the call returns after its last kernel.  With CR_GEMM_OZAKI the
 * correction is the Ozaki product of cr_krige_correct, which writes S to pooled scratch, and
 * the scan of cr_calibrate reads it.  Synchronises. */
cr_status cr_correct_calibrate(const double* d_W, int ldw, const double* d_yo, const double* d_Y,
                               int ldy, int n_p, int n_o, int M, const double* d_zhat,
                               const double* d_v, double u, double level, int negative,
                               uint8_t* d_cin, uint8_t* d_cout, int32_t* d_count, double* d_psi,
                               double* d_phi, cr_calib_info* out, cr_stream stream);

/* Kriging weights prepared for repeated conditioning corrections by the Ozaki product (the
 * paper has no counterpart; Alg.2 computes W once, steps 2-4, and applies it to the simulations
 * in step 17): the column exponents and the 8 slices of 6 bits of W (n_o x n_p column-major,
 * ldw >= n_o), made once so that the corrections of successive simulation batches with the
 * same weights do not cut W again.  cr_weights_prepare allocates 2 n_o' n_p + 4 n_p bytes
 * with cudaMalloc (n_o' = n_o rounded up to whole chunks, see CR_OPT_FP64_GEMM) and cuts the
 * slices on `stream` (asynchronous: W may change once the stream has passed this call); the
 * handle does not read W again.  cr_weights_release frees it (cudaFree, which waits for the
 * device); NULL is accepted.  The handle belongs to the device that was current at
 * cr_weights_prepare. */
typedef struct cr_weights_s* cr_weights;
cr_status cr_weights_prepare(const double* d_W, int ldw, int n_o, int n_p, cr_stream stream,
                             cr_weights* out);
cr_status cr_weights_release(cr_weights w);

/* cr_krige_correct and cr_correct_calibrate with prepared weights: always the Ozaki product
 * (whatever CR_OPT_FP64_GEMM says), with the same results, bit for bit, as those calls with
 * CR_GEMM_OZAKI on the W the handle was made from; n_o and n_p are the handle's.  Scratch,
 * synchronisation and errors as in those calls. */
cr_status cr_krige_correct_prepared(cr_weights w, const double* d_yo, const double* d_Y, int ldy,
                                    int M, double* d_S, int lds, cr_stream stream);
cr_status cr_correct_calibrate_prepared(cr_weights w, const double* d_yo, const double* d_Y,
                                        int ldy, int M, const double* d_zhat, const double* d_v,
                                        double u, double level, int negative, uint8_t* d_cin,
                                        uint8_t* d_cout, int32_t* d_count, double* d_psi,
                                        double* d_phi, cr_calib_info* out, cr_stream stream);

/* Calibration (Section V-C Eq.8-9, Alg.2 steps 18-22): t = (zhat - u)/sqrt(v);
 * psi_j = min{t_i : S_ij >= u}, phi_j = max{t_i : S_ij <= u} in one pass over d_S
 * (n_p x M column-major, lds >= n_p); per-location exceedance counts
 * count_i = #{j : S_ij >= u}; empirical quantiles q_out = Q_{1-level}(psi),
 * q_in = Q_level(phi) on the samples without empty-set sentinels; regions
 * d_cin[i] = t_i > q_in, d_cout[i] = t_i >= q_out (uint8).  d_count, d_psi, d_phi may
 * be NULL.  Returns CR_ERR_NONPOS_MSPE if some v_i <= 0 and CR_ERR_EMPTY_SAMPLE if a
 * sample is empty.  Its scratch is library-managed and shared by all calls; the call returns
 * only after its last kernel has finished, so calls made one after another (on any streams)
 * never see each other's scratch.  Synchronises. */
cr_status cr_calibrate(const double* d_S, int lds, int n_p, int M, const double* d_zhat,
                       const double* d_v, double u, double level, uint8_t* d_cin,
                       uint8_t* d_cout, int32_t* d_count, double* d_psi, double* d_phi,
                       cr_calib_info* out, cr_stream stream);

/* Calibration of the negative excursion set {Z <= u} (Section III: the method applied to the
 * sign-reversed field and threshold, -S and -u, with -zhat).  Same arguments, layouts,
 * outputs, errors and synchronisation as cr_calibrate; the outputs are those of the reversed
 * problem: t'_i = ((-zhat_i) - (-u)) / sqrt(v_i) = -t_i, psi'_j = min{t'_i : S_ij <= u},
 * phi'_j = max{t'_i : S_ij >= u}, count_i = #{j : S_ij <= u}, q_out' = Q_{1-level}(psi'),
 * q_in' = Q_level(phi'), d_cin[i] = t'_i > q_in', d_cout[i] = t'_i >= q_out'. */
cr_status cr_calibrate_negative(const double* d_S, int lds, int n_p, int M, const double* d_zhat,
                                const double* d_v, double u, double level, uint8_t* d_cin,
                                uint8_t* d_cout, int32_t* d_count, double* d_psi, double* d_phi,
                                cr_calib_info* out, cr_stream stream);

/* Calibration without any allocation.  The paper has no counterpart to this entry point:
 * it exists for callers that cannot allocate device memory themselves, for example code
 * running under a memory pool that owns every device allocation of the process (so a
 * library-side cudaMalloc would bypass or break its accounting), or embedders that must
 * keep the device footprint fixed after start-up.  It computes
 * exactly what cr_calibrate computes, with the same arguments and outputs, but its device
 * scratch (t, psi, phi and the per-block partials of the scan) lives in a fixed array
 * inside the library (CR_NOALLOC_SCRATCH_BYTES, held by every device that loads the
 * library until the process exits) and the host-side quantile samples in a fixed host
 * array; it never calls cudaMalloc, cudaFree or any allocating routine.
 * Limits: M <= CR_NOALLOC_MAX_M and 8 n_p + 16 M + 16 ceil(n_p / 2048) M + 1536 bytes
 * <= CR_NOALLOC_SCRATCH_BYTES; larger problems return CR_ERR_ARG (use cr_calibrate).
 * The first call on a device looks up the array's device address (once per device, with
 * that device current).  All calls share the one array and the one host buffer; the library
 * serialises them with a process-wide lock, and a call returns only after its last kernel
 * (the region flags, which read the array) has finished on the stream, so calls from
 * several host threads or streams never overlap on the array.  Synchronises the stream and
 * reads the quantile samples on the host: it cannot be called on a stream that is being
 * captured into a CUDA graph. */
#define CR_NOALLOC_SCRATCH_BYTES (8u << 20)
#define CR_NOALLOC_MAX_M 65536
cr_status cr_calibrate_noalloc(const double* d_S, int lds, int n_p, int M, const double* d_zhat,
                               const double* d_v, double u, double level, uint8_t* d_cin,
                               uint8_t* d_cout, int32_t* d_count, double* d_psi, double* d_phi,
                               cr_calib_info* out, cr_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* CR_H */
