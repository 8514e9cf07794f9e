// Covariance evaluation: tile statistics, generation of each tile in its precision class,
// dense extraction and dense blocks for kriging.
//
// "Mixed-Precision GPU Acceleration for Confidence Regions of Spatial Excursion Sets":
// Section V Eq.4 (joint covariance, tau^2 on the observation block only), Section VI-B.2
// (power-exponential model), Section VI-C (Matern model), Section V-D (tile Frobenius
// norms and entry extrema used by the precision checks), Alg.2 step 12 (the tiles of s^2 V
// in their selected precisions).
//
// The FP64 matrix is never stored.  cr_cov_build makes one pass that only reduces the
// per-tile statistics; the factorisation generates each tile directly in its class (FP64
// tiles in FP64, FP32 tiles rounded from a double-float evaluation, FP16 tiles from a
// single-precision one).  For the closed-form Matern orders (nu = 1/2, 3/2, 5/2) the
// statistics and the FP32 tiles are evaluated in double-float arithmetic on the FP32 units
// (about 1e-14 relative; GB300's FP64 units run at 1/60 of the FP32 rate), the FP16 tiles in
// FP32 (a few ulp, against the 2^-11 rounding of FP16); FP64 tiles and the other models use
// FP64.
#include <math.h>

#include <cmath>

#include <mutex>

#include "common.cuh"
#include "cov.cuh"
#include "df.cuh"

namespace cr {

__constant__ DfExpTables c_dfexp;

// K_nu(x) e^x by the trapezoidal rule on K_nu(x) = int_0^inf exp(-x cosh t) cosh(nu t) dt
// (the integrand is even and analytic in the strip |Im t| < pi/2, so the rule converges
// geometrically in 1/h; Trefethen & Weideman, "The exponentially convergent trapezoidal
// rule", SIAM Review 56 (2014)).  The step follows from the strip half-width a: the
// relative error is about exp(x (1 - cos a) + nu ln(1/cos a) - 2 pi a / h).
__device__ double bessel_k_scaled(double nu, double x) {
  const double a = (x > 100.0) ? 0.6 : 1.3;
  const double ca = cos(a);
  const double h = 2.0 * M_PI * a / (x * (1.0 - ca) + 38.0 + nu * log(1.0 / ca));
  const double t0 = acosh(1.0 + 40.0 / x);
  const double tmax = acosh(1.0 + (40.0 + nu * t0) / x);
  const int N = (int)ceil(tmax / h) + 1;
  const double E = exp(h), Ei = 1.0 / E, En = exp(nu * h), Eni = 1.0 / En;
  double ek = 1.0, eki = 1.0, enk = 1.0, enki = 1.0;
  double sum = 0.5;   // t = 0 term with half weight: exp(0) * cosh(0) / 2
  for (int k = 1; k <= N; ++k) {
    ek *= E; eki *= Ei; enk *= En; enki *= Eni;
    const double cm1 = 0.5 * (ek + eki) - 1.0;
    sum += exp(-x * cm1) * 0.5 * (enk + enki);
  }
  return h * sum;
}

// FP64 covariance at scaled distance x = h / range > 0.
__device__ __forceinline__ double cov_of_x(const CovK& p, double x) {
  if (p.family == CR_COV_POWEXP) return p.sigma2 * exp(-pow(x, p.nu));
  switch (p.kind) {
    case 0: return p.sigma2 * exp(-x);
    case 1: return p.sigma2 * (1.0 + x) * exp(-x);
    case 2: return p.sigma2 * (1.0 + x + x * x * (1.0 / 3.0)) * exp(-x);
    default: {
      if (x > 745.0) return 0.0;
      return p.sigma2 * p.norm * exp(p.nu * log(x) - x) * bessel_k_scaled(p.nu, x);
    }
  }
}

__device__ __forceinline__ double diag_value(const CovK& p, int gi) {
  return p.sigma2 + p.nugget + (gi >= p.n_pred ? p.tau2 : 0.0);
}

// FP64 entry V[gi, gj] (valid indices).
__device__ __forceinline__ double cov_entry64(const CovK& p, const double* __restrict__ xy, int gi, int gj) {
  if (gi == gj) return diag_value(p, gi);
  const double dx = xy[2 * gi] - xy[2 * gj], dy = xy[2 * gi + 1] - xy[2 * gj + 1];
  const double h = sqrt(dx * dx + dy * dy);
  if (h == 0.0) return p.sigma2;
  return cov_of_x(p, h * p.inv_range);
}

__device__ __noinline__ double cov_entry64_ool(const CovK& p, const double* __restrict__ xy, int gi, int gj) {
  return cov_entry64(p, xy, gi, gj);
}

// Double-float entry for an off-diagonal pair with coordinate differences (dx, dy), times
// sig; sets *fallback when the scaled distance leaves the double-float exponential's range.
__device__ __forceinline__ df cov_entry_df(const CovK& p, df dx, df dy, df sig, df inv_range, const DfExpTables& T,
                                           bool* fallback) {
  const df d2 = df_add(df_mul(dx, dx), df_mul(dy, dy));
  if (d2.hi == 0.0f) return sig;
  const df x = df_mul(df_sqrt(d2), inv_range);
  if (x.hi > 80.0f) {
    *fallback = true;
    return {0.0f, 0.0f};
  }
  df v = df_exp(df_neg(x), T);
  if (p.kind == 1) {
    v = df_mul(df_add_f(x, 1.0f), v);
  } else if (p.kind == 2) {
    const df third = {0.3333333432674408f, -9.934107e-09f};   // 1/3 = hi + lo
    v = df_mul(df_add_f(df_add(x, df_mul(df_mul(x, x), third)), 1.0f), v);
  }
  return df_mul(v, sig);
}

struct Pt {
  df x, y;
};

__device__ __forceinline__ Pt load_pt(const double* xy, int g) {
  return {df_from_double(xy[2 * g]), df_from_double(xy[2 * g + 1])};
}

__device__ __forceinline__ void tile_of(int t, int& i, int& j) {
  i = (int)floor((sqrt(8.0 * t + 1.0) - 1.0) * 0.5);
  while (i * (i + 1) / 2 > t) --i;
  while ((i + 1) * (i + 2) / 2 <= t) ++i;
  j = t - i * (i + 1) / 2;
}

// The locations as double-float pairs (x.hi, x.lo, y.hi, y.lo), once per covariance, so that
// the tile kernels load them without FP64 conversions.
__global__ void k_points_df(const double* __restrict__ xy, int n, float4* __restrict__ xy4) {
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= n) return;
  const Pt pt = load_pt(xy, g);
  xy4[g] = make_float4(pt.x.hi, pt.x.lo, pt.y.hi, pt.y.lo);
}

// Column points (nb) then the 64 row points of row block r0 of tile (i, j) into shared
// memory as (x.hi, x.lo, y.hi, y.lo); returns the thread's largest |coordinate| (high words).
__device__ __forceinline__ float load_tile_points(const float4* __restrict__ xy4, int n, int nb, int i, int j, int r0,
                                                  float4* s_pts) {
  float cmax = 0.0f;
  for (int q = threadIdx.x; q < nb + 64; q += blockDim.x) {
    const int g = q < nb ? j * nb + q : i * nb + r0 + (q - nb);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (g < n) {
      v = __ldg(xy4 + g);
      cmax = fmaxf(cmax, fmaxf(fabsf(v.x), fabsf(v.z)));
    }
    s_pts[q] = v;
  }
  return cmax;
}

// Exact statistics of row block rbk (ROWS rows, ROWS <= 64) of tile (i, j): partial sum of
// squares, min, max and 0 (an exact partial has no error bound) over valid entries, STAT_W
// doubles at sp.  Nothing is stored.
template <bool DF, int ROWS>
__device__ __forceinline__ void stats_exact(const double* __restrict__ xy, const float4* __restrict__ xy4, int n, int nb,
                                            const CovK& p, int i, int j,
                                            int rbk, double* __restrict__ sp) {
  const int r0 = rbk * ROWS;
  extern __shared__ float4 s_pts[];
  float4* s_col = s_pts;
  float4* s_row = s_pts + nb;
  load_tile_points(xy4, n, nb, i, j, r0, s_pts);
  // exponential tables in shared memory: their per-thread indices diverge
  __shared__ DfExpTables s_T;
  for (int q = threadIdx.x; q < 64; q += blockDim.x) {
    s_T.t_hi[q] = c_dfexp.t_hi[q];
    s_T.t_lo[q] = c_dfexp.t_lo[q];
  }
  if (threadIdx.x == 0) { s_T.c1 = c_dfexp.c1; s_T.c2 = c_dfexp.c2; s_T.c3 = c_dfexp.c3; }
  __syncthreads();
  const df sig = {p.sig_hi, p.sig_lo}, invr = {p.invr_hi, p.invr_lo};
  df ssq = {0.0f, 0.0f};
  df dmn = {INFINITY, 0.0f}, dmx = {-INFINITY, 0.0f};   // double-float extrema (no FP64 work per entry)
  double ssq64 = 0.0, vmn = INFINITY, vmx = -INFINITY;
  // each thread keeps one column point in registers and walks the 64 rows (the row point is
  // a broadcast read): no per-entry index division
  for (int c = threadIdx.x; c < nb; c += blockDim.x)
#pragma unroll 1
  for (int rr = 0; rr < ROWS; ++rr) {
    const int r = r0 + rr;
    const int gi = i * nb + r, gj = j * nb + c;
    if (gi >= n || gj >= n) continue;
    if (DF) {
      bool fb = gi == gj;
      df v = {0.0f, 0.0f};
      if (!fb) {
        const float4 a = s_row[rr], b = s_col[c];
        const df dx = df_add({a.x, a.y}, df_neg({b.x, b.y}));
        const df dy = df_add({a.z, a.w}, df_neg({b.z, b.w}));
        v = cov_entry_df(p, dx, dy, sig, invr, s_T, &fb);
      }
      if (__builtin_expect(fb, 0)) {
        // diagonal entries and distances outside the double-float exponential: FP64, out of
        // line, so that no FP64 instruction is predicated into the common path (GB300's FP64
        // units run at 1/64 of the FP32 rate)
        const double v64 = cov_entry64_ool(p, xy, gi, gj);
        ssq = df_add(ssq, df_from_double(v64 * v64));
        vmn = fmin(vmn, v64);
        vmx = fmax(vmx, v64);
        continue;
      }
      ssq = df_add(ssq, df_mul(v, v));
      if (df_lt(v, dmn)) dmn = v;
      if (df_lt(dmx, v)) dmx = v;
    } else {
      const double v64 = cov_entry64(p, xy, gi, gj);
      ssq64 += v64 * v64;
      vmn = fmin(vmn, v64);
      vmx = fmax(vmx, v64);
    }
  }
  if (DF) {
    vmn = fmin(vmn, df_to_double(dmn));
    vmx = fmax(vmx, df_to_double(dmx));
  }
  double s = DF ? df_to_double(ssq) : ssq64;
  __shared__ double red[3][8];
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_down_sync(0xffffffffu, s, o);
    vmn = fmin(vmn, __shfl_down_sync(0xffffffffu, vmn, o));
    vmx = fmax(vmx, __shfl_down_sync(0xffffffffu, vmx, o));
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) { red[0][w] = s; red[1][w] = vmn; red[2][w] = vmx; }
  __syncthreads();
  if (threadIdx.x == 0) {
    double a = 0.0, b = INFINITY, c = -INFINITY;
    for (int q = 0; q < (int)(blockDim.x >> 5); ++q) { a += red[0][q]; b = fmin(b, red[1][q]); c = fmax(c, red[2][q]); }
    sp[0] = a; sp[1] = b; sp[2] = c; sp[3] = 0.0;
  }
}

// Exact statistics pass over a tile list (every lower tile in order without one): one CTA
// per (listed tile, ROWS-row block).  Partials are indexed by tile, or by list position when
// by_list is set (the policy's recomputations, whose 16-row blocks keep each CTA short).
template <bool DF, int ROWS>
__global__ void __launch_bounds__(256) k_cov_stats(const double* __restrict__ xy, const float4* __restrict__ xy4, int n,
                                                   int nb, CovK p,
                                                   double* __restrict__ stat_part, const int* __restrict__ tiles,
                                                   int by_list) {
  const int tile = tiles ? tiles[blockIdx.x] : blockIdx.x;
  int i, j;
  tile_of(tile, i, j);
  const size_t slot = by_list ? blockIdx.x : tile;
  stats_exact<DF, ROWS>(xy, xy4, n, nb, p, i, j, blockIdx.y, stat_part + (slot * gridDim.y + blockIdx.y) * STAT_W);
}

// Fast statistics of row block rbk of the off-diagonal tile (i, j), closed-form Matern
// orders: every entry in FP32, distances from the FP32 roundings of the coordinates (the high
// words of their double-float pairs), the square root
// as q rsqrtf(q) (rsqrtf within 2 ulp) and the exponential by __expf (within
// 2 + floor(1.173 |x|) ulp, the documented bounds of both).  Per entry, with u = 2^-24 and
// scaled distance x:
//  - the computed x is off by at most 16.5 u x + (1/range) (C 2^-22 + 2^-70), C the largest
//    |coordinate| (each FP32 coordinate is within 2^-24 C, so each difference within
//    2^-23 C, and the distance within 2^-22.5 C; the differences' roundings 1.5 u, the
//    squares and their sum 1 u after the root, the root 5 u, the scaling 2 u, with margin;
//    squares below the FP32 range lose at most 2^-70 of the distance);
//  - |d log v / dx| <= 1 for these orders, so that error passes to v unchanged;
//  - the exponential ((4 + 2.35 x) u), the polynomial (4 u) and the products with sigma^2
//    (3 u) add (11 + 2.35 x) u.
// The sum of squares runs in FP32 over 64 ceil(nb / 256) entries per thread and then over the
// CTA (12 more additions deep), in two ranges (v^2 and (v 2^60)^2 for v < 2^-60, so that
// nothing underflows), so it adds K u to the relative error of the sum (K u / 2 to its
// square root), K = 64 ceil(nb / 256) + 12.  The partial's record holds one relative bound
// E for its sum of squares' square root, min and max:
//   E = 1.01 ((20 x_max + 16 + K) u + (1/range) (C 2^-21 + 2^-69)) + 2^-40,
// or infinity where the bound does not hold (x > 80, where the exponential leaves the
// normal range; entries below 2^-120 or above 2^56, where products, squares or their sums
// leave it).
__device__ __forceinline__ void stats_fast(const float4* __restrict__ xy4, int n, int nb, const CovK& p, int i, int j,
                                           int rbk, double* __restrict__ sp) {
  const int r0 = rbk * 64;
  extern __shared__ float4 s_pts[];
  float4* s_col = s_pts;
  float4* s_row = s_pts + nb;
  float cmax = load_tile_points(xy4, n, nb, i, j, r0, s_pts);
  __syncthreads();
  const float sig = p.sig_hi, invr = p.invr_hi;
  const int kind = p.kind;
  const float small_lim = 0x1.0p-60f, small_up = 0x1.0p60f;
  float big = 0.0f, small = 0.0f, vmn = INFINITY, vmx = -INFINITY, xmx = 0.0f;
  const int rows = min(64, n - (i * nb + r0));
  for (int c = threadIdx.x; c < nb; c += blockDim.x) {
    if (j * nb + c >= n) break;
    const float4 b = s_col[c];
#pragma unroll 4
    for (int rr = 0; rr < rows; ++rr) {
      const float4 a = s_row[rr];
      const float dx = a.x - b.x, dy = a.z - b.z;
      const float q2 = fmaf(dx, dx, dy * dy);
      const float x = (q2 > 0.0f ? q2 * rsqrtf(q2) : 0.0f) * invr;
      const float e = __expf(-x);
      const float poly = kind == 0 ? 1.0f : (kind == 1 ? 1.0f + x : fmaf(x * x, 1.0f / 3.0f, 1.0f + x));
      const float v = sig * poly * e;
      if (v >= small_lim) {
        big = fmaf(v, v, big);
      } else {
        const float w = v * small_up;
        small = fmaf(w, w, small);
      }
      vmn = fminf(vmn, v);
      vmx = fmaxf(vmx, v);
      xmx = fmaxf(xmx, x);
    }
  }
  // CTA reduction in FP32 (GB300 issues FP64 arithmetic, comparisons and conversions on its
  // slow FP64 pipe): the extrema are exact, and the two sums gain at most 5 u (warp tree)
  // and 7 u (over the 8 warps) of relative error, for 12 + K u in all
  for (int o = 16; o > 0; o >>= 1) {
    big += __shfl_down_sync(0xffffffffu, big, o);
    small += __shfl_down_sync(0xffffffffu, small, o);
    vmn = fminf(vmn, __shfl_down_sync(0xffffffffu, vmn, o));
    vmx = fmaxf(vmx, __shfl_down_sync(0xffffffffu, vmx, o));
    xmx = fmaxf(xmx, __shfl_down_sync(0xffffffffu, xmx, o));
    cmax = fmaxf(cmax, __shfl_down_sync(0xffffffffu, cmax, o));
  }
  __shared__ float red[6][8];
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) { red[0][w] = big; red[1][w] = small; red[2][w] = vmn; red[3][w] = vmx; red[4][w] = xmx; red[5][w] = cmax; }
  __syncthreads();
  if (threadIdx.x == 0) {
    float fb = 0.0f, fs = 0.0f, fmn = INFINITY, fmx = -INFINITY, fxm = 0.0f, fcm = 0.0f;
    for (int q = 0; q < (int)(blockDim.x >> 5); ++q) {
      fb += red[0][q]; fs += red[1][q]; fmn = fminf(fmn, red[2][q]); fmx = fmaxf(fmx, red[3][q]);
      fxm = fmaxf(fxm, red[4][q]); fcm = fmaxf(fcm, red[5][q]);
    }
    const double a = (double)fb + (double)fs * 0x1.0p-120, b = fmn, cc = fmx, xm = fxm, cm = fcm;
    const double u = 0x1.0p-24, K = 64.0 * ((nb + 255) / 256) + 12.0;
    double E = 1.01 * ((20.0 * xm + 16.0 + K) * u + (double)p.invr_hi * (cm * 0x1.0p-21 + 0x1.0p-69)) + 0x1.0p-40;
    const bool empty = !(b <= cc);   // no valid entry in this row block
    // entries up to 2^56 keep every partial sum of squares below 2^127 (no FP32 overflow)
    if (!empty && (!(xm <= 80.0) || !(b >= 0x1.0p-120) || !(cc <= 0x1.0p56))) E = INFINITY;
    sp[0] = a; sp[1] = b; sp[2] = cc; sp[3] = E;
  }
}

// Statistics pass of a new covariance for the closed-form Matern orders: CTAs 0 .. nt nrb - 1
// take the diagonal tiles exactly (double-float, FP64 for the diagonal entries); the others
// take the off-diagonal tiles, in row order, through the FP32 pass with its error bound.
__global__ void __launch_bounds__(256) k_cov_stats_split(const double* __restrict__ xy, const float4* __restrict__ xy4,
                                                         int n, int nb, int nt, CovK p,
                                                         double* __restrict__ stat_part) {
  const int nrb = nb / 64, ndiag = nt * nrb;
  const int b = blockIdx.x;
  int i, j, rbk;
  if (b < ndiag) {
    i = j = b / nrb;
    rbk = b % nrb;
  } else {
    const int o = (b - ndiag) / nrb;   // off-diagonal tile o in row order: row i holds i of them
    rbk = (b - ndiag) % nrb;
    i = (int)((1.0f + sqrtf(8.0f * (float)o + 1.0f)) * 0.5f);
    while (i * (i - 1) / 2 > o) --i;
    while ((i + 1) * i / 2 <= o) ++i;
    j = o - i * (i - 1) / 2;
  }
  double* sp = stat_part + ((size_t)tidx(i, j) * nrb + rbk) * STAT_W;
  if (i == j) stats_exact<true, 64>(xy, xy4, n, nb, p, i, j, rbk, sp);
  else stats_fast(xy4, n, nb, p, i, j, rbk, sp);
}

// Per-tile reduction of the partials of the tiles in the list (all tiles without one).
__global__ void k_stats_reduce(const double* __restrict__ part, int ntiles, int nrb, double* __restrict__ stats,
                               const int* __restrict__ tiles, int by_list) {
  const int q0 = blockIdx.x * blockDim.x + threadIdx.x;
  if (q0 >= ntiles) return;
  const int t = tiles ? tiles[q0] : q0;
  const size_t slot = by_list ? q0 : t;   // where the partials are
  double a = 0.0, b = INFINITY, c = -INFINITY, e = 0.0;
  for (int q = 0; q < nrb; ++q) {
    const double* sp = part + (slot * nrb + q) * STAT_W;
    a += sp[0]; b = fmin(b, sp[1]); c = fmax(c, sp[2]); e = fmax(e, sp[3]);
  }
  stats[STAT_W * t] = a; stats[STAT_W * t + 1] = b; stats[STAT_W * t + 2] = c; stats[STAT_W * t + 3] = e;
}

// Diagonal tile i (FP64 class), 16 of its rows: 8 from the top half and the mirrored 8 from
// the bottom half (rows 8q .. 8q+7 and nb-8q-8 .. nb-8q-1), so that the nb/16 CTAs of a tile
// evaluate equal parts of its lower triangle.  The upper part is stored as zeros; padding
// rows and columns are the identity (scaled by s^2).
__device__ __forceinline__ void generate_diag64(const double* __restrict__ xy, int n, int nb, const CovK& p, double s2,
                                                const TileView& v, int i, int q) {
  double* dst = v.pool64 + (size_t)v.i64[tidx(i, i)] * nb * nb;
  for (int rr = 0; rr < 16; ++rr) {
    const int r = rr < 8 ? 8 * q + rr : nb - 8 * (q + 1) + (rr - 8);
    const int gi = i * nb + r;
    for (int c = threadIdx.x; c < nb; c += blockDim.x) {
      const int gj = i * nb + c;
      double x = 0.0;
      if (gi >= n || gj >= n) x = gi == gj ? s2 : 0.0;
      else if (c <= r) x = cov_entry64(p, xy, gi, gj) * s2;
      dst[(size_t)r * nb + c] = x;
    }
  }
}

// Square root by the PTX approximation (relative error about 2^-23): enough for a distance
// whose covariance is rounded to FP16.
__device__ __forceinline__ float sqrt_approx(float x) {
  float y;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// FP16 tile, one 64-row block (off-diagonal): a single-precision evaluation, accurate to a
// few 1e-6, is far inside the 2^-11 rounding of the stored value; distances from the
// double-float coordinates, so that near points do not lose digits to cancellation.  Each
// work item is four adjacent columns, whose coordinates stay in registers, over a run of rows
// taken two at a time (eight independent evaluations in flight, no branches: MODE 0-2 the
// closed-form Matern orders nu = 1/2, 3/2, 5/2, 3 the power-exponential family); the four
// values are converted to FP16 in two packed conversions and stored as one 8-byte word, so
// that a warp writes 256 contiguous bytes of a row.
template <int MODE>
__device__ __forceinline__ void gen_fp16_tile(const CovK& p, int n, int nb, int i, int j, int r0, double s2,
                                              const float4* s_col, const float4* s_row, uint2* dst) {
  const int nq = nb / 4;
  const int splits = nq >= 256 ? 1 : (nq >= 128 ? 2 : (nq >= 64 ? 4 : 8));
  const int run = 64 / splits;
  const float sig_s2 = p.sig_hi * (float)s2, invr = p.invr_hi, nuf = (float)p.nu;
  for (int w = threadIdx.x; w < nq * splits; w += blockDim.x) {
    const int q = w % nq, rs = r0 + (w / nq) * run;
    const int c0 = 4 * q, gj0 = j * nb + c0;
    float bxh[4], bxl[4], byh[4], byl[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float4 b4 = s_col[c0 + u];
      bxh[u] = b4.x; bxl[u] = b4.y; byh[u] = b4.z; byl[u] = b4.w;
    }
#pragma unroll 1
    for (int r = rs; r < rs + run; r += 2) {
      float val[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float4 a = s_row[r + h - r0];
        const bool row_ok = i * nb + r + h < n;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float dx = (a.x - bxh[u]) + (a.y - bxl[u]), dy = (a.z - byh[u]) + (a.w - byl[u]);
          const float x = sqrt_approx(fmaf(dx, dx, dy * dy)) * invr;
          float e;
          if (MODE == 3) {
            // exp(-x^nu), x^nu = 2^(nu log2 x) (x = 0 gives 0): a few 1e-6 relative
            const float y = x > 0.0f ? exp2f(nuf * __log2f(x)) : 0.0f;
            e = __expf(-y);
          } else {
            e = __expf(-x);   // ex2-based: ~3e-6 relative at x < 50, against FP16's 4.9e-4
            if (MODE == 1) e *= 1.0f + x;
            if (MODE == 2) e *= fmaf(x * x, 1.0f / 3.0f, 1.0f + x);
          }
          val[h][u] = (row_ok && gj0 + u < n) ? sig_s2 * e : 0.0f;
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const __half2 lo = __floats2half2_rn(val[h][0], val[h][1]);
        const __half2 hi = __floats2half2_rn(val[h][2], val[h][3]);
        dst[((size_t)(r + h) * nb + c0) / 4] =
            make_uint2(*reinterpret_cast<const unsigned*>(&lo), *reinterpret_cast<const unsigned*>(&hi));
      }
    }
  }
}

// Double-float covariance of the pair (a, b) (points as (x.hi, x.lo, y.hi, y.lo)) times ss,
// to about 2^-39 relative, for values rounded to FP32 afterwards, without branches, so that
// a thread's independent evaluations interleave: the square root from the PTX approximation
// and one Newton step (as df_sqrt_lite), the exponential of df_exp_lite, the Matern order
// KIND (nu = 1/2, 3/2, 5/2) as a template argument.  far: the scaled distance is beyond the
// double-float exponential's range (the value is then to be taken in FP64).
template <int KIND>
__device__ __forceinline__ df cov_df_lite(float4 a, float4 b, df ss, df invr, const DfExpTables& T, bool& far) {
  const df dx = df_add({a.x, a.y}, df_neg({b.x, b.y}));
  const df dy = df_add({a.z, a.w}, df_neg({b.z, b.w}));
  const df d2 = df_add(df_mul(dx, dx), df_mul(dy, dy));
  float s, inv_s;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(s) : "f"(d2.hi));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv_s) : "f"(s));
  const df pp = df_two_prod(s, s);
  const float res = __fadd_rn(__fsub_rn(__fsub_rn(d2.hi, pp.hi), pp.lo), d2.lo);
  const float corr = s > 0.0f ? __fmul_rn(res, 0.5f * inv_s) : 0.0f;
  const df x = df_mul(df_quick_two_sum(s, corr), invr);
  far = x.hi > 80.0f;
  df v = df_exp_lite(df_neg(x), T);
  if (KIND == 1) v = df_mul(df_add_f(x, 1.0f), v);
  if (KIND == 2) {
    const df third = {0.3333333432674408f, -9.934107e-09f};   // 1/3 = hi + lo
    v = df_mul(df_add_f(df_add(x, df_mul(df_mul(x, x), third)), 1.0f), v);
  }
  const df out = df_mul(v, ss);
  const bool zero = d2.hi == 0.0f;   // coincident sites: the covariance is sigma^2
  return {zero ? ss.hi : out.hi, zero ? ss.lo : out.lo};
}

// FP32 tile, one block of `rows` rows (off-diagonal, closed-form Matern order KIND): double-
// float evaluations rounded once to FP32, sigma^2 s^2 folded into one factor ss, four rows
// at a time (four independent evaluation chains per thread).  The rare scaled distances
// beyond the double-float exponential's range are stored as 0 and redone in FP64 by a second
// pass of the threads that met one, so that the main loop holds no call.
template <int KIND, int GR = 4>
__device__ __forceinline__ void gen_fp32_tile(const CovK& p, const double* __restrict__ xy, int n, int nb, int i, int j,
                                              int r0, int rows, double s2, df ss, df invr, const float4* s_col,
                                              const float4* s_row, const DfExpTables& T, float* dst) {
  bool any_far = false;
  for (int c = threadIdx.x; c < nb; c += blockDim.x) {
    const float4 b = s_col[c];
    const int gj = j * nb + c;
#pragma unroll 1
    for (int r = r0; r < r0 + rows; r += GR) {
      df w[GR];
      bool far[GR];
#pragma unroll
      for (int h = 0; h < GR; ++h) w[h] = cov_df_lite<KIND>(s_row[r + h - r0], b, ss, invr, T, far[h]);
#pragma unroll
      for (int h = 0; h < GR; ++h) {
        const bool valid = i * nb + r + h < n && gj < n;
        any_far |= valid && far[h];
        dst[(size_t)(r + h) * nb + c] = (valid && !far[h]) ? __fadd_rn(w[h].hi, w[h].lo) : 0.0f;
      }
    }
  }
  if (__builtin_expect(any_far, 0)) {
    for (int c = threadIdx.x; c < nb; c += blockDim.x) {
      const float4 b = s_col[c];
      const int gj = j * nb + c;
      for (int r = r0; r < r0 + rows; ++r) {
        const int gi = i * nb + r;
        bool far;
        (void)cov_df_lite<KIND>(s_row[r - r0], b, ss, invr, T, far);
        if (far && gi < n && gj < n) dst[(size_t)r * nb + c] = (float)(cov_entry64_ool(p, xy, gi, gj) * s2);
      }
    }
  }
}

// Generation of s^2 V in each tile's class (Alg.2 step 12) over a tile list: its first ndiag
// entries are diagonal tiles, the next nheavy the tiles evaluated in FP64 or double-float
// (FP64 and FP32 classes), the rest FP16 tiles.  CTAs 0 .. ndiag nb/16 - 1 take the diagonal
// tiles, nb/16 CTAs each (generate_diag64 in FP64, or the double-float evaluation when the
// double-float executor factors them; spread wide so that they finish early); then
// nb/hrows CTAs per heavy tile, hrows rows each (16, 32 or 64: the host picks the largest
// that still gives the heavy tiles a few waves of CTAs), and nb/64 CTAs per FP16 tile, 64
// rows each.  The list fixes the issue order within a launch;
// the factorisation issues one launch per column range, so that each column is complete
// before it is needed.  Padding rows/columns are the identity (scaled by s^2).
__global__ void __launch_bounds__(256, 2) k_generate(const double* __restrict__ xy, const float4* __restrict__ xy4, int n,
                                                     int nb, CovK p, double s2,
                                                  float s2_hi, float s2_lo, TileView v, const int* __restrict__ tiles,
                                                  int ndiag, int nheavy, int hrows, int diag_df) {
  const int nrb = nb / 64, nsub = nb / 16;
  extern __shared__ float4 s_pts[];
  __shared__ DfExpTables s_T;
  if ((int)blockIdx.x < ndiag * nsub) {
    const int i = tiles[blockIdx.x / nsub] >> 16, q = blockIdx.x % nsub;
    if (!diag_df) {
      generate_diag64(xy, n, nb, p, s2, v, i, q);
      return;
    }
    // Diagonal tile for the double-float executor, which holds the tile in double-float: the
    // off-diagonal entries by the double-float evaluation of the FP32-class tiles (the same
    // ~2^-48 relative accuracy the executor keeps), the diagonal entries in FP64.  Rows as in
    // generate_diag64: 8 from the top half, the mirrored 8 from the bottom half.
    float4* s_col = s_pts;
    float4* s_row = s_pts + nb;
    auto row_of = [&](int rr) { return rr < 8 ? 8 * q + rr : nb - 8 * (q + 1) + (rr - 8); };
    for (int k = threadIdx.x; k < nb + 16; k += blockDim.x) {
      const int g = i * nb + (k < nb ? k : row_of(k - nb));
      s_pts[k] = g < n ? __ldg(xy4 + g) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int k = threadIdx.x; k < 64; k += blockDim.x) {
      s_T.t_hi[k] = c_dfexp.t_hi[k];
      s_T.t_lo[k] = c_dfexp.t_lo[k];
    }
    if (threadIdx.x == 0) { s_T.c1 = c_dfexp.c1; s_T.c2 = c_dfexp.c2; s_T.c3 = c_dfexp.c3; }
    __syncthreads();
    double* dst = v.pool64 + (size_t)v.i64[tidx(i, i)] * nb * nb;
    const df sig = {p.sig_hi, p.sig_lo}, invr = {p.invr_hi, p.invr_lo}, s2d = {s2_hi, s2_lo};
    for (int rr = 0; rr < 16; ++rr) {
      const int r = row_of(rr), gi = i * nb + r;
      const float4 a = s_row[rr];
      for (int c = threadIdx.x; c < nb; c += blockDim.x) {
        const int gj = i * nb + c;
        double x = 0.0;
        if (gi >= n || gj >= n) {
          x = gi == gj ? s2 : 0.0;
        } else if (c == r) {
          x = cov_entry64(p, xy, gi, gj) * s2;
        } else if (c < r) {
          const float4 b = s_col[c];
          const df dx = df_add({a.x, a.y}, df_neg({b.x, b.y}));
          const df dy = df_add({a.z, a.w}, df_neg({b.z, b.w}));
          bool fb = false;
          const df vd = cov_entry_df(p, dx, dy, sig, invr, s_T, &fb);
          if (__builtin_expect(fb, 0)) x = cov_entry64_ool(p, xy, gi, gj) * s2;
          else {
            const df w = df_mul(vd, s2d);
            x = (double)w.hi + (double)w.lo;
          }
        }
        dst[(size_t)r * nb + c] = x;
      }
    }
    return;
  }
  // the first nheavy tiles after the diagonal ones (FP64 and FP32 classes) in blocks of hrows
  // rows, the others in 64-row blocks
  const int b = blockIdx.x - ndiag * nsub;
  const int hsub = nb / hrows;
  int e, r0, rows;
  if (b < nheavy * hsub) {
    e = tiles[ndiag + b / hsub];
    r0 = (b % hsub) * hrows;
    rows = hrows;
  } else {
    const int b2 = b - nheavy * hsub;
    e = tiles[ndiag + nheavy + b2 / nrb];
    r0 = (b2 % nrb) * 64;
    rows = 64;
  }
  const int i = e >> 16, j = e & 0xffff;
  const int t = tidx(i, j);
  const int cls = v.cls[t];
  const bool use_df = p.use_df && cls != CR_PREC_FP64;
  // FP16 tiles take the single-precision evaluation for the closed-form Matern orders and for
  // the power-exponential family
  const bool fast16 = cls == CR_PREC_FP16 && (p.use_df || p.family == CR_COV_POWEXP);
  float4* s_col = s_pts;
  float4* s_row = s_pts + nb;
  if (use_df || fast16) {
    for (int q = threadIdx.x; q < nb + rows; q += blockDim.x) {
      const int g = q < nb ? j * nb + q : i * nb + r0 + (q - nb);
      s_pts[q] = g < n ? __ldg(xy4 + g) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  for (int q = threadIdx.x; q < 64; q += blockDim.x) {
    s_T.t_hi[q] = c_dfexp.t_hi[q];
    s_T.t_lo[q] = c_dfexp.t_lo[q];
  }
  if (threadIdx.x == 0) { s_T.c1 = c_dfexp.c1; s_T.c2 = c_dfexp.c2; s_T.c3 = c_dfexp.c3; }
  __syncthreads();
  const size_t count = (size_t)nb * nb;
  if (fast16) {
    uint2* dst = reinterpret_cast<uint2*>(v.pool16 + (size_t)v.hi16[t] * count);
    switch (p.family == CR_COV_POWEXP ? 3 : p.kind) {
      case 0: gen_fp16_tile<0>(p, n, nb, i, j, r0, s2, s_col, s_row, dst); break;
      case 1: gen_fp16_tile<1>(p, n, nb, i, j, r0, s2, s_col, s_row, dst); break;
      case 2: gen_fp16_tile<2>(p, n, nb, i, j, r0, s2, s_col, s_row, dst); break;
      default: gen_fp16_tile<3>(p, n, nb, i, j, r0, s2, s_col, s_row, dst); break;
    }
    return;
  }
  const df sig = {p.sig_hi, p.sig_lo}, invr = {p.invr_hi, p.invr_lo}, s2d = {s2_hi, s2_lo};
  if (use_df && cls == CR_PREC_FP32 && i != j) {
    float* dst = v.pool32 + (size_t)v.i32[t] * count;
    const df ss = df_mul(sig, s2d);
    switch (p.kind) {
      case 0: gen_fp32_tile<0>(p, xy, n, nb, i, j, r0, rows, s2, ss, invr, s_col, s_row, s_T, dst); break;
      case 1: gen_fp32_tile<1>(p, xy, n, nb, i, j, r0, rows, s2, ss, invr, s_col, s_row, s_T, dst); break;
      default: gen_fp32_tile<2>(p, xy, n, nb, i, j, r0, rows, s2, ss, invr, s_col, s_row, s_T, dst); break;
    }
    return;
  }
  for (int c = threadIdx.x; c < nb; c += blockDim.x)
#pragma unroll 1
  for (int r = r0; r < r0 + rows; ++r) {
    const int gi = i * nb + r, gj = j * nb + c;
    const size_t off = (size_t)r * nb + c;
    double v64 = 0.0;
    df vd = {0.0f, 0.0f};
    bool have_df = false;
    if (gi >= n || gj >= n) {
      v64 = (gi == gj) ? s2 : 0.0;
    } else if (cls == CR_PREC_FP64 && i == j && c > r) {
      v64 = 0.0;   // upper part of a diagonal tile: never read (the factorisation uses the lower part)
    } else if (use_df && gi != gj) {
      const float4 a = s_row[r - r0], b = s_col[c];
      const df dx = df_add({a.x, a.y}, df_neg({b.x, b.y}));
      const df dy = df_add({a.z, a.w}, df_neg({b.z, b.w}));
      bool fb = false;
      vd = cov_entry_df(p, dx, dy, sig, invr, s_T, &fb);
      if (__builtin_expect(fb, 0)) v64 = cov_entry64_ool(p, xy, gi, gj) * s2;
      else { vd = df_mul(vd, s2d); have_df = true; }
    } else {
      v64 = cov_entry64(p, xy, gi, gj) * s2;
    }
    if (cls == CR_PREC_FP64) {
      v.pool64[(size_t)v.i64[t] * count + off] = v64;
    } else {
      const float f = have_df ? __fadd_rn(vd.hi, vd.lo) : (float)v64;
      if (cls == CR_PREC_FP32) v.pool32[(size_t)v.i32[t] * count + off] = f;
      else v.pool16[(size_t)v.hi16[t] * count + off] = __float2half_rn(f);
    }
  }
}

// Dense column-major lower triangle of V (what = 0, FP64 evaluation) or of the working
// tiles as stored (what = 1).
__global__ void k_to_dense(const double* __restrict__ xy, CovK p, TileView v, int what, double* __restrict__ out, int ld) {
  const int n = v.n, nb = v.nb;
  const int gj = blockIdx.x * 32 + (threadIdx.x & 31);
  for (int gi = blockIdx.y * 8 + (threadIdx.x >> 5); gi < n; gi += gridDim.y * 8) {
    if (gj >= n) continue;
    double val = 0.0;
    if (gi >= gj) {
      if (what == 0) {
        val = cov_entry64(p, xy, gi, gj);
      } else {
        const int i = gi / nb, j = gj / nb, r = gi % nb, c = gj % nb;
        const int t = tidx(i, j);
        const size_t off = (size_t)r * nb + c;
        const size_t count = (size_t)nb * nb;
        const int cls = v.cls[t];
        if (cls == CR_PREC_FP64) val = v.pool64[(size_t)v.i64[t] * count + off];
        else if (cls == CR_PREC_FP32) val = (double)v.pool32[(size_t)v.i32[t] * count + off];
        else val = (double)__half2float(v.pool16[(size_t)v.hi16[t] * count + off]);
      }
    }
    out[(size_t)gj * ld + gi] = val;
  }
}

__global__ void k_cov_block(CovK p, const double* __restrict__ xy, int r0, int c0, int m, int k, double* __restrict__ out,
                            int ld) {
  const size_t total = (size_t)m * k;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const int jj = (int)(e / m), ii = (int)(e % m);
    out[(size_t)jj * ld + ii] = cov_entry64(p, xy, r0 + ii, c0 + jj);
  }
}

cr_status cov_block_launch(const CovK& p, const double* xy, int n, int r0, int c0, int m, int k, double* out, int ld,
                           cudaStream_t s) {
  (void)n;
  k_cov_block<<<2048, 256, 0, s>>>(p, xy, r0, c0, m, k, out, ld);
  CR_CHECK_LAUNCH("k_cov_block");
  return CR_OK;
}

// Per-device upload of the double-float exponential's constants.
static cr_status ensure_df_tables() {
  static std::mutex mu;
  static bool done[64] = {false};
  int dev = 0;
  CR_CUDA(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lk(mu);
  if (dev < 64 && done[dev]) return CR_OK;
  DfExpTables T;
  for (int q = 0; q < 64; ++q) {
    const df d = df_from_double(exp2((double)q / 64.0));
    T.t_hi[q] = d.hi;
    T.t_lo[q] = d.lo;
  }
  const double c = log(2.0) / 64.0;                 // in [2^-7, 2^-6): 11 significant bits -> step 2^-17
  const double c1 = nearbyint(c * 131072.0) / 131072.0;
  T.c1 = (float)c1;
  T.c2 = (float)(c - c1);
  T.c3 = (float)(c - c1 - (double)T.c2);
  CR_CUDA(cudaMemcpyToSymbol(c_dfexp, &T, sizeof(T)));
  if (dev < 64) done[dev] = true;
  return CR_OK;
}

cr_status fetch_stats(cr_tilemat V);

}  // namespace cr

using namespace cr;

extern "C" cr_status cr_cov_build(cr_tilemat V, const double* d_xy, const cr_cov_params* p, cr_stream stream) {
  if (!V || !d_xy || !p) return fail(CR_ERR_ARG, "cr_cov_build: NULL argument");
  if (p->family != CR_COV_MATERN && p->family != CR_COV_POWEXP) return fail(CR_ERR_ARG, "cr_cov_build: family");
  if (!(p->sigma2 > 0) || !(p->range > 0) || !(p->nu > 0) || !(p->nugget >= 0) || !(p->tau2 >= 0) ||
      p->n_pred < 0 || p->n_pred > V->n)
    return fail(CR_ERR_ARG, "cr_cov_build: parameter out of range");
  if (p->family == CR_COV_POWEXP && p->nu > 2.0) return fail(CR_ERR_ARG, "cr_cov_build: power-exponential needs nu <= 2");
  CR_CUDA(cudaSetDevice(V->device));
  CR_TRY(ensure_df_tables());
  CovK k{};
  k.family = p->family;
  k.sigma2 = p->sigma2;
  k.inv_range = 1.0 / p->range;
  k.nu = p->nu;
  k.nugget = p->nugget;
  k.tau2 = p->tau2;
  k.n_pred = p->n_pred;
  k.kind = 3;
  if (p->family == CR_COV_MATERN) {
    if (p->nu == 0.5) k.kind = 0;
    else if (p->nu == 1.5) k.kind = 1;
    else if (p->nu == 2.5) k.kind = 2;
    k.norm = exp((1.0 - p->nu) * log(2.0) - lgamma(p->nu));
  }
  k.use_df = (p->family == CR_COV_MATERN && k.kind <= 2) ? 1 : 0;
  {
    const df a = df_from_double(k.sigma2), b = df_from_double(k.inv_range);
    k.sig_hi = a.hi; k.sig_lo = a.lo; k.invr_hi = b.hi; k.invr_lo = b.lo;
  }
  CR_CUDA(cudaMemcpyAsync(V->xy, d_xy, (size_t)V->n * 2 * sizeof(double), cudaMemcpyDeviceToDevice, stream));
  k_points_df<<<(V->n + 255) / 256, 256, 0, stream>>>(V->xy, V->n, V->xy4);
  CR_CHECK_LAUNCH("k_points_df");
  const int nrb = V->nb / 64;
  dim3 grid(V->ntiles, nrb);
  const size_t smem = (size_t)(V->nb + 64) * sizeof(float4);
  {
    // closed-form Matern orders: diagonal tiles exact, off-diagonal tiles through the
    // error-bounded FP32 pass (the policy refines the tiles its decisions depend on);
    // the other covariances: every tile exact
    TimedScope ts("k_cov_stats", stream);
    if (k.use_df)
      k_cov_stats_split<<<(unsigned)V->ntiles * nrb, 256, smem, stream>>>(V->xy, V->xy4, V->n, V->nb, V->nt, k,
                                                                          V->stat_part);
    else
      k_cov_stats<false, 64><<<grid, 256, smem, stream>>>(V->xy, V->xy4, V->n, V->nb, k, V->stat_part, nullptr, 0);
  }
  CR_CHECK_LAUNCH("k_cov_stats");
  k_stats_reduce<<<(V->ntiles + 127) / 128, 128, 0, stream>>>(V->stat_part, V->ntiles, nrb, V->stats, nullptr, 0);
  CR_CHECK_LAUNCH("k_stats_reduce");
  V->params = *p;
  V->covk = k;
  V->built = true;
  V->stats_on_host = false;
  V->mapped = false;
  V->factored = false;
  return CR_OK;
}

namespace cr {
cr_status fetch_stats(cr_tilemat V) {
  if (!V->built) return fail(CR_ERR_STATE, "covariance not built");
  if (V->stats_on_host) return CR_OK;
  std::vector<double> st(STAT_W * (size_t)V->ntiles);
  CR_CUDA(cudaSetDevice(V->device));
  CR_CUDA(cudaDeviceSynchronize());
  CR_CUDA(cudaMemcpy(st.data(), V->stats, st.size() * sizeof(double), cudaMemcpyDeviceToHost));
  V->h_frob.resize(V->ntiles);
  V->h_vmin.resize(V->ntiles);
  V->h_vmax.resize(V->ntiles);
  V->h_stat_err.resize(V->ntiles);
  V->h_stat_exact.resize(V->ntiles);
  for (int t = 0; t < V->ntiles; ++t) {
    V->h_frob[t] = sqrt(st[STAT_W * t]);
    V->h_vmin[t] = st[STAT_W * t + 1];
    V->h_vmax[t] = st[STAT_W * t + 2];
    V->h_stat_err[t] = st[STAT_W * t + 3];
    V->h_stat_exact[t] = st[STAT_W * t + 3] == 0.0;
  }
  // A non-finite sum of squares means non-finite entries: a NaN or infinite coordinate (the
  // covariance of finite sites is finite).  Reported here, before any factorisation.
  for (int t = 0; t < V->ntiles; ++t)
    if (!std::isfinite(V->h_frob[t]))
      return fail(CR_ERR_ARG, "covariance statistics not finite (tile " + std::to_string(t) +
                                  "): a NaN or infinite site coordinate");
  V->stats_on_host = true;
  return CR_OK;
}

// Exact statistics of the listed tiles (replacing their FP32 records), then a fresh copy of
// every record on the host.
cr_status refine_stats(cr_tilemat V, const std::vector<int>& list) {
  if (list.empty()) return CR_OK;
  CR_CUDA(cudaSetDevice(V->device));
  if (!V->d_refine) CR_CUDA(cudaMalloc(&V->d_refine, (size_t)V->ntiles * sizeof(int)));
  // 16-row blocks: 4x the CTAs of the statistics pass, each 4x shorter (a few tiles only)
  constexpr int RR = 16;
  const int nrr = V->nb / RR;
  if (!V->refine_part) CR_CUDA(cudaMalloc(&V->refine_part, (size_t)V->ntiles * nrr * STAT_W * sizeof(double)));
  CR_CUDA(cudaMemcpy(V->d_refine, list.data(), list.size() * sizeof(int), cudaMemcpyHostToDevice));
  const size_t smem = (size_t)(V->nb + 64) * sizeof(float4);
  const dim3 grid((unsigned)list.size(), nrr);
  {
    TimedScope ts("k_cov_stats_refine", 0);
    if (V->covk.use_df)
      k_cov_stats<true, RR><<<grid, 256, smem, 0>>>(V->xy, V->xy4, V->n, V->nb, V->covk, V->refine_part, V->d_refine, 1);
    else
      k_cov_stats<false, RR><<<grid, 256, smem, 0>>>(V->xy, V->xy4, V->n, V->nb, V->covk, V->refine_part, V->d_refine,
                                                     1);
  }
  CR_CHECK_LAUNCH("k_cov_stats");
  k_stats_reduce<<<((unsigned)list.size() + 127) / 128, 128, 0, 0>>>(V->refine_part, (int)list.size(), nrr, V->stats,
                                                                      V->d_refine, 1);
  CR_CHECK_LAUNCH("k_stats_reduce");
  V->stats_on_host = false;
  return fetch_stats(V);
}

cr_status convert_tiles(cr_tilemat V, const int* d_tiles, int count, int ndiag, int nheavy, bool diag_df,
                        cudaStream_t stream) {
  if (count <= 0) return CR_OK;
  // heavy tiles: the largest row block (64, 32 or 16) that still gives them three waves of
  // CTAs (two CTAs per SM), so that a launch with few heavy tiles does not end on them
  int sms = 0, dev = 0;
  CR_CUDA(cudaGetDevice(&dev));
  CR_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  int hrows = 64;
  while (hrows > 16 && (long)nheavy * (V->nb / hrows) < 3L * 2 * sms) hrows /= 2;
  const unsigned grid = (unsigned)ndiag * (V->nb / 16) + (unsigned)nheavy * (V->nb / hrows) +
                        (unsigned)(count - ndiag - nheavy) * (V->nb / 64);
  const size_t smem = (size_t)(V->nb + 64) * sizeof(float4);
  const double s2 = V->s * V->s;
  const df s2d = df_from_double(s2);
  {
    TimedScope ts("k_generate", stream);
    k_generate<<<grid, 256, smem, stream>>>(V->xy, V->xy4, V->n, V->nb, V->covk, s2, s2d.hi, s2d.lo, V->view(), d_tiles, ndiag,
                                            nheavy, hrows, diag_df && V->covk.use_df ? 1 : 0);
  }
  CR_CHECK_LAUNCH("k_generate");
  return CR_OK;
}
}  // namespace cr

extern "C" cr_status cr_tile_stats(cr_tilemat V, double* h_frob, double* h_vmin, double* h_vmax) {
  if (!V) return fail(CR_ERR_ARG, "cr_tile_stats: NULL handle");
  CR_TRY(fetch_stats(V));
  {
    std::vector<int> rest;
    for (int t = 0; t < V->ntiles; ++t)
      if (!V->h_stat_exact[t]) rest.push_back(t);
    CR_TRY(refine_stats(V, rest));
  }
  const int nt = V->nt;
  for (int i = 0; i < nt; ++i)
    for (int j = 0; j < nt; ++j) {
      const bool low = j <= i;
      const int t = low ? tidx(i, j) : 0;
      if (h_frob) h_frob[i * nt + j] = low ? V->h_frob[t] : 0.0;
      if (h_vmin) h_vmin[i * nt + j] = low ? V->h_vmin[t] : 0.0;
      if (h_vmax) h_vmax[i * nt + j] = low ? V->h_vmax[t] : 0.0;
    }
  return CR_OK;
}

extern "C" cr_status cr_tile_stats_records(cr_tilemat V, double* h_frob, double* h_vmin, double* h_vmax,
                                          double* h_err) {
  if (!V) return fail(CR_ERR_ARG, "cr_tile_stats_records: NULL handle");
  CR_TRY(fetch_stats(V));
  const int nt = V->nt;
  for (int i = 0; i < nt; ++i)
    for (int j = 0; j < nt; ++j) {
      const bool low = j <= i;
      const int t = low ? tidx(i, j) : 0;
      if (h_frob) h_frob[i * nt + j] = low ? V->h_frob[t] : 0.0;
      if (h_vmin) h_vmin[i * nt + j] = low ? V->h_vmin[t] : 0.0;
      if (h_vmax) h_vmax[i * nt + j] = low ? V->h_vmax[t] : 0.0;
      if (h_err) h_err[i * nt + j] = low ? V->h_stat_err[t] : 0.0;
    }
  return CR_OK;
}

extern "C" cr_status cr_tilemat_to_dense(cr_tilemat V, int what, double* d_out, int ld, cr_stream stream) {
  if (!V || !d_out || ld < V->n || what < 0 || what > 2) return fail(CR_ERR_ARG, "cr_tilemat_to_dense: argument");
  if (what == 0 && !V->built) return fail(CR_ERR_STATE, "cr_tilemat_to_dense: covariance not built");
  if (what >= 1 && !V->mapped) return fail(CR_ERR_STATE, "cr_tilemat_to_dense: no working tiles yet");
  CR_CUDA(cudaSetDevice(V->device));
  if (what == 2) {
    // the generation step of cr_potrf_adaptive alone, over every tile: diagonal tiles first,
    // then the FP64/FP32-class tiles, then the FP16-class ones (the launch's expected order),
    // the diagonal ones in double-float when the double-float executor would factor them
    const int nt = V->nt;
    std::vector<int> list;
    for (int i = 0; i < nt; ++i) list.push_back(i << 16 | i);
    int nheavy = 0;
    for (int pass = 0; pass < 2; ++pass)
      for (int i = 0; i < nt; ++i)
        for (int j = 0; j < i; ++j) {
          const bool heavy = V->h_cls[tidx(i, j)] != CR_PREC_FP16;
          if (heavy == (pass == 0)) {
            list.push_back(i << 16 | j);
            nheavy += heavy ? 1 : 0;
          }
        }
    const int arith = option_diag_arith();
    const bool use_df = arith == CR_DIAG_DF || (arith == CR_DIAG_AUTO && V->amp);
    int* d_list = nullptr;
    CR_CUDA(cudaMallocAsync(&d_list, list.size() * sizeof(int), stream));
    const cudaError_t ce = cudaMemcpyAsync(d_list, list.data(), list.size() * sizeof(int), cudaMemcpyHostToDevice, stream);
    cr_status st = ce == cudaSuccess ? convert_tiles(V, d_list, (int)list.size(), nt, nheavy, use_df, stream)
                                     : cuda_fail(ce, "cr_tilemat_to_dense: tile list");
    cudaFreeAsync(d_list, stream);
    // the list is copied from host memory that goes out of scope here
    CR_CUDA(cudaStreamSynchronize(stream));
    CR_TRY(st);
    V->factored = false;   // the storage now holds s^2 V, not the factor
  }
  dim3 grid((V->n + 31) / 32, 64);
  k_to_dense<<<grid, 256, 0, stream>>>(V->xy, V->covk, V->view(), what == 0 ? 0 : 1, d_out, ld);
  CR_CHECK_LAUNCH("k_to_dense");
  return CR_OK;
}
