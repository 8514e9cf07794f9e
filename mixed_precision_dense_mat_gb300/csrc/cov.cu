// Covariance tile generation, tile statistics, conversion to the precision classes and
// dense extraction.
//
// "Mixed-Precision GPU Acceleration for Confidence Regions of Spatial Excursion Sets":
// Section V Eq.4 (joint covariance, tau^2 on the observation block only), Section VI-B.2
// (power-exponential model), Section VI-C (Matern model), Section V-D (tile Frobenius
// norms and entry extrema used by the precision checks), Alg.2 step 12 (scaling by s^2
// and rounding each tile to its class).
#include <math.h>

#include "common.cuh"

namespace cr {

struct CovK {
  int family;        // CR_COV_*
  int kind;          // Matern: 0 nu=1/2, 1 nu=3/2, 2 nu=5/2, 3 general (quadrature)
  double sigma2, inv_range, nu, nugget, tau2, norm;   // norm = 2^(1-nu) / Gamma(nu)
  int n_pred;
};

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

// Correlation part of the covariance at scaled distance x = h / range > 0.
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

__device__ __forceinline__ double cov_entry(const CovK& p, const double* __restrict__ xy, int n,
                                            int gi, int gj, double xi, double yi) {
  if (gi == gj) return p.sigma2 + p.nugget + (gi >= p.n_pred ? p.tau2 : 0.0);
  const double dx = xi - xy[2 * gj], dy = yi - xy[2 * gj + 1];
  const double h = sqrt(dx * dx + dy * dy);
  if (h == 0.0) return p.sigma2;
  return cov_of_x(p, h * p.inv_range);
}

// One CTA per (lower tile, 64-row block).  Writes the FP64 tile rows and partial
// statistics (sum of squares, min, max over valid entries) of its rows.
__global__ void __launch_bounds__(256) k_cov_tiles(const double* __restrict__ xy, int n, int nb,
                                                   CovK p, double* __restrict__ master,
                                                   double* __restrict__ stat_part) {
  const int t = blockIdx.x;
  const int rbk = blockIdx.y;
  const int nrb = gridDim.y;
  int i = (int)floor((sqrt(8.0 * t + 1.0) - 1.0) * 0.5);
  while (i * (i + 1) / 2 > t) --i;
  while ((i + 1) * (i + 2) / 2 <= t) ++i;
  const int j = t - i * (i + 1) / 2;

  __shared__ double s_x[64], s_y[64];
  const int r0 = rbk * 64;
  if (threadIdx.x < 64) {
    const int gi = i * nb + r0 + threadIdx.x;
    s_x[threadIdx.x] = gi < n ? xy[2 * gi] : 0.0;
    s_y[threadIdx.x] = gi < n ? xy[2 * gi + 1] : 0.0;
  }
  __syncthreads();

  double ssq = 0.0, vmn = INFINITY, vmx = -INFINITY;
  double* out = master + (size_t)t * nb * nb;
  for (int idx = threadIdx.x; idx < 64 * nb; idx += blockDim.x) {
    const int r = r0 + idx / nb, c = idx % nb;
    const int gi = i * nb + r, gj = j * nb + c;
    double v;
    if (gi >= n || gj >= n) {
      v = (gi == gj) ? 1.0 : 0.0;
    } else {
      v = cov_entry(p, xy, n, gi, gj, s_x[r - r0], s_y[r - r0]);
      ssq += v * v;
      vmn = fmin(vmn, v);
      vmx = fmax(vmx, v);
    }
    out[(size_t)r * nb + c] = v;
  }
  // block reduction
  __shared__ double red[3][8];
  for (int o = 16; o > 0; o >>= 1) {
    ssq += __shfl_down_sync(0xffffffffu, ssq, o);
    vmn = fmin(vmn, __shfl_down_sync(0xffffffffu, vmn, o));
    vmx = fmax(vmx, __shfl_down_sync(0xffffffffu, vmx, o));
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) { red[0][w] = ssq; red[1][w] = vmn; red[2][w] = vmx; }
  __syncthreads();
  if (threadIdx.x == 0) {
    double a = 0.0, b = INFINITY, c = -INFINITY;
    for (int q = 0; q < (int)(blockDim.x >> 5); ++q) { a += red[0][q]; b = fmin(b, red[1][q]); c = fmax(c, red[2][q]); }
    double* sp = stat_part + ((size_t)t * nrb + rbk) * 3;
    sp[0] = a; sp[1] = b; sp[2] = c;
  }
}

__global__ void k_stats_reduce(const double* __restrict__ part, int ntiles, int nrb, double* __restrict__ stats) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= ntiles) return;
  double a = 0.0, b = INFINITY, c = -INFINITY;
  for (int q = 0; q < nrb; ++q) {
    const double* sp = part + ((size_t)t * nrb + q) * 3;
    a += sp[0]; b = fmin(b, sp[1]); c = fmax(c, sp[2]);
  }
  stats[3 * t] = a; stats[3 * t + 1] = b; stats[3 * t + 2] = c;
}

// Scale by s^2 and round each tile to its class (Alg.2 step 12).
__global__ void __launch_bounds__(256) k_convert(const double* __restrict__ master, int nb, double s2,
                                                 TileView v) {
  const int t = blockIdx.x;
  const size_t base = (size_t)t * nb * nb;
  const size_t count = (size_t)nb * nb;
  const int cls = v.cls[t];
  const size_t chunk = count / gridDim.y;
  const size_t beg = chunk * blockIdx.y;
  const double2* src = reinterpret_cast<const double2*>(master + base + beg);
  if (cls == CR_PREC_FP64) {
    double2* dst = reinterpret_cast<double2*>(v.pool64 + (size_t)v.i64[t] * count + beg);
    for (size_t q = threadIdx.x; q < chunk / 2; q += blockDim.x) {
      double2 a = src[q];
      dst[q] = make_double2(a.x * s2, a.y * s2);
    }
  } else if (cls == CR_PREC_FP32) {
    float2* dst = reinterpret_cast<float2*>(v.pool32 + (size_t)v.i32[t] * count + beg);
    for (size_t q = threadIdx.x; q < chunk / 2; q += blockDim.x) {
      double2 a = src[q];
      dst[q] = make_float2((float)(a.x * s2), (float)(a.y * s2));
    }
  } else {
    __half2* dst = reinterpret_cast<__half2*>(v.pool16 + (size_t)v.hi16[t] * count + beg);
    for (size_t q = threadIdx.x; q < chunk / 2; q += blockDim.x) {
      double2 a = src[q];
      dst[q] = __halves2half2(__double2half(a.x * s2), __double2half(a.y * s2));
    }
  }
}

// Dense column-major copy of the lower triangle (what = 0: covariance, 1: working tiles).
__global__ void k_to_dense(const double* __restrict__ master, TileView v, int what, double* __restrict__ out, int ld) {
  const int n = v.n, nb = v.nb;
  const int gj = blockIdx.x * 32 + (threadIdx.x & 31);
  for (int gi = blockIdx.y * 8 + (threadIdx.x >> 5); gi < n; gi += gridDim.y * 8) {
    if (gj >= n) continue;
    double val = 0.0;
    if (gi >= gj) {
      const int i = gi / nb, j = gj / nb, r = gi % nb, c = gj % nb;
      const int t = tidx(i, j);
      const size_t off = (size_t)r * nb + c;
      const size_t count = (size_t)nb * nb;
      if (what == 0) {
        val = master[(size_t)t * count + off];
      } else {
        const int cls = v.cls[t];
        if (cls == CR_PREC_FP64) val = v.pool64[(size_t)v.i64[t] * count + off];
        else if (cls == CR_PREC_FP32) val = (double)v.pool32[(size_t)v.i32[t] * count + off];
        else val = (double)__half2float(v.pool16[(size_t)v.hi16[t] * count + off]);
      }
    }
    out[(size_t)gj * ld + gi] = val;
  }
}

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
  const int nrb = V->nb / 64;
  dim3 grid(V->ntiles, nrb);
  k_cov_tiles<<<grid, 256, 0, stream>>>(d_xy, V->n, V->nb, k, V->master, V->stat_part);
  CR_CHECK_LAUNCH("k_cov_tiles");
  k_stats_reduce<<<(V->ntiles + 127) / 128, 128, 0, stream>>>(V->stat_part, V->ntiles, nrb, V->stats);
  CR_CHECK_LAUNCH("k_stats_reduce");
  V->params = *p;
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
  std::vector<double> st(3 * (size_t)V->ntiles);
  CR_CUDA(cudaSetDevice(V->device));
  CR_CUDA(cudaDeviceSynchronize());
  CR_CUDA(cudaMemcpy(st.data(), V->stats, st.size() * sizeof(double), cudaMemcpyDeviceToHost));
  V->h_frob.resize(V->ntiles);
  V->h_vmin.resize(V->ntiles);
  V->h_vmax.resize(V->ntiles);
  for (int t = 0; t < V->ntiles; ++t) {
    V->h_frob[t] = sqrt(st[3 * t]);
    V->h_vmin[t] = st[3 * t + 1];
    V->h_vmax[t] = st[3 * t + 2];
  }
  V->stats_on_host = true;
  return CR_OK;
}

cr_status convert_tiles(cr_tilemat V, cudaStream_t stream) {
  dim3 grid(V->ntiles, 8);
  k_convert<<<grid, 256, 0, stream>>>(V->master, V->nb, V->s * V->s, V->view());
  CR_CHECK_LAUNCH("k_convert");
  return CR_OK;
}
}  // namespace cr

extern "C" cr_status cr_tile_stats(cr_tilemat V, double* h_frob, double* h_vmin, double* h_vmax) {
  if (!V) return fail(CR_ERR_ARG, "cr_tile_stats: NULL handle");
  CR_TRY(fetch_stats(V));
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

extern "C" cr_status cr_tilemat_to_dense(cr_tilemat V, int what, double* d_out, int ld, cr_stream stream) {
  if (!V || !d_out || ld < V->n || (what != 0 && what != 1)) return fail(CR_ERR_ARG, "cr_tilemat_to_dense: argument");
  if (what == 0 && !V->built) return fail(CR_ERR_STATE, "cr_tilemat_to_dense: covariance not built");
  if (what == 1 && !V->mapped) return fail(CR_ERR_STATE, "cr_tilemat_to_dense: no working tiles yet");
  CR_CUDA(cudaSetDevice(V->device));
  dim3 grid((V->n + 31) / 32, 64);
  k_to_dense<<<grid, 256, 0, stream>>>(V->master, V->view(), what, d_out, ld);
  CR_CHECK_LAUNCH("k_to_dense");
  return CR_OK;
}
