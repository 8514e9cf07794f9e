// Host-side precision policy and allocation of the per-precision tile storage.
//
// "Mixed-Precision GPU Acceleration for Confidence Regions of Spatial Excursion Sets":
//  - Section IV-B / VI-D: per-tile FP64/FP32/FP16 chosen by comparing each tile's norm with
//    the global norm; diagonal tiles stay FP64.  Rule used: off-diagonal tile (i, j) takes
//    the lowest p in {FP16, FP32} with ||V_ij||_F * NT <= (fixedacc / eps_p) ||V||_F, else
//    FP64 (eps_FP16 = 2^-10 as in Eq.11, eps_FP32 = 2^-23); ||V||_F over the full symmetric
//    matrix.
//  - Section V-D: automatic mode (start 1e-4, times 0.9 while a check fails, stop when both
//    pass or no FP16 tile is left); Eq.10 and Eq.11 checks over the FP16 tiles.
//  - Section V-E Eq.12: s = floor(min(65504, min_f u_f)) - 1 when above 1, else 1.
#include <float.h>
#include <math.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"

namespace cr {
cr_status fetch_stats(cr_tilemat V);
cr_status refine_stats(cr_tilemat V, const std::vector<int>& list);

namespace {

struct Checks {
  int n16 = 0;
  double R = NAN, rho1 = NAN, rho2 = NAN;
  bool c1 = true, c2 = true;
};

void make_map(const cr_tilemat V, double fixedacc, std::vector<int8_t>& cls) {
  const int nt = V->nt;
  double g2 = 0.0;
  for (int i = 0; i < nt; ++i) {
    g2 += V->h_frob[tidx(i, i)] * V->h_frob[tidx(i, i)];
    for (int j = 0; j < i; ++j) g2 += 2.0 * V->h_frob[tidx(i, j)] * V->h_frob[tidx(i, j)];
  }
  const double g = sqrt(g2);
  const double lim16 = (fixedacc / ldexp(1.0, -10)) * g;
  const double lim32 = (fixedacc / ldexp(1.0, -23)) * g;
  cls.assign(V->ntiles, CR_PREC_FP64);
  for (int i = 0; i < nt; ++i)
    for (int j = 0; j < i; ++j) {
      const double lhs = V->h_frob[tidx(i, j)] * nt;
      cls[tidx(i, j)] = lhs <= lim16 ? CR_PREC_FP16 : (lhs <= lim32 ? CR_PREC_FP32 : CR_PREC_FP64);
    }
}

Checks checks(const cr_tilemat V, const std::vector<int8_t>& cls) {
  Checks c;
  double vmax_hp = -INFINITY, vmin_hp = INFINITY, fmax_hp = -INFINITY, vmax_all = -INFINITY, fmax_all = -INFINITY;
  for (int t = 0; t < V->ntiles; ++t) {
    vmax_all = std::max(vmax_all, V->h_vmax[t]);
    fmax_all = std::max(fmax_all, V->h_frob[t]);
    if (cls[t] == CR_PREC_FP16) {
      ++c.n16;
      vmax_hp = std::max(vmax_hp, V->h_vmax[t]);
      vmin_hp = std::min(vmin_hp, V->h_vmin[t]);
      fmax_hp = std::max(fmax_hp, V->h_frob[t]);
    }
  }
  if (c.n16 == 0) return c;
  c.R = vmax_hp / vmin_hp;
  c.rho1 = vmax_hp / vmax_all;
  c.rho2 = fmax_hp / fmax_all;
  c.c1 = c.R < 65504.0 / ldexp(1.0, -24);
  c.c2 = std::max(c.rho1, c.rho2) < 1e-4 / ldexp(1.0, -10);
  return c;
}

void scale(const cr_tilemat V, const std::vector<int8_t>& cls, cr_pmap_info* info) {
  const double xmin[2] = {ldexp(1.0, -126), ldexp(1.0, -14)};   // FP32, FP16
  const double xmax[2] = {(double)FLT_MAX, 65504.0};
  const int fmt[2] = {CR_PREC_FP32, CR_PREC_FP16};
  double ell = -INFINITY, us = 65504.0;
  // every factor tile of L_s = s L enters the TRMM as an FP16 cast (Alg.1 step 15) and the
  // largest factor entry is sqrt(max V_ii): u_s also keeps s sqrt(max V_ii) inside FP16
  double vmax_all = -INFINITY;
  for (int t = 0; t < V->ntiles; ++t) vmax_all = std::max(vmax_all, V->h_vmax[t]);
  if (vmax_all > 0) us = std::min(us, 65504.0 / sqrt(vmax_all));
  bool present = false;
  for (int q = 0; q < 2; ++q) {
    double vmn = INFINITY, vmx = -INFINITY;
    bool any = false;
    for (int i = 0; i < V->nt; ++i)
      for (int j = 0; j < i; ++j)
        if (cls[tidx(i, j)] == fmt[q]) {
          any = true;
          vmn = std::min(vmn, V->h_vmin[tidx(i, j)]);
          vmx = std::max(vmx, V->h_vmax[tidx(i, j)]);
        }
    if (!any) continue;
    present = true;
    const double lf = vmn > 0 ? sqrt(xmin[q] / vmn) : INFINITY;
    const double uf = vmx > 0 ? sqrt(xmax[q] / vmx) : INFINITY;
    ell = std::max(ell, lf);
    us = std::min(us, uf);
  }
  if (!present) {
    info->s = 1.0; info->ell = NAN; info->u_s = NAN; info->range_ok = 1;
    return;
  }
  const double cand = floor(us) - 1.0;
  info->s = cand > 1.0 ? cand : 1.0;
  info->ell = ell;
  info->u_s = us;
  info->range_ok = ell <= us;
}

// ---- decisions on error-bounded statistics --------------------------------------------------
// A tile's statistics are either exact (double-float / FP64 pass) or from the FP32 pass with a
// relative bound E on each of them.  The policy runs on the point values; then every
// comparison it made is re-examined over the intervals the bounds allow, and the FP32 tiles a
// comparison or an extreme could depend on are recomputed exactly, until none is left.  The
// final map, checks and scale are then those the exact statistics of every tile give.  The
// intervals are widened by 1e-12 relative, far above the exact pass's own error, so that they
// hold the exact pass's values and not only the true ones.
struct Iv {
  double lo, hi;
};

Iv bound(double c, double e) {
  if (e == 0.0) return {c, c};
  if (!(e < 0.5) || !(c >= 0.0)) return {-INFINITY, INFINITY};
  return {c / (1.0 + e) * (1.0 - 1e-12), c / (1.0 - e) * (1.0 + 1e-12)};
}

struct Marks {
  std::vector<char> need;
  bool all = false;   // a decision turns on ||V||_F's uncertainty alone: refine every FP32 tile
  void tile(const cr_tilemat V, int t) {
    if (V->h_stat_exact[t]) all = true;
    else need[t] = 1;
  }
};

// class decisions of the map at accuracy fa that the bounds leave open
void mark_map(const cr_tilemat V, double fa, Marks& m) {
  const int nt = V->nt;
  double g2lo = 0.0, g2hi = 0.0;
  for (int i = 0; i < nt; ++i)
    for (int j = 0; j <= i; ++j) {
      const int t = tidx(i, j);
      const Iv f = bound(V->h_frob[t], V->h_stat_err[t]);
      const double w = i == j ? 1.0 : 2.0, lo = std::max(f.lo, 0.0);
      g2lo += w * lo * lo;
      g2hi += w * f.hi * f.hi;
    }
  const double glo = sqrt(g2lo) * (1.0 - 1e-12), ghi = sqrt(g2hi) * (1.0 + 1e-12);
  const double eps[2] = {ldexp(1.0, -10), ldexp(1.0, -23)};
  for (int i = 0; i < nt; ++i)
    for (int j = 0; j < i; ++j) {
      const int t = tidx(i, j);
      const Iv f = bound(V->h_frob[t], V->h_stat_err[t]);
      const double llo = std::max(f.lo, 0.0) * nt, lhi = f.hi * nt;
      for (int q = 0; q < 2; ++q) {
        const double limlo = (fa / eps[q]) * glo, limhi = (fa / eps[q]) * ghi;
        if (lhi <= limlo) break;      // below this class's limit for every value allowed
        if (llo > limhi) continue;    // above it for every value allowed
        m.tile(V, t);
        break;
      }
    }
}

// the largest (want_max) or smallest value of x over the tiles with sel[t]
template <class Sel>
void mark_extreme(const cr_tilemat V, const std::vector<double>& x, bool want_max, Sel sel, Marks& m) {
  double edge = want_max ? -INFINITY : INFINITY;
  for (int t = 0; t < V->ntiles; ++t)
    if (sel(t)) {
      const Iv b = bound(x[t], V->h_stat_err[t]);
      edge = want_max ? std::max(edge, b.lo) : std::min(edge, b.hi);
    }
  for (int t = 0; t < V->ntiles; ++t)
    if (sel(t) && !V->h_stat_exact[t]) {
      const Iv b = bound(x[t], V->h_stat_err[t]);
      if (want_max ? b.hi >= edge : b.lo <= edge) m.need[t] = 1;
    }
}

// (re)allocates *d only when the new size exceeds its capacity, so that repeated maps of the
// same matrix neither free nor allocate (cudaFree synchronises the device)
template <class T>
cr_status ensure(T** d, size_t* cap, size_t need) {
  if (need <= *cap && *d) return CR_OK;
  if (*d) cudaFree(*d);
  *d = nullptr;
  *cap = 0;
  CR_CUDA(cudaMalloc(d, std::max<size_t>(1, need) * sizeof(T)));
  *cap = need;
  return CR_OK;
}

}  // namespace

cr_status allocate_class_storage(cr_tilemat V) {
  V->mapped = false;
  V->factored = false;
  const int nt = V->nt, T = V->ntiles;
  const size_t tile = (size_t)V->nb * V->nb;
  V->h_i64.assign(T, -1); V->h_i32.assign(T, -1); V->h_hi16.assign(T, -1); V->h_lo16.assign(T, -1);
  V->n64 = V->n32 = 0;
  int off64 = 0;   // off-diagonal FP64 tiles
  for (int t = 0; t < T; ++t) {
    if (V->h_cls[t] == CR_PREC_FP64) V->h_i64[t] = V->n64++;
    else if (V->h_cls[t] == CR_PREC_FP32) V->h_i32[t] = V->n32++;
  }
  for (int i = 0; i < nt; ++i)
    for (int j = 0; j < i; ++j) off64 += V->h_cls[tidx(i, j)] == CR_PREC_FP64;
  V->n16 = 0;
  if (V->amp) {
    for (int t = 0; t < T; ++t) V->h_hi16[t] = V->n16++;
    for (int t = 0; t < T; ++t)
      if (V->h_cls[t] != CR_PREC_FP16) V->h_lo16[t] = V->n16++;
    V->ws_hi0 = V->n16; V->n16 += 2 * nt;   // two sets, by column parity
    V->ws_lo0 = V->n16; V->n16 += 2 * nt;
    V->minv_hi = V->n16; V->n16 += 2;   // by column parity
    V->minv_lo = V->n16; V->n16 += 2;
  }
  // the five per-tile tables in one device buffer and one copy: four int tables, then the
  // class bytes
  {
    const size_t ints = 4 * (size_t)T, bytes = ints * sizeof(int) + (size_t)T;
    if (!V->d_tables) CR_CUDA(cudaMalloc(&V->d_tables, bytes));
    std::vector<int> h(ints + ((size_t)T + sizeof(int) - 1) / sizeof(int), 0);
    std::copy(V->h_i64.begin(), V->h_i64.end(), h.begin());
    std::copy(V->h_i32.begin(), V->h_i32.end(), h.begin() + T);
    std::copy(V->h_hi16.begin(), V->h_hi16.end(), h.begin() + 2 * (size_t)T);
    std::copy(V->h_lo16.begin(), V->h_lo16.end(), h.begin() + 3 * (size_t)T);
    std::memcpy(h.data() + ints, V->h_cls.data(), (size_t)T);
    CR_CUDA(cudaMemcpy(V->d_tables, h.data(), bytes, cudaMemcpyHostToDevice));
    V->d_i64 = V->d_tables;
    V->d_i32 = V->d_tables + T;
    V->d_hi16 = V->d_tables + 2 * (size_t)T;
    V->d_lo16 = V->d_tables + 3 * (size_t)T;
    V->d_cls = reinterpret_cast<int8_t*>(V->d_tables + ints);
  }
  CR_TRY(ensure(&V->pool64, &V->cap64, std::max<size_t>(1, (size_t)V->n64) * tile));
  if (V->n32) CR_TRY(ensure(&V->pool32, &V->cap32, (size_t)V->n32 * tile));
  if (V->n16) {
    CR_TRY(ensure(&V->pool16, &V->cap16, (size_t)V->n16 * tile));
    CR_TRY(make_tensor_map_3d_f16(&V->tm_pool16, V->pool16, V->nb, V->nb, V->n16, 64, 128));
  }
  if (off64 > 0) CR_TRY(ensure(&V->ws64, &V->cap_ws64, 2 * (size_t)nt * tile));
  if (V->amp) CR_TRY(ensure(&V->w32, &V->cap_w32, 2 * (size_t)nt * tile));
  V->mapped = true;
  return CR_OK;
}

}  // namespace cr

using namespace cr;

extern "C" cr_status cr_precision_map(cr_tilemat V, int amp, double fixedacc, int auto_mode, int8_t* h_map,
                                      cr_pmap_info* info) {
  if (!V) return fail(CR_ERR_ARG, "cr_precision_map: NULL handle");
  if (amp && !auto_mode && !(fixedacc > 0)) return fail(CR_ERR_ARG, "cr_precision_map: fixedacc must be > 0");
  CR_CUDA(cudaSetDevice(V->device));
  CR_TRY(fetch_stats(V));
  cr_pmap_info pi{};
  std::vector<int8_t> cls;
  Checks c;
  if (!amp) {
    cls.assign(V->ntiles, CR_PREC_FP64);
    pi.fixedacc = fixedacc;
    pi.iters = 0;
    c = checks(V, cls);
    pi.s = 1.0; pi.ell = NAN; pi.u_s = NAN; pi.range_ok = 1;
  } else {
    double fa = 0.0;
    int it = 0;
    for (;;) {
      std::vector<double> visited;
      fa = auto_mode ? 1e-4 : fixedacc;
      it = 0;
      for (;;) {
        make_map(V, fa, cls);
        c = checks(V, cls);
        visited.push_back(fa);
        ++it;
        if (!auto_mode || c.n16 == 0 || (c.c1 && c.c2) || it >= 100000) break;
        fa = fa * 0.9;
      }
      // re-examine every decision taken above over the statistics' bounds
      Marks m;
      m.need.assign(V->ntiles, 0);
      std::vector<int8_t> ci;
      for (double f : visited) {
        mark_map(V, f, m);
        make_map(V, f, ci);
        auto is16 = [&](int t) { return ci[t] == CR_PREC_FP16; };
        mark_extreme(V, V->h_vmax, true, is16, m);
        mark_extreme(V, V->h_vmin, false, is16, m);
        mark_extreme(V, V->h_frob, true, is16, m);
      }
      auto every = [](int) { return true; };
      mark_extreme(V, V->h_vmax, true, every, m);
      mark_extreme(V, V->h_frob, true, every, m);
      for (int8_t q : {(int8_t)CR_PREC_FP32, (int8_t)CR_PREC_FP16}) {
        auto in_q = [&](int t) { return cls[t] == q; };
        mark_extreme(V, V->h_vmax, true, in_q, m);
        mark_extreme(V, V->h_vmin, false, in_q, m);
      }
      std::vector<int> list;
      for (int t = 0; t < V->ntiles; ++t)
        if (!V->h_stat_exact[t] && (m.all || m.need[t])) list.push_back(t);
      if (list.empty()) break;
      CR_TRY(refine_stats(V, list));
    }
    pi.fixedacc = fa;
    pi.iters = it;
    scale(V, cls, &pi);
  }
  pi.R_hp = c.R; pi.rho1 = c.rho1; pi.rho2 = c.rho2; pi.check1 = c.c1; pi.check2 = c.c2;
  pi.n_fp64 = pi.n_fp32 = pi.n_fp16 = 0;
  double vmax_all = -INFINITY;
  for (int t = 0; t < V->ntiles; ++t) {
    pi.n_fp64 += cls[t] == CR_PREC_FP64;
    pi.n_fp32 += cls[t] == CR_PREC_FP32;
    pi.n_fp16 += cls[t] == CR_PREC_FP16;
    vmax_all = std::max(vmax_all, V->h_vmax[t]);
  }
  if (h_map) {
    for (int i = 0; i < V->nt; ++i)
      for (int j = 0; j < V->nt; ++j) h_map[i * V->nt + j] = j <= i ? cls[tidx(i, j)] : (int8_t)-1;
  }
  if (info) *info = pi;
  V->h_cls = cls;
  V->amp = amp ? 1 : 0;
  V->s = pi.s;
  V->pinfo = pi;
  // Power-of-two scale for FP32-class triangular-solve inputs, which live on the s^2 V scale:
  // W 2^-eA stays below 2^14 so its FP16 high/low split cannot overflow.
  V->eA = 0;
  if (V->amp) {
    const double top = V->s * V->s * vmax_all;
    while (ldexp(top, -V->eA) > 16384.0) ++V->eA;
    // The factor L_s (magnitude up to s sqrt(max V_ii)) is read in FP16 by the simulation
    // multiply (Alg.1 casts every off-diagonal factor tile to FP16).
    if (V->s * sqrt(vmax_all) >= 65520.0)
      return fail(CR_ERR_RANGE, "cr_precision_map: s * sqrt(max V_ii) exceeds the FP16 range");
  }
  return allocate_class_storage(V);
}
