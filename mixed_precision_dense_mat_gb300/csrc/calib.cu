// Calibration of the inner and outer confidence regions.
//
// "Mixed-Precision GPU Acceleration for Confidence Regions of Spatial Excursion Sets":
//  - Alg.2 step 18 / Eq.1: t = (zhat - u) / sqrt(v), positive MSPEs required.
//  - Section V-C Eq.8 / Alg.2 step 19 (Desc_col_summary_index_both): psi_j = min{t_i : S_ij >= u},
//    phi_j = max{t_i : S_ij <= u}, both in one pass over S; sentinels +inf / -inf for empty sets.
//  - Per-location exceedance counts count_i = #{j : S_ij >= u}, fused into the same pass.
//  - Section V-C Eq.9: Q_p(a) = a_(max{1, min{N, ceil(p N)}}) on each sorted sample without
//    sentinels (ceil taken of p N - 1e-9 so a product that is an integer up to rounding stays);
//    q_out = Q_alpha(psi), q_in = Q_{1-alpha}(phi), alpha = 1 - level.
//  - Alg.2 step 22: C_in = {t_i > q_in}, C_out = {t_i >= q_out}.
// The scan streams S once from HBM: each CTA owns a 2048-row x 32-column block, keeps its
// rows' counts in registers and their t keys ranked per thread in shared memory, reduces each
// column with warp shuffles and writes one partial per column; a second kernel combines the
// partials in a fixed order (deterministic).
#include <math.h>

#include <algorithm>
#include <atomic>
#include <functional>
#include <mutex>

#include "calib.cuh"
#include "common.cuh"
#include "df.cuh"

namespace cr {

// t_i = (zhat_i - u) / sqrt(v_i); for a negative excursion set (neg != 0) the statistic of the
// sign-reversed problem, ((-zhat_i) - (-u)) / sqrt(v_i), which is exactly -t_i in IEEE arithmetic.
__global__ void k_tstat(const double* __restrict__ zhat, const double* __restrict__ v, double u, int n_p, double* __restrict__ t,
                        int* __restrict__ bad, int neg) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_p; i += gridDim.x * blockDim.x) {
    const double vi = v[i];
    if (!(vi > 0.0)) atomicOr(bad, 1);
    const double ti = (zhat[i] - u) / sqrt(vi);
    t[i] = neg ? -ti : ti;
  }
}

// Order-preserving 64-bit keys of doubles: for x, y not NaN and with -0 taken as +0,
// x < y exactly when key(x) < key(y) as unsigned integers.  The scan compares and reduces
// keys in integer arithmetic: GB300's FP64 units issue a warp instruction only every ~64
// cycles, which would bound a double-precision scan far below HBM bandwidth.
__device__ __forceinline__ unsigned long long dkey(double x) {
  unsigned long long b = (unsigned long long)__double_as_longlong(x);
  if (b == 0x8000000000000000ull) b = 0;   // -0 -> +0
  return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}
__device__ __forceinline__ double dkey_inv(unsigned long long k) {
  const unsigned long long b = (k >> 63) ? (k & 0x7fffffffffffffffull) : ~k;
  return __longlong_as_double((long long)b);
}

// High 32 bits of dkey(x), except that -0 keeps its own key (0x7fffffff): monotone in x, and
// strictly ordered whenever the high words of two keys differ.
__device__ __forceinline__ unsigned dkey_hi(double x) {
  const unsigned hi = (unsigned)__double2hiint(x);
  return hi ^ ((unsigned)((int)hi >> 31) | 0x80000000u);
}

// neg != 0: the negative excursion set (Section III's sign reversal): -S_ij >= -u is S_ij <= u and
// -S_ij <= -u is S_ij >= u, so the two decisions swap roles (t holds the reversed statistic).
__global__ void __launch_bounds__(SCAN_THREADS) k_scan(const double* __restrict__ S, int lds, int n_p, int M,
                                                       const double* __restrict__ t, double u, double* __restrict__ psi_part,
                                                       double* __restrict__ phi_part, int32_t* __restrict__ count, int neg) {
  constexpr int RPT = SCAN_ROWS / SCAN_THREADS;   // rows per thread
  constexpr unsigned long long KEY_PINF = 0xfff0000000000000ull, KEY_MINF = 0x000fffffffffffffull;
  constexpr unsigned KH_PINF = 0xfff00000u, KH_MINF = 0x000fffffu;   // high words of +-inf (and of some NaNs)
  const int rb = blockIdx.x, cbk = blockIdx.y;
  const int row0 = rb * SCAN_ROWS + threadIdx.x;
  const unsigned long long ku = dkey(u);
  // The high-word "tie band" of u: elements whose key's high word falls in it are compared
  // exactly.  For u = +-0 (or a tiny subnormal) it holds both zeros' words, which must compare
  // equal; for an infinite or NaN u it holds every word, and the whole scan is exact.
  const unsigned khu = dkey_hi(u);
  unsigned tie_lo = khu, tie_w = 0u;
  if (khu >= KH_PINF || khu <= KH_MINF) { tie_lo = 0u; tie_w = 0xffffffffu; }
  else if (khu == 0x7fffffffu || khu == 0x80000000u) { tie_lo = 0x7fffffffu; tie_w = 1u; }
  const unsigned tie_hi = tie_lo + tie_w;
  // The thread's t keys, ranked among its own RPT rows (ties by row): a column's minimum over
  // the qualifying rows is the lowest set bit of a mask in rank order, read back from shared
  // memory once per column instead of a 64-bit compare-select per element.
  __shared__ unsigned long long s_key[RPT][SCAN_THREADS];
  unsigned bit[RPT];
  int cnt[RPT];
  {
    unsigned long long tk[RPT];
#pragma unroll
    for (int q = 0; q < RPT; ++q) {
      const int r = row0 + q * SCAN_THREADS;
      tk[q] = r < n_p ? dkey(t[r]) : 0ull;
      cnt[q] = 0;
    }
#pragma unroll
    for (int q = 0; q < RPT; ++q) {
      int rank = 0;
#pragma unroll
      for (int p = 0; p < RPT; ++p) rank += (tk[p] < tk[q] || (tk[p] == tk[q] && p < q)) ? 1 : 0;
      bit[q] = 1u << rank;
      s_key[rank][threadIdx.x] = tk[q];
    }
  }
  __shared__ unsigned long long s_mn[SCAN_THREADS / 32][SCAN_COLS];
  __shared__ unsigned long long s_mx[SCAN_THREADS / 32][SCAN_COLS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this CTA's columns: a balanced share of the M columns (the grid is sized to the resident
  // CTAs, so no partial last wave), flushed in chunks of SCAN_COLS
  const int c_beg = (int)((long long)M * cbk / gridDim.y);
  const int c_end = (int)((long long)M * (cbk + 1) / gridDim.y);
  double nxt[RPT];
  auto load_col = [&](int c, double* dst) {
    const double* col = S + (size_t)c * lds;
#pragma unroll
    for (int q = 0; q < RPT; ++q) {
      const int r = row0 + q * SCAN_THREADS;
      dst[q] = r < n_p ? __ldcs(col + r) : __longlong_as_double(0x7ff8000000000000ll);   // NaN: no row
    }
  };
  if (c_beg < c_end) load_col(c_beg, nxt);
  for (int c = c_beg; c < c_end; ++c) {
    double val[RPT];
#pragma unroll
    for (int q = 0; q < RPT; ++q) val[q] = nxt[q];
    if (c + 1 < c_end) load_col(c + 1, nxt);   // next column in flight during this one's work
    // S >= u and S <= u, NaN excluded, decided on the keys' high words: a finite element whose
    // word lies outside u's tie band is above or below u.  Elements in the band, and words of
    // infinities or NaNs, are left to the exact 64-bit test below, which the warp takes only
    // when one of its lanes holds such an element.
    unsigned gmask = 0, lmask = 0, smask = 0;
#pragma unroll
    for (int q = 0; q < RPT; ++q) {
      const unsigned kh = dkey_hi(val[q]);
      const bool finite = (kh - (KH_MINF + 1u)) < (KH_PINF - KH_MINF - 1u);   // strictly between the infinities' words
      const bool slow = (kh - tie_lo) <= tie_w || !finite;
      const bool above = !slow && kh > tie_hi;
      const bool below = !slow && !above;
      const bool ge = neg ? below : above, le = neg ? above : below;
      gmask |= ge ? bit[q] : 0u;
      lmask |= le ? bit[q] : 0u;
      cnt[q] += ge ? 1 : 0;
      smask |= slow ? (1u << q) : 0u;
    }
    if (__any_sync(0xffffffffu, smask != 0u)) {
#pragma unroll
      for (int q = 0; q < RPT; ++q) {
        if (smask & (1u << q)) {
          const unsigned long long kv = dkey(val[q]);
          const bool ok = kv >= KEY_MINF && kv <= KEY_PINF;
          const bool above = ok && kv >= ku, below = ok && kv <= ku;
          const bool ge = neg ? below : above, le = neg ? above : below;
          gmask |= ge ? bit[q] : 0u;
          lmask |= le ? bit[q] : 0u;
          cnt[q] += ge ? 1 : 0;
        }
      }
    }
    unsigned long long mn = gmask ? s_key[__ffs(gmask) - 1][threadIdx.x] : KEY_PINF;
    unsigned long long mx = lmask ? s_key[31 - __clz(lmask)][threadIdx.x] : KEY_MINF;
    // warp minimum / maximum of the 64-bit keys: the high words first, then the low words of
    // the lanes that hold the extreme high word (two warp reductions each)
    {
      const unsigned h = (unsigned)(mn >> 32), hm = __reduce_min_sync(0xffffffffu, h);
      const unsigned lm = __reduce_min_sync(0xffffffffu, h == hm ? (unsigned)mn : 0xffffffffu);
      mn = ((unsigned long long)hm << 32) | lm;
    }
    {
      const unsigned h = (unsigned)(mx >> 32), hm = __reduce_max_sync(0xffffffffu, h);
      const unsigned lm = __reduce_max_sync(0xffffffffu, h == hm ? (unsigned)mx : 0u);
      mx = ((unsigned long long)hm << 32) | lm;
    }
    const int slot = (c - c_beg) % SCAN_COLS;
    if (lane == 0) { s_mn[warp][slot] = mn; s_mx[warp][slot] = mx; }
    if (slot == SCAN_COLS - 1 || c == c_end - 1) {   // the same columns in every thread
      __syncthreads();
      if (threadIdx.x <= slot) {
        unsigned long long m1 = KEY_PINF, m2 = KEY_MINF;
        for (int w = 0; w < SCAN_THREADS / 32; ++w) {
          m1 = s_mn[w][threadIdx.x] < m1 ? s_mn[w][threadIdx.x] : m1;
          m2 = s_mx[w][threadIdx.x] > m2 ? s_mx[w][threadIdx.x] : m2;
        }
        const size_t o = (size_t)rb * M + (c - slot) + threadIdx.x;
        psi_part[o] = dkey_inv(m1);   // +inf / -inf when the block's column has no qualifying row
        phi_part[o] = dkey_inv(m2);
      }
      __syncthreads();
    }
  }
  if (count) {
#pragma unroll
    for (int q = 0; q < RPT; ++q) {
      const int r = row0 + q * SCAN_THREADS;
      if (r < n_p && cnt[q]) atomicAdd(&count[r], cnt[q]);
    }
  }
}

__global__ void k_scan_reduce(const double* __restrict__ psi_part, const double* __restrict__ phi_part, int nrb, int M,
                              double* __restrict__ psi, double* __restrict__ phi) {
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < M; j += gridDim.x * blockDim.x) {
    double mn = INFINITY, mx = -INFINITY;
    for (int r = 0; r < nrb; ++r) { mn = fmin(mn, psi_part[(size_t)r * M + j]); mx = fmax(mx, phi_part[(size_t)r * M + j]); }
    psi[j] = mn;
    phi[j] = mx;
  }
}

__global__ void k_regions(const double* __restrict__ t, int n_p, double q_in, double q_out, uint8_t* __restrict__ cin,
                          uint8_t* __restrict__ cout) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_p; i += gridDim.x * blockDim.x) {
    cin[i] = t[i] > q_in ? 1 : 0;
    cout[i] = t[i] >= q_out ? 1 : 0;
  }
}

// The scan's grid: one row of CTAs per SCAN_ROWS rows, and as many column groups as fill the
// GPU's resident CTAs twice (at least one group, at most one per column).  No allocation, so
// the allocation-free entry point uses it too.
static std::atomic<int> g_scan_resident{0};
static cudaError_t scan_grid(int n_p, int M, dim3* grid) {
  int resident = g_scan_resident.load(std::memory_order_relaxed);
  if (resident == 0) {
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_scan, SCAN_THREADS, 0);
    if (e != cudaSuccess) return e;
    resident = std::max(1, sms * per_sm);
    g_scan_resident.store(resident, std::memory_order_relaxed);
  }
  const int nrb = (n_p + SCAN_ROWS - 1) / SCAN_ROWS;
  *grid = dim3((unsigned)nrb, (unsigned)std::max(1, std::min(M, 2 * resident / nrb)));
  return cudaSuccess;
}

double empirical_quantile(std::vector<double>& a, double p) {
  std::sort(a.begin(), a.end());
  const long N = (long)a.size();
  long k = (long)ceil(p * (double)N - 1e-9);
  k = std::max(1L, std::min(N, k));
  return a[k - 1];
}

cr_status calibrate_core(const double* d_S, int lds, int n_p, int M, const double* d_zhat, const double* d_v, double u,
                         double level, uint8_t* d_cin, uint8_t* d_cout, int32_t* d_count, double* d_psi, double* d_phi,
                         cr_calib_info* out, cudaStream_t stream, const CalibScratch& sc, int neg) {
  const int nrb = (n_p + SCAN_ROWS - 1) / SCAN_ROWS;
  CR_CUDA(cudaMemsetAsync(sc.bad, 0, sizeof(int), stream));
  k_tstat<<<std::min(1024, (n_p + 255) / 256), 256, 0, stream>>>(d_zhat, d_v, u, n_p, sc.t, sc.bad, neg);
  CR_CHECK_LAUNCH("k_tstat");
  if (d_count) CR_CUDA(cudaMemsetAsync(d_count, 0, (size_t)n_p * sizeof(int32_t), stream));
  dim3 grid;
  CR_CUDA(scan_grid(n_p, M, &grid));
  {
    TimedScope ts("k_scan", stream);
    k_scan<<<grid, SCAN_THREADS, 0, stream>>>(d_S, lds, n_p, M, sc.t, u, sc.psi_part, sc.phi_part, d_count, neg);
  }
  CR_CHECK_LAUNCH("k_scan");
  return calibrate_finish(sc.psi_part, sc.phi_part, nrb, n_p, M, level, sc, d_cin, d_cout, d_psi, d_phi, out, stream);
}

// Combines the per-row-block partials (nrb x M) into psi and phi in a fixed order, takes the
// quantiles of the samples without sentinels on the host and writes the regions from sc.t;
// returns only after its last kernel, which reads sc.t, has finished.
cr_status calibrate_finish(const double* psi_part, const double* phi_part, int nrb, int n_p, int M, double level,
                           const CalibScratch& sc, uint8_t* d_cin, uint8_t* d_cout, double* d_psi, double* d_phi,
                           cr_calib_info* out, cudaStream_t stream) {
  k_scan_reduce<<<std::min(1024, (M + 255) / 256), 256, 0, stream>>>(psi_part, phi_part, nrb, M, sc.psi, sc.phi);
  CR_CHECK_LAUNCH("k_scan_reduce");
  std::vector<double> psi(M), phi(M);
  int bad = 0;
  CR_CUDA(cudaMemcpyAsync(psi.data(), sc.psi, M * sizeof(double), cudaMemcpyDeviceToHost, stream));
  CR_CUDA(cudaMemcpyAsync(phi.data(), sc.phi, M * sizeof(double), cudaMemcpyDeviceToHost, stream));
  CR_CUDA(cudaMemcpyAsync(&bad, sc.bad, sizeof(int), cudaMemcpyDeviceToHost, stream));
  if (d_psi) CR_CUDA(cudaMemcpyAsync(d_psi, sc.psi, M * sizeof(double), cudaMemcpyDeviceToDevice, stream));
  if (d_phi) CR_CUDA(cudaMemcpyAsync(d_phi, sc.phi, M * sizeof(double), cudaMemcpyDeviceToDevice, stream));
  CR_CUDA(cudaStreamSynchronize(stream));
  if (bad) return fail(CR_ERR_NONPOS_MSPE, "cr_calibrate: some v_i <= 0");
  std::vector<double> a_psi, a_phi;
  a_psi.reserve(M);
  a_phi.reserve(M);
  for (int j = 0; j < M; ++j) {
    if (psi[j] != INFINITY) a_psi.push_back(psi[j]);
    if (phi[j] != -INFINITY) a_phi.push_back(phi[j]);
  }
  cr_calib_info info{};
  info.n_psi = (int)a_psi.size();
  info.n_phi = (int)a_phi.size();
  if (out) *out = info;
  if (a_psi.empty() || a_phi.empty())
    return fail(CR_ERR_EMPTY_SAMPLE, "cr_calibrate: n_psi=" + std::to_string(info.n_psi) + " n_phi=" + std::to_string(info.n_phi));
  const double alpha = 1.0 - level;
  info.q_out = empirical_quantile(a_psi, alpha);
  info.q_in = empirical_quantile(a_phi, 1.0 - alpha);
  if (out) *out = info;
  k_regions<<<std::min(1024, (n_p + 255) / 256), 256, 0, stream>>>(sc.t, n_p, info.q_in, info.q_out, d_cin, d_cout);
  CR_CHECK_LAUNCH("k_regions");
  // k_regions reads the shared scratch: return only once it is done, so that a later call on
  // another stream cannot overwrite t while this one still reads it
  CR_CUDA(cudaStreamSynchronize(stream));
  return CR_OK;
}

// Library-managed scratch for cr_calibrate, grown on demand (one per process).
static std::mutex g_mu;
static CalibScratch g_sc;
static size_t g_np = 0, g_M = 0, g_nrbM = 0;

static cr_status ensure_scratch(int n_p, int M) {
  const int nrb = (n_p + SCAN_ROWS - 1) / SCAN_ROWS;
  if ((size_t)n_p > g_np) {
    if (g_sc.t) cudaFree(g_sc.t);
    g_sc.t = nullptr;
    CR_CUDA(cudaMalloc(&g_sc.t, (size_t)n_p * sizeof(double)));
    g_np = n_p;
  }
  if ((size_t)M > g_M) {
    if (g_sc.psi) cudaFree(g_sc.psi);
    if (g_sc.phi) cudaFree(g_sc.phi);
    g_sc.psi = g_sc.phi = nullptr;
    CR_CUDA(cudaMalloc(&g_sc.psi, (size_t)M * sizeof(double)));
    CR_CUDA(cudaMalloc(&g_sc.phi, (size_t)M * sizeof(double)));
    g_M = M;
  }
  if ((size_t)nrb * M > g_nrbM) {
    if (g_sc.psi_part) cudaFree(g_sc.psi_part);
    if (g_sc.phi_part) cudaFree(g_sc.phi_part);
    g_sc.psi_part = g_sc.phi_part = nullptr;
    CR_CUDA(cudaMalloc(&g_sc.psi_part, (size_t)nrb * M * sizeof(double)));
    CR_CUDA(cudaMalloc(&g_sc.phi_part, (size_t)nrb * M * sizeof(double)));
    g_nrbM = (size_t)nrb * M;
  }
  if (!g_sc.bad) CR_CUDA(cudaMalloc(&g_sc.bad, sizeof(int)));
  return CR_OK;
}

}  // namespace cr

using namespace cr;

extern "C" cr_status cr_calibrate(const double* d_S, int lds, int n_p, int M, const double* d_zhat, const double* d_v, double u,
                                  double level, uint8_t* d_cin, uint8_t* d_cout, int32_t* d_count, double* d_psi,
                                  double* d_phi, cr_calib_info* out, cr_stream stream) {
  if (!d_S || !d_zhat || !d_v || !d_cin || !d_cout || n_p <= 0 || M <= 0 || lds < n_p || !(level > 0.0 && level < 1.0))
    return fail(CR_ERR_ARG, "cr_calibrate: argument");
  std::lock_guard<std::mutex> lk(g_mu);
  CR_TRY(ensure_scratch(n_p, M));
  return calibrate_core(d_S, lds, n_p, M, d_zhat, d_v, u, level, d_cin, d_cout, d_count, d_psi, d_phi, out, stream, g_sc, 0);
}

extern "C" cr_status cr_calibrate_negative(const double* d_S, int lds, int n_p, int M, const double* d_zhat,
                                           const double* d_v, double u, double level, uint8_t* d_cin, uint8_t* d_cout,
                                           int32_t* d_count, double* d_psi, double* d_phi, cr_calib_info* out,
                                           cr_stream stream) {
  if (!d_S || !d_zhat || !d_v || !d_cin || !d_cout || n_p <= 0 || M <= 0 || lds < n_p || !(level > 0.0 && level < 1.0))
    return fail(CR_ERR_ARG, "cr_calibrate_negative: argument");
  std::lock_guard<std::mutex> lk(g_mu);
  CR_TRY(ensure_scratch(n_p, M));
  return calibrate_core(d_S, lds, n_p, M, d_zhat, d_v, u, level, d_cin, d_cout, d_count, d_psi, d_phi, out, stream, g_sc, 1);
}

// ---------------------------------------------------------------------------------------
// Conditioning correction (Section V-B Eq.7) as a double-float GEMM, S = M_p + W^T R with
// R = y_o 1^T - M_o, and its fusion with the calibration scan.
//
// The page states the correction in FP64.  GB300's FP64 units issue 1/64 of the FP32 lanes,
// so the product runs in double-float arithmetic on the FP32 units (about 48 significant
// bits, the error-free products and sums of df.cuh; an FP64 emulation): W and R are converted
// to double-float pairs once per call, each CTA computes a 64 x 64 block of S over the whole
// inner dimension n_o, the block's value is M_p + (hi + lo) in FP64, and the epilogue either
// stores it (cr_krige_correct) or hands it to the scan's decisions (cr_correct_calibrate:
// psi/phi partials per 64-row block and per-row exceedance counts), so that S is never
// written.  Both epilogues see the same values, so the fused and unfused paths decide alike.
namespace cr {
namespace {

constexpr int CT = 64;    // rows and columns of an output block
constexpr int CK = 16;    // inner-dimension chunk staged in shared memory
constexpr int CTH = 256;  // threads: a 16 x 16 grid, 4 x 4 outputs each

// D[q + c rows] = A[q + c lda] as double-float pairs (rows x cols, column-major)
__global__ void k_to_df(const double* __restrict__ A, int lda, int rows, int cols, float2* __restrict__ D) {
  const size_t total = (size_t)rows * cols;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const size_t q = e % rows, c = e / rows;
    const double x = A[q + c * lda];
    const float h = __double2float_rn(x);
    D[e] = make_float2(h, __double2float_rn(x - (double)h));
  }
}
// R[q + j n_o] = y_o[q] - M_o[q + j ldy] (FP64), as double-float pairs
__global__ void k_resid_df(const double* __restrict__ yo, const double* __restrict__ Mo, int ldy, int n_o, int M,
                           float2* __restrict__ R) {
  const size_t total = (size_t)n_o * M;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const size_t q = e % n_o, j = e / n_o;
    const double x = yo[q] - Mo[q + j * ldy];
    const float h = __double2float_rn(x);
    R[e] = make_float2(h, __double2float_rn(x - (double)h));
  }
}

struct CAcc {
  float s, c;
};
// s + c += x y, the high products summed by two-sum, the lower-order terms in c
__device__ __forceinline__ void cmac(CAcc& a, float2 x, float2 y) {
  const float p = __fmul_rn(x.x, y.x);
  float e = __fmaf_rn(x.x, y.x, -p);
  e = __fmaf_rn(x.x, y.y, e);
  e = __fmaf_rn(x.y, y.x, e);
  const float s = __fadd_rn(a.s, p);
  const float bb = __fsub_rn(s, a.s);
  const float t = __fadd_rn(__fsub_rn(a.s, __fsub_rn(s, bb)), __fsub_rn(p, bb));
  a.s = s;
  a.c = __fadd_rn(a.c, __fadd_rn(t, e));
}

template <bool SCAN>
__global__ void __launch_bounds__(CTH) k_corr(const float2* __restrict__ Wd, const float2* __restrict__ Rd,
                                              const double* __restrict__ Mp, int ldy, int n_p, int n_o, int M,
                                              double* __restrict__ S, int lds, const double* __restrict__ t, double u, int neg,
                                              double* __restrict__ psi_part, double* __restrict__ phi_part,
                                              int32_t* __restrict__ count) {
  __shared__ float2 As[2][CK][CT + 1];   // padded: the staging stores walk k
  __shared__ float2 Bs[2][CK][CT + 1];
  // column blocks vary fastest over the grid, so the CTAs that share a block of rows of W run
  // together and read it from L2 (W is read from HBM about once, R stays in L2)
  const int i0 = blockIdx.y * CT, j0 = blockIdx.x * CT;
  const int tid = threadIdx.x, ti = tid >> 4, tj = tid & 15;
  CAcc acc[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = CAcc{0.0f, 0.0f};
  // staging: element e = tid + 256 s of a chunk is (k = e % 16, row or column e / 16); 16
  // consecutive threads read 16 consecutive inner indices (128 bytes)
  float2 ra[4], rb[4];
  auto fetch = [&](int q0) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int e = tid + CTH * s, k = e & (CK - 1), r = e >> 4, q = q0 + k;
      ra[s] = (q < n_o && i0 + r < n_p) ? Wd[(size_t)(i0 + r) * n_o + q] : make_float2(0.0f, 0.0f);
      rb[s] = (q < n_o && j0 + r < M) ? Rd[(size_t)(j0 + r) * n_o + q] : make_float2(0.0f, 0.0f);
    }
  };
  auto stash = [&](int b) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int e = tid + CTH * s, k = e & (CK - 1), r = e >> 4;
      As[b][k][r] = ra[s];
      Bs[b][k][r] = rb[s];
    }
  };
  const int nch = (n_o + CK - 1) / CK;
  fetch(0);
  stash(0);
  __syncthreads();
  for (int ch = 0; ch < nch; ++ch) {
    const int b = ch & 1;
    if (ch + 1 < nch) fetch((ch + 1) * CK);   // the next chunk in flight during this one's products
#pragma unroll
    for (int k = 0; k < CK; ++k) {
      float2 a[4], bv[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = As[b][k][ti + 16 * r];
#pragma unroll
      for (int c = 0; c < 4; ++c) bv[c] = Bs[b][k][tj + 16 * c];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) cmac(acc[r][c], a[r], bv[c]);
    }
    if (ch + 1 < nch) stash(b ^ 1);   // buffer b ^ 1 was last read before the previous barrier
    __syncthreads();
  }
  // S_ij = M_p,ij + (hi + lo), in FP64
  double sv[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = i0 + ti + 16 * r, j = j0 + tj + 16 * c;
      sv[r][c] = 0.0;
      if (i < n_p && j < M) {
        const df v = df_two_sum(acc[r][c].s, acc[r][c].c);
        sv[r][c] = Mp[i + (size_t)j * ldy] + ((double)v.hi + (double)v.lo);
      }
    }
  if (!SCAN) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int i = i0 + ti + 16 * r, j = j0 + tj + 16 * c;
        if (i < n_p && j < M) S[i + (size_t)j * lds] = sv[r][c];
      }
    return;
  }
  // The scan's decisions on the block: S >= u and S <= u (IEEE comparisons: NaN neither, the
  // two zeros equal), swapped for a negative excursion set; psi / phi partials are the
  // extreme keys of t over the qualifying rows, counts the qualifying columns of each row.
  constexpr unsigned long long KEY_PINF = 0xfff0000000000000ull, KEY_MINF = 0x000fffffffffffffull;
  __shared__ unsigned long long red_mn[CTH / 32][CT], red_mx[CTH / 32][CT];
  const int lane = tid & 31, warp = tid >> 5;
  unsigned long long tk[4];
  int cnt[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = i0 + ti + 16 * r;
    tk[r] = i < n_p ? dkey(t[i]) : 0ull;
    cnt[r] = 0;
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int j = j0 + tj + 16 * c;
    unsigned long long mn = KEY_PINF, mx = KEY_MINF;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = i0 + ti + 16 * r;
      const bool valid = i < n_p && j < M;
      const bool above = valid && sv[r][c] >= u, below = valid && sv[r][c] <= u;
      const bool ge = neg ? below : above, le = neg ? above : below;
      if (ge) mn = tk[r] < mn ? tk[r] : mn;
      if (le) mx = tk[r] > mx ? tk[r] : mx;
      cnt[r] += ge ? 1 : 0;
    }
    // lanes tj and tj + 16 of a warp hold the same column (rows of two ti)
    const unsigned long long mn2 = __shfl_xor_sync(0xffffffffu, mn, 16), mx2 = __shfl_xor_sync(0xffffffffu, mx, 16);
    mn = mn2 < mn ? mn2 : mn;
    mx = mx2 > mx ? mx2 : mx;
    if (lane < 16) {
      red_mn[warp][tj + 16 * c] = mn;
      red_mx[warp][tj + 16 * c] = mx;
    }
  }
  // counts: the 16 lanes of a half-warp share a row
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    int v = cnt[r];
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int i = i0 + ti + 16 * r;
    if (count && tj == 0 && v && i < n_p) atomicAdd(&count[i], v);
  }
  __syncthreads();
  if (tid < CT && j0 + tid < M) {
    unsigned long long m1 = KEY_PINF, m2 = KEY_MINF;
#pragma unroll
    for (int w = 0; w < CTH / 32; ++w) {
      m1 = red_mn[w][tid] < m1 ? red_mn[w][tid] : m1;
      m2 = red_mx[w][tid] > m2 ? red_mx[w][tid] : m2;
    }
    const size_t o = (size_t)blockIdx.y * M + j0 + tid;
    psi_part[o] = dkey_inv(m1);   // +inf / -inf when no row of the block qualifies
    phi_part[o] = dkey_inv(m2);
  }
}

// Converts W and R and launches the correction GEMM (stream-ordered).
cr_status correction_launch(const double* d_W, int ldw, const double* d_yo, const double* d_Y, int ldy, int n_p, int n_o,
                            int M, float2* Wd, float2* Rd, bool scan, double* d_S, int lds, const double* t, double u, int neg,
                            double* psi_part, double* phi_part, int32_t* d_count, cudaStream_t stream) {
  k_to_df<<<2048, 256, 0, stream>>>(d_W, ldw, n_o, n_p, Wd);
  CR_CHECK_LAUNCH("k_to_df");
  k_resid_df<<<1024, 256, 0, stream>>>(d_yo, d_Y + n_p, ldy, n_o, M, Rd);
  CR_CHECK_LAUNCH("k_resid_df");
  const dim3 grid((unsigned)((M + CT - 1) / CT), (unsigned)((n_p + CT - 1) / CT));
  if (scan) {
    TimedScope ts("k_corr_scan", stream);
    k_corr<true><<<grid, CTH, 0, stream>>>(Wd, Rd, d_Y, ldy, n_p, n_o, M, nullptr, 0, t, u, neg, psi_part, phi_part, d_count);
  } else {
    TimedScope ts("k_corr", stream);
    k_corr<false><<<grid, CTH, 0, stream>>>(Wd, Rd, d_Y, ldy, n_p, n_o, M, d_S, lds, nullptr, 0.0, 0, nullptr, nullptr, nullptr);
  }
  CR_CHECK_LAUNCH("k_corr");
  return CR_OK;
}

// Library-managed scratch of cr_correct_calibrate, grown on demand (one per process): the
// double-float copies of W and R, t, psi, phi, the 64-row-block partials and the MSPE flag.
std::mutex g_cc_mu;
struct CorrScratch {
  float2* W = nullptr;
  float2* R = nullptr;
  double *t = nullptr, *psi = nullptr, *phi = nullptr, *psi_part = nullptr, *phi_part = nullptr;
  int* bad = nullptr;
  size_t capW = 0, capR = 0, capT = 0, capPsi = 0, capPhi = 0, capPP = 0, capFP = 0, capBad = 0;
};
CorrScratch g_cc;

template <class T>
cr_status grow(T** p, size_t* cap, size_t need) {
  if (need <= *cap) return CR_OK;
  if (*p) cudaFree(*p);
  *p = nullptr;
  *cap = 0;
  CR_CUDA(cudaMalloc(p, need * sizeof(T)));
  *cap = need;
  return CR_OK;
}

}  // namespace

cr_status correction_async(const double* d_W, int ldw, const double* d_yo, const double* d_Y, int ldy, int n_p, int n_o,
                           int M, double* d_S, int lds, cudaStream_t stream) {
  float2 *Wd = nullptr, *Rd = nullptr;
  CR_CUDA(scratch_alloc((void**)&Wd, (size_t)n_o * n_p * sizeof(float2), stream));
  if (cudaError_t e = scratch_alloc((void**)&Rd, (size_t)n_o * M * sizeof(float2), stream)) {
    scratch_free(Wd, stream);
    return cuda_fail(e, "scratch_alloc");
  }
  const cr_status st = correction_launch(d_W, ldw, d_yo, d_Y, ldy, n_p, n_o, M, Wd, Rd, false, d_S, lds, nullptr, 0.0, 0,
                                         nullptr, nullptr, nullptr, stream);
  scratch_free(Wd, stream);
  scratch_free(Rd, stream);
  return st;
}

}  // namespace cr

// The Ozaki correction writes S (scratch from the library pool) through `correct`, then the
// scan of cr_calibrate reads it.
static cr_status correct_then_calibrate(const std::function<cr_status(double*)>& correct, int n_p, int M,
                                        const double* d_zhat, const double* d_v, double u, double level, int negative,
                                        uint8_t* d_cin, uint8_t* d_cout, int32_t* d_count, double* d_psi, double* d_phi,
                                        cr_calib_info* out, cudaStream_t stream) {
  double* S = nullptr;
  CR_CUDA(scratch_alloc((void**)&S, (size_t)n_p * M * sizeof(double), stream));
  cr_status st = correct(S);
  if (st == CR_OK) {
    std::lock_guard<std::mutex> lk(g_mu);
    st = ensure_scratch(n_p, M);
    if (st == CR_OK)
      st = calibrate_core(S, n_p, n_p, M, d_zhat, d_v, u, level, d_cin, d_cout, d_count, d_psi, d_phi, out, stream, g_sc,
                          negative ? 1 : 0);
  }
  scratch_free(S, stream);
  return st;
}

extern "C" cr_status cr_correct_calibrate_prepared(cr_weights w, const double* d_yo, const double* d_Y, int ldy, int M,
                                                   const double* d_zhat, const double* d_v, double u, double level,
                                                   int negative, uint8_t* d_cin, uint8_t* d_cout, int32_t* d_count,
                                                   double* d_psi, double* d_phi, cr_calib_info* out, cr_stream stream) {
  if (!w || !d_yo || !d_Y || !d_zhat || !d_v || !d_cin || !d_cout || M <= 0 || ldy < w->n_p + w->n_o ||
      !(level > 0.0 && level < 1.0))
    return fail(CR_ERR_ARG, "cr_correct_calibrate_prepared: argument");
  return correct_then_calibrate(
      [&](double* S) { return ozaki_correction_prepared(w, d_yo, d_Y, ldy, M, S, w->n_p, stream); }, w->n_p, M, d_zhat,
      d_v, u, level, negative, d_cin, d_cout, d_count, d_psi, d_phi, out, stream);
}

extern "C" cr_status cr_correct_calibrate(const double* d_W, int ldw, const double* d_yo, const double* d_Y, int ldy,
                                          int n_p, int n_o, int M, const double* d_zhat, const double* d_v, double u,
                                          double level, int negative, uint8_t* d_cin, uint8_t* d_cout, int32_t* d_count,
                                          double* d_psi, double* d_phi, cr_calib_info* out, cr_stream stream) {
  if (!d_W || !d_yo || !d_Y || !d_zhat || !d_v || !d_cin || !d_cout || n_p <= 0 || n_o <= 0 || M <= 0 || ldw < n_o ||
      ldy < n_p + n_o || !(level > 0.0 && level < 1.0))
    return fail(CR_ERR_ARG, "cr_correct_calibrate: argument");
  if (option_fp64_gemm() == CR_GEMM_OZAKI)
    return correct_then_calibrate(
        [&](double* S) { return ozaki_correction(d_W, ldw, d_yo, d_Y, ldy, n_p, n_o, M, S, n_p, stream); }, n_p, M, d_zhat,
        d_v, u, level, negative, d_cin, d_cout, d_count, d_psi, d_phi, out, stream);
  std::lock_guard<std::mutex> lk(g_cc_mu);
  const size_t nrb = ((size_t)n_p + CT - 1) / CT;
  CR_TRY(grow(&g_cc.W, &g_cc.capW, (size_t)n_o * n_p));
  CR_TRY(grow(&g_cc.R, &g_cc.capR, (size_t)n_o * M));
  CR_TRY(grow(&g_cc.t, &g_cc.capT, (size_t)n_p));
  CR_TRY(grow(&g_cc.psi, &g_cc.capPsi, (size_t)M));
  CR_TRY(grow(&g_cc.phi, &g_cc.capPhi, (size_t)M));
  CR_TRY(grow(&g_cc.psi_part, &g_cc.capPP, nrb * M));
  CR_TRY(grow(&g_cc.phi_part, &g_cc.capFP, nrb * M));
  CR_TRY(grow(&g_cc.bad, &g_cc.capBad, (size_t)1));
  CalibScratch sc;
  sc.t = g_cc.t;
  sc.psi = g_cc.psi;
  sc.phi = g_cc.phi;
  sc.psi_part = g_cc.psi_part;
  sc.phi_part = g_cc.phi_part;
  sc.bad = g_cc.bad;
  const int neg = negative ? 1 : 0;
  CR_CUDA(cudaMemsetAsync(sc.bad, 0, sizeof(int), stream));
  k_tstat<<<std::min(1024, (n_p + 255) / 256), 256, 0, stream>>>(d_zhat, d_v, u, n_p, sc.t, sc.bad, neg);
  CR_CHECK_LAUNCH("k_tstat");
  if (d_count) CR_CUDA(cudaMemsetAsync(d_count, 0, (size_t)n_p * sizeof(int32_t), stream));
  CR_TRY(correction_launch(d_W, ldw, d_yo, d_Y, ldy, n_p, n_o, M, g_cc.W, g_cc.R, true, nullptr, 0, sc.t, u, neg,
                           sc.psi_part, sc.phi_part, d_count, stream));
  return calibrate_finish(sc.psi_part, sc.phi_part, (int)nrb, n_p, M, level, sc, d_cin, d_cout, d_psi, d_phi, out, stream);
}

// ---------------------------------------------------------------------------------------
// Allocation-free calibration, for callers that cannot allocate device memory (code that
// runs under a memory pool which owns every device allocation, or an embedder whose device
// footprint must stay fixed after start-up).  Same kernels and results as cr_calibrate;
// the scratch is a fixed array of this file instead of library-managed allocations.
namespace cr {

cr_status fail_literal(cr_status code, const char* msg);

namespace {

// Device scratch shared by every call on a device (held until the process exits).  In host
// code this name only identifies the symbol: its device address is looked up once per
// device with cudaGetSymbolAddress and passed to the kernels as a plain pointer.
static __device__ __align__(256) unsigned char g_noalloc_scratch[CR_NOALLOC_SCRATCH_BYTES];

// Host copies of psi and phi for the quantiles (fixed, so the host side allocates nothing).
static double g_noalloc_psi[CR_NOALLOC_MAX_M];
static double g_noalloc_phi[CR_NOALLOC_MAX_M];

constexpr int kNoallocMaxDevices = 64;
static unsigned char* g_noalloc_dev[kNoallocMaxDevices];   // device address per device
static std::mutex g_noalloc_mu;

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// Q_p of the sorted prefix a[0, N) (N >= 1), same rule as empirical_quantile.
double quantile_sorted(const double* a, long N, double p) {
  long k = (long)ceil(p * (double)N - 1e-9);
  k = std::max(1L, std::min(N, k));
  return a[k - 1];
}

}  // namespace
}  // namespace cr

extern "C" cr_status cr_calibrate_noalloc(const double* d_S, int lds, int n_p, int M, const double* d_zhat,
                                          const double* d_v, double u, double level, uint8_t* d_cin, uint8_t* d_cout,
                                          int32_t* d_count, double* d_psi, double* d_phi, cr_calib_info* out,
                                          cr_stream stream) {
  if (!d_S || !d_zhat || !d_v || !d_cin || !d_cout || n_p <= 0 || M <= 0 || lds < n_p || !(level > 0.0 && level < 1.0))
    return fail_literal(CR_ERR_ARG, "cr_calibrate_noalloc: argument");
  if (M > CR_NOALLOC_MAX_M) return fail_literal(CR_ERR_ARG, "cr_calibrate_noalloc: M exceeds CR_NOALLOC_MAX_M");
  const size_t nrb = ((size_t)n_p + SCAN_ROWS - 1) / SCAN_ROWS;
  const size_t need = 8 * (size_t)n_p + 16 * (size_t)M + 16 * nrb * (size_t)M + 1536;
  if (need > CR_NOALLOC_SCRATCH_BYTES)
    return fail_literal(CR_ERR_ARG, "cr_calibrate_noalloc: problem needs more than CR_NOALLOC_SCRATCH_BYTES of scratch");
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_literal(CR_ERR_CUDA, cudaGetErrorName(e));
  if (dev < 0 || dev >= kNoallocMaxDevices) return fail_literal(CR_ERR_ARG, "cr_calibrate_noalloc: device index too large");
  if (!g_noalloc_dev[dev]) {   // once per device, with that device current
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return fail_literal(CR_ERR_CUDA, cudaGetErrorName(e));
    g_noalloc_dev[dev] = static_cast<unsigned char*>(p);
  }
  // carve the array: t | psi | phi | psi_part | phi_part | flag
  unsigned char* base = g_noalloc_dev[dev];
  size_t off = 0;
  auto take = [&](size_t bytes) {
    unsigned char* q = base + off;
    off += round256(bytes);
    return q;
  };
  double* t = reinterpret_cast<double*>(take(8 * (size_t)n_p));
  double* psi = reinterpret_cast<double*>(take(8 * (size_t)M));
  double* phi = reinterpret_cast<double*>(take(8 * (size_t)M));
  double* psi_part = reinterpret_cast<double*>(take(8 * nrb * M));
  double* phi_part = reinterpret_cast<double*>(take(8 * nrb * M));
  int* bad = reinterpret_cast<int*>(take(sizeof(int)));

  // The array keeps the previous call's contents: clear what is accumulated (the MSPE flag
  // and the caller's counts); t, psi, phi and the partials are fully overwritten.
#define NA_CUDA(call)                                                 \
  do {                                                                \
    cudaError_t e__ = (call);                                         \
    if (e__ != cudaSuccess) return fail_literal(CR_ERR_CUDA, cudaGetErrorName(e__)); \
  } while (0)
  NA_CUDA(cudaMemsetAsync(bad, 0, sizeof(int), stream));
  if (d_count) NA_CUDA(cudaMemsetAsync(d_count, 0, (size_t)n_p * sizeof(int32_t), stream));
  k_tstat<<<std::min(1024, (n_p + 255) / 256), 256, 0, stream>>>(d_zhat, d_v, u, n_p, t, bad, 0);
  count_launch();
  NA_CUDA(cudaGetLastError());
  dim3 grid;
  NA_CUDA(scan_grid(n_p, M, &grid));
  k_scan<<<grid, SCAN_THREADS, 0, stream>>>(d_S, lds, n_p, M, t, u, psi_part, phi_part, d_count, 0);
  count_launch();
  NA_CUDA(cudaGetLastError());
  k_scan_reduce<<<std::min(1024, (M + 255) / 256), 256, 0, stream>>>(psi_part, phi_part, (int)nrb, M, psi, phi);
  count_launch();
  NA_CUDA(cudaGetLastError());
  int h_bad = 0;
  NA_CUDA(cudaMemcpyAsync(g_noalloc_psi, psi, (size_t)M * sizeof(double), cudaMemcpyDeviceToHost, stream));
  NA_CUDA(cudaMemcpyAsync(g_noalloc_phi, phi, (size_t)M * sizeof(double), cudaMemcpyDeviceToHost, stream));
  NA_CUDA(cudaMemcpyAsync(&h_bad, bad, sizeof(int), cudaMemcpyDeviceToHost, stream));
  if (d_psi) NA_CUDA(cudaMemcpyAsync(d_psi, psi, (size_t)M * sizeof(double), cudaMemcpyDeviceToDevice, stream));
  if (d_phi) NA_CUDA(cudaMemcpyAsync(d_phi, phi, (size_t)M * sizeof(double), cudaMemcpyDeviceToDevice, stream));
  NA_CUDA(cudaStreamSynchronize(stream));
  if (h_bad) return fail_literal(CR_ERR_NONPOS_MSPE, "cr_calibrate_noalloc: some v_i <= 0");
  long n_psi = 0, n_phi = 0;   // drop the empty-set sentinels in place
  for (int j = 0; j < M; ++j) {
    if (g_noalloc_psi[j] != INFINITY) g_noalloc_psi[n_psi++] = g_noalloc_psi[j];
    if (g_noalloc_phi[j] != -INFINITY) g_noalloc_phi[n_phi++] = g_noalloc_phi[j];
  }
  cr_calib_info info{};
  info.n_psi = (int)n_psi;
  info.n_phi = (int)n_phi;
  if (out) *out = info;
  if (n_psi == 0 || n_phi == 0) return fail_literal(CR_ERR_EMPTY_SAMPLE, "cr_calibrate_noalloc: empty psi or phi sample");
  std::sort(g_noalloc_psi, g_noalloc_psi + n_psi);
  std::sort(g_noalloc_phi, g_noalloc_phi + n_phi);
  const double alpha = 1.0 - level;
  info.q_out = quantile_sorted(g_noalloc_psi, n_psi, alpha);
  info.q_in = quantile_sorted(g_noalloc_phi, n_phi, 1.0 - alpha);
  if (out) *out = info;
  k_regions<<<std::min(1024, (n_p + 255) / 256), 256, 0, stream>>>(t, n_p, info.q_in, info.q_out, d_cin, d_cout);
  count_launch();
  NA_CUDA(cudaGetLastError());
  // k_regions reads t from the shared array: wait for it while still holding the lock, so that
  // the next call (on any stream) starts only after this one has stopped using the array
  NA_CUDA(cudaStreamSynchronize(stream));
#undef NA_CUDA
  return CR_OK;
}
