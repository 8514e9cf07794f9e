// Universal kriging, pointwise MSPE and the conditioning correction (FP64).
//
// "Mixed-Precision GPU Acceleration for Confidence Regions of Spatial Excursion Sets":
//  - Section V-A Eq.5 and Alg.2 steps 2-5: factor Sigma_y = L_o L_o^T and solve
//    Sigma_y F = X_o; G = X_o^T F; solve G H = F^T V_op - X_p^T; solve L_o Y = V_op - X_o H,
//    then L_o^T W = Y (reusing L_o); z_hat = W^T y_o.  The kriging stage is FP64.
//  - Section V-A Eq.6: v = theta0 1 + colsum(W .* U) - 2 colsum(V_op .* W) with U = Sigma_y W
//    and theta0 = sigma^2.  Since Sigma_y W = L_o Y, colsum(W .* U) = colsum(Y .* Y): the
//    same quantity without the symmetric product (exact in exact arithmetic).
//  - Section V-B Eq.7: S = M_p + W^T (y_o 1^T - M_o): one double-float GEMM with the residual
//    formed in its operand conversion (calib.cu, shared with the fused correction + scan).
// Sigma_y is factored as its own all-FP64 tile matrix by the library's Cholesky (which keeps
// each diagonal tile's inverse here); the many-right-hand-side triangular solves are blocked
// substitutions over tile rows whose products run on the FP64 tile GEMM, or, with
// CR_OPT_FP64_GEMM = CR_GEMM_OZAKI, as Ozaki products on the FP16 tensor cores (ozaki.cu) over
// dense copies of the factor.
#include <functional>

#include "calib.cuh"
#include "common.cuh"
#include "cov.cuh"
#include "fp64.cuh"

namespace cr {

// out[i] = sum_q A[q + i lda] B[q + i ldb] (ldb = 0: B is one vector)
__global__ void __launch_bounds__(256) k_coldot(const double* __restrict__ A, int lda, const double* __restrict__ B, int ldb,
                                                int rows, double* __restrict__ out) {
  const int i = blockIdx.x;
  double s = 0.0;
  for (int q = threadIdx.x; q < rows; q += 256) s = fma(A[(size_t)i * lda + q], B[(size_t)i * ldb + q], s);
  __shared__ double red[8];
  for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    double a = 0.0;
    for (int w = 0; w < 8; ++w) a += red[w];
    out[i] = a;
  }
}

// Q (3 x n_p, column-major) = -X_p^T
__global__ void k_neg_xpT(const double* __restrict__ Xp, int n_p, double* __restrict__ Q) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_p; i += gridDim.x * blockDim.x)
    for (int m = 0; m < 3; ++m) Q[3 * i + m] = -Xp[(size_t)m * n_p + i];
}

// H[:, i] = G^-1 Q[:, i] for the 3 x 3 symmetric positive definite G (column-major), by its
// Cholesky factor (the page's second POSV on the small trend system)
__global__ void k_solve3(const double* __restrict__ G, const double* __restrict__ Q, int n_p, double* __restrict__ H,
                         int* __restrict__ bad) {
  const double g00 = G[0], g10 = G[1], g20 = G[2], g11 = G[4], g21 = G[5], g22 = G[8];
  const double l00 = sqrt(g00);
  const double l10 = g10 / l00, l20 = g20 / l00;
  const double d1 = g11 - l10 * l10;
  const double l11 = sqrt(d1);
  const double l21 = (g21 - l20 * l10) / l11;
  const double d2 = g22 - l20 * l20 - l21 * l21;
  const double l22 = sqrt(d2);
  if (blockIdx.x == 0 && threadIdx.x == 0 && !(g00 > 0 && d1 > 0 && d2 > 0)) atomicOr(bad, 1);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_p; i += gridDim.x * blockDim.x) {
    const double b0 = Q[3 * i], b1 = Q[3 * i + 1], b2 = Q[3 * i + 2];
    const double z0 = b0 / l00, z1 = (b1 - l10 * z0) / l11, z2 = (b2 - l20 * z0 - l21 * z1) / l22;
    const double x2 = z2 / l22, x1 = (z1 - l21 * x2) / l11, x0 = (z0 - l10 * x1 - l20 * x2) / l00;
    H[3 * i] = x0; H[3 * i + 1] = x1; H[3 * i + 2] = x2;
  }
}

__global__ void k_mspe(const double* __restrict__ c1, const double* __restrict__ c2, double theta0, int n_p, double* __restrict__ v) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_p; i += gridDim.x * blockDim.x) v[i] = theta0 + c1[i] - 2.0 * c2[i];
}

// Dense copies of the strictly lower tiles of an all-FP64 tile factor (row-major tiles in
// pool64): Lr row-major (Lr[r n + c] = L(r, c)) and Lc column-major (Lc[c n + r] = L(r, c)).
// The diagonal blocks and the upper part are not written (the solves never read them).  One
// CTA of 32 x 8 threads per 32 x 32 piece of a tile; the transposed copy goes through shared
// memory so that both stores are coalesced.  blockIdx.z enumerates the tiles (I, J), I > J.
__global__ void __launch_bounds__(256) k_dense_lower(const double* __restrict__ pool64, const int* __restrict__ i64, int n,
                                                     int nb, double* __restrict__ Lr, double* __restrict__ Lc) {
  const int t = blockIdx.z;
  int I = (int)((1.0 + sqrt(1.0 + 8.0 * (double)t)) * 0.5);
  while (I * (I - 1) / 2 > t) --I;
  while ((I + 1) * I / 2 <= t) ++I;
  const int J = t - I * (I - 1) / 2;
  const double* tile = pool64 + (size_t)i64[tidx(I, J)] * nb * nb;
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  __shared__ double sm[32][33];
  for (int q = threadIdx.y; q < 32; q += 8) {
    const int r = r0 + q, c = c0 + threadIdx.x;
    const int gr = I * nb + r, gc = J * nb + c;
    if (r < nb && c < nb && gr < n && gc < n) {
      const double x = tile[(size_t)r * nb + c];
      Lr[(size_t)gr * n + gc] = x;
      sm[q][threadIdx.x] = x;
    }
  }
  __syncthreads();
  for (int q = threadIdx.y; q < 32; q += 8) {
    const int c = c0 + q, r = r0 + threadIdx.x;
    const int gr = I * nb + r, gc = J * nb + c;
    if (r < nb && c < nb && gr < n && gc < n) Lc[(size_t)gc * n + gr] = sm[threadIdx.x][q];
  }
}

// Mt_i = M_i^T for every row-major nb x nb tile M_i of `src` (Mt_i[c nb + r] = M_i[r nb + c]).
__global__ void __launch_bounds__(256) k_transpose_tiles(const double* __restrict__ src, int nb, double* __restrict__ dst) {
  const double* a = src + (size_t)blockIdx.z * nb * nb;
  double* b = dst + (size_t)blockIdx.z * nb * nb;
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  __shared__ double sm[32][33];
  for (int q = threadIdx.y; q < 32; q += 8) {
    const int r = r0 + q, c = c0 + threadIdx.x;
    if (r < nb && c < nb) sm[q][threadIdx.x] = a[(size_t)r * nb + c];
  }
  __syncthreads();
  for (int q = threadIdx.y; q < 32; q += 8) {
    const int c = c0 + q, r = r0 + threadIdx.x;
    if (r < nb && c < nb) b[(size_t)c * nb + r] = sm[threadIdx.x][q];
  }
}

namespace {

// Slices per operand in the solves' Ozaki products: 9 x 6 = 54 bits below each column's power
// of two, about FP64's 53 (the solution columns span several orders of magnitude, and the
// scheme's error is relative to each column's largest entry).
constexpr int KRIGE_OZ_SLICES = 9;

// Blocked solve of the factor's triangular systems with the Ozaki product: forward L X = B or
// backward L^T X = B, in place on B (n x r, column-major, ld ldb).  Per tile row i:
// B_i -= L_(i, <i) B_(<i) (forward) or L_(>i, i)^T B_(>i) (backward), then B_i = M_i B_i or
// M_i^T B_i with M_i the inverse of the diagonal factor.  Lr, Lc are the dense copies of
// k_dense_lower; Mt holds the transposed inverse tiles.
cr_status ozaki_trsm(cr_tilemat L, const double* Lr, const double* Lc, const double* Mt, double* B, int ldb, int r,
                     bool backward, cudaStream_t s) {
  const int nt = L->nt, nb = L->nb, n = L->n;
  const size_t nb2 = (size_t)nb * nb;
  for (int step = 0; step < nt; ++step) {
    const int i = backward ? nt - 1 - step : step;
    const int ri = std::min(nb, n - i * nb);
    double* Bi = B + (size_t)i * nb;
    if (!backward && i > 0)   // A(k, c) = L(i nb + c, k) = Lr[(i nb + c) n + k]
      CR_TRY(ozaki_gemm_tn(Lr + (size_t)i * nb * n, n, B, ldb, i * nb, ri, r, -1.0, Bi, ldb, Bi, ldb, KRIGE_OZ_SLICES, s));
    if (backward && i < nt - 1) {   // A(k, c) = L(k0 + k, i nb + c) = Lc[(i nb + c) n + k0 + k]
      const int k0 = (i + 1) * nb;
      CR_TRY(ozaki_gemm_tn(Lc + (size_t)i * nb * n + k0, n, B + k0, ldb, n - k0, ri, r, -1.0, Bi, ldb, Bi, ldb,
                                KRIGE_OZ_SLICES, s));
    }
    // forward: A(k, c) = M_i(c, k) = M_i[c nb + k]; backward: A(k, c) = M_i(k, c) = Mt_i[c nb + k]
    const double* Md = (backward ? Mt : L->minv_all) + (size_t)i * nb2;
    CR_TRY(ozaki_gemm_tn(Md, nb, Bi, ldb, ri, ri, r, 1.0, nullptr, 0, Bi, ldb, KRIGE_OZ_SLICES, s));
  }
  return CR_OK;
}

// FP64 GEMM jobs over an m x r column-major output, 64 x 64 blocks.
void add_jobs(std::vector<DJob>& js, double* C, int ldc, int m, int r, int pbeg, int pcnt, double alpha, double beta, int kmax) {
  for (int i0 = 0; i0 < m; i0 += 64)
    for (int j0 = 0; j0 < r; j0 += 64) {
      DJob jb{};
      jb.C = C + (size_t)j0 * ldc + i0;
      jb.sCm = 1; jb.sCn = ldc;
      jb.m = std::min(64, m - i0); jb.n = std::min(64, r - j0);
      jb.pbeg = pbeg; jb.pcnt = pcnt; jb.alpha = alpha; jb.beta = beta;
      jb.arow = i0; jb.brow = j0; jb.kmax = kmax;
      js.push_back(jb);
    }
}

struct Seq {
  std::vector<DJob> jobs;
  std::vector<DPair> pairs;
  std::vector<std::function<cr_status(cudaStream_t, const DJob*, const DPair*)>> ops;
  void gemm(const std::vector<DJob>& js) {
    if (js.empty()) return;
    const int off = (int)jobs.size(), cnt = (int)js.size();
    jobs.insert(jobs.end(), js.begin(), js.end());
    ops.push_back([=](cudaStream_t s, const DJob* dj, const DPair* dp) { return dgemm_launch(64, dj + off, dp, cnt, s); });
  }
  cr_status run(cudaStream_t s) {
    DJob* dj = nullptr;
    DPair* dp = nullptr;
    cr_status st = CR_OK;
    if (!jobs.empty()) CR_CUDA(cudaMalloc(&dj, jobs.size() * sizeof(DJob)));
    if (!pairs.empty()) CR_CUDA(cudaMalloc(&dp, pairs.size() * sizeof(DPair)));
    if (dj) CR_CUDA(cudaMemcpyAsync(dj, jobs.data(), jobs.size() * sizeof(DJob), cudaMemcpyHostToDevice, s));
    if (dp) CR_CUDA(cudaMemcpyAsync(dp, pairs.data(), pairs.size() * sizeof(DPair), cudaMemcpyHostToDevice, s));
    for (size_t q = 0; st == CR_OK && q < ops.size(); ++q) st = ops[q](s, dj, dp);
    cudaError_t e = cudaStreamSynchronize(s);
    if (dj) cudaFree(dj);
    if (dp) cudaFree(dp);
    if (st == CR_OK && e != cudaSuccess) st = cuda_fail(e, "kriging solve");
    return st;
  }
};

// Blocked solve with the FP64 tile factor L (diagonal inverses in minv_all):
// forward L X = B, or backward L^T X = B, in place on B (n x r, column-major, ld ldb);
// T is an nb x r scratch (ld nb).
void plan_trsm(Seq& S, cr_tilemat L, double* B, int ldb, int r, bool backward, double* T) {
  const int nt = L->nt, nb = L->nb, n = L->n;
  const size_t nb2 = (size_t)nb * nb;
  auto tile = [&](int i, int j) { return L->pool64 + (size_t)L->h_i64[tidx(i, j)] * nb2; };
  auto rows = [&](int i) { return std::min(nb, n - i * nb); };
  for (int s = 0; s < nt; ++s) {
    const int i = backward ? nt - 1 - s : s;
    const int ri = rows(i);
    double* Bi = B + (size_t)i * nb;
    std::vector<DJob> js;
    const int pbeg = (int)S.pairs.size();
    if (!backward) {
      for (int k = 0; k < i; ++k) S.pairs.push_back(DPair{tile(i, k), B + (size_t)k * nb, nb, 1, ldb, 1, nb});
    } else {
      for (int k = i + 1; k < nt; ++k) S.pairs.push_back(DPair{tile(k, i), B + (size_t)k * nb, 1, nb, ldb, 1, rows(k)});
    }
    const int pcnt = (int)S.pairs.size() - pbeg;
    if (pcnt > 0) add_jobs(js, Bi, ldb, ri, r, pbeg, pcnt, -1.0, 1.0, nb);
    S.gemm(js);
    js.clear();
    const double* Mi = L->minv_all + (size_t)i * nb2;
    const int p = (int)S.pairs.size();
    if (!backward) S.pairs.push_back(DPair{Mi, Bi, nb, 1, ldb, 1, ri});
    else S.pairs.push_back(DPair{Mi, Bi, 1, nb, ldb, 1, ri});
    add_jobs(js, T, nb, ri, r, p, 1, 1.0, 0.0, ri);
    S.gemm(js);
    S.ops.push_back([=](cudaStream_t st, const DJob*, const DPair*) -> cr_status {
      CR_CUDA(cudaMemcpy2DAsync(Bi, (size_t)ldb * sizeof(double), T, (size_t)nb * sizeof(double), (size_t)ri * sizeof(double), r,
                                cudaMemcpyDeviceToDevice, st));
      return CR_OK;
    });
  }
}

}  // namespace
}  // namespace cr

using namespace cr;

extern "C" cr_status cr_krige(cr_tilemat V, const double* d_Xo, const double* d_Xp, const double* d_yo, double* d_W, int ldw,
                              double* d_zhat, double* d_v, cr_stream stream, int* info) {
  if (info) *info = 0;
  if (!V || !d_Xo || !d_Xp || !d_yo || !d_W || !d_zhat || !d_v) return fail(CR_ERR_ARG, "cr_krige: NULL argument");
  if (!V->built) return fail(CR_ERR_STATE, "cr_krige: call cr_cov_build first");
  const int n_p = V->params.n_pred, n_o = V->n - n_p;
  if (n_p <= 0 || n_o <= 0 || ldw < n_o) return fail(CR_ERR_ARG, "cr_krige: needs prediction and observation sites, ldw >= n_o");
  CR_CUDA(cudaSetDevice(V->device));
  cudaStream_t s = stream;
  // Sigma_y = V_o + tau^2 I: the covariance of the observation sites with every diagonal entry
  // carrying the observation variance (n_pred = 0 in that sub-problem)
  cr_tilemat So = nullptr;
  CR_TRY(cr_tilemat_create(n_o, V->nb, &So));
  struct Guard {
    cr_tilemat m;
    std::vector<void*> bufs;
    ~Guard() {
      for (void* b : bufs) cudaFree(b);
      cr_tilemat_destroy(m);
    }
  } guard{So, {}};
  auto alloc = [&](size_t bytes) -> double* {
    void* p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) return nullptr;
    guard.bufs.push_back(p);
    return static_cast<double*>(p);
  };
  cr_cov_params po = V->params;
  po.n_pred = 0;
  CR_TRY(cr_cov_build(So, V->xy + (size_t)2 * n_p, &po, s));
  CR_TRY(cr_precision_map(So, 0, 1.0, 0, nullptr, nullptr));
  So->minv_all = alloc((size_t)So->nt * So->nb * So->nb * sizeof(double));
  if (!So->minv_all) return fail(CR_ERR_NOMEM, "cr_krige: inverse tiles");
  guard.bufs.pop_back();   // owned by So from here (freed by cr_tilemat_destroy)
  int inf = 0;
  cr_status st = cr_potrf_adaptive(So, s, &inf);
  if (info) *info = inf;
  if (st != CR_OK) return st;

  const int nb = V->nb;
  double* F = alloc((size_t)n_o * 3 * sizeof(double));
  double* T = alloc((size_t)nb * std::max(3, n_p) * sizeof(double));
  double* G = alloc(9 * sizeof(double));
  double* Q = alloc((size_t)3 * n_p * sizeof(double));
  double* H = alloc((size_t)3 * n_p * sizeof(double));
  double* Vop = alloc((size_t)n_o * n_p * sizeof(double));
  double* c1 = alloc((size_t)n_p * sizeof(double));
  double* c2 = alloc((size_t)n_p * sizeof(double));
  int* bad = reinterpret_cast<int*>(alloc(sizeof(int)));
  if (!F || !T || !G || !Q || !H || !Vop || !c1 || !c2 || !bad) return fail(CR_ERR_NOMEM, "cr_krige: workspace");
  CR_CUDA(cudaMemsetAsync(bad, 0, sizeof(int), s));

  // step 2: F = Sigma_y^-1 X_o
  CR_CUDA(cudaMemcpyAsync(F, d_Xo, (size_t)n_o * 3 * sizeof(double), cudaMemcpyDeviceToDevice, s));
  {
    Seq S;
    plan_trsm(S, So, F, n_o, 3, false, T);
    plan_trsm(S, So, F, n_o, 3, true, T);
    CR_TRY(S.run(s));
  }
  // step 3: G = X_o^T F; Q = F^T V_op - X_p^T; H = G^-1 Q
  CR_TRY(cov_block_launch(V->covk, V->xy, V->n, n_p, 0, n_o, n_p, Vop, n_o, s));
  k_neg_xpT<<<std::min(1024, (n_p + 255) / 256), 256, 0, s>>>(d_Xp, n_p, Q);
  CR_CHECK_LAUNCH("k_neg_xpT");
  {
    Seq S;
    S.pairs.push_back(DPair{d_Xo, F, n_o, 1, n_o, 1, n_o});   // G(m, c) = sum_q Xo[q, m] F[q, c]
    S.pairs.push_back(DPair{F, Vop, n_o, 1, n_o, 1, n_o});    // Q(m, i) += sum_q F[q, m] Vop[q, i]
    std::vector<DJob> js;
    add_jobs(js, G, 3, 3, 3, 0, 1, 1.0, 0.0, n_o);
    add_jobs(js, Q, 3, 3, n_p, 1, 1, 1.0, 1.0, n_o);
    S.gemm(js);
    CR_TRY(S.run(s));
  }
  k_solve3<<<std::min(1024, (n_p + 255) / 256), 256, 0, s>>>(G, Q, n_p, H, bad);
  CR_CHECK_LAUNCH("k_solve3");
  // step 4: W = V_op - X_o H; forward solve (Y), colsum(Y .* Y); backward solve (W)
  CR_CUDA(cudaMemcpy2DAsync(d_W, (size_t)ldw * sizeof(double), Vop, (size_t)n_o * sizeof(double), (size_t)n_o * sizeof(double), n_p,
                            cudaMemcpyDeviceToDevice, s));
  const bool oz = option_fp64_gemm() == CR_GEMM_OZAKI;
  double *Lr = nullptr, *Lc = nullptr, *Mt = nullptr;
  if (oz) {
    const size_t nn = (size_t)n_o * n_o;
    Lr = alloc(nn * sizeof(double));
    Lc = alloc(nn * sizeof(double));
    Mt = alloc((size_t)So->nt * nb * nb * sizeof(double));
    if (!Lr || !Lc || !Mt) return fail(CR_ERR_NOMEM, "cr_krige: dense factor copies");
    const int nstrict = So->nt * (So->nt - 1) / 2;
    const dim3 blk(32, 8), gt((nb + 31) / 32, (nb + 31) / 32, 1);
    if (nstrict > 0) {
      k_dense_lower<<<dim3(gt.x, gt.y, nstrict), blk, 0, s>>>(So->pool64, So->d_i64, n_o, nb, Lr, Lc);
      CR_CHECK_LAUNCH("k_dense_lower");
    }
    k_transpose_tiles<<<dim3(gt.x, gt.y, So->nt), blk, 0, s>>>(So->minv_all, nb, Mt);
    CR_CHECK_LAUNCH("k_transpose_tiles");
  }
  {
    Seq S;
    S.pairs.push_back(DPair{d_Xo, H, 1, n_o, 3, 1, 3});       // (X_o H)(q, i) = sum_m Xo[q, m] H[m, i]
    std::vector<DJob> js;
    add_jobs(js, d_W, ldw, n_o, n_p, 0, 1, -1.0, 1.0, 3);
    S.gemm(js);
    if (!oz) plan_trsm(S, So, d_W, ldw, n_p, false, T);
    CR_TRY(S.run(s));
  }
  if (oz) CR_TRY(ozaki_trsm(So, Lr, Lc, Mt, d_W, ldw, n_p, false, s));
  k_coldot<<<n_p, 256, 0, s>>>(d_W, ldw, d_W, ldw, n_o, c1);
  CR_CHECK_LAUNCH("k_coldot");
  if (oz) {
    CR_TRY(ozaki_trsm(So, Lr, Lc, Mt, d_W, ldw, n_p, true, s));
  } else {
    Seq S;
    plan_trsm(S, So, d_W, ldw, n_p, true, T);
    CR_TRY(S.run(s));
  }
  // step 5 and Eq.6
  k_coldot<<<n_p, 256, 0, s>>>(d_W, ldw, d_yo, 0, n_o, d_zhat);
  CR_CHECK_LAUNCH("k_coldot");
  k_coldot<<<n_p, 256, 0, s>>>(Vop, n_o, d_W, ldw, n_o, c2);
  CR_CHECK_LAUNCH("k_coldot");
  k_mspe<<<std::min(1024, (n_p + 255) / 256), 256, 0, s>>>(c1, c2, V->params.sigma2, n_p, d_v);
  CR_CHECK_LAUNCH("k_mspe");
  int h_bad = 0;
  CR_CUDA(cudaMemcpyAsync(&h_bad, bad, sizeof(int), cudaMemcpyDeviceToHost, s));
  CR_CUDA(cudaStreamSynchronize(s));
  if (h_bad) return fail(CR_ERR_NOT_SPD, "cr_krige: the trend system X_o^T Sigma_y^-1 X_o is not positive definite");
  return CR_OK;
}

extern "C" cr_status cr_krige_correct(const double* d_W, int ldw, const double* d_yo, const double* d_Y, int ldy, int n_p,
                                      int n_o, int M, double* d_S, int lds, cr_stream stream) {
  if (!d_W || !d_yo || !d_Y || !d_S || n_p <= 0 || n_o <= 0 || M <= 0 || ldw < n_o || ldy < n_p + n_o || lds < n_p)
    return fail(CR_ERR_ARG, "cr_krige_correct: argument");
  if (option_fp64_gemm() == CR_GEMM_OZAKI) return ozaki_correction(d_W, ldw, d_yo, d_Y, ldy, n_p, n_o, M, d_S, lds, stream);
  return correction_async(d_W, ldw, d_yo, d_Y, ldy, n_p, n_o, M, d_S, lds, stream);
}
