// Adaptive mixed-precision tile Cholesky driver (left-looking, one tile column at a time).
//
// "Mixed-Precision GPU Acceleration for Confidence Regions of Spatial Excursion Sets",
// Section IV-B and Alg.2 step 12: L_s = chol(s^2 V) with the tile precisions of the map;
// diagonal tiles FP64.  For tile column j:
//   1. FP64 products (destination and both operands FP64) on the FP64 units;
//   2. every other product on the tensor cores (FP16, or FP16 high/low parts for FP32-class
//      accuracy), accumulated in FP32 and applied to the destination in its own precision;
//   3. the FP64 diagonal tile is factored together with its inverse (recursive 2 x 2 blocks
//      down to 64 x 64, the GEMMs spread over many SMs);
//   4. the off-diagonal tiles of the column are solved, L_ij = A_ij L_jj^-T, as a product with
//      the inverse factor, in the tile's precision.
// The schedule depends only on the map, so it is built once on the host (all job lists are
// uploaded in one copy) and then replayed in stream order.
#include <functional>

#include "common.cuh"
#include "fp64.cuh"
#include "tc.cuh"

namespace cr {

cr_status convert_tiles(cr_tilemat V, cudaStream_t stream);

__global__ void k_zero_upper(double* A, int nb) {
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < nb * nb; idx += gridDim.x * blockDim.x) {
    const int r = idx / nb, c = idx % nb;
    if (c > r) A[idx] = 0.0;
  }
}

namespace {

using Op = std::function<cr_status(cudaStream_t, const DJob*, const DPair*)>;

struct Plan {
  std::vector<DJob> jobs;
  std::vector<DPair> pairs;
  std::vector<Op> ops;

  int add_pair(const double* A, const double* B, int sAm, int sAk, int sBn, int sBk, int K) {
    pairs.push_back(DPair{A, B, sAm, sAk, sBn, sBk, K});
    return (int)pairs.size() - 1;
  }
  void dgemm(int block, const std::vector<DJob>& js) {
    if (js.empty()) return;
    const int off = (int)jobs.size(), cnt = (int)js.size();
    jobs.insert(jobs.end(), js.begin(), js.end());
    ops.push_back([=](cudaStream_t s, const DJob* dj, const DPair* dp) -> cr_status { return dgemm_launch(block, dj + off, dp, cnt, s); });
  }
};

DJob job(double* C, int sCm, int sCn, int m, int n, int pbeg, int pcnt, double alpha, double beta, int arow, int brow,
         int kmax) {
  DJob j;
  j.C = C; j.sCm = sCm; j.sCn = sCn; j.m = m; j.n = n; j.pbeg = pbeg; j.pcnt = pcnt;
  j.alpha = alpha; j.beta = beta; j.arow = arow; j.brow = brow; j.kmax = kmax;
  return j;
}

// Cholesky and inverse of the n x n diagonal block at offset `off` of the FP64 tile A
// (row-major, ld nb); inverse into M (same layout), temporaries in T.
void plan_chol_inv(Plan& P, cr_tilemat V, double* A, double* M, double* T, int off, int n, int gcol0) {
  const int nb = V->nb;
  int* status = V->d_status;
  if (n == 64) {
    double* a = A + (size_t)off * nb + off;
    double* m = M + (size_t)off * nb + off;
    const int g = gcol0 + off;
    P.ops.push_back([=](cudaStream_t s, const DJob*, const DPair*) -> cr_status { return potrf64_base_launch(a, nb, m, nb, g, status, s); });
    return;
  }
  const int h = n / 2;
  const int bs = 16;
  const int nbk = h / bs;
  plan_chol_inv(P, V, A, M, T, off, h, gcol0);
  double* A21 = A + (size_t)(off + h) * nb + off;
  double* A22 = A + (size_t)(off + h) * nb + off + h;
  double* M11 = M + (size_t)off * nb + off;
  double* M21 = M + (size_t)(off + h) * nb + off;
  double* M22 = M + (size_t)(off + h) * nb + off + h;
  double* U = T + h;   // second h x h scratch block
  std::vector<DJob> js;
  // T = A21 M11^T
  int p = P.add_pair(A21, M11, nb, 1, nb, 1, h);
  for (int bi = 0; bi < nbk; ++bi)
    for (int bj = 0; bj < nbk; ++bj)
      js.push_back(job(T + (size_t)bi * bs * nb + bj * bs, nb, 1, bs, bs, p, 1, 1.0, 0.0, bi * bs, bj * bs, h));
  P.dgemm(bs, js);
  js.clear();
  // A22 -= T T^T (lower blocks)
  p = P.add_pair(T, T, nb, 1, nb, 1, h);
  for (int bi = 0; bi < nbk; ++bi)
    for (int bj = 0; bj <= bi; ++bj)
      js.push_back(job(A22 + (size_t)bi * bs * nb + bj * bs, nb, 1, bs, bs, p, 1, -1.0, 1.0, bi * bs, bj * bs, h));
  P.dgemm(bs, js);
  js.clear();
  // A21 = T
  P.ops.push_back([=](cudaStream_t s, const DJob*, const DPair*) -> cr_status {
    CR_CUDA(cudaMemcpy2DAsync(A21, nb * sizeof(double), T, nb * sizeof(double), h * sizeof(double), h,
                              cudaMemcpyDeviceToDevice, s));
    return CR_OK;
  });
  plan_chol_inv(P, V, A, M, T, off + h, h, gcol0);
  // U = L21 M11 (B(n, k) = M11[k][n])
  p = P.add_pair(A21, M11, nb, 1, 1, nb, h);
  for (int bi = 0; bi < nbk; ++bi)
    for (int bj = 0; bj < nbk; ++bj)
      js.push_back(job(U + (size_t)bi * bs * nb + bj * bs, nb, 1, bs, bs, p, 1, 1.0, 0.0, bi * bs, bj * bs, h));
  P.dgemm(bs, js);
  js.clear();
  // M21 = -M22 U (B(n, k) = U[k][n])
  p = P.add_pair(M22, U, nb, 1, 1, nb, h);
  for (int bi = 0; bi < nbk; ++bi)
    for (int bj = 0; bj < nbk; ++bj)
      js.push_back(job(M21 + (size_t)bi * bs * nb + bj * bs, nb, 1, bs, bs, p, 1, -1.0, 0.0, bi * bs, bj * bs, h));
  P.dgemm(bs, js);
}

}  // namespace

cr_status build_and_run_cholesky(cr_tilemat V, cudaStream_t stream) {
  const int nt = V->nt, nb = V->nb;
  const size_t nb2 = (size_t)nb * nb;
  const int nsb = nb / TC_BM;
  const auto& cls = V->h_cls;
  auto t64 = [&](int i, int j) { return V->pool64 + (size_t)V->h_i64[tidx(i, j)] * nb2; };
  Plan P;
  int* status = V->d_status;
  P.ops.push_back([=](cudaStream_t s, const DJob*, const DPair*) -> cr_status { return status_init_launch(status, s); });
  P.ops.push_back([=](cudaStream_t s, const DJob*, const DPair*) -> cr_status { return convert_tiles(V, s); });

  // rows solved on the tensor cores, per column
  std::vector<int> rows_flat;
  std::vector<int> rows_off(nt + 1, 0);
  for (int j = 0; j < nt; ++j) {
    rows_off[j] = (int)rows_flat.size();
    for (int i = j + 1; i < nt; ++i)
      if (cls[tidx(i, j)] != CR_PREC_FP64) rows_flat.push_back(i);
  }
  rows_off[nt] = (int)rows_flat.size();
  int* d_rows = nullptr;
  if (!rows_flat.empty()) {
    CR_CUDA(cudaMalloc(&d_rows, rows_flat.size() * sizeof(int)));
    CR_CUDA(cudaMemcpy(d_rows, rows_flat.data(), rows_flat.size() * sizeof(int), cudaMemcpyHostToDevice));
  }

  TcParams base{};
  base.v = V->view();
  base.ws_hi0 = V->ws_hi0;
  base.ws_lo0 = V->ws_lo0;
  base.minv_hi = V->minv_hi;
  base.minv_lo = V->minv_lo;
  base.eA = V->eA;
  base.status = V->d_status;
  base.err = V->d_status;
  base.ws64 = V->ws64;

  for (int j = 0; j < nt; ++j) {
    // 1. FP64 products
    {
      std::vector<DJob> js;
      for (int i = j; i < nt; ++i) {
        if (cls[tidx(i, j)] != CR_PREC_FP64) continue;
        const int pbeg = (int)P.pairs.size();
        for (int k = 0; k < j; ++k)
          if (cls[tidx(i, k)] == CR_PREC_FP64 && cls[tidx(j, k)] == CR_PREC_FP64)
            P.add_pair(t64(i, k), t64(j, k), nb, 1, nb, 1, nb);
        const int pcnt = (int)P.pairs.size() - pbeg;
        if (pcnt == 0) continue;
        double* C = t64(i, j);
        for (int bi = 0; bi < nb / 64; ++bi)
          for (int bj = 0; bj < nb / 64; ++bj) {
            if (i == j && bj > bi) continue;
            js.push_back(job(C + (size_t)bi * 64 * nb + bj * 64, nb, 1, 64, 64, pbeg, pcnt, -1.0, 1.0, bi * 64, bj * 64, nb));
          }
      }
      P.dgemm(64, js);
    }
    // 2. tensor-core products (also stages the solve inputs), or plain copies without AMP
    if (V->amp) {
      TcParams tp = base;
      tp.mode = TC_UPDATE;
      tp.j = j;
      tp.rows = nullptr;
      const int grid = (nt - j) * nsb * nsb;
      const CUtensorMap* tm = &V->tm_pool16;
      P.ops.push_back([=](cudaStream_t s, const DJob*, const DPair*) -> cr_status { return tc_launch(tp, *tm, *tm, grid, s); });
    } else {
      for (int i = j + 1; i < nt; ++i) {
        double* dst = V->ws64 + (size_t)i * nb2;
        const double* src = t64(i, j);
        P.ops.push_back([=](cudaStream_t s, const DJob*, const DPair*) -> cr_status {
          CR_CUDA(cudaMemcpyAsync(dst, src, nb2 * sizeof(double), cudaMemcpyDeviceToDevice, s));
          return CR_OK;
        });
      }
    }
    // 3. diagonal factor and its inverse
    double* Ajj = t64(j, j);
    double* Minv = V->minv;
    double* T = V->scratch64;
    P.ops.push_back([=](cudaStream_t s, const DJob*, const DPair*) -> cr_status {
      CR_CUDA(cudaMemsetAsync(Minv, 0, nb2 * sizeof(double), s));
      return CR_OK;
    });
    plan_chol_inv(P, V, Ajj, Minv, T, 0, nb, j * nb);
    P.ops.push_back([=](cudaStream_t s, const DJob*, const DPair*) -> cr_status {
      k_zero_upper<<<64, 256, 0, s>>>(Ajj, nb);
      CR_CHECK_LAUNCH("k_zero_upper");
      return CR_OK;
    });
    if (V->amp) {
      __half* mh = V->pool16 + (size_t)V->minv_hi * nb2;
      __half* ml = V->pool16 + (size_t)V->minv_lo * nb2;
      __half* dh = V->pool16 + (size_t)V->h_hi16[tidx(j, j)] * nb2;
      __half* dl = V->pool16 + (size_t)V->h_lo16[tidx(j, j)] * nb2;
      P.ops.push_back([=](cudaStream_t s, const DJob*, const DPair*) -> cr_status {
        CR_TRY(split_minv_launch(Minv, nb, mh, ml, status, s));
        return split_tile_launch(Ajj, nb, dh, dl, 1, s);
      });
    }
    // 4. off-diagonal solves
    const int ntc = rows_off[j + 1] - rows_off[j];
    if (ntc > 0) {
      TcParams tp = base;
      tp.mode = TC_TRSM;
      tp.j = j;
      tp.rows = d_rows + rows_off[j];
      const int grid = ntc * nsb * nsb;
      const CUtensorMap* tm = &V->tm_pool16;
      P.ops.push_back([=](cudaStream_t s, const DJob*, const DPair*) -> cr_status { return tc_launch(tp, *tm, *tm, grid, s); });
    }
    {
      std::vector<DJob> js;
      std::vector<int> fp64_rows;
      for (int i = j + 1; i < nt; ++i) {
        if (cls[tidx(i, j)] != CR_PREC_FP64) continue;
        fp64_rows.push_back(i);
        const int p = P.add_pair(V->ws64 + (size_t)i * nb2, Minv, nb, 1, nb, 1, nb);
        double* C = t64(i, j);
        for (int bi = 0; bi < nb / 64; ++bi)
          for (int bj = 0; bj < nb / 64; ++bj)
            js.push_back(job(C + (size_t)bi * 64 * nb + bj * 64, nb, 1, 64, 64, p, 1, 1.0, 0.0, bi * 64, bj * 64, (bj + 1) * 64));
      }
      P.dgemm(64, js);
      if (V->amp) {
        for (int i : fp64_rows) {
          const double* src = t64(i, j);
          __half* h = V->pool16 + (size_t)V->h_hi16[tidx(i, j)] * nb2;
          __half* l = V->pool16 + (size_t)V->h_lo16[tidx(i, j)] * nb2;
          P.ops.push_back([=](cudaStream_t s, const DJob*, const DPair*) -> cr_status { return split_tile_launch(src, nb, h, l, 0, s); });
        }
      }
    }
  }

  // upload job lists and replay
  DJob* d_jobs = nullptr;
  DPair* d_pairs = nullptr;
  cr_status st = CR_OK;
  if (!P.jobs.empty() && cudaMalloc(&d_jobs, P.jobs.size() * sizeof(DJob)) != cudaSuccess) st = fail(CR_ERR_NOMEM, "job list");
  if (st == CR_OK && !P.pairs.empty() && cudaMalloc(&d_pairs, P.pairs.size() * sizeof(DPair)) != cudaSuccess)
    st = fail(CR_ERR_NOMEM, "pair list");
  if (st == CR_OK && d_jobs)
    if (cudaMemcpyAsync(d_jobs, P.jobs.data(), P.jobs.size() * sizeof(DJob), cudaMemcpyHostToDevice, stream) != cudaSuccess)
      st = fail(CR_ERR_CUDA, "job upload");
  if (st == CR_OK && d_pairs)
    if (cudaMemcpyAsync(d_pairs, P.pairs.data(), P.pairs.size() * sizeof(DPair), cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
      st = fail(CR_ERR_CUDA, "pair upload");
  for (size_t q = 0; st == CR_OK && q < P.ops.size(); ++q) st = P.ops[q](stream, d_jobs, d_pairs);
  cudaError_t e = cudaStreamSynchronize(stream);
  if (st == CR_OK && e != cudaSuccess) st = cuda_fail(e, "cholesky");
  if (d_jobs) cudaFree(d_jobs);
  if (d_pairs) cudaFree(d_pairs);
  if (d_rows) cudaFree(d_rows);
  return st;
}

}  // namespace cr

using namespace cr;

extern "C" cr_status cr_potrf_adaptive(cr_tilemat V, cr_stream stream, int* info) {
  if (!V) return fail(CR_ERR_ARG, "cr_potrf_adaptive: NULL handle");
  if (info) *info = 0;
  if (!V->mapped) return fail(CR_ERR_STATE, "cr_potrf_adaptive: call cr_precision_map first");
  CR_CUDA(cudaSetDevice(V->device));
  CR_TRY(build_and_run_cholesky(V, stream));
  int h[4];
  CR_CUDA(cudaMemcpy(h, V->d_status, sizeof(h), cudaMemcpyDeviceToHost));
  V->info = h[1] == 0x7fffffff ? 0 : h[1];
  if (info) *info = V->info;
  if (h[0] & DEV_ERR_TIMEOUT) return fail(CR_ERR_TIMEOUT, "cr_potrf_adaptive: a device-side wait timed out");
  if (V->info) return fail(CR_ERR_NOT_SPD, "cr_potrf_adaptive: leading minor not positive definite at column " + std::to_string(V->info));
  V->factored = true;
  return CR_OK;
}
