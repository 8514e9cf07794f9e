// Universal kriging and the conditioning correction (FP64).
//
// "Mixed-Precision GPU Acceleration for Confidence Regions of Spatial Excursion Sets":
// Section V-A Eq.5-6 (weights, prediction, pointwise MSPE; the kriging stage is FP64) and
// Section V-B Eq.7 (S = M_p + W^T (y_o 1^T - M_o): the residual is formed by negating M_o
// and broadcasting y_o, then one GEMM applies the correction).
#include "common.cuh"
#include "fp64.cuh"

namespace cr {

__global__ void k_residual(const double* __restrict__ yo, const double* __restrict__ Mo, int ldy, int n_o, int M,
                           double* __restrict__ R) {
  const size_t total = (size_t)n_o * M;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const int j = (int)(e / n_o), q = (int)(e % n_o);
    R[e] = yo[q] - Mo[(size_t)j * ldy + q];
  }
}

}  // namespace cr

using namespace cr;

extern "C" cr_status cr_krige(cr_tilemat V, const double* d_Xo, const double* d_Xp, const double* d_yo, double* d_W, int ldw,
                              double* d_zhat, double* d_v, cr_stream stream, int* info) {
  (void)V; (void)d_Xo; (void)d_Xp; (void)d_yo; (void)d_W; (void)ldw; (void)d_zhat; (void)d_v; (void)stream;
  if (info) *info = 0;
  return fail(CR_ERR_NOT_IMPLEMENTED, "cr_krige: not built yet");
}

extern "C" cr_status cr_krige_correct(const double* d_W, int ldw, const double* d_yo, const double* d_Y, int ldy, int n_p,
                                      int n_o, int M, double* d_S, int lds, cr_stream stream) {
  if (!d_W || !d_yo || !d_Y || !d_S || n_p <= 0 || n_o <= 0 || M <= 0 || ldw < n_o || ldy < n_p + n_o || lds < n_p)
    return fail(CR_ERR_ARG, "cr_krige_correct: argument");
  double* R = nullptr;
  CR_CUDA(cudaMallocAsync(&R, (size_t)n_o * M * sizeof(double), stream));
  k_residual<<<1216, 256, 0, stream>>>(d_yo, d_Y + n_p, ldy, n_o, M, R);
  CR_CHECK_LAUNCH("k_residual");
  CR_CUDA(cudaMemcpy2DAsync(d_S, (size_t)lds * sizeof(double), d_Y, (size_t)ldy * sizeof(double), (size_t)n_p * sizeof(double), M,
                            cudaMemcpyDeviceToDevice, stream));
  // S += W^T R : A(m = site i, k = obs q) = W[i ldw + q], B(n = sim j, k = obs q) = R[j n_o + q]
  const int bs = 64;
  std::vector<DJob> jobs;
  DPair pr{d_W, R, ldw, 1, n_o, 1, n_o};
  for (int i0 = 0; i0 < n_p; i0 += bs)
    for (int j0 = 0; j0 < M; j0 += bs) {
      DJob jb{};
      jb.C = d_S + (size_t)j0 * lds + i0;
      jb.sCm = 1; jb.sCn = lds;
      jb.m = std::min(bs, n_p - i0); jb.n = std::min(bs, M - j0);
      jb.pbeg = 0; jb.pcnt = 1; jb.alpha = 1.0; jb.beta = 1.0;
      jb.arow = i0; jb.brow = j0; jb.kmax = n_o;
      jobs.push_back(jb);
    }
  DJob* dj = nullptr;
  DPair* dp = nullptr;
  CR_CUDA(cudaMallocAsync(&dj, jobs.size() * sizeof(DJob), stream));
  CR_CUDA(cudaMallocAsync(&dp, sizeof(DPair), stream));
  CR_CUDA(cudaMemcpyAsync(dj, jobs.data(), jobs.size() * sizeof(DJob), cudaMemcpyHostToDevice, stream));
  CR_CUDA(cudaMemcpyAsync(dp, &pr, sizeof(DPair), cudaMemcpyHostToDevice, stream));
  CR_TRY(dgemm_launch(bs, dj, dp, (int)jobs.size(), stream));
  CR_CUDA(cudaFreeAsync(dj, stream));
  CR_CUDA(cudaFreeAsync(dp, stream));
  CR_CUDA(cudaFreeAsync(R, stream));
  // pageable host-to-device copies are staged before cudaMemcpyAsync returns, so the host
  // job vector may go out of scope here
  return CR_OK;
}
