// FP64 kernel interfaces (fp64.cu).
#pragma once
#include "common.cuh"

namespace cr {

// One product term A (m x K) times B^T (B is n x K); element (m, k) of A at
// A[m * sAm + k * sAk], element (n, k) of B at B[n * sBn + k * sBk].
struct DPair {
  const double* A;
  const double* B;
  int sAm, sAk, sBn, sBk, K;
};

// One output block C (m x n, m, n <= block size), element (m, n) at C[m * sCm + n * sCn]:
// C = beta C + alpha sum over pairs [pbeg, pbeg + pcnt) of A B^T, where this block reads
// rows arow + m of every A and rows brow + n of every B, and K is capped at kmax.
struct DJob {
  double* C;
  int sCm, sCn, m, n, pbeg, pcnt;
  double alpha, beta;
  int arow, brow, kmax;
};

cr_status dgemm_launch(int block, const DJob* d_jobs, const DPair* d_pairs, int njobs, cudaStream_t stream);
cr_status potrf64_base_launch(double* A, int lda, double* Minv, int ldm, int gcol0, int* status, cudaStream_t s);
cr_status split_tile_launch(const double* src, int nb, __half* hi, __half* lo, int lower_only, cudaStream_t s);
// part: 64 doubles of device scratch
// FP16 high/low splits of the inverse factor (scaled by 2^eM, status[2] = eM, from the maximum
// in *amax) and of the diagonal factor's lower part, in one launch.
cr_status split_diag_launch(const double* Minv, const double* L, int nb, const unsigned long long* amax, __half* mh, __half* ml,
                            __half* lh, __half* ll, int* status, cudaStream_t s);
cr_status status_init_launch(int* status, cudaStream_t s);

}  // namespace cr
