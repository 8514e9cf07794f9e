// Covariance evaluation shared by the covariance, conversion and kriging kernels (cov.cu).
#pragma once
#include "common.cuh"

namespace cr {

// Dense column-major block V[r0 + i, c0 + j] (i < m, j < k), FP64, from locations xy (n x 2).
cr_status cov_block_launch(const CovK& p, const double* xy, int n, int r0, int c0, int m, int k, double* out, int ld,
                           cudaStream_t s);

}  // namespace cr
