// Dataflow factorisation of one FP64 diagonal tile (diag.cu).
#pragma once
#include <vector>

#include "common.cuh"

namespace cr {

// Flag words needed by diag_chol_launch for a tile of size nb and block size db (16 or 32):
// ver, fac, inv, tfl (NB^2 each), the abort flag, the task counter and the role counter.
inline int diag_flag_words(int nb, int db) {
  const int NB = nb / db;
  return 4 * NB * NB + 3;
}

// Fixed topological task order for NB x NB blocks (type, i, j, k / s).
void diag_task_list(int NB, std::vector<int4>& tasks);

// A (nb x nb row-major, ld nb): lower part overwritten by L; Minv (same layout) receives
// L^-1 (lower; the caller zeroes it beforehand); T: nb x nb FP64 scratch.  flags:
// diag_flag_words(nb, db) ints of device scratch, cleared by this call.
cr_status diag_chol_launch(int db, double* A, double* Minv, double* T, int nb, int gcol0, int* status, int* flags,
                           const int4* d_tasks, int ntasks, int grid, cudaStream_t s);

}  // namespace cr
