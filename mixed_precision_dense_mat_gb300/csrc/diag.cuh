// Dataflow factorisation of one FP64 diagonal tile (diag.cu).
#pragma once
#include <vector>

#include "common.cuh"

namespace cr {

// Flag words needed by diag_chol_launch for a tile of size nb and block size db (16):
// ver, fac, inv, iver (NB^2 each), the abort flag, the task counter and the role counter.
inline int diag_flag_words(int nb, int db) {
  const int NB = nb / db;
  return 4 * NB * NB + 3;
}

// Doubles of the publication buffers: two parities of (M_kk, L_{k+1,k}) for every block k.
inline size_t diag_pub_doubles(int nb, int db) {
  const int NB = nb / db;
  return 2 * 2 * (size_t)NB * db * db;
}

// Task list for NB x NB blocks (type, i, j, k): the factorisation and the inverse, in an
// order under which every wait of the executor ends; false if that check fails.
bool diag_task_list(int NB, std::vector<int4>& tasks);

// A (nb x nb row-major, ld nb): lower part overwritten by L, upper part zeroed; Minv (same
// layout) receives L^-1 with its upper part zeroed; W: nb x nb FP64 scratch.
// flags: two sets of diag_flag_words(nb, db) ints; set `par` must be zero on entry and is
// used, set 1 - par is cleared for the next call.  amax: two words; amax[par] (zero on entry)
// receives the IEEE bits of max |L^-1|, amax[1 - par] is cleared.  pub: diag_pub_doubles
// doubles; parity par must be all-ones bytes on entry and receives the chain's published
// blocks, parity 1 - par is refilled with all-ones bytes.  Calls alternate par, and every
// set is in its entry state before the first call.
cr_status diag_chol_launch(int db, double* A, double* Minv, double* W, int nb, int gcol0, int* status, int* flags,
                           int par, double* pub, const int4* d_tasks, int ntasks, int grid, unsigned long long* amax,
                           cudaStream_t s);

}  // namespace cr
