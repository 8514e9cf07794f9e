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
// wait_ns: limit of every device-side wait (the executor aborts with the timeout bit).
cr_status diag_chol_launch(int db, double* A, double* Minv, double* W, int nb, int gcol0, int* status, int* flags,
                           int par, double* pub, const int4* d_tasks, int ntasks, int grid, unsigned long long* amax,
                           unsigned long long wait_ns, cudaStream_t s);

// The same factorisation in double-float arithmetic (FP64 emulated on the FP32 units, about
// 48 significant bits).  A (FP64, nb x nb row-major, lower part) is only read.  Ldf and Mdf
// (nb x nb float2 pairs hi, lo, row-major) receive L and L^-1 in their lower parts (the
// strictly upper 16 x 16 blocks are left as they were), Wdf is nb x nb float2 scratch.
// amax[par] (zero on entry) receives the FP32 bits of max |L^-1| over the high parts; flags,
// pub and the parity rule as for diag_chol_launch (the same buffers serve both).
cr_status diag_chol_df_launch(int db, const double* A, float2* Ldf, float2* Mdf, float2* Wdf, int nb, int gcol0,
                              int* status, int* flags, int par, double* pub, const int4* d_tasks, int ntasks, int grid,
                              unsigned long long* amax, unsigned long long wait_ns, cudaStream_t s);

// After diag_chol_df_launch: L64 and M64 (FP64 nb x nb row-major) receive the factor and the
// inverse with zero upper parts; when mh is not NULL, mh/ml receive the FP16 high/low parts of
// L^-1 2^eM and lh/ll those of L, with eM (status[2]) chosen from *amax so that
// max |L^-1| 2^eM < 2^14.
cr_status split_diag_df_launch(const float2* Mdf, const float2* Ldf, int nb, const unsigned long long* amax, double* M64,
                               double* L64, __half* mh, __half* ml, __half* lh, __half* ll, int* status, cudaStream_t s);

}  // namespace cr
