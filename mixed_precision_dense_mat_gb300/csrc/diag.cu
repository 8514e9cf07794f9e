// FP64 factorisation of one diagonal tile, L_jj = chol(A_jj), together with its inverse
// M = L_jj^-1, as an on-device dataflow executor.
//
// The nb x nb tile is cut into DB x DB blocks.  The blocked Cholesky DAG (the tile-DAG
// formulation of Section IV-A of "Mixed-Precision GPU Acceleration for Confidence Regions
// of Spatial Excursion Sets", here inside one tile and on one GPU) is listed in a fixed
// topological order:
//   POTRF(k)      factor block (k,k) and invert it                   needs ver(k,k) = k
//   TRSM(i,k)     L_ik = A_ik M_kk^T                                 needs POTRF(k), ver(i,k) = k
//   UPDATE(i,j,k) A_ij -= L_ik L_jk^T  (k < j <= i)                   needs TRSM(i,k), TRSM(j,k), ver(i,j) = k
// The inverse is assembled by recursive doubling: for every aligned pair of diagonal
// super-blocks of s blocks each, [[L11, 0], [L21, L22]]^-1 has lower-left part
// M21 = -M22 (L21 M11), computed block by block as
//   TMUL(R,C,s)   T_RC = sum_m L_Rm M_mC      (m over the M11 half)
//   MMUL(R,C,s)   M_RC = -sum_m M_Rm T_mC     (m over the M22 half)
// so the inverse's dependent chain is about 2 NB block products instead of NB^2.  The
// inverse tasks of a pair are listed right after the factorisation step that finishes the
// pair's last diagonal block.
// A fixed grid of CTAs takes tasks from a global counter in that order and waits (bounded,
// wall-clock limited) on per-block flags released by the producers.  A task only waits on
// tasks earlier in the order, which were taken by CTAs that are already running, so the
// scheme needs no co-residency guarantee.  On GB300 the FP64 units give about two FMA lanes
// per SM per clock, so small blocks and many SMs keep the dependent chain short; the CTAs
// use little shared memory and can share SMs with tensor-core kernels.
#include <math.h>

#include "common.cuh"
#include "diag.cuh"
#include "ptx.cuh"

namespace cr {

namespace {

enum { T_POTRF = 0, T_TRSM = 1, T_UPDATE = 2, T_TMUL = 3, T_MMUL = 4 };

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

struct Ctx {
  double* A;
  double* Minv;
  double* T;   // products L21 M11 of the doubling steps (same block positions as M21)
  int nb, NB;
  int* ver;    // NB x NB: updates applied to block (i, j)
  int* fac;    // NB x NB: L block (i, j) final (for i == j also the inverse block M_ii)
  int* inv;    // NB x NB: inverse block (i, j), i > j, final
  int* tfl;    // NB x NB: T block (i, j) final
  int* abort_flag;
  int* status;
  int gcol0;
};

// Thread 0 waits until *p >= v; false on timeout (sets the abort flag and the error bit).
__device__ bool wait_ge(const Ctx& c, const int* p, int v) {
  if (ld_acquire(p) >= v) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (ld_acquire(p) >= v) return true;
    if (ld_acquire(c.abort_flag)) return false;
    if (global_timer_ns() - t0 > 2000000000ull) {
      atomicOr(&c.status[0], DEV_ERR_TIMEOUT);
      atomicExch(c.abort_flag, 1);
      return false;
    }
  }
}

template <int DB>
__device__ __forceinline__ void load_block(double (*S)[DB + 1], const double* src, int ld, bool lower_only = false) {
  for (int idx = threadIdx.x; idx < DB * DB; idx += blockDim.x) {
    const int r = idx / DB, q = idx % DB;
    S[r][q] = (lower_only && q > r) ? 0.0 : __ldcg(src + (size_t)r * ld + q);
  }
}
// S[col][q] = src[q][col]
template <int DB>
__device__ __forceinline__ void load_block_t(double (*S)[DB + 1], const double* src, int ld) {
  for (int idx = threadIdx.x; idx < DB * DB; idx += blockDim.x) {
    const int r = idx / DB, q = idx % DB;
    S[q][r] = __ldcg(src + (size_t)r * ld + q);
  }
}

// Cholesky of the DB x DB block k held (lower part) in L, in place, with its inverse in X;
// then both are written to the tile (factor, lower part) and to Minv (inverse, upper zero).
template <int DB>
__device__ void potrf_block(const Ctx& c, int k, double (*L)[DB + 1], double (*X)[DB + 1], double* s_r) {
  double* a = c.A + (size_t)(k * DB) * c.nb + k * DB;
  for (int idx = threadIdx.x; idx < DB * DB; idx += blockDim.x) {
    const int r = idx / DB, q = idx % DB;
    X[r][q] = (r == q) ? 1.0 : 0.0;
  }
  __syncthreads();
  for (int col = 0; col < DB; ++col) {
    if (threadIdx.x == 0) {
      const double d = L[col][col];
      if (!(d > 0.0)) atomicMin(&c.status[1], c.gcol0 + k * DB + col + 1);
      const double r = rsqrt(d);
      L[col][col] = d * r;
      *s_r = r;
    }
    __syncthreads();
    const double rc = *s_r;
    for (int i = threadIdx.x; i < DB; i += blockDim.x) {
      if (i > col) L[i][col] *= rc;
      if (i <= col) X[col][i] *= rc;
    }
    __syncthreads();
    // L[r][q] -= L[r][col] L[q][col] (col < q <= r);  X[r][q] -= L[r][col] X[col][q] (q <= col < r)
    const int rows = DB - col - 1;
    for (int idx = threadIdx.x; idx < rows * DB; idx += blockDim.x) {
      const int r = col + 1 + idx / DB, q = idx % DB;
      const double lrc = L[r][col];
      if (q > col) {
        if (q <= r) L[r][q] -= lrc * L[q][col];
      } else {
        X[r][q] -= lrc * X[col][q];
      }
    }
    __syncthreads();
  }
  double* m = c.Minv + (size_t)(k * DB) * c.nb + k * DB;
  for (int idx = threadIdx.x; idx < DB * DB; idx += blockDim.x) {
    const int r = idx / DB, q = idx % DB;
    if (q <= r) a[(size_t)r * c.nb + q] = L[r][q];
    m[(size_t)r * c.nb + q] = (q <= r) ? X[r][q] : 0.0;
  }
}

template <int DB>
struct Frag {
  static constexpr int PER = (DB * DB) / 256;   // outputs per thread (1 for DB = 16, 4 for DB = 32)
  double acc[PER];
  __device__ void zero() {
#pragma unroll
    for (int x = 0; x < PER; ++x) acc[x] = 0.0;
  }
  // acc(r, col) += sum_q P[r][q] Q[col][q]
  __device__ void mac(double (*P)[DB + 1], double (*Q)[DB + 1]) {
    const int r = threadIdx.x / (DB / PER), c0 = threadIdx.x % (DB / PER);
#pragma unroll 8
    for (int q = 0; q < DB; ++q) {
      const double a = P[r][q];
#pragma unroll
      for (int x = 0; x < PER; ++x) acc[x] = fma(a, Q[c0 + x * (DB / PER)][q], acc[x]);
    }
  }
  // S(r, col) += alpha acc (lower part only when asked)
  __device__ void add_to(double (*S)[DB + 1], double alpha, bool lower_only) {
    const int r = threadIdx.x / (DB / PER), c0 = threadIdx.x % (DB / PER);
#pragma unroll
    for (int x = 0; x < PER; ++x) {
      const int col = c0 + x * (DB / PER);
      if (!(lower_only && col > r)) S[r][col] += alpha * acc[x];
    }
  }
  // S(r, col) = acc and dst(r, col) = acc
  __device__ void put(double (*S)[DB + 1], double* dst, int ld) {
    const int r = threadIdx.x / (DB / PER), c0 = threadIdx.x % (DB / PER);
#pragma unroll
    for (int x = 0; x < PER; ++x) {
      const int col = c0 + x * (DB / PER);
      S[r][col] = acc[x];
      dst[(size_t)r * ld + col] = acc[x];
    }
  }
  // dst(r, col) = alpha acc (+ dst when accumulate)
  __device__ void store(double* dst, int ld, double alpha, bool accumulate, bool lower_only) {
    const int r = threadIdx.x / (DB / PER), c0 = threadIdx.x % (DB / PER);
#pragma unroll
    for (int x = 0; x < PER; ++x) {
      const int col = c0 + x * (DB / PER);
      if (lower_only && col > r) continue;
      double* o = dst + (size_t)r * ld + col;
      *o = accumulate ? __ldcg(o) + alpha * acc[x] : alpha * acc[x];
    }
  }
};

// dst = alpha sum_{m = m0}^{m1 - 1} P_m Q_m with P_m the block at Prow + m DB (ld nb) and Q_m
// the block at Qcol + m DB nb (ld nb).
template <int DB>
__device__ void chain_product(const Ctx& c, const double* Prow, const double* Qcol, int m0, int m1, double* dst, double alpha,
                              double (*S0)[DB + 1], double (*S1)[DB + 1]) {
  Frag<DB> f;
  f.zero();
  for (int m = m0; m < m1; ++m) {
    load_block<DB>(S0, Prow + (size_t)m * DB, c.nb);
    load_block_t<DB>(S1, Qcol + (size_t)m * DB * c.nb, c.nb);
    __syncthreads();
    f.mac(S0, S1);
    __syncthreads();
  }
  f.store(dst, c.nb, alpha, false, false);
}

// The critical chain, run by one CTA with the blocks kept in shared memory:
// POTRF(0); then for k = 0 .. NB-2: TRSM(k+1,k), SYRK(k+1,k+1,k), POTRF(k+1).
template <int DB>
__device__ void run_chain(const Ctx& c, double (*S0)[DB + 1], double (*S1)[DB + 1], double (*S2)[DB + 1],
                          double (*S3)[DB + 1], double* s_r, int* s_ok) {
  const int NB = c.NB;
  const size_t rowstride = (size_t)DB * c.nb;
  load_block<DB>(S0, c.A, c.nb, true);
  potrf_block<DB>(c, 0, S0, S1, s_r);   // S1 = M_00
  __syncthreads();
  if (threadIdx.x == 0) st_release(&c.fac[0], 1);
  for (int k = 0; k + 1 < NB; ++k) {
    const int i = k + 1;
    // TRSM(i, k): L_ik = A_ik M_kk^T, M_kk in S1
    if (threadIdx.x == 0) *s_ok = wait_ge(c, &c.ver[i * NB + k], k) ? 1 : 0;
    __syncthreads();
    if (!*s_ok) return;
    load_block<DB>(S2, c.A + i * rowstride + k * DB, c.nb);
    __syncthreads();
    Frag<DB> f;
    f.zero();
    f.mac(S2, S1);
    f.put(S3, c.A + i * rowstride + k * DB, c.nb);   // S3 = L_ik
    __syncthreads();
    if (threadIdx.x == 0) st_release(&c.fac[i * NB + k], 1);
    // SYRK(i, i, k) into the diagonal block, then POTRF(i)
    if (threadIdx.x == 0) *s_ok = wait_ge(c, &c.ver[i * NB + i], k) ? 1 : 0;
    __syncthreads();
    if (!*s_ok) return;
    load_block<DB>(S0, c.A + i * rowstride + i * DB, c.nb, true);
    __syncthreads();
    Frag<DB> g;
    g.zero();
    g.mac(S3, S3);
    g.add_to(S0, -1.0, true);
    __syncthreads();
    potrf_block<DB>(c, i, S0, S1, s_r);   // S1 = M_ii
    __syncthreads();
    if (threadIdx.x == 0) st_release(&c.fac[i * NB + i], 1);
  }
}

template <int DB>
__global__ void __launch_bounds__(256) k_diag_chol(Ctx c, const int4* __restrict__ tasks, int ntasks, int* counter,
                                                   int* role) {
  __shared__ double S0[DB][DB + 1];
  __shared__ double S1[DB][DB + 1];
  __shared__ double S2[DB][DB + 1];
  __shared__ double S3[DB][DB + 1];
  __shared__ double s_r;
  __shared__ int s_task;
  __shared__ int s_ok;
  const int NB = c.NB;
  const size_t rowstride = (size_t)DB * c.nb;
  // the first CTA to start takes the critical chain: it is resident, so the chain progresses
  if (threadIdx.x == 0) s_task = atomicAdd(role, 1);
  __syncthreads();
  if (s_task == 0) {
    run_chain<DB>(c, S0, S1, S2, S3, &s_r, &s_ok);
    return;
  }
  while (true) {
    if (threadIdx.x == 0) s_task = atomicAdd(counter, 1);
    __syncthreads();
    const int t = s_task;
    if (t >= ntasks) break;
    const int4 tk = tasks[t];
    const int type = tk.x;
    if (threadIdx.x == 0) {
      bool ok = true;
      if (type == T_POTRF) {
        const int k = tk.w;
        ok = wait_ge(c, &c.ver[k * NB + k], k);
      } else if (type == T_TRSM) {
        const int i = tk.y, k = tk.w;
        ok = wait_ge(c, &c.fac[k * NB + k], 1) && wait_ge(c, &c.ver[i * NB + k], k);
      } else if (type == T_UPDATE) {
        const int i = tk.y, j = tk.z, k = tk.w;
        ok = wait_ge(c, &c.fac[i * NB + k], 1) && wait_ge(c, &c.fac[j * NB + k], 1) && wait_ge(c, &c.ver[i * NB + j], k);
      } else {
        const int R = tk.y, C = tk.z, s = tk.w;
        const int base = C - C % (2 * s);
        if (type == T_TMUL) {
          for (int m = C; ok && m < base + s; ++m)
            ok = wait_ge(c, &c.fac[R * NB + m], 1) && (m == C ? wait_ge(c, &c.fac[C * NB + C], 1) : wait_ge(c, &c.inv[m * NB + C], 1));
        } else {
          for (int m = base + s; ok && m <= R; ++m)
            ok = (m == R ? wait_ge(c, &c.fac[R * NB + R], 1) : wait_ge(c, &c.inv[R * NB + m], 1)) && wait_ge(c, &c.tfl[m * NB + C], 1);
        }
      }
      s_ok = ok ? 1 : 0;
    }
    __syncthreads();
    if (!s_ok) break;
    if (type == T_TRSM) {
      const int i = tk.y, k = tk.w;
      double* a = c.A + i * rowstride + k * DB;
      load_block<DB>(S0, a, c.nb);
      load_block<DB>(S1, c.Minv + k * rowstride + k * DB, c.nb);
      __syncthreads();
      Frag<DB> f;
      f.zero();
      f.mac(S0, S1);
      f.store(a, c.nb, 1.0, false, false);
    } else if (type == T_UPDATE) {
      const int i = tk.y, j = tk.z, k = tk.w;
      load_block<DB>(S0, c.A + i * rowstride + k * DB, c.nb);
      load_block<DB>(S1, c.A + j * rowstride + k * DB, c.nb);
      __syncthreads();
      Frag<DB> f;
      f.zero();
      f.mac(S0, S1);
      f.store(c.A + i * rowstride + j * DB, c.nb, -1.0, true, i == j);
    } else if (type == T_TMUL) {
      const int R = tk.y, C = tk.z, s = tk.w;
      const int base = C - C % (2 * s);
      chain_product<DB>(c, c.A + R * rowstride, c.Minv + C * DB, C, base + s, c.T + R * rowstride + C * DB, 1.0, S0, S1);
    } else {
      const int R = tk.y, C = tk.z, s = tk.w;
      const int base = C - C % (2 * s);
      chain_product<DB>(c, c.Minv + R * rowstride, c.T + C * DB, base + s, R + 1, c.Minv + R * rowstride + C * DB, -1.0, S0,
                        S1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      // the barrier orders the CTA's stores before this thread's release store, which makes
      // them visible at GPU scope to an acquiring reader of the flag
      if (type == T_TRSM) st_release(&c.fac[tk.y * NB + tk.w], 1);
      else if (type == T_UPDATE) st_release(&c.ver[tk.y * NB + tk.z], tk.w + 1);
      else if (type == T_TMUL) st_release(&c.tfl[tk.y * NB + tk.z], 1);
      else st_release(&c.inv[tk.y * NB + tk.z], 1);
    }
  }
}

}  // namespace

void diag_task_list(int NB, std::vector<int4>& tasks) {
  tasks.clear();
  // POTRF(k), TRSM(k+1,k) and UPDATE(k+1,k+1,k) belong to the chain CTA and are not queued
  for (int k = 0; k < NB; ++k) {
    for (int i = k + 2; i < NB; ++i) tasks.push_back(make_int4(T_TRSM, i, k, k));
    for (int j = k + 1; j < NB; ++j)
      for (int i = j; i < NB; ++i)
        if (!(i == k + 1 && j == k + 1)) tasks.push_back(make_int4(T_UPDATE, i, j, k));
    // doubling steps whose pair ends with diagonal block k, smallest pairs first
    for (int s = 1; 2 * s <= NB; s *= 2) {
      const int base = k + 1 - 2 * s;
      if (base < 0 || base % (2 * s) != 0) continue;
      for (int a = 0; a < s; ++a)
        for (int b = 0; b < s; ++b) tasks.push_back(make_int4(T_TMUL, base + s + a, base + b, s));
      for (int a = 0; a < s; ++a)
        for (int b = 0; b < s; ++b) tasks.push_back(make_int4(T_MMUL, base + s + a, base + b, s));
    }
  }
}

cr_status diag_chol_launch(int db, double* A, double* Minv, double* T, int nb, int gcol0, int* status, int* flags,
                           const int4* d_tasks, int ntasks, int grid, cudaStream_t s) {
  const int NB = nb / db;
  Ctx c;
  c.A = A; c.Minv = Minv; c.T = T; c.nb = nb; c.NB = NB;
  c.ver = flags; c.fac = flags + NB * NB; c.inv = flags + 2 * NB * NB; c.tfl = flags + 3 * NB * NB;
  c.abort_flag = flags + 4 * NB * NB;
  int* counter = flags + 4 * NB * NB + 1;
  int* role = flags + 4 * NB * NB + 2;
  c.status = status; c.gcol0 = gcol0;
  CR_CUDA(cudaMemsetAsync(flags, 0, diag_flag_words(nb, db) * sizeof(int), s));
  static bool configured = false;
  if (!configured) {
    // same shared-memory carveout as the tensor-core kernel, so these small CTAs can share
    // SMs with it instead of waiting for SMs to be reconfigured
    CR_CUDA(cudaFuncSetAttribute(k_diag_chol<16>, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared));
    CR_CUDA(cudaFuncSetAttribute(k_diag_chol<32>, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared));
    configured = true;
  }
  if (db == 16) k_diag_chol<16><<<grid, 256, 0, s>>>(c, d_tasks, ntasks, counter, role);
  else if (db == 32) k_diag_chol<32><<<grid, 256, 0, s>>>(c, d_tasks, ntasks, counter, role);
  else return fail(CR_ERR_ARG, "diag_chol_launch: block size");
  CR_CHECK_LAUNCH("k_diag_chol");
  return CR_OK;
}

}  // namespace cr
