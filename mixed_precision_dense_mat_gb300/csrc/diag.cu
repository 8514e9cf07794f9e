// FP64 factorisation of one diagonal tile, L_jj = chol(A_jj), together with its inverse
// M = L_jj^-1, as an on-device dataflow executor.
//
// The nb x nb tile is cut into 16 x 16 blocks.  The blocked Cholesky DAG (the tile-DAG
// formulation of Section IV-A of "Mixed-Precision GPU Acceleration for Confidence Regions
// of Spatial Excursion Sets", here inside one tile and on one GPU) and the blocked forward
// substitution L M = I that gives the inverse are listed in a fixed order:
//   POTRF(k)       factor block (k,k), invert it                     needs ver(k,k) = k
//   TRSM(i,k)      L_ik = A_ik M_kk^T                                needs POTRF(k), ver(i,k) = k
//   UPDATE(i,j,k)  A_ij -= L_ik L_jk^T  (k < j <= i)                  needs TRSM(i,k), TRSM(j,k), ver(i,j) = k
//   IUPD(R,C,m)    W_RC += L_Rm M_mC    (C <= m < R)                  needs TRSM(R,m), M_mC, iver(R,C) = m - C
//   ISOLVE(R,C)    M_RC = -M_RR W_RC    (C < R)                       needs POTRF(R), iver(R,C) = R - C
// Every task is one 16 x 16 x 16 product.  The inverse tasks are listed shortly after their
// inputs can exist, so the substitution runs behind the factorisation and only a few
// products remain once the last diagonal block is factored.
//
// One CTA, the first to start, runs the critical chain POTRF(0), then per k TRSM(k+1,k),
// UPDATE(k+1,k+1,k) and POTRF(k+1) with its blocks in shared memory.  The other CTAs take
// the listed tasks from a global counter and wait (bounded, wall-clock limited) on per-block
// flags released by the producers.  The list is ordered so that a task only waits on
// earlier tasks, or on chain steps whose own inputs are earlier tasks; every waited-on task
// is therefore held by a running CTA, and the scheme needs no co-residency guarantee
// (checked on the host when the list is built).
//
// On GB300 an FP64 FMA has a dependent latency of about 64 cycles, each SM sub-partition
// issues one warp-wide FP64 instruction per ~64 cycles, and a double reciprocal square root
// or division costs over 400 cycles.  The kernels therefore keep FP64 instructions off
// control flow (exponent tests in integer arithmetic), spread FP64 work evenly over the four
// sub-partitions, and factor diagonal blocks without divisions (fraction-free elimination).
#include <math.h>

#include <algorithm>
#include <vector>

#include "common.cuh"
#include "df.cuh"
#include "diag.cuh"
#include "ptx.cuh"

namespace cr {

namespace {

// T_UPDATE2(i, j, k): UPDATE(i, j, k) and UPDATE(i, j+1, k) in one task (they share L_ik)
enum { T_TRSM = 1, T_UPDATE = 2, T_IUPD = 3, T_ISOLVE = 4, T_UPDATE2 = 5 };

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
  double* W;   // accumulators W_RC of the substitution (same block positions as M_RC)
  int nb, NB;
  int* ver;    // NB x NB: updates applied to block (i, j)
  int* fac;    // NB x NB: L block (i, j) final (for i == j also the inverse block M_ii)
  int* inv;    // NB x NB: inverse block (R, C), R > C, final
  int* iver;   // NB x NB: products accumulated into W_RC
  int* abort_flag;
  int* status;
  int gcol0;
  unsigned long long* amax;   // IEEE bits of max |M| over the inverse (non-negative doubles order as unsigned)
  int* clear_flags;           // the next call's flag set, cleared here
  int clear_words;
  unsigned long long* clear_amax;
  // Blocks the chain CTA produces, published without a release fence: pub_m[k] = M_kk and
  // pub_l[k] = L_{k+1,k} (16 x 16 row-major each), pre-filled with PUB_EMPTY; readers poll
  // the data itself until no element is PUB_EMPTY.  clear_pub: the next call's set.
  double* pub_m;
  double* pub_l;
  double* clear_pub;
  unsigned long long wait_ns;   // limit of every wait (wall clock)
};

// NaN bit pattern marking an unpublished element; a produced value with this pattern is
// stored as the quiet NaN 0x7ff8... instead, so that readers never wait on it.
constexpr unsigned long long PUB_EMPTY = 0xffffffffffffffffull;

__device__ __forceinline__ void st_pub(double* p, double x) {
  unsigned long long b = (unsigned long long)__double_as_longlong(x);
  if (b == PUB_EMPTY) b = 0x7ff8000000000000ull;
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(b) : "memory");
}
__device__ __forceinline__ unsigned long long ld_pub(const double* p) {
  unsigned long long b;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(b) : "l"(p) : "memory");
  return b;
}

// Folds the calling warp's |x| into the inverse's running maximum (one atomic per warp).
__device__ __forceinline__ void fold_amax(const Ctx& c, double x) {
  unsigned long long b = (unsigned long long)__double_as_longlong(x) & 0x7fffffffffffffffull;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, b, o);
    b = y > b ? y : b;
  }
  if ((threadIdx.x & 31) == 0) atomicMax(c.amax, b);
}

// Lane `lane` of the polling warp gets the flag (p, v) it waits on for task tk (p = nullptr:
// nothing); lanes 0-2 cover every task type.
template <class C>
__device__ __forceinline__ void task_flag(const C& c, int4 tk, int lane, const int*& p, int& v) {
  const int NB = c.NB;
  p = nullptr;
  v = 1;
  // the chain's blocks (M_kk, L_{k+1,k}) have no flag: they are read from the publication
  // buffers, which the operand loads poll
  if (tk.x == T_TRSM) {
    const int i = tk.y, k = tk.w;
    if (lane == 1) { p = &c.ver[i * NB + k]; v = k; }
  } else if (tk.x == T_UPDATE || tk.x == T_UPDATE2) {
    const int i = tk.y, j = tk.z, k = tk.w;
    if (lane == 0) p = &c.fac[i * NB + k];
    else if (lane == 1 && j != k + 1) p = &c.fac[j * NB + k];
    else if (lane == 2) { p = &c.ver[i * NB + j]; v = k; }
    else if (tk.x == T_UPDATE2 && lane == 3) p = &c.fac[(j + 1) * NB + k];
    else if (tk.x == T_UPDATE2 && lane == 4) { p = &c.ver[i * NB + j + 1]; v = k; }
  } else if (tk.x == T_IUPD) {
    const int R = tk.y, C = tk.z, m = tk.w;
    if (lane == 0 && R != m + 1) p = &c.fac[R * NB + m];
    else if (lane == 1 && m != C) p = &c.inv[m * NB + C];
    else if (lane == 2) { p = &c.iver[R * NB + C]; v = m - C; }
  } else {
    const int R = tk.y, C = tk.z;
    if (lane == 1) { p = &c.iver[R * NB + C]; v = R - C; }
  }
}

// All 32 lanes of a warp: waits until *p >= v for every lane with p != nullptr (the lanes
// poll side by side).  False when the kernel's abort flag is set, or after the context's wait
// limit (2 s unless the caller set another), which sets the abort flag and the timeout bit.
template <class C>
__device__ bool warp_wait_ge(const C& c, const int* p, int v) {
  bool done = p == nullptr || ld_acquire(p) >= v;
  if (__all_sync(0xffffffffu, done)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (!done) done = ld_acquire(p) >= v;
    if (__all_sync(0xffffffffu, done)) return true;
    int stop = 0;
    if ((threadIdx.x & 31) == 0) {
      stop = ld_acquire(c.abort_flag);
      if (!stop && global_timer_ns() - t0 > c.wait_ns) {
        atomicOr(&c.status[0], DEV_ERR_TIMEOUT);
        atomicExch(c.abort_flag, 1);
        stop = 1;
      }
    }
    if (__shfl_sync(0xffffffffu, stop, 0)) return false;
  }
}

constexpr int DB = 16;                        // block size: 256 threads, one element of a block each
constexpr int NT_LOWER = DB * (DB + 1) / 2;   // 136 lower-triangle elements
typedef double Blk[DB + 1];                   // padded shared-memory row

__device__ __forceinline__ void load_block(Blk* S, const double* src, int ld) {
  for (int idx = threadIdx.x; idx < DB * DB; idx += blockDim.x) {
    const int r = idx / DB, q = idx % DB;
    S[r][q] = __ldcg(src + (size_t)r * ld + q);
  }
}
// S[col][q] = src[q][col]
__device__ __forceinline__ void load_block_t(Blk* S, const double* src, int ld) {
  for (int idx = threadIdx.x; idx < DB * DB; idx += blockDim.x) {
    const int r = idx / DB, q = idx % DB;
    S[q][r] = __ldcg(src + (size_t)r * ld + q);
  }
}

// All 256 threads: S (or its transpose) receives the published block at pub once none of its
// elements is PUB_EMPTY.  False when the kernel's abort flag is set, or after the wait limit,
// which sets the abort flag and the timeout error bit.
__device__ bool load_pub(const Ctx& c, Blk* S, const double* pub, bool transpose) {
  const int r = threadIdx.x / DB, q = threadIdx.x % DB;
  uint64_t t0 = 0;
  for (int it = 0;; ++it) {
    const unsigned long long b = ld_pub(pub + threadIdx.x);
    if (!__syncthreads_or(b == PUB_EMPTY)) {
      const double x = __longlong_as_double((long long)b);
      if (transpose) S[q][r] = x;
      else S[r][q] = x;
      return true;
    }
    int stop = 0;
    if (threadIdx.x == 0) {
      if (it == 0) t0 = global_timer_ns();
      stop = ld_acquire(c.abort_flag);
      if (!stop && global_timer_ns() - t0 > c.wait_ns) {
        atomicOr(&c.status[0], DEV_ERR_TIMEOUT);
        atomicExch(c.abort_flag, 1);
        stop = 1;
      }
    }
    if (__syncthreads_or(stop)) return false;
  }
}

// x 2^e by integer exponent adjustment, exact for normal x and results; zero, subnormal
// and non-finite x are returned unchanged (the callers keep magnitudes in the normal range,
// and a non-finite pivot is reported as a failed factorisation).  Branch-free, with no FP64
// instruction.
__device__ __forceinline__ double scale2(double x, int e) {
  const int hi = __double2hiint(x), lo = __double2loint(x);
  const int ex = (hi >> 20) & 0x7ff;
  const double y = __hiloint2double(hi + (e << 20), lo);
  return (ex == 0 || ex == 0x7ff) ? x : y;
}
// unbiased binary exponent of a positive normal number, 0 for anything else (integer tests)
__device__ __forceinline__ int expo_pos(double x) {
  const int hi = __double2hiint(x);
  const int ex = (hi >> 20) & 0x7ff;
  return (hi > 0 && ex != 0 && ex != 0x7ff) ? ex - 1023 : 0;
}
// Row of element e of a row-by-row lower triangle (e = i (i + 1) / 2 + j, j <= i), in closed
// form: a data-dependent loop would diverge across the lanes of a warp.
__device__ __forceinline__ int tri_row(int e) {
  int i = (int)((sqrtf(8.0f * (float)e + 1.0f) - 1.0f) * 0.5f);
  if ((i + 1) * (i + 2) / 2 <= e) ++i;
  if (i * (i + 1) / 2 > e) --i;
  return i;
}
// x > 0 without an FP64 comparison (NaN and zero give false)
__device__ __forceinline__ bool positive(double x) {
  const int hi = __double2hiint(x), lo = __double2loint(x);
  const int ex = (hi >> 20) & 0x7ff;
  const bool nan = ex == 0x7ff && (((hi & 0xfffff) | lo) != 0);
  return hi >= 0 && ((hi | lo) != 0) && !nan;
}


// Fraction-free factorisation of one N x N diagonal block by N^2 threads: threads
// 0 .. N(N+1)/2-1 own the lower triangle of the working matrix (row by row), the others the
// strict lower triangle of the transformed identity.  N = 16 uses the whole CTA and
// __syncthreads; N = 8 would use warps 0-1 and named barrier 1 (measured on GB300: splitting
// a 16 x 16 block into 8 x 8 halves is slower than eliminating it whole).
template <int N>
struct FFS {
  double col[2][N];   // column c of the working matrix, double-buffered by step parity
  double row[2][N];   // row c of the transformed identity (unit-diagonal form)
  double piv[N];      // t_cc
  double alpha[N];    // alpha_c
  double r[N];        // 1 / sqrt(alpha_c t_cc)
};

template <int N>
__device__ __forceinline__ void ffbar() {
  if (N == DB) __syncthreads();
  else asm volatile("bar.sync 1, 64;" ::: "memory");
}

// Division-free (fraction-free) elimination of the SPD block src (lower part, row stride
// DB + 1): the Schur complement is carried as T = alpha_c S, and step c performs
//   T <- 2^-k_c (t_cc T - t_c t_c^T)      with 2^-k_c t_cc in [1, 2),
// so alpha_{c+1} = alpha_c t_cc 2^-k_c.  The same row operations applied to the identity,
// carried with unit diagonal (Z = U^-1, A = U D U^T with U unit lower), give
//   L_ic = t_ic r_c   and   L^-1 = diag(r) Z diag(alpha),   r_c = 1 / sqrt(alpha_c t_cc).
// Every element's step is the same predicated multiply, FMA and exponent adjustment (no
// divergent paths, no division or square root); the power of two comes from the pivot's
// owner.  The alpha_c are a prefix product of the normalised pivots, taken by a shuffle scan
// after the last step, followed by the N reciprocal square roots.  Lout receives L (lower
// part), Xout L^-1 (upper part zero).  gcol: global column of the block's first column, for
// the failure report.
// Which element each of the 256 threads carries through the elimination of a 16 x 16 block:
// code = isT << 8 | i << 4 | j.  Working-matrix element (i, j), i >= j, is updated at steps
// col < j; transformed-identity element (i, j), i > j, at steps j <= col < i.  Threads are
// ordered by the last step that updates their element (then the first), so the elements
// still live at a step sit in few warps, spread over the four sub-partitions, and the other
// warps skip the step's FP64 instructions.
struct ElemMap {
  unsigned short code[DB * DB];
};
constexpr ElemMap make_elem_map() {
  ElemMap m{};
  int key[DB * DB] = {};
  int n = 0;
  for (int i = 0; i < DB; ++i)
    for (int j = 0; j <= i; ++j) {   // working matrix: steps 0 .. j-1
      m.code[n] = (unsigned short)(1 << 8 | i << 4 | j);
      key[n++] = (j - 1) * 64 + 0;
    }
  for (int i = 1; i < DB; ++i)
    for (int j = 0; j < i; ++j) {    // transformed identity: steps j .. i-1
      m.code[n] = (unsigned short)(i << 4 | j);
      key[n++] = (i - 1) * 64 + j;
    }
  for (int a = 1; a < n; ++a)        // stable insertion sort by key
    for (int b = a; b > 0 && key[b - 1] > key[b]; --b) {
      const int tk = key[b]; key[b] = key[b - 1]; key[b - 1] = tk;
      const unsigned short tc = m.code[b]; m.code[b] = m.code[b - 1]; m.code[b - 1] = tc;
    }
  return m;
}
__constant__ ElemMap c_elem_map = make_elem_map();

template <int N>
__device__ void ffN(const Ctx& c, int gcol, const double* src, double* Lout, double* Xout, FFS<N>& f) {
  const int t = threadIdx.x;   // 0 .. N*N-1
  const int code = c_elem_map.code[t];
  const bool isT = (code >> 8) != 0;
  const int i = (code >> 4) & 15, j = code & 15;
  double v = isT ? src[i * (DB + 1) + j] : 0.0;
  for (int col = 0; col < N; ++col) {
    const int par = col & 1;
    // the owners of column col publish it (the pivot owner also into piv); nothing else
    // stands between the last step's result and the barrier
    if (isT && j == col) {
      f.col[par][i] = v;
      if (i == col) f.piv[col] = v;
    }
    if (!isT && i == col) f.row[par][j] = v;
    ffbar<N>();
    const double d = f.col[par][col];
    const double a = f.col[par][i];
    const double b = isT ? f.col[par][j] : (j == col ? 1.0 : f.row[par][j]);
    const bool act = isT ? (j > col) : (i > col && j <= col);
    const int e = -expo_pos(d);   // integer work that overlaps the FP64 latency below
    if (__any_sync(0xffffffffu, act)) {   // warp-uniform: idle warps issue no FP64 work
      const double nv = scale2(fma(-a, b, d * v), e);
      v = act ? nv : v;                     // a select: divergent branches cost ~100 cycles a step
    }
  }
  ffbar<N>();
  if (t < 32) {
    // alpha_t = prod_{c < t} 2^-k_c t_cc, inclusive shuffle scan over lanes 0 .. N-1
    double x = 1.0;
    // every pivot is checked (lane t: the block's column t, reported 1-based)
    if (t < N && !positive(f.piv[t])) atomicMin(&c.status[1], gcol + t + 1);
    if (t >= 1 && t < N) {
      const double p = f.piv[t - 1];
      x = scale2(p, -expo_pos(p));
    }
#pragma unroll
    for (int o = 1; o < N; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, x, o);
      if (t >= o) x *= y;
    }
    if (t < N) {
      f.alpha[t] = x;
      f.r[t] = rsqrt(x * f.piv[t]);
    }
  }
  ffbar<N>();
  if (isT) {
    Lout[i * (DB + 1) + j] = v * f.r[j];
    if (i != j) Xout[j * (DB + 1) + i] = 0.0;
    else Xout[i * (DB + 1) + i] = f.r[i] * f.alpha[i];
  } else {
    Xout[i * (DB + 1) + j] = f.r[i] * v * f.alpha[j];
  }
  ffbar<N>();
}

struct FFShared {
  union {
    double part[2][NT_LOWER];   // halves of the fused symmetric update (before the factorisation)
    Blk l16[DB];                // the factor of the diagonal block
  };
  FFS<DB> f;
};

// Lower element t (row by row, t < 136) of diagonal block k, 0 for the other threads.
__device__ __forceinline__ double diag_elem(const Ctx& c, int k) {
  const int t = threadIdx.x;
  if (t >= NT_LOWER) return 0.0;
  const int i = tri_row(t);
  const int j = t - i * (i + 1) / 2;
  return __ldcg(c.A + (size_t)(k * DB + i) * c.nb + k * DB + j);
}

// Cholesky factor and inverse of diagonal block k, after subtracting P P^T when P is given
// (the last symmetric update of the block, fused).  v: the block's element from diag_elem,
// read by the caller ahead of time.  A16 is shared-memory scratch; the factor (lower part)
// is written to the tile, the inverse (upper part zero) to Minv and to X.
__device__ void potrf16(const Ctx& c, int k, double v, const Blk* P, Blk* A16, Blk* X, FFShared& sh) {
  const int t = threadIdx.x;
  double* a = c.A + (size_t)(k * DB) * c.nb + k * DB;
  if (P) {
    // lower element e = ii (ii + 1) / 2 + jj of P P^T, inner dimension in halves: thread t
    // sums half (t & 1) of element t >> 1 (elements 0..127); lanes 0..15 of warp 0 also sum
    // the halves of elements 128..135
    auto half_sum = [&](int item) {
      const int e = item >> 1, q0 = (item & 1) * (DB / 2);
      const int ii = tri_row(e);
      const int jj = e - ii * (ii + 1) / 2;
      double s0 = 0.0, s1 = 0.0;
#pragma unroll
      for (int q = 0; q < DB / 2; q += 2) {
        s0 = fma(P[ii][q0 + q], P[jj][q0 + q], s0);
        s1 = fma(P[ii][q0 + q + 1], P[jj][q0 + q + 1], s1);
      }
      sh.part[item & 1][e] = s0 + s1;
    };
    half_sum(t);
    if (t < 2 * (NT_LOWER - 128)) half_sum(256 + t);
    __syncthreads();
  }
  if (t < NT_LOWER) {
    const int i = tri_row(t);
    const int j = t - i * (i + 1) / 2;
    if (P) v -= sh.part[0][t] + sh.part[1][t];
    A16[i][j] = v;
  }
  __syncthreads();
  ffN<DB>(c, c.gcol0 + k * DB, &A16[0][0], &sh.l16[0][0], &X[0][0], sh.f);
  double* m = c.Minv + (size_t)(k * DB) * c.nb + k * DB;
  {
    const int i = t / DB, j = t % DB;
    m[(size_t)i * c.nb + j] = X[i][j];
    st_pub(c.pub_m + k * DB * DB + t, X[i][j]);
    a[(size_t)i * c.nb + j] = j <= i ? sh.l16[i][j] : 0.0;
    fold_amax(c, X[i][j]);
  }
}

// Output element (r, cc) of the triangular product P M^T (M lower) owned by this thread.
// Warp w takes the column pair p(w) = w (w < 4) or 11 - w (w >= 4), so the two warps of
// each sub-partition hold pairs whose inner lengths add up to the same total.
__device__ __forceinline__ void trsm_owner(int& r, int& cc) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = w < 4 ? w : 11 - w;
  r = lane & 15;
  cc = 2 * pair + (lane >> 4);
}
// sum over q <= cc of P[r][q] M[cc][q]; the extra term at q = cc + 1 (cc even) multiplies
// a zero of M's upper part
__device__ __forceinline__ double trsm_elem(const Blk* P, const Blk* M, int r, int cc) {
  double s0 = 0.0, s1 = 0.0;
  for (int q = 0; q <= (cc | 1); q += 2) {
    s0 = fma(P[r][q], M[cc][q], s0);
    s1 = fma(P[r][q + 1], M[cc][q + 1], s1);
  }
  return s0 + s1;
}

// sum_q P[r][q] Q[col][q] for (r, col) = (tid / 16, tid % 16), two accumulation chains to
// halve the FP64 latency of the sum
__device__ __forceinline__ double gemm_elem(const Blk* P, const Blk* Q) {
  const int r = threadIdx.x / DB, col = threadIdx.x % DB;
  double s0 = 0.0, s1 = 0.0;
#pragma unroll
  for (int q = 0; q < DB; q += 2) {
    s0 = fma(P[r][q], Q[col][q], s0);
    s1 = fma(P[r][q + 1], Q[col][q + 1], s1);
  }
  return s0 + s1;
}

// The critical chain, run by one CTA with the blocks kept in shared memory:
// POTRF(0); then for k = 0 .. NB-2: TRSM(k+1,k), then UPDATE(k+1,k+1,k) fused into POTRF(k+1).
__device__ void run_chain(const Ctx& c, Blk* S0, Blk* S1, Blk* S2, Blk* S3, FFShared& sh, int* s_ok) {
  const int NB = c.NB;
  const size_t rowstride = (size_t)DB * c.nb;
  potrf16(c, 0, diag_elem(c, 0), nullptr, S0, S1, sh);   // S1 = M_00, published
  __syncthreads();
  int r, cc;
  trsm_owner(r, cc);
  for (int k = 0; k + 1 < NB; ++k) {
    const int i = k + 1;
    // the inputs of TRSM(i, k) and of the fused UPDATE(i, i, k) are waited for and read
    // together: the updates of step k - 1 that complete them are adjacent in the list
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      const bool ok = warp_wait_ge(c, lane < 2 ? &c.ver[i * NB + (lane ? i : k)] : nullptr, k);
      if (lane == 0) *s_ok = ok ? 1 : 0;
    }
    __syncthreads();
    if (!*s_ok) return;
    double* aik = c.A + i * rowstride + k * DB;
    const double vii = diag_elem(c, i);
    load_block(S2, aik, c.nb);
    __syncthreads();
    // TRSM(i, k): L_ik = A_ik M_kk^T, M_kk in S1
    const double l = trsm_elem(S2, S1, r, cc);
    S3[r][cc] = l;                     // S3 = L_ik
    aik[(size_t)r * c.nb + cc] = l;
    st_pub(c.pub_l + k * DB * DB + r * DB + cc, l);
    __syncthreads();
    // UPDATE(i, i, k) fused into POTRF(i)
    potrf16(c, i, vii, S3, S0, S1, sh);   // S1 = M_ii, published
    __syncthreads();
  }
}

__global__ void __launch_bounds__(256) k_diag_chol(Ctx c, const int4* __restrict__ tasks, int ntasks, int* counter, int* role) {
  __shared__ Blk S0[DB];
  __shared__ Blk S1[DB];
  __shared__ Blk S2[DB];
  __shared__ Blk S3[DB];
  __shared__ FFShared sh;
  __shared__ int s_task;
  __shared__ int s_ok;
  __shared__ int4 s_tk;
  const int NB = c.NB;
  const size_t rowstride = (size_t)DB * c.nb;
  // the first CTA to start takes the critical chain: it is resident, so the chain progresses
  if (threadIdx.x == 0) s_task = atomicAdd(role, 1);
  __syncthreads();
  if (s_task == 0) {
    run_chain(c, S0, S1, S2, S3, sh, &s_ok);
    return;
  }
  {
    // Housekeeping the queue CTAs do while the chain factors the first block: clear the next
    // call's flags and abs-max, and zero the strictly upper 16 x 16 blocks of the factor
    // tile and of the inverse (no task reads them).
    const int q = s_task - 1, nq = gridDim.x - 1;
    for (int w = q * 256 + threadIdx.x; w < c.clear_words; w += nq * 256) c.clear_flags[w] = 0;
    if (q == 0 && threadIdx.x == 0) *c.clear_amax = 0ull;
    for (int w = q * 256 + threadIdx.x; w < 2 * NB * DB * DB; w += nq * 256)
      c.clear_pub[w] = __longlong_as_double((long long)PUB_EMPTY);
    const int r = threadIdx.x / DB, col = threadIdx.x % DB;
    for (int blk = q; blk < NB * NB; blk += nq) {
      const int bi = blk / NB, bj = blk % NB;
      if (bj <= bi) continue;
      const size_t o = (size_t)(bi * DB + r) * c.nb + bj * DB + col;
      c.A[o] = 0.0;
      c.Minv[o] = 0.0;
    }
  }
  // Warp 1 runs the queue: lane 0 claims task indices one ahead (the claim's round trip
  // overlaps the current task) and lanes 0-2 poll the current task's flags side by side
  // while warp 0 releases the previous task's flag.  A claimed task waits only behind the
  // task its CTA is running, which is earlier in the list, so the progress argument above
  // still holds.
  const int lane = threadIdx.x & 31;
  int claim = 0;
  if (threadIdx.x == 32) claim = atomicAdd(counter, 1);
  while (true) {
    if (threadIdx.x >= 32 && threadIdx.x < 64) {
      int t = 0;
      if (lane == 0) {
        t = claim;
        if (t < ntasks) claim = atomicAdd(counter, 1);
      }
      t = __shfl_sync(0xffffffffu, t, 0);
      bool ok = true;
      if (t < ntasks) {
        const int4 tk = tasks[t];
        const int* fp = nullptr;
        int fv = 0;
        task_flag(c, tk, lane, fp, fv);
        ok = warp_wait_ge(c, fp, fv);
        if (lane == 0) s_tk = tk;
      }
      if (lane == 0) {
        s_task = t;
        s_ok = ok ? 1 : 0;
      }
    }
    __syncthreads();
    const int t = s_task;
    if (t >= ntasks || !s_ok) break;
    const int4 tk = s_tk;
    const int type = tk.x;
    if (type == T_TRSM) {
      const int i = tk.y, k = tk.w;
      double* a = c.A + i * rowstride + k * DB;
      load_block(S0, a, c.nb);
      if (!load_pub(c, S1, c.pub_m + k * DB * DB, false)) break;
      __syncthreads();
      int r, cc;
      trsm_owner(r, cc);
      a[(size_t)r * c.nb + cc] = trsm_elem(S0, S1, r, cc);
    } else {
      const int r = threadIdx.x / DB, col = threadIdx.x % DB;
      if (type == T_UPDATE) {
        const int i = tk.y, j = tk.z, k = tk.w;
        double* o = c.A + i * rowstride + j * DB + (size_t)r * c.nb + col;
        const bool live = !(i == j && col > r);
        // the destination is read with the operands: only this task writes it until its flag
        const double d = live ? __ldcg(o) : 0.0;
        load_block(S0, c.A + i * rowstride + k * DB, c.nb);
        if (j == k + 1) {
          if (!load_pub(c, S1, c.pub_l + k * DB * DB, false)) break;
        } else {
          load_block(S1, c.A + j * rowstride + k * DB, c.nb);
        }
        __syncthreads();
        const double p = gemm_elem(S0, S1);
        if (live) *o = d - p;
      } else if (type == T_UPDATE2) {
        // A_ij -= L_ik L_jk^T and A_i,j+1 -= L_ik L_j+1,k^T (block j + 1 <= i is the diagonal one
        // at most, lower part only)
        const int i = tk.y, j = tk.z, k = tk.w;
        double* o = c.A + i * rowstride + j * DB + (size_t)r * c.nb + col;
        const bool live2 = !(i == j + 1 && col > r);
        const double d1 = __ldcg(o);
        const double d2 = live2 ? __ldcg(o + DB) : 0.0;
        load_block(S0, c.A + i * rowstride + k * DB, c.nb);
        if (j == k + 1) {
          if (!load_pub(c, S1, c.pub_l + k * DB * DB, false)) break;
        } else {
          load_block(S1, c.A + j * rowstride + k * DB, c.nb);
        }
        load_block(S2, c.A + (j + 1) * rowstride + k * DB, c.nb);
        __syncthreads();
        double a0 = 0.0, a1 = 0.0, b0 = 0.0, b1 = 0.0;
#pragma unroll
        for (int q = 0; q < DB; q += 2) {
          const double x0 = S0[r][q], x1 = S0[r][q + 1];
          a0 = fma(x0, S1[col][q], a0);
          a1 = fma(x1, S1[col][q + 1], a1);
          b0 = fma(x0, S2[col][q], b0);
          b1 = fma(x1, S2[col][q + 1], b1);
        }
        *o = d1 - (a0 + a1);
        if (live2) o[DB] = d2 - (b0 + b1);
      } else if (type == T_IUPD) {
        // W_RC (+)= L_Rm M_mC
        const int R = tk.y, C = tk.z, m = tk.w;
        double* o = c.W + R * rowstride + C * DB + (size_t)r * c.nb + col;
        const double d = (m == C) ? 0.0 : __ldcg(o);
        if (R == m + 1) {
          if (!load_pub(c, S0, c.pub_l + m * DB * DB, false)) break;
        } else {
          load_block(S0, c.A + R * rowstride + m * DB, c.nb);
        }
        if (m == C) {
          if (!load_pub(c, S1, c.pub_m + C * DB * DB, true)) break;
        } else {
          load_block_t(S1, c.Minv + m * rowstride + C * DB, c.nb);
        }
        __syncthreads();
        const double p = gemm_elem(S0, S1);
        *o = (m == C) ? p : d + p;
      } else {
        // M_RC = -M_RR W_RC
        const int R = tk.y, C = tk.z;
        if (!load_pub(c, S0, c.pub_m + R * DB * DB, false)) break;
        load_block_t(S1, c.W + R * rowstride + C * DB, c.nb);
        __syncthreads();
        const double mv = -gemm_elem(S0, S1);
        c.Minv[R * rowstride + C * DB + (size_t)r * c.nb + col] = mv;
        fold_amax(c, mv);
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      // the barrier orders the CTA's stores before this thread's release store, which makes
      // them visible at GPU scope to an acquiring reader of the flag
      if (type == T_TRSM) st_release(&c.fac[tk.y * NB + tk.w], 1);
      else if (type == T_UPDATE) st_release(&c.ver[tk.y * NB + tk.z], tk.w + 1);
      else if (type == T_UPDATE2) {
        st_release(&c.ver[tk.y * NB + tk.z], tk.w + 1);
        st_release(&c.ver[tk.y * NB + tk.z + 1], tk.w + 1);
      }
      else if (type == T_IUPD) st_release(&c.iver[tk.y * NB + tk.z], tk.w - tk.z + 1);
      else st_release(&c.inv[tk.y * NB + tk.z], 1);
    }
  }
}


// =======================================================================================
// Double-float executor: the same dataflow (task list, flags, publication buffers, chain
// CTA), with every block held as a double-float pair hi + lo of FP32 numbers (about 48
// significant bits; the error-free two-product and two-sum of df.cuh).  It emulates the
// FP64 diagonal tile on the FP32 units, which on GB300 issue 64 times as many lanes per
// cycle as the FP64 units and have a dependent latency of a few cycles instead of ~64.
// The updated tile is read in FP64 where a block is first touched (the tasks of step 0 and
// the chain's first two blocks); factor, Schur complements, inverse and the substitution's
// accumulators live in double-float buffers, which k_split_diag_df turns into the FP64
// factor and inverse and into the FP16 high/low parts the tensor cores read.

struct CtxD {
  const double* A;        // the updated diagonal tile, FP64 row-major (ld nb); read only
  float2* L;              // running Schur complements, then the factor's blocks (ld nb)
  float2* Minv;           // the inverse's blocks (ld nb)
  float2* W;              // accumulators W_RC of the substitution (ld nb)
  int nb, NB;
  int* ver;
  int* fac;
  int* inv;
  int* iver;
  int* abort_flag;
  int* status;
  int gcol0;
  unsigned long long* amax;   // FP32 bits of max |M| over the high parts (non-negative floats order as unsigned)
  int* clear_flags;
  int clear_words;
  unsigned long long* clear_amax;
  unsigned long long* pub_m;  // publication buffers as in Ctx, one 64-bit word (hi, lo) per element
  unsigned long long* pub_l;
  unsigned long long* clear_pub;
  unsigned long long wait_ns;
};

typedef df BlkD[DB + 1];   // padded shared-memory row (17 pairs: conflict-free column reads)

__device__ __forceinline__ df to_df(float2 v) { return {v.x, v.y}; }
__device__ __forceinline__ float2 to_f2(df v) { return make_float2(v.hi, v.lo); }
// An FP64 value as a double-float pair: hi = its nearest FP32 number, lo = the FP32 rounding
// of the remainder (FP64 conversions; only where an original block is first read).
__device__ __forceinline__ df df_of(double x) {
  const float h = __double2float_rn(x);
  return {h, __double2float_rn(x - (double)h)};
}
// unbiased exponent of a positive normal FP32 number, 0 for anything else (integer tests)
__device__ __forceinline__ int expo_f(float x) {
  const int b = __float_as_int(x);
  const int ex = (b >> 23) & 0xff;
  return (b > 0 && ex != 0 && ex != 0xff) ? ex - 127 : 0;
}
// 2^e as an FP32 number, -126 <= e <= 127
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

// Dot-product accumulator: the high parts of the products are summed with two-sum (a 4-cycle
// dependent chain through s), every lower-order term (the products' errors, cross terms and
// the two-sum errors) in the plain FP32 compensation c.  For K terms the result is accurate
// to about K 2^-48 of the largest partial sum.
struct DAcc {
  float s, c;
};
__device__ __forceinline__ void mac(DAcc& a, df x, df y) {
  const float p = __fmul_rn(x.hi, y.hi);
  float e = __fmaf_rn(x.hi, y.hi, -p);
  e = __fmaf_rn(x.hi, y.lo, e);
  e = __fmaf_rn(x.lo, y.hi, e);
  const float s = __fadd_rn(a.s, p);
  const float bb = __fsub_rn(s, a.s);
  const float t = __fadd_rn(__fsub_rn(a.s, __fsub_rn(s, bb)), __fsub_rn(p, bb));
  a.s = s;
  a.c = __fadd_rn(a.c, __fadd_rn(t, e));
}
__device__ __forceinline__ df acc_df(DAcc a) { return df_two_sum(a.s, a.c); }
// x - y and x + y, closed by a full two-sum: a Schur complement cancels, and the faster
// closing step of df_add assumes the sum's high part dominates
__device__ __forceinline__ df df_sub(df x, df y) {
  const df s = df_two_sum(x.hi, -y.hi);
  return df_two_sum(s.hi, __fadd_rn(s.lo, __fsub_rn(x.lo, y.lo)));
}
__device__ __forceinline__ df df_sum(df x, df y) {
  const df s = df_two_sum(x.hi, y.hi);
  return df_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo)));
}

// 1/sqrt(x) of a positive double-float: an FP32 estimate and one FP32 Newton step (about 24
// bits), then one double-float Newton step whose residual 1 - x r^2 is formed from exact
// products (about 47 bits).
__device__ __forceinline__ df df_rsqrt(df x) {
  float r = rsqrtf(x.hi);
  r = __fmaf_rn(0.5f * r, __fmaf_rn(-__fmul_rn(x.hi, r), r, 1.0f), r);
  const df y = df_mul_f(x, r);
  const df z = df_mul_f(y, r);
  const float h = __fsub_rn(__fsub_rn(1.0f, z.hi), z.lo);
  return df_quick_two_sum(r, __fmul_rn(__fmul_rn(0.5f, r), h));
}

// One fraction-free elimination step 2^e (d v - a b) in double-float: the high products split
// exactly, their difference by two-sum, the cross terms by FMA; sc = 2^e (exact scaling).
__device__ __forceinline__ df ff_step(df d, df v, df a, df b, float sc) {
  const float ph = __fmul_rn(d.hi, v.hi);
  const float pe = __fmaf_rn(d.hi, v.hi, -ph);
  const float qh = __fmul_rn(a.hi, b.hi);
  const float qe = __fmaf_rn(a.hi, b.hi, -qh);
  const df s = df_two_sum(ph, -qh);
  float lo = __fsub_rn(pe, qe);
  lo = __fmaf_rn(d.hi, v.lo, lo);
  lo = __fmaf_rn(d.lo, v.hi, lo);
  lo = __fmaf_rn(-a.hi, b.lo, lo);
  lo = __fmaf_rn(-a.lo, b.hi, lo);
  const df r = df_two_sum(s.hi, __fadd_rn(s.lo, lo));
  return {__fmul_rn(r.hi, sc), __fmul_rn(r.lo, sc)};
}

__device__ __forceinline__ unsigned long long df_bits(df x) {
  return (unsigned long long)__float_as_uint(x.hi) | ((unsigned long long)__float_as_uint(x.lo) << 32);
}
__device__ __forceinline__ void st_pub_d(unsigned long long* p, df x) {
  unsigned long long b = df_bits(x);
  if (b == PUB_EMPTY) b = 0x7fc000007fc00000ull;   // both halves the quiet NaN
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(b) : "memory");
}
__device__ __forceinline__ unsigned long long ld_pub_u(const unsigned long long* p) {
  unsigned long long b;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(b) : "l"(p) : "memory");
  return b;
}

__device__ __forceinline__ void fold_amax_d(const CtxD& c, df x) {
  const unsigned b = __reduce_max_sync(0xffffffffu, __float_as_uint(x.hi) & 0x7fffffffu);
  if ((threadIdx.x & 31) == 0) atomicMax(c.amax, (unsigned long long)b);
}

// an original block (FP64) into shared memory as double-float pairs
__device__ __forceinline__ void load_b64(BlkD* S, const double* src, int ld) {
  for (int idx = threadIdx.x; idx < DB * DB; idx += blockDim.x) {
    const int r = idx / DB, q = idx % DB;
    S[r][q] = df_of(__ldcg(src + (size_t)r * ld + q));
  }
}
__device__ __forceinline__ void load_bdf(BlkD* S, const float2* src, int ld) {
  for (int idx = threadIdx.x; idx < DB * DB; idx += blockDim.x) {
    const int r = idx / DB, q = idx % DB;
    S[r][q] = to_df(__ldcg(src + (size_t)r * ld + q));
  }
}
// S[col][q] = src[q][col]
__device__ __forceinline__ void load_bdf_t(BlkD* S, const float2* src, int ld) {
  for (int idx = threadIdx.x; idx < DB * DB; idx += blockDim.x) {
    const int r = idx / DB, q = idx % DB;
    S[q][r] = to_df(__ldcg(src + (size_t)r * ld + q));
  }
}

// All 256 threads: S (or its transpose) receives the published block once none of its words
// is PUB_EMPTY; false on abort or after the wait limit (which sets abort and timeout).
__device__ bool load_pub_d(const CtxD& c, BlkD* S, const unsigned long long* pub, bool transpose) {
  const int r = threadIdx.x / DB, q = threadIdx.x % DB;
  uint64_t t0 = 0;
  for (int it = 0;; ++it) {
    const unsigned long long b = ld_pub_u(pub + threadIdx.x);
    if (!__syncthreads_or(b == PUB_EMPTY)) {
      const df x = {__uint_as_float((unsigned)b), __uint_as_float((unsigned)(b >> 32))};
      if (transpose) S[q][r] = x;
      else S[r][q] = x;
      return true;
    }
    int stop = 0;
    if (threadIdx.x == 0) {
      if (it == 0) t0 = global_timer_ns();
      stop = ld_acquire(c.abort_flag);
      if (!stop && global_timer_ns() - t0 > c.wait_ns) {
        atomicOr(&c.status[0], DEV_ERR_TIMEOUT);
        atomicExch(c.abort_flag, 1);
        stop = 1;
      }
    }
    if (__syncthreads_or(stop)) return false;
  }
}

struct FFSD {
  df cr[2][2][DB];   // [step parity][0: column c of the working matrix, 1: row c of the transformed identity]
  df piv[DB];        // t_cc
  float sc[DB];      // 2^-k_c with 2^-k_c t_cc in [1, 2), published by the pivot's owner
  df alpha[DB];
  df r[DB];
};

// The fraction-free factorisation of ffN (same element map, same steps, same closing scan of
// the normalised pivots) in double-float arithmetic, arranged for few instructions per step:
// each element is published at one step (working (i, j) into the column buffer at step j,
// identity (i, j) into the row buffer at step i), the pivot's owner also publishes the step's
// power of two and the identity's unit diagonal entry, so that every active element reads its
// operands from fixed slots, and each element's active steps are a bit mask.  src: the block
// (lower part), Lout receives L (lower part), Xout L^-1 (upper part zero).
__device__ void ffD(const CtxD& c, int gcol, const BlkD* src, BlkD* Lout, BlkD* Xout, FFSD& f) {
  const int t = threadIdx.x;
  const int code = c_elem_map.code[t];
  const bool isT = (code >> 8) != 0;
  const int i = (code >> 4) & 15, j = code & 15;
  // active steps: working (i, j) at col < j; identity (i, j) at j <= col < i
  const unsigned act = isT ? ((1u << j) - 1u) : (((1u << i) - 1u) & ~((1u << j) - 1u));
  const int pub_step = isT ? j : i;
  const int kind = isT ? 0 : 1, pub_idx = isT ? i : j;
  const bool piv_owner = isT && i == j;
  df v = isT ? src[i][j] : df{0.0f, 0.0f};
  for (int col = 0; col < DB; ++col) {
    const int par = col & 1;
    if (pub_step == col) {
      f.cr[par][kind][pub_idx] = v;
      if (piv_owner) {
        f.piv[col] = v;
        f.sc[col] = pow2f(max(-expo_f(v.hi), -126));
        f.cr[par][1][col] = df{1.0f, 0.0f};
      }
    }
    __syncthreads();
    const bool on = (act >> col) & 1u;
    if (__any_sync(0xffffffffu, on)) {   // warp-uniform: idle warps issue no work
      const df d = f.cr[par][0][col];
      const df a = f.cr[par][0][i];
      const df b = f.cr[par][kind][j];
      const df nv = ff_step(d, v, a, b, f.sc[col]);
      if (on) v = nv;
    }
  }
  __syncthreads();
  if (t < 32) {
    df x = {1.0f, 0.0f};
    // every pivot is checked (lane t: the block's column t, reported 1-based)
    if (t < DB && !(f.piv[t].hi > 0.0f)) atomicMin(&c.status[1], gcol + t + 1);
    if (t >= 1 && t < DB) {
      const df p = f.piv[t - 1];
      const float s = f.sc[t - 1];
      x = {__fmul_rn(p.hi, s), __fmul_rn(p.lo, s)};
    }
#pragma unroll
    for (int o = 1; o < DB; o <<= 1) {
      const df y = {__shfl_up_sync(0xffffffffu, x.hi, o), __shfl_up_sync(0xffffffffu, x.lo, o)};
      if (t >= o) x = df_mul(x, y);
    }
    if (t < DB) {
      f.alpha[t] = x;
      f.r[t] = df_rsqrt(df_mul(x, f.piv[t]));
    }
  }
  __syncthreads();
  if (isT) {
    Lout[i][j] = df_mul(v, f.r[j]);
    if (i != j) Xout[j][i] = df{0.0f, 0.0f};
    else Xout[i][i] = df_mul(f.r[i], f.alpha[i]);
  } else {
    Xout[i][j] = df_mul(df_mul(f.r[i], v), f.alpha[j]);
  }
  __syncthreads();
}

struct FFSharedD {
  BlkD l16[DB];   // the factor of the diagonal block
  FFSD f;
};

// Lower element t of diagonal block k, 0 for the other threads: from the FP64 tile for the
// two blocks nothing has updated yet (k <= 1), else from the double-float buffer.
__device__ __forceinline__ df diag_elem_d(const CtxD& c, int k) {
  const int t = threadIdx.x;
  if (t >= NT_LOWER) return {0.0f, 0.0f};
  const int i = tri_row(t);
  const int j = t - i * (i + 1) / 2;
  const size_t o = (size_t)(k * DB + i) * c.nb + k * DB + j;
  return k <= 1 ? df_of(__ldcg(c.A + o)) : to_df(__ldcg(c.L + o));
}

// potrf16 in double-float: factor and inverse of diagonal block k after subtracting P P^T.
__device__ void potrf16_d(const CtxD& c, int k, df v, const BlkD* P, BlkD* A16, BlkD* X, FFSharedD& sh) {
  const int t = threadIdx.x;
  if (t < NT_LOWER) {
    // lower element t: its whole update, in two interleaved accumulators
    const int i = tri_row(t);
    const int j = t - i * (i + 1) / 2;
    if (P) {
      DAcc a{0.0f, 0.0f}, b{0.0f, 0.0f};
#pragma unroll
      for (int q = 0; q < DB; q += 2) {
        mac(a, P[i][q], P[j][q]);
        mac(b, P[i][q + 1], P[j][q + 1]);
      }
      v = df_sub(v, df_sum(acc_df(a), acc_df(b)));
    }
    A16[i][j] = v;
  }
  __syncthreads();
  ffD(c, c.gcol0 + k * DB, A16, sh.l16, X, sh.f);
  {
    const int i = t / DB, j = t % DB;
    const size_t o = (size_t)(k * DB + i) * c.nb + k * DB + j;
    c.Minv[o] = to_f2(X[i][j]);
    st_pub_d(c.pub_m + k * DB * DB + t, X[i][j]);
    c.L[o] = j <= i ? to_f2(sh.l16[i][j]) : make_float2(0.0f, 0.0f);
    fold_amax_d(c, X[i][j]);
  }
}

// sum over q <= cc of P[r][q] M[cc][q] (M lower)
__device__ __forceinline__ df trsm_elem_d(const BlkD* P, const BlkD* M, int r, int cc) {
  DAcc a{0.0f, 0.0f};
  for (int q = 0; q <= cc; ++q) mac(a, P[r][q], M[cc][q]);
  return acc_df(a);
}
// sum_q P[r][q] Q[col][q] for (r, col) = (tid / 16, tid % 16)
__device__ __forceinline__ df gemm_elem_d(const BlkD* P, const BlkD* Q) {
  const int r = threadIdx.x / DB, col = threadIdx.x % DB;
  DAcc a{0.0f, 0.0f};
#pragma unroll
  for (int q = 0; q < DB; ++q) mac(a, P[r][q], Q[col][q]);
  return acc_df(a);
}

// The critical chain of run_chain in double-float.
__device__ void run_chain_d(const CtxD& c, BlkD* S0, BlkD* S1, BlkD* S2, BlkD* S3, FFSharedD& sh, int* s_ok) {
  const int NB = c.NB;
  potrf16_d(c, 0, diag_elem_d(c, 0), nullptr, S0, S1, sh);   // S1 = M_00, published
  __syncthreads();
  int r, cc;
  trsm_owner(r, cc);
  for (int k = 0; k + 1 < NB; ++k) {
    const int i = k + 1;
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      const bool ok = warp_wait_ge(c, lane < 2 ? &c.ver[i * NB + (lane ? i : k)] : nullptr, k);
      if (lane == 0) *s_ok = ok ? 1 : 0;
    }
    __syncthreads();
    if (!*s_ok) return;
    const size_t oik = (size_t)(i * DB) * c.nb + k * DB;
    const df vii = diag_elem_d(c, i);
    if (k == 0) load_b64(S2, c.A + oik, c.nb);
    else load_bdf(S2, c.L + oik, c.nb);
    __syncthreads();
    const df l = trsm_elem_d(S2, S1, r, cc);   // L_ik = A_ik M_kk^T
    S3[r][cc] = l;
    c.L[oik + (size_t)r * c.nb + cc] = to_f2(l);
    st_pub_d(c.pub_l + k * DB * DB + r * DB + cc, l);
    __syncthreads();
    potrf16_d(c, i, vii, S3, S0, S1, sh);       // UPDATE(i,i,k) fused; S1 = M_ii, published
    __syncthreads();
  }
}

__global__ void __launch_bounds__(256) k_diag_chol_df(CtxD c, const int4* __restrict__ tasks, int ntasks, int* counter,
                                                      int* role) {
  __shared__ BlkD S0[DB];
  __shared__ BlkD S1[DB];
  __shared__ BlkD S2[DB];
  __shared__ BlkD S3[DB];
  __shared__ FFSharedD sh;
  __shared__ int s_task;
  __shared__ int s_ok;
  __shared__ int4 s_tk;
  const int NB = c.NB;
  const size_t rowstride = (size_t)DB * c.nb;
  if (threadIdx.x == 0) s_task = atomicAdd(role, 1);
  __syncthreads();
  if (s_task == 0) {
    run_chain_d(c, S0, S1, S2, S3, sh, &s_ok);
    return;
  }
  {
    // the next call's flags, abs-max and publication buffers (no zeroing of upper blocks:
    // nothing reads them, and the FP64 outputs are written by the split kernel)
    const int q = s_task - 1, nq = gridDim.x - 1;
    for (int w = q * 256 + threadIdx.x; w < c.clear_words; w += nq * 256) c.clear_flags[w] = 0;
    if (q == 0 && threadIdx.x == 0) *c.clear_amax = 0ull;
    for (int w = q * 256 + threadIdx.x; w < 2 * NB * DB * DB; w += nq * 256) c.clear_pub[w] = PUB_EMPTY;
  }
  const int lane = threadIdx.x & 31;
  int claim = 0;
  if (threadIdx.x == 32) claim = atomicAdd(counter, 1);
  while (true) {
    if (threadIdx.x >= 32 && threadIdx.x < 64) {
      int t = 0;
      if (lane == 0) {
        t = claim;
        if (t < ntasks) claim = atomicAdd(counter, 1);
      }
      t = __shfl_sync(0xffffffffu, t, 0);
      bool ok = true;
      if (t < ntasks) {
        const int4 tk = tasks[t];
        const int* fp = nullptr;
        int fv = 0;
        task_flag(c, tk, lane, fp, fv);
        ok = warp_wait_ge(c, fp, fv);
        if (lane == 0) s_tk = tk;
      }
      if (lane == 0) {
        s_task = t;
        s_ok = ok ? 1 : 0;
      }
    }
    __syncthreads();
    const int t = s_task;
    if (t >= ntasks || !s_ok) break;
    const int4 tk = s_tk;
    const int type = tk.x;
    if (type == T_TRSM) {
      const int i = tk.y, k = tk.w;
      const size_t o = i * rowstride + k * DB;
      if (k == 0) load_b64(S0, c.A + o, c.nb);
      else load_bdf(S0, c.L + o, c.nb);
      if (!load_pub_d(c, S1, c.pub_m + k * DB * DB, false)) break;
      __syncthreads();
      int r, cc;
      trsm_owner(r, cc);
      c.L[o + (size_t)r * c.nb + cc] = to_f2(trsm_elem_d(S0, S1, r, cc));
    } else {
      const int r = threadIdx.x / DB, col = threadIdx.x % DB;
      if (type == T_UPDATE) {
        const int i = tk.y, j = tk.z, k = tk.w;
        const size_t o = i * rowstride + j * DB + (size_t)r * c.nb + col;
        const bool live = !(i == j && col > r);
        // the destination is read with the operands: only this task writes it until its flag
        df d = {0.0f, 0.0f};
        if (live) d = k == 0 ? df_of(__ldcg(c.A + o)) : to_df(__ldcg(c.L + o));
        load_bdf(S0, c.L + i * rowstride + k * DB, c.nb);
        if (j == k + 1) {
          if (!load_pub_d(c, S1, c.pub_l + k * DB * DB, false)) break;
        } else {
          load_bdf(S1, c.L + j * rowstride + k * DB, c.nb);
        }
        __syncthreads();
        const df p = gemm_elem_d(S0, S1);
        if (live) c.L[o] = to_f2(df_sub(d, p));
      } else if (type == T_UPDATE2) {
        const int i = tk.y, j = tk.z, k = tk.w;
        const size_t o = i * rowstride + j * DB + (size_t)r * c.nb + col;
        const bool live2 = !(i == j + 1 && col > r);
        df d1, d2 = {0.0f, 0.0f};
        if (k == 0) {
          d1 = df_of(__ldcg(c.A + o));
          if (live2) d2 = df_of(__ldcg(c.A + o + DB));
        } else {
          d1 = to_df(__ldcg(c.L + o));
          if (live2) d2 = to_df(__ldcg(c.L + o + DB));
        }
        load_bdf(S0, c.L + i * rowstride + k * DB, c.nb);
        if (j == k + 1) {
          if (!load_pub_d(c, S1, c.pub_l + k * DB * DB, false)) break;
        } else {
          load_bdf(S1, c.L + j * rowstride + k * DB, c.nb);
        }
        load_bdf(S2, c.L + (j + 1) * rowstride + k * DB, c.nb);
        __syncthreads();
        DAcc a{0.0f, 0.0f}, b{0.0f, 0.0f};
#pragma unroll
        for (int q = 0; q < DB; ++q) {
          const df x = S0[r][q];
          mac(a, x, S1[col][q]);
          mac(b, x, S2[col][q]);
        }
        c.L[o] = to_f2(df_sub(d1, acc_df(a)));
        if (live2) c.L[o + DB] = to_f2(df_sub(d2, acc_df(b)));
      } else if (type == T_IUPD) {
        // W_RC (+)= L_Rm M_mC
        const int R = tk.y, C = tk.z, m = tk.w;
        const size_t o = R * rowstride + C * DB + (size_t)r * c.nb + col;
        const df d = (m == C) ? df{0.0f, 0.0f} : to_df(__ldcg(c.W + o));
        if (R == m + 1) {
          if (!load_pub_d(c, S0, c.pub_l + m * DB * DB, false)) break;
        } else {
          load_bdf(S0, c.L + R * rowstride + m * DB, c.nb);
        }
        if (m == C) {
          if (!load_pub_d(c, S1, c.pub_m + C * DB * DB, true)) break;
        } else {
          load_bdf_t(S1, c.Minv + m * rowstride + C * DB, c.nb);
        }
        __syncthreads();
        const df p = gemm_elem_d(S0, S1);
        c.W[o] = to_f2((m == C) ? p : df_sum(d, p));
      } else {
        // M_RC = -M_RR W_RC
        const int R = tk.y, C = tk.z;
        if (!load_pub_d(c, S0, c.pub_m + R * DB * DB, false)) break;
        load_bdf_t(S1, c.W + R * rowstride + C * DB, c.nb);
        __syncthreads();
        const df mv = df_neg(gemm_elem_d(S0, S1));
        c.Minv[R * rowstride + C * DB + (size_t)r * c.nb + col] = to_f2(mv);
        fold_amax_d(c, mv);
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      if (type == T_TRSM) st_release(&c.fac[tk.y * NB + tk.w], 1);
      else if (type == T_UPDATE) st_release(&c.ver[tk.y * NB + tk.z], tk.w + 1);
      else if (type == T_UPDATE2) {
        st_release(&c.ver[tk.y * NB + tk.z], tk.w + 1);
        st_release(&c.ver[tk.y * NB + tk.z + 1], tk.w + 1);
      }
      else if (type == T_IUPD) st_release(&c.iver[tk.y * NB + tk.z], tk.w - tk.z + 1);
      else st_release(&c.inv[tk.y * NB + tk.z], 1);
    }
  }
}

// The double-float factor and inverse of one tile into FP64 (lower parts; zero above) and
// into the FP16 high/low parts of M 2^eM and of L, as k_split_diag does from FP64: eM with
// max|M| 2^eM < 2^14 (status[2] = eM) from the executor's maximum (FP32 bits of the high
// parts).  Elements [0, nb^2) are M, [nb^2, 2 nb^2) are L, two adjacent ones per thread.
// The FP16 parts of an element x = hi + lo (scaled) are h = fp16(hi) and fp16((hi - h) + lo).
__global__ void __launch_bounds__(256) k_split_diag_df(const float2* __restrict__ Mdf, const float2* __restrict__ Ldf,
                                                       int nb, const unsigned long long* __restrict__ amax,
                                                       double* __restrict__ M64, double* __restrict__ L64,
                                                       __half* __restrict__ mh, __half* __restrict__ ml,
                                                       __half* __restrict__ lh, __half* __restrict__ ll, int* status) {
  const unsigned bits = (unsigned)*amax;
  const int ef = (int)((bits >> 23) & 0xff);   // max |M| in [2^(ef-127), 2^(ef-126))
  const int e = (bits == 0 || ef == 0 || ef == 0xff) ? 0 : 14 - (ef - 126);
  if (blockIdx.x == 0 && threadIdx.x == 0) status[2] = e;
  const float sc = ldexpf(1.0f, e);
  const size_t half_count = (size_t)nb * nb / 2;
  for (size_t pidx = blockIdx.x * 256 + threadIdx.x; pidx < 2 * half_count; pidx += (size_t)gridDim.x * 256) {
    const bool isM = pidx < half_count;
    const size_t q = isM ? pidx : pidx - half_count;
    const int r = (int)(2 * q / nb), c0 = (int)(2 * q % nb);
    const float4 v = reinterpret_cast<const float4*>(isM ? Mdf : Ldf)[q];
    const bool z0 = c0 > r, z1 = c0 + 1 > r;
    const double d0 = z0 ? 0.0 : (double)v.x + (double)v.y;
    const double d1 = z1 ? 0.0 : (double)v.z + (double)v.w;
    reinterpret_cast<double2*>(isM ? M64 : L64)[q] = make_double2(d0, d1);
    __half* h = isM ? mh : lh;
    __half* l = isM ? ml : ll;
    if (h) {
      const float s = isM ? sc : 1.0f;
      const float x0 = z0 ? 0.0f : v.x * s, x1 = z1 ? 0.0f : v.z * s;
      const float y0 = z0 ? 0.0f : v.y * s, y1 = z1 ? 0.0f : v.w * s;
      const __half2 hv = __floats2half2_rn(x0, x1);
      const float2 hf = __half22float2(hv);
      reinterpret_cast<__half2*>(h)[q] = hv;
      reinterpret_cast<__half2*>(l)[q] = __floats2half2_rn((x0 - hf.x) + y0, (x1 - hf.y) + y1);
    }
  }
}

}  // namespace

bool diag_task_list(int NB, std::vector<int4>& tasks) {
  // Step k lists what POTRF(k) and the k-th block column of the factor enable; POTRF(k),
  // TRSM(k+1,k) and UPDATE(k+1,k+1,k) belong to the chain CTA and are not listed.
  // The inverse tasks of step k are listed after the factorisation tasks of step k + 2, so
  // that they fill idle CTAs instead of delaying the updates the chain waits for.  (Measured
  // on GB300: ordering the list by an estimate of each task's latest start, so that rows
  // near the diagonal of later steps overtake far rows of earlier steps, is slower: the
  // overtaking tasks park CTAs until the chain reaches them.)
  tasks.clear();
  const int lag = 2;
  auto inverse_step = [&](int k) {
    for (int C = 0; C < k; ++C) tasks.push_back(make_int4(T_ISOLVE, k, C, 0));
    for (int C = 0; C <= k; ++C)
      for (int R = k + 1; R < NB; ++R) tasks.push_back(make_int4(T_IUPD, R, C, k));
  };
  for (int k = 0; k < NB; ++k) {
    // all solves of the step first (they run side by side), then the updates row by row,
    // nearest the diagonal first, in pairs of adjacent blocks: UPDATE(k+2,k+1,k) and
    // UPDATE(k+2,k+2,k) (one task) feed the chain's next step
    for (int i = k + 2; i < NB; ++i) tasks.push_back(make_int4(T_TRSM, i, k, k));
    for (int i = k + 2; i < NB; ++i)
      for (int j = k + 1; j <= i; j += 2) tasks.push_back(make_int4(j + 1 <= i ? T_UPDATE2 : T_UPDATE, i, j, k));
    if (k >= lag) inverse_step(k - lag);
  }
  for (int k = std::max(0, NB - lag); k < NB; ++k) inverse_step(k);
  // Progress check.  Chain node times: POTRF(k) = 3k, TRSM(k+1,k) = 3k+1,
  // UPDATE(k+1,k+1,k) = 3k+2.  A listed task waits on earlier listed tasks and on chain
  // nodes; chain nodes wait on listed tasks.  Every wait ends if each chain node a task
  // waits on needs, through the chain up to it, only tasks listed before that task.
  const int Q = (int)tasks.size();
  std::vector<int> pos_trsm(NB * NB, -1), pos_isolve(NB * NB, -1);
  std::vector<int> pos_upd((size_t)NB * NB * NB, -1), pos_iupd((size_t)NB * NB * NB, -1);
  for (int t = 0; t < Q; ++t) {
    const int4 tk = tasks[t];
    if (tk.x == T_TRSM) pos_trsm[tk.y * NB + tk.w] = t;
    else if (tk.x == T_UPDATE) pos_upd[((size_t)tk.y * NB + tk.z) * NB + tk.w] = t;
    else if (tk.x == T_UPDATE2) {
      pos_upd[((size_t)tk.y * NB + tk.z) * NB + tk.w] = t;
      pos_upd[((size_t)tk.y * NB + tk.z + 1) * NB + tk.w] = t;
    }
    else if (tk.x == T_IUPD) pos_iupd[((size_t)tk.y * NB + tk.z) * NB + tk.w] = t;
    else pos_isolve[tk.y * NB + tk.z] = t;
  }
  auto upd = [&](int i, int j, int k) { return pos_upd[((size_t)i * NB + j) * NB + k]; };
  auto iupd = [&](int R, int C, int m) { return pos_iupd[((size_t)R * NB + C) * NB + m]; };
  auto before = [](int p, int t) { return p >= 0 && p < t; };
  const int nchain = 3 * NB;
  std::vector<int> need(nchain, -1);   // last listed position the chain needs up to time tau
  for (int tau = 0; tau < nchain; ++tau) {
    int p = tau > 0 ? need[tau - 1] : -1;
    const int k = tau / 3, kind = tau % 3;
    if (kind != 0 && k >= 1 && k + 1 < NB) {
      const int q = kind == 1 ? upd(k + 1, k, k - 1) : upd(k + 1, k + 1, k - 1);
      if (q < 0) return false;
      p = std::max(p, q);
    }
    need[tau] = p;
  }
  auto chain_ok = [&](int tau, int t) { return tau < nchain && need[tau] < t; };
  auto fac_ok = [&](int i, int k, int t) {
    if (i == k) return chain_ok(3 * k, t);
    if (i == k + 1) return chain_ok(3 * k + 1, t);
    return before(pos_trsm[i * NB + k], t);
  };
  for (int t = 0; t < Q; ++t) {
    const int4 tk = tasks[t];
    bool ok;
    if (tk.x == T_TRSM) {
      const int i = tk.y, k = tk.w;
      ok = chain_ok(3 * k, t) && (k == 0 || before(upd(i, k, k - 1), t));
    } else if (tk.x == T_UPDATE || tk.x == T_UPDATE2) {
      const int i = tk.y, j = tk.z, k = tk.w;
      ok = fac_ok(i, k, t) && fac_ok(j, k, t) && (k == 0 || before(upd(i, j, k - 1), t));
      if (tk.x == T_UPDATE2)
        ok = ok && fac_ok(j + 1, k, t) && (k == 0 || before(upd(i, j + 1, k - 1), t));
    } else if (tk.x == T_IUPD) {
      const int R = tk.y, C = tk.z, m = tk.w;
      ok = fac_ok(R, m, t) && (m == C ? chain_ok(3 * C, t) : before(pos_isolve[m * NB + C], t)) &&
           (m == C || before(iupd(R, C, m - 1), t));
    } else {
      const int R = tk.y, C = tk.z;
      ok = chain_ok(3 * R, t) && before(iupd(R, C, R - 1), t);
    }
    if (!ok) return false;
  }
  return true;
}

cr_status diag_chol_launch(int db, double* A, double* Minv, double* W, int nb, int gcol0, int* status, int* flags,
                           int par, double* pub, const int4* d_tasks, int ntasks, int grid, unsigned long long* amax,
                           unsigned long long wait_ns, cudaStream_t s) {
  if (db != DB || nb % DB != 0 || grid < 2) return fail(CR_ERR_ARG, "diag_chol_launch: block size 16 dividing nb and at least 2 CTAs");
  const int NB = nb / db;
  const int words = diag_flag_words(nb, db);
  int* cur = flags + (size_t)(par & 1) * words;
  Ctx c;
  c.A = A; c.Minv = Minv; c.W = W; c.nb = nb; c.NB = NB;
  c.clear_flags = flags + (size_t)((par & 1) ^ 1) * words;
  c.clear_words = words;
  c.clear_amax = amax + ((par & 1) ^ 1);
  c.pub_m = pub + (size_t)(par & 1) * diag_pub_doubles(nb, db) / 2;
  c.pub_l = c.pub_m + (size_t)NB * DB * DB;
  c.clear_pub = pub + (size_t)((par & 1) ^ 1) * diag_pub_doubles(nb, db) / 2;
  amax += par & 1;
  flags = cur;
  c.ver = flags; c.fac = flags + NB * NB; c.inv = flags + 2 * NB * NB; c.iver = flags + 3 * NB * NB;
  c.abort_flag = flags + 4 * NB * NB;
  int* counter = flags + 4 * NB * NB + 1;
  int* role = flags + 4 * NB * NB + 2;
  c.status = status; c.gcol0 = gcol0; c.amax = amax;
  c.wait_ns = wait_ns;
  static bool configured = false;
  if (!configured) {
    // same shared-memory carveout as the tensor-core kernel, so these small CTAs can share
    // SMs with it instead of waiting for SMs to be reconfigured
    CR_CUDA(cudaFuncSetAttribute(k_diag_chol, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared));
    configured = true;
  }
  {
    TimedScope ts("k_diag_chol", s);
    k_diag_chol<<<grid, 256, 0, s>>>(c, d_tasks, ntasks, counter, role);
  }
  CR_CHECK_LAUNCH("k_diag_chol");
  return CR_OK;
}

cr_status diag_chol_df_launch(int db, const double* A, float2* Ldf, float2* Mdf, float2* Wdf, int nb, int gcol0,
                              int* status, int* flags, int par, double* pub, const int4* d_tasks, int ntasks, int grid,
                              unsigned long long* amax, unsigned long long wait_ns, cudaStream_t s) {
  if (db != DB || nb % DB != 0 || grid < 2) return fail(CR_ERR_ARG, "diag_chol_df_launch: block size 16 dividing nb and at least 2 CTAs");
  const int NB = nb / db;
  const int words = diag_flag_words(nb, db);
  CtxD c;
  c.A = A; c.L = Ldf; c.Minv = Mdf; c.W = Wdf; c.nb = nb; c.NB = NB;
  int* cur = flags + (size_t)(par & 1) * words;
  c.clear_flags = flags + (size_t)((par & 1) ^ 1) * words;
  c.clear_words = words;
  c.clear_amax = amax + ((par & 1) ^ 1);
  unsigned long long* pub64 = reinterpret_cast<unsigned long long*>(pub);
  c.pub_m = pub64 + (size_t)(par & 1) * diag_pub_doubles(nb, db) / 2;
  c.pub_l = c.pub_m + (size_t)NB * DB * DB;
  c.clear_pub = pub64 + (size_t)((par & 1) ^ 1) * diag_pub_doubles(nb, db) / 2;
  c.amax = amax + (par & 1);
  c.ver = cur; c.fac = cur + NB * NB; c.inv = cur + 2 * NB * NB; c.iver = cur + 3 * NB * NB;
  c.abort_flag = cur + 4 * NB * NB;
  int* counter = cur + 4 * NB * NB + 1;
  int* role = cur + 4 * NB * NB + 2;
  c.status = status; c.gcol0 = gcol0;
  c.wait_ns = wait_ns;
  static bool configured = false;
  if (!configured) {
    CR_CUDA(cudaFuncSetAttribute(k_diag_chol_df, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared));
    configured = true;
  }
  {
    TimedScope ts("k_diag_chol_df", s);
    k_diag_chol_df<<<grid, 256, 0, s>>>(c, d_tasks, ntasks, counter, role);
  }
  CR_CHECK_LAUNCH("k_diag_chol_df");
  return CR_OK;
}

cr_status split_diag_df_launch(const float2* Mdf, const float2* Ldf, int nb, const unsigned long long* amax, double* M64,
                               double* L64, __half* mh, __half* ml, __half* lh, __half* ll, int* status, cudaStream_t s) {
  const unsigned grid = (unsigned)(((size_t)nb * nb + 255) / 256);   // 2 nb^2 / 2 pairs, 256 per CTA
  {
    TimedScope ts("k_split_diag_df", s);
    k_split_diag_df<<<grid, 256, 0, s>>>(Mdf, Ldf, nb, amax, M64, L64, mh, ml, lh, ll, status);
  }
  CR_CHECK_LAUNCH("k_split_diag_df");
  return CR_OK;
}

}  // namespace cr
