// FP64-class matrix product on the FP16 tensor cores by the Ozaki scheme (Ozaki, Ogita, Oishi
// and Rump, "Error-free transformations of matrix multiplication by using fast routines of
// matrix multiplication and its applications", Numerical Algorithms 59 (2012)), for two steps of
// "Mixed-Precision GPU Acceleration for Confidence Regions of Spatial Excursion Sets": the
// conditioning correction (Section V-B Eq.7: S = M_p + W^T (y_o 1^T - M_o)) and the triangular
// solves of the kriging weights with many right-hand sides (Section V-A, Alg.2 steps 2-4).
//
// C = A^T B with A (k x m) and B (k x n) column-major FP64, S slices per operand column:
//  - each column c of A gets a power of two 2^Ea_c above its largest |entry| (B likewise), and
//    |A_rc| 2^(6 S - Ea_c), truncated to an integer below 2^(6 S), is cut into S slices of 6
//    bits: A_rc = sum_s a_s,rc 2^(Ea_c - 6 s) + d with |a_s,rc| <= 63 and |d| < 2^(Ea_c - 6 S);
//  - the slice products with s + t = L share the scale 2^(Ea_i + Eb_j - 6 L), so for each
//    level L = 2 .. S + 1 the L - 1 products are one product over the concatenated rows
//    [A_1; ...; A_(L-1)]^T [B_(L-1); ...; B_1] (the slices of A stored in order, those of B in
//    reverse, so that both ranges are contiguous);
//  - that product over a chunk of at most 4096 rows is a sum of at most 4096 integers of
//    magnitude <= 63^2, below 2^24, so an FP16 tensor-core GEMM with FP32 accumulation computes
//    it exactly (whatever its summation order);
//  - the products with s + t <= S + 1 are kept (36 of 64 for S = 8): the rest, and the
//    truncations, are below k 8.95 2^-48 2^(Ea_i + Eb_j) per output for S = 8 (derived in the
//    tests);
//  - each level's chunk sums, added in 32-bit integers (exact), are scaled by 2^-6L (exact)
//    and added to a double-float accumulator held in units of 2^(Ea_i + Eb_j), the least
//    significant level first; the last addition writes Cout = Cin + alpha 2^(Ea_i + Eb_j) C in
//    FP64 (so the product's range is FP64's);
//  - a column holding an infinity or a NaN makes every output it touches NaN.
// The slice GEMMs are plain FP16 x FP16 -> FP32 library GEMMs (cuBLAS, strided-batched over the
// K chunks); slicing, exact accumulation and the final sum are this file's kernels.
#include <cublas_v2.h>
#include <math.h>

#include <algorithm>
#include <mutex>

#include "calib.cuh"
#include "common.cuh"
#include "df.cuh"

namespace cr {

namespace {

// slice width; slice counts supported (S slices keep 6 S bits below each column's power of
// two: 48 for the correction, 54 for the kriging solves); chunk rows with 4096 * 63^2 < 2^24;
// chunks per GEMM call at most
constexpr int OZ_BITS = 6, OZ_MIN_SLICES = 2, OZ_MAX_SLICES = 10, OZ_KC_MAX = 4096, OZ_GROUP = 32;
constexpr unsigned long long OZ_MASK = (1ull << OZ_BITS) - 1ull;
constexpr int OZ_CORR_SLICES = 8;   // the conditioning correction's slices (48 bits)

// Exponent marking a column with an infinite or NaN entry: its slices are zero and every output
// it touches is NaN (as in an FP64 product, where the entry reaches all of them).
constexpr int OZ_NONFINITE = 0x7fffffff;

// E_c with max_r |X_rc| < 2^E_c (positive doubles order as their bit patterns); 0 for a zero
// column (its slices are all zero); OZ_NONFINITE for a column holding an infinity or a NaN.
// One CTA per column.
__global__ void __launch_bounds__(256) k_oz_colexp(const double* __restrict__ X, int ld, int rows, int* __restrict__ E) {
  const int c = blockIdx.x;
  unsigned long long m = 0ull;
  for (int r = threadIdx.x; r < rows; r += 256) {
    const unsigned long long b = (unsigned long long)__double_as_longlong(X[(size_t)c * ld + r]) & 0x7fffffffffffffffull;
    m = b > m ? b : m;
  }
  __shared__ unsigned long long red[8];
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long y = __shfl_down_sync(0xffffffffu, m, o);
    m = y > m ? y : m;
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w) m = red[w] > m ? red[w] : m;
    const int eb = (int)(m >> 52);   // biased exponent of the largest |entry|
    // a normal value lies in [2^(eb-1023), 2^(eb-1022)); a subnormal one below 2^-1022
    E[c] = m == 0ull ? 0 : (eb == 0x7ff ? OZ_NONFINITE : (eb == 0 ? -1022 : eb - 1022));
  }
}

// Slices of X (rows x cols, column-major, ld), OZ_SLICES of them: column c of out holds, at
// out + c * S * rows_pad + slot * rows_pad, slice s + 1 (s = 0 the most significant) in slot s,
// or in slot S - 1 - s when `reversed`, as rows_pad FP16 integers in [-63, 63], rows beyond
// `rows` zero.  Integer arithmetic on the FP64 bit pattern only.
template <int OZ_SLICES>
__global__ void __launch_bounds__(256) k_oz_slice(const double* __restrict__ X, int ld, int rows, int rows_pad, int cols,
                                                  const int* __restrict__ E, int reversed, __half* __restrict__ out) {
  for (int c = blockIdx.y; c < cols; c += gridDim.y) {
    const int Ec = E[c];
    __half* oc = out + (size_t)c * OZ_SLICES * rows_pad;
    for (int r = blockIdx.x * 256 + threadIdx.x; r < rows_pad; r += gridDim.x * 256) {
      unsigned long long q = 0ull;
      bool neg = false;
      if (r < rows && Ec != OZ_NONFINITE) {
        const unsigned long long b = (unsigned long long)__double_as_longlong(X[(size_t)c * ld + r]);
        neg = (b >> 63) != 0;
        const int eb = (int)((b >> 52) & 0x7ff);
        const unsigned long long mant = (b & 0x000fffffffffffffull) | (eb ? 0x0010000000000000ull : 0ull);
        // |x| = mant 2^(e2);  q = floor(|x| 2^(6 S - E_c)) < 2^(6 S) <= 2^60
        const int e2 = (eb ? eb : 1) - 1075;
        const int shift = e2 + OZ_BITS * OZ_SLICES - Ec;
        if (shift >= 0) q = shift < 64 ? mant << shift : 0ull;
        else q = -shift < 64 ? mant >> (-shift) : 0ull;
      }
#pragma unroll
      for (int s = 0; s < OZ_SLICES; ++s) {
        const int a = (int)((q >> (OZ_BITS * (OZ_SLICES - 1 - s))) & OZ_MASK);
        const int slot = reversed ? OZ_SLICES - 1 - s : s;
        oc[(size_t)slot * rows_pad + r] = __int2half_rn(neg ? -a : a);
      }
    }
  }
}

// R = y_o 1^T - M_o (k x n column-major, ld k), the right-hand factor of the correction.
__global__ void __launch_bounds__(256) k_oz_resid(const double* __restrict__ yo, const double* __restrict__ Y, int ldy,
                                                  int n_p, int n_o, int M, double* __restrict__ R) {
  const size_t total = (size_t)n_o * M;
  for (size_t e = blockIdx.x * (size_t)256 + threadIdx.x; e < total; e += (size_t)gridDim.x * 256) {
    const int r = (int)(e % n_o), j = (int)(e / n_o);
    R[e] = yo[r] - Y[(size_t)j * ldy + n_p + r];
  }
}

// One level's contribution for `nb` chunk products P_b (m x n FP32 exact integers below 2^24):
// v = sum_b P_b(i, j), exact in 32-bit integers (nb <= 32), split exactly into two floats,
// scaled by 2^-shift (shift = 6 L <= 66: an exact normal FP32 factor) and added to the
// double-float C (C = the term when `first`).  C holds the product in units of
// 2^(Ea_i + Eb_j), so its range is FP64's, not FP32's.  With `last`, Cout = Cin +
// alpha 2^(Ea_i + Eb_j) C in FP64 is written instead of C (Cin = NULL: zero; hi + lo of a
// double-float value is exact in FP64, the power of two exact unless the result is subnormal);
// Cout may be Cin (each entry is read, then written, by one thread).
__global__ void __launch_bounds__(256) k_oz_accum(const float* __restrict__ P, int nb, int m, int n,
                                                  const int* __restrict__ Ea, const int* __restrict__ Eb, int shift,
                                                  float2* __restrict__ C, int first, int last, double alpha,
                                                  const double* Cin, int ldci, double* Cout, int ldco) {
  const size_t mn = (size_t)m * n;
  const float lev_scale = __int_as_float((127 - shift) << 23);   // 2^-shift
  for (int j = blockIdx.y; j < n; j += gridDim.y) {
    const int eb = Eb[j];
    for (int i = blockIdx.x * 256 + threadIdx.x; i < m; i += gridDim.x * 256) {
      const size_t e = (size_t)j * m + i;
      const float* p = P + e;
      int v = 0;
#pragma unroll 8
      for (int b = 0; b < nb; ++b) v += __float2int_rn(p[(size_t)b * mn]);
      const float h = (float)v;                   // nearest FP32 of v (|v| < 2^29)
      const float l = (float)(v - (int)h);        // the rest, below 2^5: exact
      const int ea = Ea[i];
      const bool nonfinite = ea == OZ_NONFINITE || eb == OZ_NONFINITE;
      df acc = {h * lev_scale, l * lev_scale};
      if (nonfinite) acc = {__int_as_float(0x7fc00000), 0.0f};   // NaN
      if (!first) {
        const float2 c = C[e];
        acc = df_add({c.x, c.y}, acc);
      }
      if (last) {
        const double base = Cin ? Cin[(size_t)j * ldci + i] : 0.0;
        const double prod = nonfinite ? (double)acc.hi : ldexp((double)acc.hi + (double)acc.lo, ea + eb);
        Cout[(size_t)j * ldco + i] = base + alpha * prod;
      } else {
        C[e] = make_float2(acc.hi, acc.lo);
      }
    }
  }
}

// Cout = Cin (or 0) when the inner dimension is empty.
__global__ void __launch_bounds__(256) k_oz_copy(const double* Cin, int ldci, int m, int n, double* Cout, int ldco) {
  for (int j = blockIdx.y; j < n; j += gridDim.y)
    for (int i = blockIdx.x * 256 + threadIdx.x; i < m; i += gridDim.x * 256)
      Cout[(size_t)j * ldco + i] = Cin ? Cin[(size_t)j * ldci + i] : 0.0;
}

std::mutex g_cublas_mu;
cublasHandle_t g_cublas[64] = {};

cr_status cublas_for(cudaStream_t stream, cublasHandle_t* h) {
  int dev = 0;
  CR_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(CR_ERR_ARG, "Ozaki product: device index too large");
  if (!g_cublas[dev]) {
    if (cublasCreate(&g_cublas[dev]) != CUBLAS_STATUS_SUCCESS) return fail(CR_ERR_CUDA, "cublasCreate failed");
  }
  if (cublasSetStream(g_cublas[dev], stream) != CUBLAS_STATUS_SUCCESS) return fail(CR_ERR_CUDA, "cublasSetStream failed");
  *h = g_cublas[dev];
  return CR_OK;
}

// 2-D grid for the column-wise kernels: blocks of 256 rows times columns, about 16 CTAs per SM
dim3 grid2d(int rows, int cols) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int gx = std::max(1, (rows + 255) / 256);
  const long long want_y = std::max(1LL, (long long)sms * 16 / gx);
  const int gy = (int)std::min<long long>({(long long)std::max(cols, 1), want_y * 4, 65535LL});
  return dim3((unsigned)gx, (unsigned)gy);
}

unsigned grid_for(size_t total) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t want = (total + 255) / 256, cap = (size_t)sms * 16;
  return (unsigned)std::max<size_t>(1, std::min(want, cap));
}

}  // namespace

namespace {

// Geometry of one Ozaki product's inner dimension: c = ceil(K / 4096) chunks of kc rows
// (K / c rounded up to 128, so at most 4096) per slice, K' = c kc padded rows, S slices.
struct OzGeom {
  int K, S, cpk, kc, kpad;
  size_t ldk;   // S K': the halves of one column's slices
};

OzGeom oz_geom(int K, int S) {
  OzGeom g;
  g.K = K;
  g.S = S;
  g.cpk = (K + OZ_KC_MAX - 1) / OZ_KC_MAX;
  g.kc = ((K + g.cpk - 1) / g.cpk + 127) / 128 * 128;
  g.kpad = g.cpk * g.kc;
  g.ldk = (size_t)S * g.kpad;
  return g;
}

void oz_slice_launch(const OzGeom& g, const double* X, int ld, int cols, const int* E, int rev, __half* out,
                     cudaStream_t stream) {
  const dim3 grid = grid2d(g.kpad, cols);
  const int K = g.K, kpad = g.kpad;
  switch (g.S) {
    case 2: k_oz_slice<2><<<grid, 256, 0, stream>>>(X, ld, K, kpad, cols, E, rev, out); break;
    case 3: k_oz_slice<3><<<grid, 256, 0, stream>>>(X, ld, K, kpad, cols, E, rev, out); break;
    case 4: k_oz_slice<4><<<grid, 256, 0, stream>>>(X, ld, K, kpad, cols, E, rev, out); break;
    case 5: k_oz_slice<5><<<grid, 256, 0, stream>>>(X, ld, K, kpad, cols, E, rev, out); break;
    case 6: k_oz_slice<6><<<grid, 256, 0, stream>>>(X, ld, K, kpad, cols, E, rev, out); break;
    case 7: k_oz_slice<7><<<grid, 256, 0, stream>>>(X, ld, K, kpad, cols, E, rev, out); break;
    case 8: k_oz_slice<8><<<grid, 256, 0, stream>>>(X, ld, K, kpad, cols, E, rev, out); break;
    case 9: k_oz_slice<9><<<grid, 256, 0, stream>>>(X, ld, K, kpad, cols, E, rev, out); break;
    default: k_oz_slice<10><<<grid, 256, 0, stream>>>(X, ld, K, kpad, cols, E, rev, out); break;
  }
  count_launch();
}

// The left operand's column exponents (Ea, m) and slices (As, ldk x m halves, in order).
cr_status oz_slice_left(const OzGeom& g, const double* A, int lda, int m, int* Ea, __half* As, cudaStream_t stream) {
  TimedScope ts("k_oz_slice", stream);
  k_oz_colexp<<<(unsigned)m, 256, 0, stream>>>(A, lda, g.K, Ea);
  count_launch();
  oz_slice_launch(g, A, lda, m, Ea, 0, As, stream);
  if (cudaError_t e = cudaGetLastError()) return fail(CR_ERR_CUDA, cudaGetErrorName(e));
  return CR_OK;
}

// Cout = Cin + alpha A^T B with A already sliced (Ea, As for m columns, geometry g): B is sliced
// per block of output columns, the blocks as wide as keeps one level's chunk products within
// 2 GiB; scratch from the library pool (the slices of a block, its chunk products, at most 32
// m nbc FP32, and the accumulator, m nbc double-float pairs).
cr_status oz_product(const OzGeom& g, const int* Ea, const __half* As, int m_, const double* B, int ldb, int n_,
                     double alpha, const double* Cin, int ldci, double* Cout, int ldco, cudaStream_t stream) {
  const size_t m = (size_t)m_;
  std::lock_guard<std::mutex> lk(g_cublas_mu);
  cublasHandle_t h = nullptr;
  CR_TRY(cublas_for(stream, &h));
  const int S = g.S, cpk = g.cpk, kc = g.kc, kpad = g.kpad;
  const size_t ldk = g.ldk;
  const int group = std::min(OZ_GROUP, S * cpk);                     // chunks per GEMM call
  const size_t budget = (size_t)1 << 31;
  const int nbc = (int)std::max<size_t>(1, std::min<size_t>((size_t)n_, budget / (m * group * sizeof(float))));
  int* Eb = nullptr;
  __half* Bs = nullptr;
  float* P = nullptr;
  float2* C = nullptr;
  auto alloc = [&](void** p, size_t bytes) { return scratch_alloc(p, bytes, stream); };
  cudaError_t e = cudaSuccess;
  if ((e = alloc((void**)&Eb, nbc * sizeof(int))) != cudaSuccess ||
      (e = alloc((void**)&Bs, ldk * nbc * sizeof(__half))) != cudaSuccess ||
      (e = alloc((void**)&P, (size_t)group * m * nbc * sizeof(float))) != cudaSuccess ||
      (e = alloc((void**)&C, m * nbc * sizeof(float2))) != cudaSuccess) {
    for (void* p : {(void*)Eb, (void*)Bs, (void*)P, (void*)C}) scratch_free(p, stream);
    return fail(CR_ERR_NOMEM, std::string("Ozaki product: scratch: ") + cudaGetErrorName(e));
  }
  cr_status st = CR_OK;
  const float one = 1.0f, zero = 0.0f;
  for (int j0 = 0; j0 < n_ && st == CR_OK; j0 += nbc) {
    const int w = std::min(nbc, n_ - j0);
    const double* Bj = B + (size_t)j0 * ldb;
    {
      TimedScope ts("k_oz_slice", stream);   // exponents and slices of this block of B
      k_oz_colexp<<<(unsigned)w, 256, 0, stream>>>(Bj, ldb, g.K, Eb);
      count_launch();
      oz_slice_launch(g, Bj, ldb, w, Eb, 1, Bs, stream);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) { st = fail(CR_ERR_CUDA, cudaGetErrorName(e)); break; }
    const dim3 ga = grid2d(m_, w);
    const double* Cin_j = Cin ? Cin + (size_t)j0 * ldci : nullptr;
    double* Cout_j = Cout + (size_t)j0 * ldco;
    bool first = true;
    // least significant level first
    for (int lev = S + 1; lev >= 2 && st == CR_OK; --lev) {
      // rows of the concatenated product: A slots 0 .. lev-2, B slots S-lev+1 .. S-1
      const int nchunk = (lev - 1) * cpk;
      const __half* a0 = As;
      const __half* b0 = Bs + (size_t)(S - lev + 1) * kpad;
      for (int g0 = 0; g0 < nchunk; g0 += group) {
        const int cnt = std::min(group, nchunk - g0);
        // P_c = A_lev[chunk g0 + c]^T B_lev[chunk g0 + c], c < cnt (m x w each, exact)
        cublasStatus_t cs;
        {
          TimedScope tg("oz_gemm", stream);
          cs = cublasGemmStridedBatchedEx(h, CUBLAS_OP_T, CUBLAS_OP_N, m_, w, kc, &one, a0 + (size_t)g0 * kc, CUDA_R_16F,
                                          (int)ldk, kc, b0 + (size_t)g0 * kc, CUDA_R_16F, (int)ldk, kc, &zero, P,
                                          CUDA_R_32F, m_, (long long)(m * w), cnt, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
        }
        if (cs != CUBLAS_STATUS_SUCCESS) {
          st = fail(CR_ERR_CUDA, "Ozaki product: cublasGemmStridedBatchedEx failed (" + std::to_string((int)cs) + ")");
          break;
        }
        const bool last = lev == 2 && g0 + cnt >= nchunk;
        TimedScope ts("k_oz_accum", stream);
        k_oz_accum<<<ga, 256, 0, stream>>>(P, cnt, m_, w, Ea, Eb, OZ_BITS * lev, C, first ? 1 : 0, last ? 1 : 0, alpha,
                                           Cin_j, ldci, Cout_j, ldco);
        count_launch();
        first = false;
      }
    }
  }
  if (st == CR_OK && (e = cudaGetLastError()) != cudaSuccess) st = fail(CR_ERR_CUDA, cudaGetErrorName(e));
  for (void* p : {(void*)Eb, (void*)Bs, (void*)P, (void*)C}) scratch_free(p, stream);
  return st;
}

// R = y_o 1^T - M_o into pool scratch (n_o x M, ld n_o); *R_out NULL on failure.
cr_status oz_residual(const double* d_yo, const double* d_Y, int ldy, int n_p, int n_o, int M, double** R_out,
                      cudaStream_t stream) {
  *R_out = nullptr;
  double* R = nullptr;
  CR_CUDA(scratch_alloc((void**)&R, (size_t)n_o * M * sizeof(double), stream));
  {
    TimedScope ts("k_oz_slice", stream);
    k_oz_resid<<<grid_for((size_t)n_o * M), 256, 0, stream>>>(d_yo, d_Y, ldy, n_p, n_o, M, R);
    count_launch();
  }
  if (cudaError_t e = cudaGetLastError()) {
    scratch_free(R, stream);
    return fail(CR_ERR_CUDA, cudaGetErrorName(e));
  }
  *R_out = R;
  return CR_OK;
}

}  // namespace

// Cout = Cin + alpha A^T B by the Ozaki product with S slices of 6 bits per operand column
// (A: K x m, ld lda; B: K x n, ld ldb; Cin, Cout: m x n, ld ldci / ldco; Cin NULL for zero;
// Cout may equal Cin with the same ld, and may overlap A or B, which are sliced before Cout is
// written).  The kept products are those with s + t <= S + 1, one GEMM per level.  A's slices
// (S K' m FP16, pool scratch) are made once, B's per block of output columns (oz_product).
cr_status ozaki_gemm_tn(const double* A, int lda, const double* B, int ldb, int K, int m_, int n_, double alpha,
                        const double* Cin, int ldci, double* Cout, int ldco, int S, cudaStream_t stream) {
  if (S < OZ_MIN_SLICES || S > OZ_MAX_SLICES) return fail(CR_ERR_ARG, "Ozaki product: slice count");
  if (m_ <= 0 || n_ <= 0) return CR_OK;
  if (K <= 0) {
    k_oz_copy<<<grid2d(m_, n_), 256, 0, stream>>>(Cin, ldci, m_, n_, Cout, ldco);
    CR_CHECK_LAUNCH("k_oz_copy");
    return CR_OK;
  }
  const OzGeom g = oz_geom(K, S);
  int* Ea = nullptr;
  __half* As = nullptr;
  cudaError_t e = scratch_alloc((void**)&Ea, (size_t)m_ * sizeof(int), stream);
  if (e == cudaSuccess) e = scratch_alloc((void**)&As, g.ldk * m_ * sizeof(__half), stream);
  cr_status st = e == cudaSuccess ? CR_OK : fail(CR_ERR_NOMEM, std::string("Ozaki product: scratch: ") + cudaGetErrorName(e));
  if (st == CR_OK) st = oz_slice_left(g, A, lda, m_, Ea, As, stream);
  if (st == CR_OK) st = oz_product(g, Ea, As, m_, B, ldb, n_, alpha, Cin, ldci, Cout, ldco, stream);
  scratch_free(Ea, stream);
  scratch_free(As, stream);
  return st;
}

// The correction S = M_p + W^T (y_o 1^T - M_o) (W: n_o x n_p, ld ldw; Y: (n_p + n_o) x M, ld
// ldy; S: n_p x M, ld lds): R = y_o 1^T - M_o (n_o M FP64, pool scratch), then the Ozaki
// product with Cin = M_p.
cr_status ozaki_correction(const double* d_W, int ldw, const double* d_yo, const double* d_Y, int ldy, int n_p, int n_o,
                           int M, double* d_S, int lds, cudaStream_t stream) {
  double* R = nullptr;
  CR_TRY(oz_residual(d_yo, d_Y, ldy, n_p, n_o, M, &R, stream));
  const cr_status st = ozaki_gemm_tn(d_W, ldw, R, n_o, n_o, n_p, M, 1.0, d_Y, ldy, d_S, lds, OZ_CORR_SLICES, stream);
  scratch_free(R, stream);
  return st;
}

// The correction with W's slices prepared by cr_weights_prepare (same arithmetic as
// ozaki_correction on the W the handle was made from).
cr_status ozaki_correction_prepared(cr_weights w, const double* d_yo, const double* d_Y, int ldy, int M, double* d_S, int lds,
                                    cudaStream_t stream) {
  CR_CUDA(cudaSetDevice(w->device));
  double* R = nullptr;
  CR_TRY(oz_residual(d_yo, d_Y, ldy, w->n_p, w->n_o, M, &R, stream));
  const OzGeom g = oz_geom(w->n_o, w->slices);
  const cr_status st = oz_product(g, w->Ea, w->As, w->n_p, R, w->n_o, M, 1.0, d_Y, ldy, d_S, lds, stream);
  scratch_free(R, stream);
  return st;
}

}  // namespace cr

using namespace cr;

extern "C" cr_status cr_weights_prepare(const double* d_W, int ldw, int n_o, int n_p, cr_stream stream, cr_weights* out) {
  if (!out) return fail(CR_ERR_ARG, "cr_weights_prepare: NULL output");
  *out = nullptr;
  if (!d_W || n_o <= 0 || n_p <= 0 || ldw < n_o) return fail(CR_ERR_ARG, "cr_weights_prepare: argument");
  int dev = 0;
  CR_CUDA(cudaGetDevice(&dev));
  cr_weights w = new cr_weights_s();
  w->device = dev;
  w->n_o = n_o;
  w->n_p = n_p;
  w->slices = OZ_CORR_SLICES;
  const OzGeom g = oz_geom(n_o, w->slices);
  cudaError_t e = cudaMalloc(&w->Ea, (size_t)n_p * sizeof(int));
  if (e == cudaSuccess) e = cudaMalloc(&w->As, g.ldk * n_p * sizeof(__half));
  cr_status st = e == cudaSuccess ? CR_OK : cuda_fail(e, "cr_weights_prepare: slices");
  if (st == CR_OK) st = oz_slice_left(g, d_W, ldw, n_p, w->Ea, w->As, stream);
  if (st != CR_OK) {
    cr_weights_release(w);
    return st;
  }
  *out = w;
  return CR_OK;
}

extern "C" cr_status cr_weights_release(cr_weights w) {
  if (!w) return CR_OK;
  cudaSetDevice(w->device);
  if (w->Ea) cudaFree(w->Ea);
  if (w->As) cudaFree(w->As);
  delete w;
  return CR_OK;
}

extern "C" cr_status cr_krige_correct_prepared(cr_weights w, const double* d_yo, const double* d_Y, int ldy, int M,
                                               double* d_S, int lds, cr_stream stream) {
  if (!w || !d_yo || !d_Y || !d_S || M <= 0 || ldy < w->n_p + w->n_o || lds < w->n_p)
    return fail(CR_ERR_ARG, "cr_krige_correct_prepared: argument");
  return ozaki_correction_prepared(w, d_yo, d_Y, ldy, M, d_S, lds, stream);
}
