// FP64-class matrix product on the FP16 tensor cores by the Ozaki scheme (Ozaki, Ogita, Oishi
// and Rump, "Error-free transformations of matrix multiplication by using fast routines of
// matrix multiplication and its applications", Numerical Algorithms 59 (2012)), for the
// conditioning correction of "Mixed-Precision GPU Acceleration for Confidence Regions of
// Spatial Excursion Sets" (Section V-B Eq.7: S = M_p + W^T (y_o 1^T - M_o)).
//
// C = A^T B with A (k x m) and B (k x n) column-major FP64:
//  - each column c of A gets a power of two 2^Ea_c above its largest |entry| (B likewise), and
//    |A_rc| 2^(7 S - Ea_c), truncated to an integer below 2^(7 S), is cut into S = 7 slices of
//    7 bits: A_rc = sum_s a_s,rc 2^(Ea_c - 7 s) + d with |a_s,rc| <= 127 and
//    |d| < 2^(Ea_c - 49);
//  - a slice product A_s^T B_t over K <= 1024 rows is a sum of at most 1024 integers of
//    magnitude <= 127^2 < 2^14, an integer below 2^24, so an FP16 tensor-core GEMM with FP32
//    accumulation computes it exactly (whatever its summation order);
//  - the products with s + t <= S + 1 (28 of the 49) are kept: the rest, and the truncations,
//    are below (k (2 + 8 2^-7) 2^-49) 2^(Ea_i + Eb_j) per output (derived in the tests);
//  - each kept product, summed over the K chunks in 64-bit integers (exact), is scaled by
//    2^(Ea_i + Eb_j - 7 (s + t)) (exact) and added to a double-float accumulator.
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

constexpr int OZ_BITS = 7, OZ_SLICES = 7, OZ_KC = 1024;

// E_c with max_r |X_rc| < 2^E_c (positive doubles order as their bit patterns); 0 for a zero
// column (its slices are all zero).  One CTA per column.
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
    E[c] = m == 0ull ? 0 : (eb == 0 ? -1022 : eb - 1022);
  }
}

// Slices of X (rows x cols, column-major, ld): out + s * rows_pad * cols holds slice s + 1
// (the most significant first) as a rows_pad x cols column-major FP16 matrix of integers in
// [-127, 127], rows beyond `rows` zero.  Integer arithmetic on the FP64 bit pattern only.
__global__ void __launch_bounds__(256) k_oz_slice(const double* __restrict__ X, int ld, int rows, int rows_pad, int cols,
                                                  const int* __restrict__ E, __half* __restrict__ out) {
  const size_t total = (size_t)rows_pad * cols, plane = total;
  for (size_t e = blockIdx.x * (size_t)256 + threadIdx.x; e < total; e += (size_t)gridDim.x * 256) {
    const int r = (int)(e % rows_pad), c = (int)(e / rows_pad);
    unsigned long long q = 0ull;
    bool neg = false;
    if (r < rows) {
      const unsigned long long b = (unsigned long long)__double_as_longlong(X[(size_t)c * ld + r]);
      neg = (b >> 63) != 0;
      const int eb = (int)((b >> 52) & 0x7ff);
      const unsigned long long mant = (b & 0x000fffffffffffffull) | (eb ? 0x0010000000000000ull : 0ull);
      // |x| = mant 2^(e2);  q = floor(|x| 2^(7 S - E_c)) < 2^(7 S)
      const int e2 = (eb ? eb : 1) - 1075;
      const int shift = e2 + OZ_BITS * OZ_SLICES - E[c];
      if (shift >= 0) q = shift < 64 ? mant << shift : 0ull;
      else q = -shift < 64 ? mant >> (-shift) : 0ull;
    }
#pragma unroll
    for (int s = 0; s < OZ_SLICES; ++s) {
      const int a = (int)((q >> (OZ_BITS * (OZ_SLICES - 1 - s))) & 127ull);
      out[(size_t)s * plane + e] = __int2half_rn(neg ? -a : a);
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

// C += 2^(Ea_i + Eb_j - 7 lev) sum_b P_b(i, j) for one slice pair (C = that term when first):
// the chunk products are exact integers below 2^24, their sum (below 2^28) is exact in 64-bit
// integers and as a double-float pair, and the power-of-two scaling is exact.
__global__ void __launch_bounds__(256) k_oz_accum(const float* __restrict__ P, int nchunk, int m, int n,
                                                  const int* __restrict__ Ea, const int* __restrict__ Eb, int lev,
                                                  float2* __restrict__ C, int first) {
  const size_t total = (size_t)m * n;
  for (size_t e = blockIdx.x * (size_t)256 + threadIdx.x; e < total; e += (size_t)gridDim.x * 256) {
    long long v = 0;
    for (int b = 0; b < nchunk; ++b) v += (long long)__float2ll_rn(P[(size_t)b * total + e]);
    const int i = (int)(e % m), j = (int)(e / m);
    const int ex = Ea[i] + Eb[j] - OZ_BITS * lev;
    const float h = (float)v;                          // nearest FP32 of v (|v| < 2^28)
    const float l = (float)(v - (long long)h);         // the rest, below 2^5: exact
    const df term = {ldexpf(h, ex), ldexpf(l, ex)};
    if (first) {
      C[e] = make_float2(term.hi, term.lo);
    } else {
      const float2 c = C[e];
      const df s = df_add({c.x, c.y}, term);
      C[e] = make_float2(s.hi, s.lo);
    }
  }
}

// S = M_p + C (FP64), C the double-float product.
__global__ void __launch_bounds__(256) k_oz_final(const float2* __restrict__ C, int m, int n, const double* __restrict__ Y,
                                                  int ldy, double* __restrict__ S, int lds) {
  const size_t total = (size_t)m * n;
  for (size_t e = blockIdx.x * (size_t)256 + threadIdx.x; e < total; e += (size_t)gridDim.x * 256) {
    const int i = (int)(e % m), j = (int)(e / m);
    const float2 c = C[e];
    S[(size_t)j * lds + i] = Y[(size_t)j * ldy + i] + ((double)c.x + (double)c.y);
  }
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

unsigned grid_for(size_t total) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t want = (total + 255) / 256, cap = (size_t)sms * 16;
  return (unsigned)std::max<size_t>(1, std::min(want, cap));
}

}  // namespace

// The correction S = M_p + W^T (y_o 1^T - M_o) by the Ozaki product (W: n_o x n_p, ld ldw;
// Y: (n_p + n_o) x M, ld ldy; S: n_p x M, ld lds).  Stream-ordered scratch: the slices
// (7 (n_o' n_p + n_o' M) FP16, n_o' = n_o rounded up to 1024), the chunk products
// (n_o' / 1024 n_p M FP32), R (n_o M FP64) and the accumulator (n_p M double-float pairs).
cr_status ozaki_correction(const double* d_W, int ldw, const double* d_yo, const double* d_Y, int ldy, int n_p, int n_o,
                           int M, double* d_S, int lds, cudaStream_t stream) {
  std::lock_guard<std::mutex> lk(g_cublas_mu);
  cublasHandle_t h = nullptr;
  CR_TRY(cublas_for(stream, &h));
  const int kpad = (n_o + OZ_KC - 1) / OZ_KC * OZ_KC, nchunk = kpad / OZ_KC;
  const size_t m = (size_t)n_p, n = (size_t)M;
  double* R = nullptr;
  int *Ea = nullptr, *Eb = nullptr;
  __half *As = nullptr, *Bs = nullptr;
  float* P = nullptr;
  float2* C = nullptr;
  auto alloc = [&](void** p, size_t bytes) { return cudaMallocAsync(p, bytes, stream); };
  cudaError_t e = cudaSuccess;
  if ((e = alloc((void**)&R, (size_t)n_o * n * sizeof(double))) != cudaSuccess ||
      (e = alloc((void**)&Ea, m * sizeof(int))) != cudaSuccess || (e = alloc((void**)&Eb, n * sizeof(int))) != cudaSuccess ||
      (e = alloc((void**)&As, (size_t)OZ_SLICES * kpad * m * sizeof(__half))) != cudaSuccess ||
      (e = alloc((void**)&Bs, (size_t)OZ_SLICES * kpad * n * sizeof(__half))) != cudaSuccess ||
      (e = alloc((void**)&P, (size_t)nchunk * m * n * sizeof(float))) != cudaSuccess ||
      (e = alloc((void**)&C, m * n * sizeof(float2))) != cudaSuccess) {
    for (void* p : {(void*)R, (void*)Ea, (void*)Eb, (void*)As, (void*)Bs, (void*)P, (void*)C})
      if (p) cudaFreeAsync(p, stream);
    return fail(CR_ERR_NOMEM, std::string("Ozaki product: scratch: ") + cudaGetErrorName(e));
  }
  cr_status st = CR_OK;
  do {
    k_oz_resid<<<grid_for((size_t)n_o * n), 256, 0, stream>>>(d_yo, d_Y, ldy, n_p, n_o, M, R);
    count_launch();
    k_oz_colexp<<<(unsigned)m, 256, 0, stream>>>(d_W, ldw, n_o, Ea);
    count_launch();
    k_oz_colexp<<<(unsigned)n, 256, 0, stream>>>(R, n_o, n_o, Eb);
    count_launch();
    k_oz_slice<<<grid_for((size_t)kpad * m), 256, 0, stream>>>(d_W, ldw, n_o, kpad, (int)m, Ea, As);
    count_launch();
    k_oz_slice<<<grid_for((size_t)kpad * n), 256, 0, stream>>>(R, n_o, n_o, kpad, (int)n, Eb, Bs);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) { st = fail(CR_ERR_CUDA, cudaGetErrorName(e)); break; }
    const float one = 1.0f, zero = 0.0f;
    bool first = true;
    for (int lev = 2; lev <= OZ_SLICES + 1 && st == CR_OK; ++lev) {
      for (int s = 1; s <= OZ_SLICES; ++s) {
        const int t = lev - s;
        if (t < 1 || t > OZ_SLICES) continue;
        const __half* a = As + (size_t)(s - 1) * kpad * m;
        const __half* b = Bs + (size_t)(t - 1) * kpad * n;
        // P_c = A_s[chunk c]^T B_t[chunk c], c = 0 .. nchunk-1 (m x n each, exact)
        const cublasStatus_t cs = cublasGemmStridedBatchedEx(
            h, CUBLAS_OP_T, CUBLAS_OP_N, (int)m, (int)n, OZ_KC, &one, a, CUDA_R_16F, kpad, OZ_KC, b, CUDA_R_16F, kpad,
            OZ_KC, &zero, P, CUDA_R_32F, (int)m, (long long)(m * n), nchunk, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
        if (cs != CUBLAS_STATUS_SUCCESS) {
          st = fail(CR_ERR_CUDA, "Ozaki product: cublasGemmStridedBatchedEx failed (" + std::to_string((int)cs) + ")");
          break;
        }
        TimedScope ts("k_oz_accum", stream);
        k_oz_accum<<<grid_for(m * n), 256, 0, stream>>>(P, nchunk, (int)m, (int)n, Ea, Eb, lev, C, first ? 1 : 0);
        count_launch();
        first = false;
      }
    }
    if (st != CR_OK) break;
    k_oz_final<<<grid_for(m * n), 256, 0, stream>>>(C, (int)m, (int)n, d_Y, ldy, d_S, lds);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) st = fail(CR_ERR_CUDA, cudaGetErrorName(e));
  } while (false);
  for (void* p : {(void*)R, (void*)Ea, (void*)Eb, (void*)As, (void*)Bs, (void*)P, (void*)C}) cudaFreeAsync(p, stream);
  return st;
}

}  // namespace cr
