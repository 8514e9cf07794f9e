// FP64 kernels: batched strided tile GEMM (C = beta C + alpha sum_p A_p B_p^T), the 64 x 64
// Cholesky-plus-inverse base block, and conversions of FP64 tiles to FP16 high/low parts.
//
// On GB300 the FP64 units deliver about 1.2 TFLOP/s (two FMA lanes per SM per clock), so
// these kernels are bound by the FP64 pipe and need no elaborate data staging; what matters
// is spreading the work over many SMs (small output blocks) on the critical path.
#include <math.h>

#include "common.cuh"
#include "fp64.cuh"

namespace cr {

template <int BM, int BN>
__global__ void __launch_bounds__(256) k_dgemm(const DJob* __restrict__ jobs, const DPair* __restrict__ pairs) {
  constexpr int KB = 16;
  constexpr int TM = BM / 16, TN = BN / 16;
  __shared__ double As[KB][BM + 1];
  __shared__ double Bs[KB][BN + 1];
  const DJob jb = jobs[blockIdx.x];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  double acc[TM][TN];
#pragma unroll
  for (int a = 0; a < TM; ++a)
#pragma unroll
    for (int b = 0; b < TN; ++b) acc[a][b] = 0.0;
  for (int pi = 0; pi < jb.pcnt; ++pi) {
    const DPair pr = pairs[jb.pbeg + pi];
    const int K = min(pr.K, jb.kmax);
    const double* Ab = pr.A + (size_t)jb.arow * pr.sAm;
    const double* Bb = pr.B + (size_t)jb.brow * pr.sBn;
    for (int k0 = 0; k0 < K; k0 += KB) {
      for (int idx = threadIdx.x; idx < BM * KB; idx += 256) {
        const int m = idx / KB, k = idx % KB;
        As[k][m] = (m < jb.m && k0 + k < K) ? Ab[(size_t)m * pr.sAm + (size_t)(k0 + k) * pr.sAk] : 0.0;
      }
      for (int idx = threadIdx.x; idx < BN * KB; idx += 256) {
        const int nn = idx / KB, k = idx % KB;
        Bs[k][nn] = (nn < jb.n && k0 + k < K) ? Bb[(size_t)nn * pr.sBn + (size_t)(k0 + k) * pr.sBk] : 0.0;
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < KB; ++k) {
        double a[TM], b[TN];
#pragma unroll
        for (int q = 0; q < TM; ++q) a[q] = As[k][ty + 16 * q];
#pragma unroll
        for (int q = 0; q < TN; ++q) b[q] = Bs[k][tx + 16 * q];
#pragma unroll
        for (int x = 0; x < TM; ++x)
#pragma unroll
          for (int y = 0; y < TN; ++y) acc[x][y] = fma(a[x], b[y], acc[x][y]);
      }
      __syncthreads();
    }
  }
#pragma unroll
  for (int x = 0; x < TM; ++x)
#pragma unroll
    for (int y = 0; y < TN; ++y) {
      const int m = ty + 16 * x, nn = tx + 16 * y;
      if (m < jb.m && nn < jb.n) {
        double* c = jb.C + (size_t)m * jb.sCm + (size_t)nn * jb.sCn;
        const double prev = jb.beta != 0.0 ? jb.beta * *c : 0.0;
        *c = prev + jb.alpha * acc[x][y];
      }
    }
}

cr_status dgemm_launch(int bm, const DJob* d_jobs, const DPair* d_pairs, int njobs, cudaStream_t stream) {
  if (njobs <= 0) return CR_OK;
  switch (bm) {
    case 16: k_dgemm<16, 16><<<njobs, 256, 0, stream>>>(d_jobs, d_pairs); break;
    case 32: k_dgemm<32, 32><<<njobs, 256, 0, stream>>>(d_jobs, d_pairs); break;
    case 64: k_dgemm<64, 64><<<njobs, 256, 0, stream>>>(d_jobs, d_pairs); break;
    default: return fail(CR_ERR_ARG, "dgemm_launch: block size");
  }
  CR_CHECK_LAUNCH("k_dgemm");
  return CR_OK;
}

// Cholesky of the 64 x 64 block at A (row-major, leading dimension lda; lower part read,
// lower part overwritten with L) and its inverse M = L^-1 written (lower, upper zeroed) at
// Minv.  A non-positive pivot records its 1-based global column (gcol0 + c + 1) in
// status[1] with atomicMin.
__global__ void __launch_bounds__(256) k_potrf64_base(double* A, int lda, double* Minv, int ldm, int gcol0, int* status) {
  // L holds the factor in its lower triangle; the inverse M is kept transposed in the strict
  // upper triangle (M[r][c] at L[c][r], r > c) with its diagonal in dg.
  __shared__ double L[64][65];
  __shared__ double dg[64];
  for (int idx = threadIdx.x; idx < 64 * 64; idx += 256) {
    const int r = idx / 64, c = idx % 64;
    L[r][c] = r >= c ? A[(size_t)r * lda + c] : 0.0;
  }
  __syncthreads();
  for (int c = 0; c < 64; ++c) {
    if (threadIdx.x == 0) {
      const double d = L[c][c];
      if (!(d > 0.0)) atomicMin(&status[1], gcol0 + c + 1);
      L[c][c] = sqrt(d);
    }
    __syncthreads();
    const double dc = L[c][c];
    for (int r = c + 1 + threadIdx.x; r < 64; r += 256) L[r][c] /= dc;
    __syncthreads();
    // trailing update of the lower part: rows r > c, columns q in (c, r]
    const int m = 63 - c;
    for (int idx = threadIdx.x; idx < m * m; idx += 256) {
      const int r = c + 1 + idx / m, q = c + 1 + idx % m;
      if (q <= r) L[r][q] -= L[r][c] * L[q][c];
    }
    __syncthreads();
  }
  // inverse by forward substitution, one column of M per thread
  if (threadIdx.x < 64) {
    const int c = threadIdx.x;
    dg[c] = 1.0 / L[c][c];
    for (int r = c + 1; r < 64; ++r) {
      double sum = L[r][c] * dg[c];
      for (int q = c + 1; q < r; ++q) sum = fma(L[r][q], L[c][q], sum);
      L[c][r] = -sum / L[r][r];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < 64 * 64; idx += 256) {
    const int r = idx / 64, c = idx % 64;
    if (r >= c) A[(size_t)r * lda + c] = L[r][c];
    Minv[(size_t)r * ldm + c] = r > c ? L[c][r] : (r == c ? dg[c] : 0.0);
  }
}

// FP64 tile -> FP16 high and low parts (x = hi + lo to ~2^-22), optionally zeroing the
// strict upper triangle (diagonal factor tiles).
__global__ void __launch_bounds__(256) k_split_tile(const double* __restrict__ src, int nb, __half* __restrict__ hi,
                                                    __half* __restrict__ lo, int lower_only) {
  const size_t count = (size_t)nb * nb;
  for (size_t idx = blockIdx.x * 256 + threadIdx.x; idx < count; idx += (size_t)gridDim.x * 256) {
    const int r = (int)(idx / nb), c = (int)(idx % nb);
    // via FP32: the pair keeps the leading 22 bits, which is all an FP16 pair can hold
    const float x = (lower_only && c > r) ? 0.0f : (float)src[idx];
    const __half h = __float2half_rn(x);
    hi[idx] = h;
    lo[idx] = __float2half_rn(x - __half2float(h));
  }
}

// FP64 -> FP32 rounded to nearest (ties to even) from the IEEE 754 fields, in integer
// arithmetic: GB300 issues the F2F conversion on its slow FP64/conversion pipe.  Results
// below 2^-126 come out as signed zero (the FP16 pairs made from them are zero either way:
// FP16 holds nothing below 2^-24); infinities and NaN map to infinity and NaN.
__device__ __forceinline__ float narrow(double x) {
  const unsigned long long b = (unsigned long long)__double_as_longlong(x);
  const unsigned sign = (unsigned)(b >> 32) & 0x80000000u;
  const int e = (int)((b >> 52) & 0x7ff);
  const unsigned long long frac = b & 0xfffffffffffffull;
  if (e == 0x7ff) return __uint_as_float(sign | 0x7f800000u | (frac ? 0x400000u : 0u));
  const int fe = e - 1023 + 127;
  if (fe < 1) return __uint_as_float(sign);
  if (fe > 254) return __uint_as_float(sign | 0x7f800000u);
  const unsigned m = (unsigned)(frac >> 29);
  const unsigned rest = (unsigned)(frac & 0x1fffffffull);   // the 29 dropped bits
  const unsigned up = (rest > 0x10000000u || (rest == 0x10000000u && (m & 1u))) ? 1u : 0u;
  // a carry out of the fraction raises the exponent, as rounding should
  return __uint_as_float((sign | ((unsigned)fe << 23) | m) + up);
}

// Splits the inverse factor and the diagonal factor of one column in one launch:
//  - eM with max|M| 2^eM < 2^14 (status[2] = eM), from the running maximum the diagonal
//    executor accumulated (IEEE bits of max |M|), and the FP16 high/low parts of M 2^eM;
//  - the FP16 high/low parts of the diagonal factor L (lower part; zero above).
// Elements [0, nb^2) are M, [nb^2, 2 nb^2) are L; both through FP32, whose 24 bits cover
// everything an FP16 pair can hold.  Each thread takes pairs of adjacent elements (nb is
// even, so a pair never straddles a row or the M / L boundary): 16-byte loads, packed
// FP16 conversions and 4-byte stores.
__global__ void __launch_bounds__(256) k_split_diag(const double* __restrict__ Minv, const double* __restrict__ L, int nb,
                                                    const unsigned long long* __restrict__ amax, __half* __restrict__ mh,
                                                    __half* __restrict__ ml, __half* __restrict__ lh, __half* __restrict__ ll,
                                                    int* status) {
  const unsigned long long bits = *amax;
  const int ef = (int)((bits >> 52) & 0x7ff);   // max |M| in [2^(ef-1023), 2^(ef-1022))
  const int e = (bits == 0 || ef == 0 || ef == 0x7ff) ? 0 : 14 - (ef - 1022);
  if (blockIdx.x == 0 && threadIdx.x == 0) status[2] = e;
  const float sc = ldexpf(1.0f, e);
  const size_t half_count = (size_t)nb * nb / 2;
  for (size_t pidx = blockIdx.x * 256 + threadIdx.x; pidx < 2 * half_count; pidx += (size_t)gridDim.x * 256) {
    float x0, x1;
    __half2 *h, *l;
    size_t q;
    if (pidx < half_count) {
      q = pidx;
      const double2 v = reinterpret_cast<const double2*>(Minv)[q];
      x0 = narrow(v.x) * sc;
      x1 = narrow(v.y) * sc;
      h = reinterpret_cast<__half2*>(mh);
      l = reinterpret_cast<__half2*>(ml);
    } else {
      q = pidx - half_count;
      const int r = (int)(2 * q / nb), c = (int)(2 * q % nb);
      const double2 v = reinterpret_cast<const double2*>(L)[q];
      x0 = c > r ? 0.0f : narrow(v.x);
      x1 = c + 1 > r ? 0.0f : narrow(v.y);
      h = reinterpret_cast<__half2*>(lh);
      l = reinterpret_cast<__half2*>(ll);
    }
    const __half2 hv = __floats2half2_rn(x0, x1);
    const float2 hf = __half22float2(hv);
    h[q] = hv;
    l[q] = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
  }
}

__global__ void k_status_init(int* status) {
  status[0] = 0;
  status[1] = 0x7fffffff;
  status[2] = 0;
  status[3] = 0;
}

cr_status potrf64_base_launch(double* A, int lda, double* Minv, int ldm, int gcol0, int* status, cudaStream_t s) {
  k_potrf64_base<<<1, 256, 0, s>>>(A, lda, Minv, ldm, gcol0, status);
  CR_CHECK_LAUNCH("k_potrf64_base");
  return CR_OK;
}
cr_status split_tile_launch(const double* src, int nb, __half* hi, __half* lo, int lower_only, cudaStream_t s) {
  k_split_tile<<<128, 256, 0, s>>>(src, nb, hi, lo, lower_only);
  CR_CHECK_LAUNCH("k_split_tile");
  return CR_OK;
}
cr_status split_diag_launch(const double* Minv, const double* L, int nb, const unsigned long long* amax, __half* mh, __half* ml,
                            __half* lh, __half* ll, int* status, cudaStream_t s) {
  // one element pair per thread: the kernel is latency-bound, so every load is in flight at once
  const unsigned grid = (unsigned)(((size_t)nb * nb + 255) / 256);   // 2 nb^2 / 2 pairs, 256 per CTA
  k_split_diag<<<grid, 256, 0, s>>>(Minv, L, nb, amax, mh, ml, lh, ll, status);
  CR_CHECK_LAUNCH("k_split_diag");
  return CR_OK;
}
cr_status status_init_launch(int* status, cudaStream_t s) {
  k_status_init<<<1, 1, 0, s>>>(status);
  CR_CHECK_LAUNCH("k_status_init");
  return CR_OK;
}

}  // namespace cr
