// Standard-normal generation, input compensation and the simulation multiply.
//
// "Mixed-Precision GPU Acceleration for Confidence Regions of Spatial Excursion Sets":
//  - Section V-B (Desc_rnorm): seeded N(0,1) draws generated on the GPU with a Box-Muller
//    ordering.  The stream here is the library's own: SplitMix64 (Steele, Lea, Flood, OOPSLA
//    2014) on seed + (c + 1) * 0x9E3779B97F4A7C15 gives 64 random bits per counter c; element
//    e = offset + j n + i of an n x M column-major matrix uses counters 2p and 2p + 1 with
//    p = floor(e / 2); Box-Muller (1958) gives r cos(2 pi u2) for even e, r sin(2 pi u2) for odd.
//  - Alg.1 steps 5-8 and Section V-F: B = M_rand / s before the FP16 rounding; ||B||_F is a
//    diagnostic only.
//  - Section IV-C Eq.3 / Alg.1: Y = L_s B (tensor cores) or, without AMP, Y = L M_rand in FP64.
#include <math.h>

#include "common.cuh"
#include "fp64.cuh"
#include "tc.cuh"

namespace cr {

__device__ __forceinline__ uint64_t splitmix64(uint64_t seed, uint64_t c) {
  uint64_t z = seed + (c + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ double normal64(uint64_t seed, uint64_t e) {
  const uint64_t p = e >> 1;
  const double u1 = ((double)(splitmix64(seed, 2 * p) >> 11) + 0.5) * 0x1.0p-53;
  const double u2 = ((double)(splitmix64(seed, 2 * p + 1) >> 11) + 0.5) * 0x1.0p-53;
  const double r = sqrt(-2.0 * log(u1));
  return (e & 1ull) ? r * sinpi(2.0 * u2) : r * cospi(2.0 * u2);
}

// FP32 variant: 24-bit uniforms from the same 64-bit draws.
__device__ __forceinline__ float normal32(uint64_t seed, uint64_t e) {
  const uint64_t p = e >> 1;
  const float u1 = ((float)(splitmix64(seed, 2 * p) >> 40) + 0.5f) * 0x1.0p-24f;
  const float u2 = ((float)(splitmix64(seed, 2 * p + 1) >> 40) + 0.5f) * 0x1.0p-24f;
  const float r = sqrtf(-2.0f * logf(u1));
  return (e & 1ull) ? r * sinpif(2.0f * u2) : r * cospif(2.0f * u2);
}

__global__ void k_rnorm(double* __restrict__ Z, int ldz, int n, int M, uint64_t seed, uint64_t offset) {
  const size_t total = (size_t)n * M;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const int j = (int)(e / n), i = (int)(e % n);
    Z[(size_t)j * ldz + i] = normal64(seed, offset + e);
  }
}

// B (npad x M, column-major, ld npad) = fp16(Z / s), zero padding rows; optional partial
// sums of (Z/s)^2 per block (before rounding).
__global__ void __launch_bounds__(256) k_compensate(const double* __restrict__ Z, int ldz, int n, int npad, int M, double inv_s,
                                                    int generate, uint64_t seed, uint64_t offset, __half* __restrict__ B,
                                                    double* __restrict__ part) {
  double ssq = 0.0;
  const size_t total = (size_t)npad * M;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const int j = (int)(e / npad), i = (int)(e % npad);
    double b = 0.0;
    if (i < n) {
      if (generate) b = (double)(normal32(seed, offset + (uint64_t)j * n + i) * (float)inv_s);
      else b = Z[(size_t)j * ldz + i] * inv_s;
    }
    ssq += b * b;
    B[e] = __double2half(b);
  }
  if (part) {
    __shared__ double red[8];
    for (int o = 16; o > 0; o >>= 1) ssq += __shfl_down_sync(0xffffffffu, ssq, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ssq;
    __syncthreads();
    if (threadIdx.x == 0) {
      double a = 0.0;
      for (int q = 0; q < 8; ++q) a += red[q];
      part[blockIdx.x] = a;
    }
  }
}

// Generated stream with n and offset even: the two elements of a Box-Muller pair are rows
// i, i+1 (i even) of one column, so each thread draws a pair once, converts it to FP16 with
// one packed conversion and stores it as one half2; squares are summed in FP32 (the norm is
// a diagnostic).  Columns are walked with row pairs, so no index division is needed.
__global__ void __launch_bounds__(256) k_compensate_pairs(int n, int npad, int M, float inv_s, uint64_t seed,
                                                          uint64_t offset, __half* __restrict__ B, double* __restrict__ part) {
  float ssq = 0.0f;
  const int pairs = npad / 2;
  for (int j = blockIdx.x; j < M; j += gridDim.x) {
    __half2* col = reinterpret_cast<__half2*>(B + (size_t)j * npad);
    const uint64_t e0 = offset + (uint64_t)j * n;   // even
    for (int ip = threadIdx.x; ip < pairs; ip += blockDim.x) {
      const int i = 2 * ip;
      float z0 = 0.0f, z1 = 0.0f;
      if (i < n) {
        const uint64_t p = (e0 + (uint64_t)i) >> 1;
        const float u1 = ((float)(splitmix64(seed, 2 * p) >> 40) + 0.5f) * 0x1.0p-24f;
        const float u2 = ((float)(splitmix64(seed, 2 * p + 1) >> 40) + 0.5f) * 0x1.0p-24f;
        const float r = sqrtf(-2.0f * logf(u1));
        float sn, cs;
        sincospif(2.0f * u2, &sn, &cs);
        z0 = r * cs * inv_s;
        z1 = (i + 1 < n) ? r * sn * inv_s : 0.0f;
      }
      ssq = fmaf(z0, z0, fmaf(z1, z1, ssq));
      col[ip] = __floats2half2_rn(z0, z1);
    }
  }
  if (part) {
    __shared__ double red[8];
    double a = ssq;
    for (int o = 16; o > 0; o >>= 1) a += __shfl_down_sync(0xffffffffu, a, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
    __syncthreads();
    if (threadIdx.x == 0) {
      double t = 0.0;
      for (int q = 0; q < 8; ++q) t += red[q];
      part[blockIdx.x] = t;
    }
  }
}

constexpr int COMP_BLOCKS = 1216;   // 8 per SM on 152 SMs

}  // namespace cr

using namespace cr;

extern "C" cr_status cr_rnorm(double* d_Z, int ldz, int n, int M, uint64_t seed, uint64_t offset, cr_stream stream) {
  if (!d_Z || n <= 0 || M <= 0 || ldz < n) return fail(CR_ERR_ARG, "cr_rnorm: argument");
  k_rnorm<<<COMP_BLOCKS, 256, 0, stream>>>(d_Z, ldz, n, M, seed, offset);
  CR_CHECK_LAUNCH("k_rnorm");
  return CR_OK;
}

namespace cr {

static cr_status trmm64(cr_tilemat L, const double* d_Z, int ldz, int M, double* d_Y, int ldy, cudaStream_t stream) {
  const int nt = L->nt, nb = L->nb, n = L->n;
  const size_t nb2 = (size_t)nb * nb;
  std::vector<DPair> pairs;
  std::vector<DJob> jobs;
  const int bs = 64;
  for (int i = 0; i < nt; ++i) {
    const int pbeg = (int)pairs.size();
    for (int k = 0; k <= i; ++k) {
      const int K = std::min(nb, n - k * nb);
      pairs.push_back(DPair{L->pool64 + (size_t)L->h_i64[tidx(i, k)] * nb2, d_Z + (size_t)k * nb, nb, 1, ldz, 1, K});
    }
    for (int rb = 0; rb < nb / bs; ++rb) {
      const int row0 = i * nb + rb * bs;
      if (row0 >= n) break;
      for (int cb = 0; cb * bs < M; ++cb) {
        DJob j{};
        j.C = d_Y + (size_t)cb * bs * ldy + row0;
        j.sCm = 1; j.sCn = ldy;
        j.m = std::min(bs, n - row0); j.n = std::min(bs, M - cb * bs);
        j.pbeg = pbeg; j.pcnt = i + 1;
        j.alpha = 1.0; j.beta = 0.0;
        j.arow = rb * bs; j.brow = cb * bs; j.kmax = nb;
        jobs.push_back(j);
      }
    }
    // the diagonal pair only needs K up to the block's last row: handled by the zero upper
    // triangle of the factor tile
  }
  DJob* dj = nullptr;
  DPair* dp = nullptr;
  CR_CUDA(cudaMalloc(&dj, jobs.size() * sizeof(DJob)));
  CR_CUDA(cudaMalloc(&dp, pairs.size() * sizeof(DPair)));
  CR_CUDA(cudaMemcpyAsync(dj, jobs.data(), jobs.size() * sizeof(DJob), cudaMemcpyHostToDevice, stream));
  CR_CUDA(cudaMemcpyAsync(dp, pairs.data(), pairs.size() * sizeof(DPair), cudaMemcpyHostToDevice, stream));
  cr_status st = dgemm_launch(bs, dj, dp, (int)jobs.size(), stream);
  cudaStreamSynchronize(stream);
  cudaFree(dj);
  cudaFree(dp);
  return st;
}

}  // namespace cr

extern "C" cr_status cr_trmm_sim(cr_tilemat L, const double* d_Z, int ldz, int M, uint64_t seed, uint64_t offset, double* d_Y,
                                 int ldy, int flags, double* h_bnorm, cr_stream stream) {
  if (!L || !d_Y || M <= 0 || ldy < L->n) return fail(CR_ERR_ARG, "cr_trmm_sim: argument");
  const bool gen = (flags & CR_TRMM_GENERATE) != 0;
  if (!gen && (!d_Z || ldz < L->n)) return fail(CR_ERR_ARG, "cr_trmm_sim: d_Z / ldz");
  if (!L->factored) return fail(CR_ERR_STATE, "cr_trmm_sim: factor first (cr_potrf_adaptive)");
  CR_CUDA(cudaSetDevice(L->device));
  if (!L->amp) {
    if (gen) return fail(CR_ERR_ARG, "cr_trmm_sim: the FP64 path needs d_Z (use cr_rnorm)");
    if (h_bnorm) *h_bnorm = NAN;
    return trmm64(L, d_Z, ldz, M, d_Y, ldy, stream);
  }
  const size_t need = (size_t)L->npad * M;
  if (need > L->b16_elems) {
    if (L->b16) cudaFree(L->b16);
    L->b16 = nullptr;
    L->b16_elems = 0;
    CR_CUDA(cudaMalloc(&L->b16, need * sizeof(__half)));
    L->b16_elems = need;
    L->b16_M = -1;
  }
  if (L->b16_M != M) {
    CR_TRY(make_tensor_map_2d_f16(&L->tm_b16, L->b16, L->npad, M, L->npad, 64, 128));
    L->b16_M = M;
  }
  if (!L->bnorm_part) CR_CUDA(cudaMalloc(&L->bnorm_part, COMP_BLOCKS * sizeof(double)));
  if (gen && L->n % 2 == 0 && offset % 2 == 0 && L->npad % 2 == 0) {
    k_compensate_pairs<<<COMP_BLOCKS, 256, 0, stream>>>(L->n, L->npad, M, (float)(1.0 / L->s), seed, offset, L->b16,
                                                        h_bnorm ? L->bnorm_part : nullptr);
    CR_CHECK_LAUNCH("k_compensate_pairs");
  } else {
    k_compensate<<<COMP_BLOCKS, 256, 0, stream>>>(d_Z, ldz, L->n, L->npad, M, 1.0 / L->s, gen ? 1 : 0, seed, offset, L->b16,
                                                  h_bnorm ? L->bnorm_part : nullptr);
    CR_CHECK_LAUNCH("k_compensate");
  }
  TcParams tp{};
  tp.v = L->view();
  tp.mode = TC_TRMM;
  tp.err = L->d_status;
  tp.status = L->d_status;
  tp.Y = d_Y;
  tp.ldy = ldy;
  tp.M = M;
  tp.ncb = (M + TC_BN - 1) / TC_BN;
  tp.flags = flags;
  if (flags & CR_TRMM_FP16_PER_GEMM) {
    const size_t need16 = (size_t)L->npad * tp.ncb * TC_BN;   // one 128 x 256 tile per output block
    if (need16 > L->y16_elems) {
      if (L->y16) cudaFree(L->y16);
      L->y16 = nullptr;
      L->y16_elems = 0;
      CR_CUDA(cudaMalloc(&L->y16, need16 * sizeof(__half)));
      L->y16_elems = need16;
    }
    tp.y16 = L->y16;
  }
  CR_TRY(tc_launch(tp, L->tm_pool16, L->tm_b16, stream));
  if (h_bnorm) {
    std::vector<double> part(COMP_BLOCKS);
    CR_CUDA(cudaMemcpyAsync(part.data(), L->bnorm_part, COMP_BLOCKS * sizeof(double), cudaMemcpyDeviceToHost, stream));
    CR_CUDA(cudaStreamSynchronize(stream));
    double a = 0.0;
    for (double x : part) a += x;
    *h_bnorm = sqrt(a);
    int h[4];
    CR_CUDA(cudaMemcpy(h, L->d_status, sizeof(h), cudaMemcpyDeviceToHost));
    if (h[0] & DEV_ERR_TIMEOUT) return fail(CR_ERR_TIMEOUT, "cr_trmm_sim: a device-side wait timed out");
  }
  return CR_OK;
}
