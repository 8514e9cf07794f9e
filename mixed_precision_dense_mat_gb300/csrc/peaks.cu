// Throughput probes of the arithmetic units the factorisation runs on, for the roofline
// denominators of the measurement (the paper has no counterpart): FP64 FMA, FP32 FMA, the FP64
// tensor-core MMA (mma.sync m8n8k4, FP64), and the double-float multiply-accumulate of the
// diagonal executor (an emulated FP64 FMA on the FP32 units).  Each thread runs CHAINS
// independent dependency chains so that latency is hidden and the units' issue rate bounds
// the loop; the grid fills every SM several times.
#include "common.cuh"
#include "df.cuh"

namespace cr {
namespace {

constexpr int CHAINS = 8;
constexpr int PROBE_THREADS = 256;

__global__ void __launch_bounds__(PROBE_THREADS) k_peak_dfma(int iters, double seed, double* sink) {
  double a[CHAINS];
#pragma unroll
  for (int q = 0; q < CHAINS; ++q) a[q] = seed + threadIdx.x * 1e-9 + q;
  const double m = 0.9999999, s = 1e-7;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int q = 0; q < CHAINS; ++q) a[q] = fma(a[q], m, s);
  }
  double r = 0.0;
#pragma unroll
  for (int q = 0; q < CHAINS; ++q) r += a[q];
  if (r == 12345.678) *sink = r;   // keeps the loop; never true for these inputs
}

__global__ void __launch_bounds__(PROBE_THREADS) k_peak_ffma(int iters, float seed, double* sink) {
  float a[CHAINS];
#pragma unroll
  for (int q = 0; q < CHAINS; ++q) a[q] = seed + threadIdx.x * 1e-6f + q;
  const float m = 0.9999f, s = 1e-4f;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int q = 0; q < CHAINS; ++q) a[q] = fmaf(a[q], m, s);
  }
  float r = 0.0f;
#pragma unroll
  for (int q = 0; q < CHAINS; ++q) r += a[q];
  if (r == 12345.678f) *sink = r;
}

// The diagonal executor's accumulate step: s + c += x * y with x, y double-float pairs (the
// high products summed by two-sum, all lower-order terms in the FP32 compensation).
__global__ void __launch_bounds__(PROBE_THREADS) k_peak_dfmac(int iters, float seed, double* sink) {
  float s[CHAINS], c[CHAINS];
#pragma unroll
  for (int q = 0; q < CHAINS; ++q) { s[q] = seed + q; c[q] = 0.0f; }
  // products near 1: the sums grow to about iters, far inside the FP32 range
  const df x = {1.0000001f + threadIdx.x * 1e-7f, 3e-9f}, y = {0.9999999f, -2e-9f};
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int q = 0; q < CHAINS; ++q) {
      const float p = __fmul_rn(x.hi, y.hi);
      float e = __fmaf_rn(x.hi, y.hi, -p);
      e = __fmaf_rn(x.hi, y.lo, e);
      e = __fmaf_rn(x.lo, y.hi, e);
      const float t = __fadd_rn(s[q], p);
      const float bb = __fsub_rn(t, s[q]);
      const float err = __fadd_rn(__fsub_rn(s[q], __fsub_rn(t, bb)), __fsub_rn(p, bb));
      s[q] = t;
      c[q] = __fadd_rn(c[q], __fadd_rn(err, e));
    }
  }
  float r = 0.0f;
#pragma unroll
  for (int q = 0; q < CHAINS; ++q) r += s[q] + c[q];
  if (r == 12345.678f) *sink = r;
}

// FP64 tensor-core MMA: D(8x8) = A(8x4) B(4x8) + C, FP64 throughout (mma.sync.m8n8k4).
__global__ void __launch_bounds__(PROBE_THREADS) k_peak_dmma(int iters, double seed, double* sink) {
  double acc[CHAINS][2];
#pragma unroll
  for (int q = 0; q < CHAINS; ++q) { acc[q][0] = seed + q; acc[q][1] = seed - q; }
  const double a = 1.0 + threadIdx.x * 1e-9, b = 0.999999;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int q = 0; q < CHAINS; ++q)
      asm volatile("mma.sync.aligned.m8n8k4.row.col.f64.f64.f64.f64 {%0, %1}, {%2}, {%3}, {%0, %1};"
                   : "+d"(acc[q][0]), "+d"(acc[q][1])
                   : "d"(a), "d"(b));
  }
  double r = 0.0;
#pragma unroll
  for (int q = 0; q < CHAINS; ++q) r += acc[q][0] + acc[q][1];
  if (r == 12345.678) *sink = r;
}

}  // namespace
}  // namespace cr

using namespace cr;

extern "C" cr_status cr_peak_probe(int kind, int iters, double* tflops, cr_stream stream) {
  if (!tflops || iters <= 0 || iters > (1 << 24)) return fail(CR_ERR_ARG, "cr_peak_probe: argument");
  int dev = 0, sms = 0;
  CR_CUDA(cudaGetDevice(&dev));
  CR_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int grid = sms * 8;
  static double* sink = nullptr;
  if (!sink) CR_CUDA(cudaMalloc(&sink, sizeof(double)));
  cudaEvent_t a = nullptr, b = nullptr;
  CR_CUDA(cudaEventCreate(&a));
  CR_CUDA(cudaEventCreate(&b));
  double flops_per_iter_thread = 0.0;
  auto launch = [&]() -> cudaError_t {
    switch (kind) {
      case CR_PEAK_DFMA: k_peak_dfma<<<grid, PROBE_THREADS, 0, stream>>>(iters, 1.0, sink); break;
      case CR_PEAK_FFMA: k_peak_ffma<<<grid, PROBE_THREADS, 0, stream>>>(iters, 1.0f, sink); break;
      case CR_PEAK_DF_MAC: k_peak_dfmac<<<grid, PROBE_THREADS, 0, stream>>>(iters, 1.0f, sink); break;
      case CR_PEAK_DMMA: k_peak_dmma<<<grid, PROBE_THREADS, 0, stream>>>(iters, 1.0, sink); break;
      default: return cudaErrorInvalidValue;
    }
    count_launch();
    return cudaGetLastError();
  };
  switch (kind) {
    case CR_PEAK_DFMA: case CR_PEAK_FFMA: case CR_PEAK_DF_MAC: flops_per_iter_thread = 2.0 * CHAINS; break;
    // one m8n8k4 per warp: 2 * 8 * 8 * 4 flops over 32 threads
    case CR_PEAK_DMMA: flops_per_iter_thread = 2.0 * 8 * 8 * 4 / 32.0 * CHAINS; break;
    default:
      cudaEventDestroy(a);
      cudaEventDestroy(b);
      return fail(CR_ERR_ARG, "cr_peak_probe: unknown kind");
  }
  cudaError_t e = launch();   // warm-up
  if (e == cudaSuccess) e = cudaEventRecord(a, stream);
  if (e == cudaSuccess) e = launch();
  if (e == cudaSuccess) e = cudaEventRecord(b, stream);
  if (e == cudaSuccess) e = cudaEventSynchronize(b);
  float ms = 0.0f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, a, b);
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  if (e != cudaSuccess) return cuda_fail(e, "cr_peak_probe");
  *tflops = (double)grid * PROBE_THREADS * iters * flops_per_iter_thread / (ms * 1e-3) / 1e12;
  return CR_OK;
}
