// Status codes, error reporting, tile-matrix lifetime and TMA descriptor creation.
#include <stdio.h>

#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <vector>
#include <mutex>

#include "common.cuh"

namespace cr {

static thread_local std::string g_detail;
// Message set without allocating (a string with static storage), used by the allocation-free
// entry point; any other error clears it.
static thread_local const char* g_literal = nullptr;
static std::atomic<uint64_t> g_launches{0};

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static std::atomic<long long> g_opt_wait_us{2000000};
static std::atomic<int> g_opt_diag{CR_DIAG_AUTO};
static std::atomic<int> g_opt_gemm{CR_GEMM_DF};
unsigned long long option_wait_ns() { return 1000ull * (unsigned long long)g_opt_wait_us.load(std::memory_order_relaxed); }
int option_diag_arith() { return g_opt_diag.load(std::memory_order_relaxed); }
int option_fp64_gemm() { return g_opt_gemm.load(std::memory_order_relaxed); }

namespace {
struct TimingState {
  std::mutex mu;
  bool on = false;
  std::vector<cudaEvent_t> free_events;
  struct Pending { std::string name; cudaEvent_t a, b; };
  std::vector<Pending> pending;
  std::map<std::string, std::pair<double, uint64_t>> totals;
  // an event from the pool made by cr_timing_enable; when the pool runs dry the launch is
  // simply not timed (no event is created between launches)
  cudaEvent_t get() {
    if (free_events.empty()) return nullptr;
    cudaEvent_t e = free_events.back();
    free_events.pop_back();
    return e;
  }
  void fold() {
    for (auto& p : pending) {
      float ms = 0.0f;
      if (cudaEventSynchronize(p.b) == cudaSuccess && cudaEventElapsedTime(&ms, p.a, p.b) == cudaSuccess) {
        auto& t = totals[p.name];
        t.first += ms;
        t.second += 1;
      }
      free_events.push_back(p.a);
      free_events.push_back(p.b);
    }
    pending.clear();
  }
};
TimingState& timing() {
  static TimingState t;
  return t;
}
}  // namespace

TimedScope::TimedScope(const char* n, cudaStream_t s) : name(n), stream(s) {
  auto& T = timing();
  std::lock_guard<std::mutex> lk(T.mu);
  if (!T.on) return;
  start = T.get();
  if (start && cudaEventRecord(start, stream) != cudaSuccess) start = nullptr;
}

TimedScope::~TimedScope() {
  if (!start) return;
  auto& T = timing();
  std::lock_guard<std::mutex> lk(T.mu);
  cudaEvent_t stop = T.get();
  if (stop && cudaEventRecord(stop, stream) == cudaSuccess) T.pending.push_back({name, start, stop});
  else T.free_events.push_back(start);
}

void set_error(const std::string& msg) {
  g_literal = nullptr;
  g_detail = msg;
}

cr_status fail_literal(cr_status code, const char* msg) {
  g_literal = msg;
  return code;
}

cr_status fail(cr_status code, const std::string& msg) {
  g_literal = nullptr;
  g_detail = msg;
  return code;
}

cr_status cuda_fail(cudaError_t e, const char* what) {
  g_literal = nullptr;
  g_detail = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return e == cudaErrorMemoryAllocation ? CR_ERR_NOMEM : CR_ERR_CUDA;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point, so the library does not
// link libcuda directly and loads on machines without a driver.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

cr_status make_tensor_map_3d_f16(CUtensorMap* tm, void* base, int inner, int rows, int slots, int box_inner,
                                 int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(CR_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)slots};
  cuuint64_t strides[2] = {(cuuint64_t)inner * 2, (cuuint64_t)inner * rows * 2};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(CR_ERR_CUDA, "cuTensorMapEncodeTiled (3d) failed: " + std::to_string((int)r));
  return CR_OK;
}

cr_status make_tensor_map_2d_f16(CUtensorMap* tm, void* base, int inner, int outer, int ld, int box_inner,
                                 int box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(CR_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(CR_ERR_CUDA, "cuTensorMapEncodeTiled (2d) failed: " + std::to_string((int)r));
  return CR_OK;
}

template <class T>
static void dfree(T*& p) {
  if (p) cudaFree((void*)p);
  p = nullptr;
}

cr_status free_class_storage(cr_tilemat V) {
  dfree(V->d_tables);
  V->d_cls = nullptr; V->d_i64 = V->d_i32 = V->d_hi16 = V->d_lo16 = nullptr;
  dfree(V->pool64); dfree(V->pool32); dfree(V->pool16); dfree(V->ws64); dfree(V->w32);
  V->cap64 = V->cap32 = V->cap16 = V->cap_ws64 = V->cap_w32 = 0;
  V->mapped = false;
  V->factored = false;
  return CR_OK;
}

}  // namespace cr

using namespace cr;

extern "C" const char* cr_status_str(cr_status code) {
  switch (code) {
    case CR_OK: return "CR_OK";
    case CR_ERR_ARG: return "CR_ERR_ARG";
    case CR_ERR_CUDA: return "CR_ERR_CUDA";
    case CR_ERR_NOMEM: return "CR_ERR_NOMEM";
    case CR_ERR_NOT_SPD: return "CR_ERR_NOT_SPD";
    case CR_ERR_EMPTY_SAMPLE: return "CR_ERR_EMPTY_SAMPLE";
    case CR_ERR_NONPOS_MSPE: return "CR_ERR_NONPOS_MSPE";
    case CR_ERR_TIMEOUT: return "CR_ERR_TIMEOUT";
    case CR_ERR_STATE: return "CR_ERR_STATE";
    case CR_ERR_NOT_IMPLEMENTED: return "CR_ERR_NOT_IMPLEMENTED";
    case CR_ERR_RANGE: return "CR_ERR_RANGE";
    default: return "CR_ERR_UNKNOWN";
  }
}

extern "C" const char* cr_last_error_detail(void) { return g_literal ? g_literal : g_detail.c_str(); }

extern "C" cr_status cr_version(int* major, int* minor) {
  if (major) *major = 0;
  if (minor) *minor = 1;
  return CR_OK;
}

extern "C" cr_status cr_timing_enable(int on) {
  auto& T = timing();
  std::lock_guard<std::mutex> lk(T.mu);
  if (on) {
    // events are created here, not between launches: creating them while the library
    // enqueues its schedule would hold back the launches it is timing
    T.fold();
    while (T.free_events.size() < 16384) {
      cudaEvent_t e = nullptr;
      if (cudaEventCreate(&e) != cudaSuccess) return fail(CR_ERR_CUDA, "cr_timing_enable: cudaEventCreate");
      T.free_events.push_back(e);
    }
  }
  T.on = on != 0;
  return CR_OK;
}

extern "C" cr_status cr_timing_read(const char* kernel, double* total_ms, uint64_t* launches) {
  if (!kernel || !total_ms || !launches) return fail(CR_ERR_ARG, "cr_timing_read: NULL argument");
  auto& T = timing();
  std::lock_guard<std::mutex> lk(T.mu);
  T.fold();
  auto it = T.totals.find(kernel);
  *total_ms = it == T.totals.end() ? 0.0 : it->second.first;
  *launches = it == T.totals.end() ? 0 : it->second.second;
  return CR_OK;
}

extern "C" cr_status cr_timing_reset(void) {
  auto& T = timing();
  std::lock_guard<std::mutex> lk(T.mu);
  T.fold();
  T.totals.clear();
  return CR_OK;
}

extern "C" cr_status cr_set_option(int option, long long value) {
  if (option == CR_OPT_WAIT_LIMIT_US) {
    if (value < 0 || value > 600000000ll) return fail(CR_ERR_ARG, "cr_set_option: wait limit outside [0, 600 s]");
    g_opt_wait_us.store(value);
    return CR_OK;
  }
  if (option == CR_OPT_DIAG_ARITH) {
    if (value != CR_DIAG_AUTO && value != CR_DIAG_FP64 && value != CR_DIAG_DF)
      return fail(CR_ERR_ARG, "cr_set_option: diagonal arithmetic must be CR_DIAG_AUTO, CR_DIAG_FP64 or CR_DIAG_DF");
    g_opt_diag.store((int)value);
    return CR_OK;
  }
  if (option == CR_OPT_FP64_GEMM) {
    if (value != CR_GEMM_DF && value != CR_GEMM_OZAKI)
      return fail(CR_ERR_ARG, "cr_set_option: FP64 product arithmetic must be CR_GEMM_DF or CR_GEMM_OZAKI");
    g_opt_gemm.store((int)value);
    return CR_OK;
  }
  return fail(CR_ERR_ARG, "cr_set_option: unknown option");
}

extern "C" cr_status cr_get_option(int option, long long* value) {
  if (!value) return fail(CR_ERR_ARG, "cr_get_option: NULL value");
  if (option == CR_OPT_WAIT_LIMIT_US) *value = g_opt_wait_us.load();
  else if (option == CR_OPT_DIAG_ARITH) *value = g_opt_diag.load();
  else if (option == CR_OPT_FP64_GEMM) *value = g_opt_gemm.load();
  else return fail(CR_ERR_ARG, "cr_get_option: unknown option");
  return CR_OK;
}

namespace cr {
namespace {
std::mutex g_pool_mu;
cudaMemPool_t g_pool[64] = {};
}  // namespace

cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaMemPool_t pool = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_pool_mu);
    if (!g_pool[dev]) {
      cudaMemPoolProps props = {};
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      if ((e = cudaMemPoolCreate(&g_pool[dev], &props)) != cudaSuccess) {
        g_pool[dev] = nullptr;
        return e;
      }
      uint64_t keep = ~0ull;
      if ((e = cudaMemPoolSetAttribute(g_pool[dev], cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) return e;
    }
    pool = g_pool[dev];
  }
  return cudaMallocFromPoolAsync(p, bytes, pool, stream);
}

void scratch_free(void* p, cudaStream_t stream) {
  if (p) cudaFreeAsync(p, stream);
}
}  // namespace cr

extern "C" cr_status cr_workspace_trim(void) {
  std::lock_guard<std::mutex> lk(g_pool_mu);
  for (cudaMemPool_t pool : g_pool)
    if (pool) CR_CUDA(cudaMemPoolTrimTo(pool, 0));
  return CR_OK;
}

extern "C" cr_status cr_kernel_launches(uint64_t* count) {
  if (!count) return fail(CR_ERR_ARG, "cr_kernel_launches: NULL");
  *count = g_launches.load(std::memory_order_relaxed);
  return CR_OK;
}

extern "C" cr_status cr_tilemat_create(int n, int nb, cr_tilemat* out) {
  if (!out) return fail(CR_ERR_ARG, "cr_tilemat_create: NULL out");
  *out = nullptr;
  if (n <= 0 || nb < 128 || nb > 1024 || nb % 128 != 0) return fail(CR_ERR_ARG, "cr_tilemat_create: n > 0, nb in {128..1024} step 128");
  cr_tilemat V = new cr_tilemat_s();
  V->n = n;
  V->nb = nb;
  V->nt = (n + nb - 1) / nb;
  V->npad = V->nt * nb;
  V->ntiles = V->nt * (V->nt + 1) / 2;
  cudaGetDevice(&V->device);
  const size_t tile = (size_t)nb * nb;
  cudaError_t e;
  if ((e = cudaMalloc(&V->xy, (size_t)n * 2 * sizeof(double))) != cudaSuccess ||
      (e = cudaMalloc(&V->xy4, (size_t)n * sizeof(float4))) != cudaSuccess ||
      (e = cudaMalloc(&V->stat_part, (size_t)V->ntiles * (nb / 64) * STAT_W * sizeof(double))) != cudaSuccess ||
      (e = cudaMalloc(&V->stats, (size_t)V->ntiles * STAT_W * sizeof(double))) != cudaSuccess ||
      (e = cudaMalloc(&V->minv, 2 * tile * sizeof(double))) != cudaSuccess ||
      (e = cudaMalloc(&V->scratch64, tile * sizeof(double))) != cudaSuccess ||
      (e = cudaMalloc(&V->d_status, 4 * sizeof(int))) != cudaSuccess) {
    cr_status st = cuda_fail(e, "cr_tilemat_create: cudaMalloc");
    cr_tilemat_destroy(V);
    return st;
  }
  cudaMemset(V->d_status, 0, 4 * sizeof(int));
  *out = V;
  return CR_OK;
}

extern "C" cr_status cr_tilemat_destroy(cr_tilemat V) {
  if (!V) return CR_OK;
  cudaSetDevice(V->device);
  cudaDeviceSynchronize();
  free_class_storage(V);
  dfree(V->b16); dfree(V->y16); dfree(V->bnorm_part); dfree(V->minv_all); dfree(V->diag_tasks); dfree(V->diag_flags); dfree(V->diag_pub); dfree(V->minv_part); dfree(V->diag_df);
  dfree(V->xy); dfree(V->xy4); dfree(V->stat_part); dfree(V->d_refine); dfree(V->refine_part); dfree(V->stats); dfree(V->minv); dfree(V->scratch64); dfree(V->d_status);
  if (V->s_hi) cudaStreamDestroy(V->s_hi);
  if (V->s_lo) cudaStreamDestroy(V->s_lo);
  if (V->s_mid) cudaStreamDestroy(V->s_mid);
  if (V->s_gen) cudaStreamDestroy(V->s_gen);
  for (cudaEvent_t e : V->sched_ev) cudaEventDestroy(e);
  dfree(V->sched_ints);
  if (V->sched_jobs) cudaFree(V->sched_jobs);
  delete V;
  return CR_OK;
}

extern "C" cr_status cr_tilemat_info(cr_tilemat V, int* n, int* nb, int* nt) {
  if (!V) return fail(CR_ERR_ARG, "cr_tilemat_info: NULL handle");
  if (n) *n = V->n;
  if (nb) *nb = V->nb;
  if (nt) *nt = V->nt;
  return CR_OK;
}

// ---------------------------------------------------------------------------------------
// Spatial ordering of the locations (host only).  The pages' precision maps (Section VI-D,
// Fig. 5) are banded: nearby sites sit in nearby tiles.  The locations are therefore put in
// Z-order (Morton order) before the covariance is built: each coordinate is quantised to
// 16 bits, q = clamp(floor(65536 x), 0, 65535), the key interleaves the bits of q_x (even
// positions) and q_y (odd positions), and the permutation sorts the keys stably (equal keys
// keep their input order).
namespace cr {
namespace {
uint32_t spread16(uint32_t v) {
  v &= 0xffffu;
  v = (v | (v << 8)) & 0x00ff00ffu;
  v = (v | (v << 4)) & 0x0f0f0f0fu;
  v = (v | (v << 2)) & 0x33333333u;
  v = (v | (v << 1)) & 0x55555555u;
  return v;
}
uint32_t quant16(double x) {
  const double q = floor(x * 65536.0);   // exact: a power-of-two scale, then an integer part
  return q <= 0.0 ? 0u : (q >= 65535.0 ? 65535u : (uint32_t)q);
}
}  // namespace
}  // namespace cr

#include <algorithm>
#include <cmath>

extern "C" cr_status cr_morton_order(const double* h_xy, int n, int32_t* h_perm) {
  using namespace cr;
  if (n < 0 || (n > 0 && (!h_xy || !h_perm))) return fail(CR_ERR_ARG, "cr_morton_order: argument");
  std::vector<uint32_t> key((size_t)n);
  for (int i = 0; i < n; ++i) {
    const double x = h_xy[2 * (size_t)i], y = h_xy[2 * (size_t)i + 1];
    if (std::isnan(x) || std::isnan(y)) return fail(CR_ERR_ARG, "cr_morton_order: NaN coordinate at site " + std::to_string(i));
    key[i] = spread16(quant16(x)) | (spread16(quant16(y)) << 1);
  }
  for (int i = 0; i < n; ++i) h_perm[i] = i;
  std::stable_sort(h_perm, h_perm + n, [&](int32_t a, int32_t b) { return key[a] < key[b]; });
  return CR_OK;
}
