// Internal definitions shared by the translation units of libcr.so.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/cr.h"

namespace cr {

// ----------------------------------------------------------------- errors
void set_error(const std::string& msg);
cr_status fail(cr_status code, const std::string& msg);
cr_status cuda_fail(cudaError_t e, const char* what);

#define CR_CUDA(call)                                               \
  do {                                                              \
    cudaError_t e__ = (call);                                       \
    if (e__ != cudaSuccess) return ::cr::cuda_fail(e__, #call);     \
  } while (0)

void count_launch();

// Stream-ordered scratch from the library's memory pool of the current device, which keeps
// freed memory for the next call (unlimited release threshold) instead of returning it to
// the driver at every synchronisation; cr_workspace_trim returns it.
cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t stream);
void scratch_free(void* p, cudaStream_t stream);

// Process-wide options (cr_set_option): the limit of every bounded device-side wait of the
// factorisation, and the arithmetic of the diagonal-tile executor (CR_DIAG_*).
unsigned long long option_wait_ns();
int option_diag_arith();
int option_fp64_gemm();

// Opt-in device timing of named kernels (cr_timing_enable): a scope object records an event
// on the launch stream before and after the launch it brackets.
struct TimedScope {
  TimedScope(const char* name, cudaStream_t s);
  ~TimedScope();
  const char* name;
  cudaStream_t stream;
  cudaEvent_t start = nullptr;
};

// Every kernel launch is followed by this check, which also counts the launch.
#define CR_CHECK_LAUNCH(what)                                       \
  do {                                                              \
    ::cr::count_launch();                                           \
    cudaError_t e__ = cudaGetLastError();                           \
    if (e__ != cudaSuccess) return ::cr::cuda_fail(e__, what);      \
  } while (0)

#define CR_TRY(expr)                                                \
  do {                                                              \
    cr_status s__ = (expr);                                         \
    if (s__ != CR_OK) return s__;                                   \
  } while (0)

// Device status word bits (written by kernels, read by the host after a sync).
enum : int { DEV_ERR_TIMEOUT = 1, DEV_ERR_BOUNDS = 2 };

// ----------------------------------------------------------------- tile indexing
__host__ __device__ inline int tidx(int i, int j) { return i * (i + 1) / 2 + j; }  // i >= j

// Covariance model as the kernels see it.
// Doubles per tile statistics record: sum of squares, min, max, and the relative error bound
// of an FP32-evaluated record (0 for an exact record, infinity where no bound holds).
constexpr int STAT_W = 4;

struct CovK {
  int family;        // CR_COV_*
  int kind;          // Matern: 0 nu=1/2, 1 nu=3/2, 2 nu=5/2, 3 general (quadrature)
  double sigma2, inv_range, nu, nugget, tau2, norm;   // norm = 2^(1-nu) / Gamma(nu)
  int n_pred;
  int use_df;        // closed-form Matern orders: statistics and reduced-precision tiles in double-float
  float sig_hi, sig_lo, invr_hi, invr_lo;   // sigma2 and 1/range as double-float pairs
};

// Kernel-side view of the tile storage.
struct TileView {
  int n, nb, nt;
  int8_t* cls;     // [ntiles] CR_PREC_*
  int* i64;        // [ntiles] slot in pool64 or -1
  int* i32;        // [ntiles] slot in pool32 or -1
  int* hi16;       // [ntiles] FP16 slot of the value (FP16 class) or of its high part
  int* lo16;       // [ntiles] FP16 slot of the low part (FP32/FP64 classes) or -1
  double* pool64;
  float* pool32;
  __half* pool16;
};

}  // namespace cr

struct cr_tilemat_s {
  int n = 0, nb = 0, nt = 0, npad = 0, ntiles = 0;
  int device = 0;
  // covariance model, locations and tile statistics (tiles are generated on demand)
  double* xy = nullptr;          // n x 2 locations (copy of the caller's)
  float4* xy4 = nullptr;         // the locations as double-float pairs (x.hi, x.lo, y.hi, y.lo)
  cr::CovK covk{};
  double* stat_part = nullptr;   // ntiles * (nb/64) * STAT_W partials
  double* stats = nullptr;       // ntiles * STAT_W : sum of squares, min, max, error parameter
  cr_cov_params params{};
  bool built = false;
  std::vector<double> h_frob, h_vmin, h_vmax;   // ntiles each, after cr_tile_stats
  std::vector<double> h_stat_err;  // per tile: relative error bound of its statistics (0: exact)
  std::vector<char> h_stat_exact;  // per tile: statistics from the exact (double-float / FP64) pass
  int* d_refine = nullptr;         // tile list of the exact pass (ntiles ints)
  double* refine_part = nullptr;   // its partials: ntiles x (nb/16) x STAT_W
  bool stats_on_host = false;
  // precision map and class storage
  bool mapped = false;
  int amp = 1;
  double s = 1.0;
  int eA = 0;                     // power-of-two scale of FP32-class TRSM inputs
  cr_pmap_info pinfo{};
  std::vector<int8_t> h_cls;
  std::vector<int> h_i64, h_i32, h_hi16, h_lo16;
  int n64 = 0, n32 = 0, n16 = 0;  // slots per pool
  size_t cap64 = 0, cap32 = 0, cap16 = 0, cap_ws64 = 0, cap_w32 = 0;   // allocated elements, kept across maps
  int ws_hi0 = 0, ws_lo0 = 0, minv_hi = 0, minv_lo = 0;
  int* d_tables = nullptr;        // 4 ntiles ints (i64, i32, hi16, lo16) then ntiles class bytes
  int8_t* d_cls = nullptr;        // views into d_tables
  int *d_i64 = nullptr, *d_i32 = nullptr, *d_hi16 = nullptr, *d_lo16 = nullptr;
  double* pool64 = nullptr;
  float* pool32 = nullptr;
  __half* pool16 = nullptr;
  double* ws64 = nullptr;         // 2 * nt * nb * nb: FP64-class solve inputs (double-buffered by column parity)
  float* w32 = nullptr;           // 2 * nt * nb * nb: FP32 intermediate of FP16/FP32-class tiles (same)
  cudaStream_t s_hi = nullptr, s_lo = nullptr, s_mid = nullptr;   // critical chain / bulk updates / lookahead rows
  cudaStream_t s_gen = nullptr;   // tile generation ahead of the factorisation
  // the factorisation schedule's events and device lists, kept across calls (sized by capacity)
  std::vector<cudaEvent_t> sched_ev;
  int* sched_ints = nullptr;      // solve rows, then the generation list
  size_t sched_ints_cap = 0;
  void* sched_jobs = nullptr;     // job list, then the pair list
  size_t sched_jobs_cap = 0;
  double* minv = nullptr;         // 2 * nb * nb: inverse of the diagonal factor, by column parity
  double* minv_all = nullptr;     // nt * nb * nb: every diagonal factor's inverse (kept on request)
  double* scratch64 = nullptr;    // nb * nb: temporaries of the diagonal factorisation
  int* d_status = nullptr;        // [0] device error bits, [1] first failing column (1-based) or 0, [2] Minv exponent
  CUtensorMap tm_pool16;          // 3-D map over pool16 (slot, row, col)
  // simulation right-hand side B = fp16(M_rand / s), npad x M column-major
  __half* b16 = nullptr;
  size_t b16_elems = 0;
  __half* y16 = nullptr;          // FP16 destination of the per-product rounding mode (npad x M)
  size_t y16_elems = 0;
  int b16_M = -1;
  CUtensorMap tm_b16;
  double* bnorm_part = nullptr;   // per-block partial sums of ||B||_F^2
  // diagonal-tile dataflow factorisation: task list and flag scratch
  int4* diag_tasks = nullptr;
  int diag_ntasks = 0, diag_db = 0;
  int* diag_flags = nullptr;
  double* diag_pub = nullptr;     // the diagonal executor's publication buffers (diag_pub_doubles)
  double* minv_part = nullptr;    // per-block partial maxima of |L_jj^-1|
  float2* diag_df = nullptr;      // 2 * nb * nb double-float pairs: factor, then inverse, of the diagonal tile
  bool factored = false;
  int info = 0;

  cr::TileView view() const {
    cr::TileView v;
    v.n = n; v.nb = nb; v.nt = nt;
    v.cls = d_cls; v.i64 = d_i64; v.i32 = d_i32; v.hi16 = d_hi16; v.lo16 = d_lo16;
    v.pool64 = pool64; v.pool32 = pool32; v.pool16 = pool16;
    return v;
  }
};

namespace cr {
// Implemented in the translation units.
cr_status free_class_storage(cr_tilemat V);
cr_status make_tensor_map_3d_f16(CUtensorMap* tm, void* base, int inner, int rows, int slots,
                                 int box_inner, int box_rows);
cr_status make_tensor_map_2d_f16(CUtensorMap* tm, void* base, int inner, int outer, int ld,
                                 int box_inner, int box_outer);
}  // namespace cr
