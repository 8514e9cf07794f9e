// Parameters of the tensor-core tile kernel (tc.cu).
#pragma once
#include "common.cuh"

namespace cr {

constexpr int TC_BM = 128, TC_BN = 256, TC_BK = 64;            // output block 128 x 256, K chunk 64
constexpr int TC_STAGES = 4;
constexpr int TC_STAGE_BYTES = (TC_BM + TC_BN) * TC_BK * 2;     // A and B, FP16, 48 KB
constexpr int TC_THREADS = 192;
constexpr int TC_KT_INTS = 5;                                   // ints per k-term table entry
constexpr int TC_TMEM_COLS = 2 * TC_BN;                         // two accumulators
constexpr int TC_EPI_BYTES = 4 * 32 * 33 * 4;                   // epilogue staging, one 32 x 32 chunk per warp
// stages, 1 KB alignment slack, barriers, epilogue staging; the two k-term tables come on top
constexpr size_t TC_SMEM = (size_t)TC_STAGES * TC_STAGE_BYTES + 1024 + 256 + TC_EPI_BYTES;

// TC_UPD_OLD: products k in [kbeg, kend) from the class storage into the intermediate
//             (FP32 workspace w32, FP64 workspace ws64, diagonal FP64 in place);
// TC_UPD_NEW: products k in [kbeg, kend) from the intermediate into the solve inputs
//             (FP16 / FP16 high-low workspace slots, ws64, diagonal in place).
enum { TC_UPD_OLD = 0, TC_TRSM = 1, TC_TRMM = 2, TC_UPD_NEW = 3 };

struct TcParams {
  TileView v;
  int mode;
  int j;              // tile column (update / triangular solve)
  int kbeg, kend;     // update terms
  float* w32;         // FP32 intermediate of FP16/FP32-class tiles (tile row i at i nb^2)
  const int* rows;    // tile rows of this launch (triangular solve)
  int row0, nrows;    // updates: tile rows row0 .. row0+nrows-1 (row0 = j includes the diagonal tile);
                      // triangular solve: nrows entries of rows
  int ws_hi0, ws_lo0, minv_hi, minv_lo;
  int eA;             // FP32-class inputs were scaled by 2^-eA
  const int* status;  // status[2]: exponent eM of the scaled inverse factor
  int* err;           // device error bits
  double* ws64;       // FP64-class triangular-solve inputs
  double* Y;          // simulation output (n x M column-major)
  int ldy, M, ncb, flags;
  __half* y16;        // CR_TRMM_FP16_PER_GEMM: FP16 destination between products, one 128 x 256
                      // row-major tile per output block (npad x ncb 256 halves)
  int max_ctas;       // grid cap (0: one CTA per SM); background launches leave SMs free for
                      // the critical stream, whose CTAs cannot preempt persistent ones
  int esplit;         // update and solve modes: 1, or CTAs per output block (each repeats the
                      // block's products and writes 1/esplit of its columns), which spreads
                      // the epilogue of a launch with few blocks over more SMs
};

// Launches the persistent kernel over every output block of the launch described by p (one
// CTA per SM at most).
cr_status tc_launch(const TcParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, cudaStream_t stream);

}  // namespace cr
