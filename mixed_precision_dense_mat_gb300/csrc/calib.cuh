// Calibration scan interfaces (calib.cu).
#pragma once
#include "common.cuh"

namespace cr {

constexpr int SCAN_THREADS = 256;
constexpr int SCAN_ROWS = 2048;   // rows per CTA (8 per thread)
constexpr int SCAN_COLS = 32;     // simulation columns per CTA

// Device scratch of one calibration: t (n_p), psi/phi (M), per-row-block partials
// (ceil(n_p / SCAN_ROWS) x M each) and an MSPE flag.
struct CalibScratch {
  double* t = nullptr;
  double* psi = nullptr;
  double* phi = nullptr;
  double* psi_part = nullptr;
  double* phi_part = nullptr;
  int* bad = nullptr;
};

cr_status calibrate_core(const double* d_S, int lds, int n_p, int M, const double* d_zhat, const double* d_v, double u,
                         double level, uint8_t* d_cin, uint8_t* d_cout, int32_t* d_count, double* d_psi, double* d_phi,
                         cr_calib_info* out, cudaStream_t stream, const CalibScratch& sc, int neg);

// Tail of a calibration: partials (nrb x M) -> psi, phi -> host quantiles -> regions from sc.t.
cr_status calibrate_finish(const double* psi_part, const double* phi_part, int nrb, int n_p, int M, double level,
                           const CalibScratch& sc, uint8_t* d_cin, uint8_t* d_cout, double* d_psi, double* d_phi,
                           cr_calib_info* out, cudaStream_t stream);

// Conditioning correction S = M_p + W^T (y_o 1^T - M_o) in double-float arithmetic, into d_S
// (stream-ordered; allocates its double-float copies of W and R with cudaMallocAsync).
cr_status correction_async(const double* d_W, int ldw, const double* d_yo, const double* d_Y, int ldy, int n_p, int n_o,
                           int M, double* d_S, int lds, cudaStream_t stream);

// Cout = Cin + alpha A^T B (A: K x m, B: K x n, column-major FP64; Cin NULL for zero; Cout may
// be Cin) by the Ozaki scheme with S slices of 6 bits (2 <= S <= 10) on the FP16 tensor cores
// (ozaki.cu); pool scratch, asynchronous.
cr_status ozaki_gemm_tn(const double* A, int lda, const double* B, int ldb, int K, int m, int n, double alpha,
                        const double* Cin, int ldci, double* Cout, int ldco, int S, cudaStream_t stream);

// The conditioning correction S = M_p + W^T (y_o 1^T - M_o) by the Ozaki product on the FP16
// tensor cores (ozaki.cu); stream-ordered scratch, asynchronous.  The _prepared form takes W's
// slices from a cr_weights handle.
cr_status ozaki_correction(const double* d_W, int ldw, const double* d_yo, const double* d_Y, int ldy, int n_p, int n_o,
                           int M, double* d_S, int lds, cudaStream_t stream);
cr_status ozaki_correction_prepared(cr_weights w, const double* d_yo, const double* d_Y, int ldy, int M, double* d_S, int lds,
                                    cudaStream_t stream);

}  // namespace cr

// Kriging weights prepared for the Ozaki correction (cr_weights_prepare): W's column exponents
// and slices, with the geometry they were cut for.
struct cr_weights_s {
  int device = 0, n_o = 0, n_p = 0, slices = 0;
  int* Ea = nullptr;
  __half* As = nullptr;
};
