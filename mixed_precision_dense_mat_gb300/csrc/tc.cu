// Tensor-core tile kernel: tcgen05.mma kind::f16 with FP32 accumulation in TMEM, fed by TMA
// through a 4-stage shared-memory ring; persistent (one CTA per SM at most, output blocks
// taken round-robin), warp-specialised (warp 0 TMA producer and k-term table, warp 1 MMA
// issuer and TMEM owner, warps 2-5 epilogue), with two TMEM accumulators so that the
// epilogue of one 128 x 256 output block overlaps the main loop of the next.
//
// Three uses, all from "Mixed-Precision GPU Acceleration for Confidence Regions of Spatial
// Excursion Sets":
//  TC_UPD_*   Cholesky column update A_ij -= sum_k L_ik L_jk^T (Section IV-B) for the
//             products whose lowest operand precision is FP16 (one FP16 MMA) or FP32 (three
//             MMAs on FP16 high/low parts: hi*hi + hi*lo + lo*hi).  Products between FP64
//             tiles are left to the FP64 kernel.
//  TC_TRSM    L_ij = A_ij L_jj^-T for FP16/FP32-class tiles, as A_ij times the FP64 inverse of
//             the diagonal factor split into FP16 high/low parts (2^eM scaled).
//  TC_TRMM    Alg.1: Y_i = sum_{k<i} cast16(L_ik) B_k + L_ii B_i with B = fp16(M_rand / s); the
//             diagonal factor enters as its FP16 high/low split (FP32-class accuracy, Alg.1
//             steps 11-13), every off-diagonal factor tile as its FP16 cast (step 15).
#include "common.cuh"
#include "ptx.cuh"
#include <algorithm>

#include "tc.cuh"

namespace cr {

namespace {

struct Job {
  int i, rb, cb;
};

__host__ __device__ inline int tc_nsbm(int nb) { return nb / TC_BM; }
__host__ __device__ inline int tc_nsbn(int nb) { return (nb + TC_BN - 1) / TC_BN; }
// output blocks (rb, cb) of a diagonal tile that hold part of its lower triangle
__host__ __device__ inline int tc_diag_blocks(int nb) {
  int d = 0;
  for (int rb = 0; rb < tc_nsbm(nb); ++rb) d += ((rb + 1) * TC_BM + TC_BN - 1) / TC_BN;
  return d;
}

__host__ __device__ inline int tc_num_blocks(const TcParams& p) {
  const int nb = p.v.nb, per = tc_nsbm(nb) * tc_nsbn(nb);
  if (p.mode == TC_TRMM) return p.v.nt * tc_nsbm(nb) * p.ncb;
  if (p.mode == TC_TRSM) return p.nrows * per;
  if (p.nrows <= 0) return 0;
  return p.row0 == p.j ? tc_diag_blocks(nb) + (p.nrows - 1) * per : p.nrows * per;
}

__device__ __forceinline__ Job decode(const TcParams& p, int t) {
  const int nb = p.v.nb, nsbm = tc_nsbm(nb), nsbn = tc_nsbn(nb);
  Job jb;
  if (p.mode == TC_TRMM) {
    const int per_row = nsbm * p.ncb;
    jb.i = p.v.nt - 1 - t / per_row;   // longest K-chains first
    const int rem = t % per_row;
    jb.rb = rem / p.ncb;
    jb.cb = rem % p.ncb;
  } else if (p.mode == TC_TRSM) {
    const int per = nsbm * nsbn;
    jb.i = p.rows[t / per];
    jb.rb = (t % per) / nsbn;
    jb.cb = (t % per) % nsbn;
  } else {
    const int d = p.row0 == p.j ? tc_diag_blocks(nb) : 0;
    if (t < d) {
      // diagonal tile: the blocks of row rb that reach the lower triangle
      jb.i = p.j;
      int rb = 0, left = t;
      while (true) {
        const int in_row = ((rb + 1) * TC_BM + TC_BN - 1) / TC_BN;
        if (left < in_row) break;
        left -= in_row;
        ++rb;
      }
      jb.rb = rb;
      jb.cb = left;
    } else {
      const int per = nsbm * nsbn, u = t - d;
      jb.i = p.row0 + (d > 0 ? 1 : 0) + u / per;
      jb.rb = (u % per) / nsbn;
      jb.cb = (u % per) % nsbn;
    }
  }
  return jb;
}

// Per-k metadata of one output block, gathered by the 32 lanes of warp 0 into shared memory
// so that the step enumeration below does no global loads: for the update modes entry
// k - kbeg holds (product class, A hi slot, B hi slot, A lo slot, B lo slot); for the
// simulation multiply entry k holds the slot of the factor tile (i, k) in field 1 and the slot
// of its low part in field 3 (-1 for FP16-class tiles, which have none).
__device__ __forceinline__ void fill_ktable(const TcParams& p, const Job& jb, int* kt) {
  const TileView& v = p.v;
  const int lane = threadIdx.x & 31;
  if (p.mode == TC_UPD_OLD || p.mode == TC_UPD_NEW) {
    const int i = jb.i, j = p.j;
    const int cd = v.cls[tidx(i, j)];
    for (int k = p.kbeg + lane; k < p.kend; k += 32) {
      const int ti = tidx(i, k), tj = tidx(j, k);
      const int pc = max(cd, max((int)v.cls[ti], (int)v.cls[tj]));
      int* e = kt + TC_KT_INTS * (k - p.kbeg);
      e[0] = pc;
      e[1] = v.hi16[ti];
      e[2] = v.hi16[tj];
      e[3] = pc == CR_PREC_FP32 ? v.lo16[ti] : 0;
      e[4] = pc == CR_PREC_FP32 ? v.lo16[tj] : 0;
    }
  } else if (p.mode == TC_TRMM) {
    const int i = jb.i;
    for (int k = lane; k <= i; k += 32) {
      int* e = kt + TC_KT_INTS * k;
      e[1] = v.hi16[tidx(i, k)];
      e[3] = v.lo16[tidx(i, k)];
    }
  }
}

// Enumerates the pipeline steps of one output block.  Each step is one 64-wide K chunk of an
// (A, B) pair of FP16 operands; f(a_slot, a_k, b_slot, b_k, b_row).  A is read from the FP16
// tile pool at rows [rb*128, +128); B (256 rows from b_row) from the pool (b_slot >= 0) or
// from the 2-D right-hand-side map (b_slot < 0, b_k the global row of the simulation
// matrix).  kt is the table of fill_ktable.  Returns the number of steps.
// seg (simulation multiply with CR_TRMM_FP16_PER_GEMM): -1 enumerates the whole chain; 0 only
// the diagonal factor tile's product; s >= 1 only the product of the factor tile k = i - s.
template <class F>
__device__ __forceinline__ int for_each_step(const TcParams& p, const Job& jb, const int* kt, F&& f, int seg = -1) {
  const TileView& v = p.v;
  const int nq = v.nb / TC_BK;
  const int brow = jb.cb * TC_BN;
  int s = 0;
  if (p.mode == TC_UPD_OLD || p.mode == TC_UPD_NEW) {
    for (int k = p.kbeg; k < p.kend; ++k) {
      const int* e = kt + TC_KT_INTS * (k - p.kbeg);
      const int pc = e[0];
      if (pc == CR_PREC_FP64) continue;
      const int ahi = e[1], bhi = e[2];
      if (pc == CR_PREC_FP16) {
        for (int q = 0; q < nq; ++q, ++s) f(ahi, q * TC_BK, bhi, q * TC_BK, brow);
      } else {
        const int alo = e[3], blo = e[4];
        for (int q = 0; q < nq; ++q) {
          f(ahi, q * TC_BK, bhi, q * TC_BK, brow);
          f(ahi, q * TC_BK, blo, q * TC_BK, brow);
          f(alo, q * TC_BK, bhi, q * TC_BK, brow);
          s += 3;
        }
      }
    }
  } else if (p.mode == TC_TRSM) {
    const int i = jb.i;
    const int cd = v.cls[tidx(i, p.j)];
    const int nqk = min(nq, (jb.cb + 1) * (TC_BN / TC_BK));   // the inverse factor is lower triangular
    const int wh = p.ws_hi0 + i, wl = p.ws_lo0 + i;
    for (int q = 0; q < nqk; ++q) {
      f(wh, q * TC_BK, p.minv_hi, q * TC_BK, brow);
      f(wh, q * TC_BK, p.minv_lo, q * TC_BK, brow);
      s += 2;
      if (cd == CR_PREC_FP32) {
        f(wl, q * TC_BK, p.minv_hi, q * TC_BK, brow);
        ++s;
      }
    }
  } else {
    const int i = jb.i;
    const bool split = (p.flags & CR_TRMM_SPLIT_L) != 0;
    for (int k = 0; k < i; ++k) {
      if (seg >= 0 && k != i - seg) continue;
      const int a = kt[TC_KT_INTS * k + 1], alo = split ? kt[TC_KT_INTS * k + 3] : -1;
      for (int q = 0; q < nq; ++q, ++s) {
        f(a, q * TC_BK, -1, k * v.nb + q * TC_BK, brow);
        if (alo >= 0) {   // the tile's low part (FP32/FP64 class)
          f(alo, q * TC_BK, -1, k * v.nb + q * TC_BK, brow);
          ++s;
        }
      }
    }
    const int nqd = (jb.rb + 1) * (TC_BM / TC_BK);    // the diagonal factor is lower triangular
    const int dh = kt[TC_KT_INTS * i + 1], dl = kt[TC_KT_INTS * i + 3];
    for (int q = 0; q < (seg > 0 ? 0 : nqd); ++q) {
      f(dh, q * TC_BK, -1, i * v.nb + q * TC_BK, brow);
      f(dl, q * TC_BK, -1, i * v.nb + q * TC_BK, brow);
      s += 2;
    }
  }
  return s;
}

struct NoOp {
  __device__ void operator()(int, int, int, int, int) const {}
};

// The jobs of one CTA: output blocks t = blockIdx.x, + gridDim.x, ...; with
// CR_TRMM_FP16_PER_GEMM each block of tile row i is i + 1 consecutive jobs (segments: the
// diagonal product, then k = i-1 down to 0), each with its own accumulator and epilogue, so
// that the FP16 destination is rounded after every product as in Alg.1's task sequence.
struct JobIter {
  int t, seg, nseg, nblocks;
  bool perk, started;
  __device__ JobIter(const TcParams& p, int nb_)
      : t(blockIdx.x), seg(-1), nseg(1), nblocks(nb_),
        perk(p.mode == TC_TRMM && (p.flags & CR_TRMM_FP16_PER_GEMM) != 0), started(false) {}
  __device__ bool next(const TcParams& p) {
    if (!started) {
      started = true;
    } else if (perk && seg + 1 < nseg) {
      ++seg;
      return true;
    } else {
      t += gridDim.x;
    }
    if (t >= nblocks) return false;
    seg = perk ? 0 : -1;
    nseg = perk ? decode(p, t).i + 1 : 1;
    return true;
  }
};

// FP32 -> FP64 widening from the IEEE 754 fields (exponent rebiased by 1023 - 127, fraction
// shifted up by 29 bits) on the integer units: on GB300 the conversion instruction issues on
// the slow FP64/conversion pipe, which bounds the epilogues that widen every accumulator.
// Zeros, subnormals and non-finite values (rare here) use the conversion instruction.
__device__ __forceinline__ double widen(float f) {
  const unsigned u = __float_as_uint(f);
  const unsigned ex = (u >> 23) & 0xffu;
  if (__builtin_expect(ex == 0u || ex == 0xffu, 0)) return (double)f;
  const unsigned hi = (u & 0x80000000u) | ((ex + (1023u - 127u)) << 20) | ((u & 0x7fffffu) >> 3);
  return __hiloint2double((int)hi, (int)(u << 29));
}

// Output of the simulation multiply for the thread's row r_local and 16 columns from c0:
// Y is column-major, so the 32 lanes of a warp (32 consecutive rows) write contiguously.
__device__ __forceinline__ void trmm_store(const TcParams& p, const Job& jb, int r_local, int c0, const float* acc) {
  const TileView& v = p.v;
  const int row = jb.i * v.nb + jb.rb * TC_BM + r_local;
  if (row >= v.n) return;
  const bool f16 = (p.flags & CR_TRMM_FP16_DEST) != 0;
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int col = jb.cb * TC_BN + c0 + q;
    if (col < p.M) {
      const float a = f16 ? __half2float(__float2half_rn(acc[q])) : acc[q];
      p.Y[(size_t)col * p.ldy + row] = widen(a);
    }
  }
}

// CR_TRMM_FP16_PER_GEMM: segment seg of nseg of output block t's products.  The running
// result is kept in the FP16 destination y16 and rounded after every product:
// y = fp16(y + acc) (y = 0 before the first); the last segment widens y into Y.  y16 holds
// each output block as its own 128 x 256 row-major FP16 tile (block t at t 128 256), so a
// thread's 16 columns are two 16-byte words.
__device__ __forceinline__ void trmm_store_per_gemm(const TcParams& p, const Job& jb, int t, int r_local, int c0,
                                                    const float* acc, int seg, int nseg) {
  const TileView& v = p.v;
  const int row = jb.i * v.nb + jb.rb * TC_BM + r_local;
  if (row >= v.n) return;
  uint4* y = reinterpret_cast<uint4*>(p.y16 + ((size_t)t * TC_BM + r_local) * TC_BN + c0);
  unsigned w[8];   // 16 FP16 values as 8 packed pairs
  if (seg == 0) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const __half2 h = __floats2half2_rn(acc[2 * q], acc[2 * q + 1]);
      memcpy(&w[q], &h, 4);
    }
  } else {
    const uint4 a = y[0], b = y[1];
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      __half2 h;
      memcpy(&h, &w[q], 4);
      const float2 f = __half22float2(h);
      h = __floats2half2_rn(f.x + acc[2 * q], f.y + acc[2 * q + 1]);
      memcpy(&w[q], &h, 4);
    }
  }
  if (seg + 1 < nseg) {
    y[0] = make_uint4(w[0], w[1], w[2], w[3]);
    y[1] = make_uint4(w[4], w[5], w[6], w[7]);
    return;
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    __half2 h;
    memcpy(&h, &w[q], 4);
    const float2 f = __half22float2(h);
    const int col = jb.cb * TC_BN + c0 + 2 * q;
    if (col < p.M) p.Y[(size_t)col * p.ldy + row] = widen(f.x);
    if (col + 1 < p.M) p.Y[(size_t)(col + 1) * p.ldy + row] = widen(f.y);
  }
}

// Where the epilogue of a tile-update or triangular-solve block reads and writes; resolved
// once per block.  All tiles are row-major nb x nb; off is the element offset in the tile.
enum {
  EK_OLD64,   // dst64 = src64 - acc          (diagonal in place, or FP64 class into ws64)
  EK_OLD32,   // f32 = src32 - acc            (FP32 class into w32)
  EK_OLD16,   // f32 = src16 - acc            (FP16 class into w32)
  EK_NEW64,   // dst64 -= acc
  EK_NEW32,   // w = (w32 - acc) 2^-eA, split into FP16 high/low solve inputs
  EK_NEW16,   // FP16 solve input = w32 - acc
  EK_TRSM16,  // FP16 factor tile = acc 2^-eM
  EK_TRSM32   // x = acc 2^(eA - eM): FP32 tile, FP16 high/low shadows
};
struct Epi {
  int kind;
  double* d64;
  const double* s64;
  float* f32;
  const float* s32;
  const __half* s16;
  __half* h;
  __half* l;
  float sc;
};

__device__ __forceinline__ Epi make_epi(const TcParams& p, const Job& jb) {
  const TileView& v = p.v;
  const size_t nb2 = (size_t)v.nb * v.nb;
  const int i = jb.i, j = p.j;
  const int t = tidx(i, j);
  const int cd = v.cls[t];
  Epi e{};
  if (p.mode == TC_UPD_OLD) {
    if (i == j || cd == CR_PREC_FP64) {
      e.kind = EK_OLD64;
      e.s64 = v.pool64 + (size_t)v.i64[t] * nb2;
      e.d64 = (i == j) ? const_cast<double*>(e.s64) : p.ws64 + (size_t)i * nb2;
    } else if (cd == CR_PREC_FP32) {
      e.kind = EK_OLD32;
      e.f32 = p.w32 + (size_t)i * nb2;
      e.s32 = v.pool32 + (size_t)v.i32[t] * nb2;
    } else {
      e.kind = EK_OLD16;
      e.f32 = p.w32 + (size_t)i * nb2;
      e.s16 = v.pool16 + (size_t)v.hi16[t] * nb2;
    }
  } else if (p.mode == TC_UPD_NEW) {
    if (i == j || cd == CR_PREC_FP64) {
      e.kind = EK_NEW64;
      e.d64 = (i == j) ? v.pool64 + (size_t)v.i64[t] * nb2 : p.ws64 + (size_t)i * nb2;
    } else if (cd == CR_PREC_FP32) {
      e.kind = EK_NEW32;
      e.s32 = p.w32 + (size_t)i * nb2;
      e.h = v.pool16 + (size_t)(p.ws_hi0 + i) * nb2;
      e.l = v.pool16 + (size_t)(p.ws_lo0 + i) * nb2;
      e.sc = ldexpf(1.0f, -p.eA);
    } else {
      e.kind = EK_NEW16;
      e.s32 = p.w32 + (size_t)i * nb2;
      e.h = v.pool16 + (size_t)(p.ws_hi0 + i) * nb2;
    }
  } else {   // TC_TRSM
    const int eM = p.status[2];
    if (cd == CR_PREC_FP16) {
      e.kind = EK_TRSM16;
      e.h = v.pool16 + (size_t)v.hi16[t] * nb2;
      e.sc = ldexpf(1.0f, -eM);
    } else {
      e.kind = EK_TRSM32;
      e.f32 = v.pool32 + (size_t)v.i32[t] * nb2;
      e.h = v.pool16 + (size_t)v.hi16[t] * nb2;
      e.l = v.pool16 + (size_t)v.lo16[t] * nb2;
      e.sc = ldexpf(1.0f, p.eA - eM);
    }
  }
  return e;
}

// FP16 high/low split of the values of rows r and r + 1 at element offset o (and o + nb),
// two at a time: one packed conversion serves both rows (conversions issue on GB300's slow
// conversion pipe).  with32 also stores the FP32 values.
__device__ __forceinline__ void split_pair(const Epi& e, size_t o, int nb, float a, float b, bool with32) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
  if (with32) {
    e.f32[o] = a;
    e.f32[o + nb] = b;
  }
  e.h[o] = __low2half(h);
  e.h[o + nb] = __high2half(h);
  e.l[o] = __low2half(l);
  e.l[o + nb] = __high2half(l);
}

// One 32 x 32 chunk of a row-major tile: lane `lane` handles column col0 + lane of the 32
// rows from row offset base (element offsets off(r) = base + r nb + lane); st holds the
// accumulator chunk (st[r][lane]).  The reads of all 32 rows are issued before any store,
// so that each lane keeps 32 loads in flight.
__device__ __forceinline__ void epi_chunk(const Epi& e, size_t base, int nb, int lane, const float (*st)[33]) {
  const size_t o = base + lane;
  switch (e.kind) {
    case EK_OLD64: {
      double x[32];
#pragma unroll
      for (int r = 0; r < 32; ++r) x[r] = e.s64[o + (size_t)r * nb];
#pragma unroll
      for (int r = 0; r < 32; ++r) e.d64[o + (size_t)r * nb] = x[r] - widen(st[r][lane]);
      break;
    }
    case EK_NEW64: {
      double x[32];
#pragma unroll
      for (int r = 0; r < 32; ++r) x[r] = e.d64[o + (size_t)r * nb];
#pragma unroll
      for (int r = 0; r < 32; ++r) e.d64[o + (size_t)r * nb] = x[r] - widen(st[r][lane]);
      break;
    }
    case EK_OLD32: {
      float x[32];
#pragma unroll
      for (int r = 0; r < 32; ++r) x[r] = e.s32[o + (size_t)r * nb];
#pragma unroll
      for (int r = 0; r < 32; ++r) e.f32[o + (size_t)r * nb] = x[r] - st[r][lane];
      break;
    }
    case EK_OLD16: {
      __half x[32];
#pragma unroll
      for (int r = 0; r < 32; ++r) x[r] = e.s16[o + (size_t)r * nb];
#pragma unroll
      for (int r = 0; r < 32; r += 2) {
        const float2 f = __half22float2(__halves2half2(x[r], x[r + 1]));
        e.f32[o + (size_t)r * nb] = f.x - st[r][lane];
        e.f32[o + (size_t)(r + 1) * nb] = f.y - st[r + 1][lane];
      }
      break;
    }
    case EK_NEW32: {
      float x[32];
#pragma unroll
      for (int r = 0; r < 32; ++r) x[r] = e.s32[o + (size_t)r * nb];
#pragma unroll
      for (int r = 0; r < 32; r += 2)
        split_pair(e, o + (size_t)r * nb, nb, (x[r] - st[r][lane]) * e.sc, (x[r + 1] - st[r + 1][lane]) * e.sc, false);
      break;
    }
    case EK_NEW16: {
      float x[32];
#pragma unroll
      for (int r = 0; r < 32; ++r) x[r] = e.s32[o + (size_t)r * nb];
#pragma unroll
      for (int r = 0; r < 32; r += 2) {
        const __half2 h = __floats2half2_rn(x[r] - st[r][lane], x[r + 1] - st[r + 1][lane]);
        e.h[o + (size_t)r * nb] = __low2half(h);
        e.h[o + (size_t)(r + 1) * nb] = __high2half(h);
      }
      break;
    }
    case EK_TRSM16: {
#pragma unroll
      for (int r = 0; r < 32; r += 2) {
        const __half2 h = __floats2half2_rn(st[r][lane] * e.sc, st[r + 1][lane] * e.sc);
        e.h[o + (size_t)r * nb] = __low2half(h);
        e.h[o + (size_t)(r + 1) * nb] = __high2half(h);
      }
      break;
    }
    default: {
#pragma unroll
      for (int r = 0; r < 32; r += 2)
        split_pair(e, o + (size_t)r * nb, nb, st[r][lane] * e.sc, st[r + 1][lane] * e.sc, true);
    }
  }
}

// Shared-memory layout after the stage ring (offsets from the 1 KB aligned base).
struct TcBars {
  uint64_t full[TC_STAGES], empty[TC_STAGES];   // stage ring
  uint64_t tfull[2], tempty[2];                 // TMEM accumulators
  uint64_t kfull[2], kempty[2];                 // k-term tables
  int steps[2];                                 // step count of the block in each accumulator
  uint32_t tmem;
  int abort;
};
static_assert(sizeof(TcBars) <= 256, "barrier area");

}  // namespace

// One kernel for every mode; MODE only names the instantiation (equal to p.mode), so that a
// profiler can tell the modes apart.
template <int MODE>
__global__ void __launch_bounds__(TC_THREADS, 1)
    k_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const TcParams p, int nblocks) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  TcBars* bars = reinterpret_cast<TcBars*>(smem + TC_STAGES * TC_STAGE_BYTES);
  float* estage = reinterpret_cast<float*>(smem + TC_STAGES * TC_STAGE_BYTES + 256);   // 4 warps x 32 x 33
  int* ktab = reinterpret_cast<int*>(smem + TC_STAGES * TC_STAGE_BYTES + 256 + TC_EPI_BYTES);
  const int kt_ints = TC_KT_INTS * p.v.nt;
  volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int es = p.mode == TC_TRMM ? 1 : max(1, p.esplit);   // nblocks counts es CTAs per output block

  if (threadIdx.x == 0) {
    for (int s = 0; s < TC_STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->tfull[b], 2);       // the MMA thread's arrival and the MMA completion
      mbar_init(&bars->tempty[b], 128);    // every epilogue thread
      mbar_init(&bars->kfull[b], 1);
      mbar_init(&bars->kempty[b], 1);
    }
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&bars->tmem, TC_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;

  if (warp == 0) {
    // k-term tables and TMA producer
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
    }
    uint32_t gs = 0;   // global step count of this CTA
    int u = 0;
    for (JobIter it(p, nblocks); it.next(p); ++u) {
      const int t = it.t;
      const int b = u & 1;
      const uint32_t ph = (uint32_t)(u >> 1) & 1u;
      int* kt = ktab + b * kt_ints;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&bars->kempty[b], ph ^ 1u);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok || *abort_flag) {
        if (lane == 0 && !ok) {
          *abort_flag = 1;
          atomicOr(p.err, DEV_ERR_TIMEOUT);
        }
        break;
      }
      const Job jb = decode(p, t / es);
      fill_ktable(p, jb, kt);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars->kfull[b]);
        for_each_step(p, jb, kt, [&](int aslot, int ak, int bslot, int bk, int brow) {
          if (*abort_flag) return;
          const int st = gs % TC_STAGES;
          const uint32_t sph = (gs / TC_STAGES) & 1u;
          ++gs;
          if (!mbar_wait(&bars->empty[st], sph ^ 1u)) {
            *abort_flag = 1;
            atomicOr(p.err, DEV_ERR_TIMEOUT);
            return;
          }
          mbar_arrive_expect_tx(&bars->full[st], TC_STAGE_BYTES);
          uint8_t* sa = smem + st * TC_STAGE_BYTES;
          uint8_t* sb = sa + TC_BM * TC_BK * 2;
          tma_load_3d(sa, &tmA, &bars->full[st], ak, jb.rb * TC_BM, aslot);
          if (bslot >= 0) {
            tma_load_3d(sb, &tmA, &bars->full[st], bk, brow, bslot);
            tma_load_3d(sb + 128 * TC_BK * 2, &tmA, &bars->full[st], bk, brow + 128, bslot);
          } else {
            tma_load_2d(sb, &tmB, &bars->full[st], bk, brow);
            tma_load_2d(sb + 128 * TC_BK * 2, &tmB, &bars->full[st], bk, brow + 128);
          }
        }, it.seg);
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(TC_BM, TC_BN);
      uint32_t gs = 0;
      int u = 0;
      for (JobIter it(p, nblocks); it.next(p); ++u) {
        const int t = it.t;
        const int b = u & 1;
        const uint32_t ph = (uint32_t)(u >> 1) & 1u;
        if (*abort_flag) break;
        if (!mbar_wait(&bars->kfull[b], ph) || !mbar_wait(&bars->tempty[b], ph ^ 1u)) {
          *abort_flag = 1;
          atomicOr(p.err, DEV_ERR_TIMEOUT);
          break;
        }
        const Job jb = decode(p, t / es);
        const int S = for_each_step(p, jb, ktab + b * kt_ints, NoOp(), it.seg);
        mbar_arrive(&bars->kempty[b]);
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(b * TC_BN);
        bool ok = true;
        for (int s = 0; s < S; ++s, ++gs) {
          const int st = gs % TC_STAGES;
          const uint32_t sph = (gs / TC_STAGES) & 1u;
          if (*abort_flag || !mbar_wait(&bars->full[st], sph)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + st * TC_STAGE_BYTES);
          const uint32_t sb = sa + TC_BM * TC_BK * 2;
          const uint64_t da = desc_sw128(sa), db = desc_sw128(sb);
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk)
            mma_f16(acc, da + (uint64_t)((kk * 32) >> 4), db + (uint64_t)((kk * 32) >> 4), idesc, (s | kk) != 0);
          mma_commit(&bars->empty[st]);
        }
        if (!ok) {
          *abort_flag = 1;
          atomicOr(p.err, DEV_ERR_TIMEOUT);
          break;
        }
        bars->steps[b] = S;
        mbar_arrive(&bars->tfull[b]);
        if (S > 0) mma_commit(&bars->tfull[b]);
        else mbar_arrive(&bars->tfull[b]);
      }
    }
  } else {
    // epilogue: warp w reads TMEM lanes of quadrant (w % 4)
    const int quad = warp & 3;
    const int r_local = quad * 32 + lane;
    int u = 0;
    for (JobIter it(p, nblocks); it.next(p); ++u) {
      const int t = it.t;
      const int b = u & 1;
      const uint32_t ph = (uint32_t)(u >> 1) & 1u;
      if (*abort_flag) break;
      if (!mbar_wait(&bars->tfull[b], ph)) {
        if (lane == 0) atomicOr(p.err, DEV_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const Job jb = decode(p, t / es);
      const int part = t % es;
      const int S = bars->steps[b];
      const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(b * TC_BN);
      if (p.mode == TC_TRMM) {
        for (int c0 = 0; c0 < TC_BN; c0 += 16) {
          float acc[16];
          if (S > 0) {
            tmem_ld16(tq + (uint32_t)c0, acc);
          } else {
#pragma unroll
            for (int q = 0; q < 16; ++q) acc[q] = 0.0f;
          }
          if (it.perk) trmm_store_per_gemm(p, jb, t, r_local, c0, acc, it.seg, it.nseg);
          else trmm_store(p, jb, r_local, c0, acc);
        }
      } else {
        // row-major tiles: each 32 x 32 chunk of the warp's quadrant goes through shared
        // memory so that consecutive lanes handle consecutive columns of one row
        const Epi e = make_epi(p, jb);
        const int ncols = min(TC_BN, p.v.nb - jb.cb * TC_BN);
        const int per = ((ncols / 32 + es - 1) / es) * 32;   // this CTA's share of the columns
        const int g_end = min(ncols, (part + 1) * per);
        float(*st)[33] = reinterpret_cast<float(*)[33]>(estage + (warp - 2) * 32 * 33);
        const size_t base = (size_t)(jb.rb * TC_BM + quad * 32) * p.v.nb + jb.cb * TC_BN;
        for (int g = part * per; g < g_end; g += 32) {
          float acc[32];
          if (S > 0) {
            tmem_ld16(tq + (uint32_t)g, acc);
            tmem_ld16(tq + (uint32_t)(g + 16), acc + 16);
          } else {
#pragma unroll
            for (int q = 0; q < 32; ++q) acc[q] = 0.0f;
          }
#pragma unroll
          for (int q = 0; q < 32; ++q) st[lane][q] = acc[q];
          __syncwarp();
          epi_chunk(e, base + g, p.v.nb, lane, st);
          __syncwarp();
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->tempty[b]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TC_TMEM_COLS);
  }
}

cr_status tc_launch(const TcParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, cudaStream_t stream) {
  constexpr int kMaxSmem = 227 * 1024;
  static bool configured = false;
  if (!configured) {
    for (auto* fn : {k_tc<TC_UPD_OLD>, k_tc<TC_TRSM>, k_tc<TC_TRMM>, k_tc<TC_UPD_NEW>}) {
      CR_CUDA(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem));
      CR_CUDA(cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared));
    }
    configured = true;
  }
  const int es = p.mode == TC_TRMM ? 1 : std::max(1, p.esplit);
  const int nblocks = tc_num_blocks(p) * es;
  if (nblocks <= 0) return CR_OK;
  int dev = 0, sms = 0;
  CR_CUDA(cudaGetDevice(&dev));
  CR_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const size_t smem = TC_SMEM + 2 * (((size_t)TC_KT_INTS * sizeof(int) * p.v.nt + 15) & ~(size_t)15);
  if (smem > (size_t)kMaxSmem) return fail(CR_ERR_ARG, "tensor-core kernel: too many tiles per column for the k-term tables");
  const int cap = (p.max_ctas > 0 && p.max_ctas < sms) ? p.max_ctas : sms;
  const int grid = nblocks < cap ? nblocks : cap;
  {
    static const char* names[4] = {"k_tc_old", "k_tc_trsm", "k_tc_trmm", "k_tc_new"};
    TimedScope ts(names[p.mode & 3], stream);
    switch (p.mode) {
      case TC_UPD_OLD: k_tc<TC_UPD_OLD><<<grid, TC_THREADS, smem, stream>>>(tmA, tmB, p, nblocks); break;
      case TC_TRSM: k_tc<TC_TRSM><<<grid, TC_THREADS, smem, stream>>>(tmA, tmB, p, nblocks); break;
      case TC_TRMM: k_tc<TC_TRMM><<<grid, TC_THREADS, smem, stream>>>(tmA, tmB, p, nblocks); break;
      case TC_UPD_NEW: k_tc<TC_UPD_NEW><<<grid, TC_THREADS, smem, stream>>>(tmA, tmB, p, nblocks); break;
      default: return fail(CR_ERR_ARG, "tensor-core kernel: mode");
    }
  }
  CR_CHECK_LAUNCH("k_tc");
  return CR_OK;
}

}  // namespace cr
