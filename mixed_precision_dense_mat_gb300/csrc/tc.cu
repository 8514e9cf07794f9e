// Tensor-core tile kernel (tcgen05.mma kind::f16, FP32 accumulation in TMEM, TMA-fed
// 6-stage shared-memory ring, warp-specialised: warp 0 TMA producer, warp 1 MMA issuer and
// TMEM owner, warps 2-5 epilogue).  One CTA computes one 128 x 128 output block.
//
// Three uses, all from "Mixed-Precision GPU Acceleration for Confidence Regions of Spatial
// Excursion Sets":
//  TC_UPDATE  Cholesky column update A_ij -= sum_k L_ik L_jk^T (Section IV-B) for the
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
#include "tc.cuh"

namespace cr {

namespace {

struct Job {
  int i, rb, cb;
  bool skip;
};

__device__ __forceinline__ Job decode(const TcParams& p) {
  const int nsb = p.v.nb / TC_BM;
  Job jb;
  jb.skip = false;
  if (p.mode == TC_TRMM) {
    const int per_row = nsb * p.ncb;
    jb.i = p.v.nt - 1 - (int)blockIdx.x / per_row;   // longest K-chains first
    const int rem = blockIdx.x % per_row;
    jb.rb = rem / p.ncb;
    jb.cb = rem % p.ncb;
  } else {
    const int per = nsb * nsb;
    const int ri = blockIdx.x / per;
    jb.i = p.rows ? p.rows[ri] : p.j + ri;
    const int rem = blockIdx.x % per;
    jb.rb = rem / nsb;
    jb.cb = rem % nsb;
    jb.skip = (jb.i == p.j && jb.cb > jb.rb);
  }
  return jb;
}

// Enumerates the pipeline steps of one CTA.  Each step is one 64-wide K chunk of an
// (A, B) pair of FP16 operand tiles; f(step, a_slot, a_k, b_slot, b_c0, b_c1).  A is read
// from the FP16 tile pool at rows [rb*128, rb*128+128); B from the pool (b_slot >= 0, rows
// [cb*128, +128), K offset b_c0) or from the 2-D right-hand-side map (b_slot < 0).
template <class F>
__device__ __forceinline__ int for_each_step(const TcParams& p, const Job& jb, F&& f) {
  const TileView& v = p.v;
  const int nq = v.nb / TC_BK;
  int s = 0;
  if (p.mode == TC_UPD_OLD || p.mode == TC_UPD_NEW) {
    const int i = jb.i, j = p.j;
    const int cd = v.cls[tidx(i, j)];
    for (int k = p.kbeg; k < p.kend; ++k) {
      const int ti = tidx(i, k), tj = tidx(j, k);
      const int pc = max(cd, max((int)v.cls[ti], (int)v.cls[tj]));
      if (pc == CR_PREC_FP64) continue;
      const int ahi = v.hi16[ti], bhi = v.hi16[tj];
      if (pc == CR_PREC_FP16) {
        for (int q = 0; q < nq; ++q) f(s++, ahi, q * TC_BK, bhi, q * TC_BK, jb.cb * TC_BN);
      } else {
        const int alo = v.lo16[ti], blo = v.lo16[tj];
        for (int q = 0; q < nq; ++q) {
          f(s++, ahi, q * TC_BK, bhi, q * TC_BK, jb.cb * TC_BN);
          f(s++, ahi, q * TC_BK, blo, q * TC_BK, jb.cb * TC_BN);
          f(s++, alo, q * TC_BK, bhi, q * TC_BK, jb.cb * TC_BN);
        }
      }
    }
  } else if (p.mode == TC_TRSM) {
    const int i = jb.i;
    const int cd = v.cls[tidx(i, p.j)];
    const int nqk = (jb.cb + 1) * (TC_BN / TC_BK);   // inverse factor is lower triangular
    const int wh = p.ws_hi0 + i, wl = p.ws_lo0 + i;
    for (int q = 0; q < nqk; ++q) {
      f(s++, wh, q * TC_BK, p.minv_hi, q * TC_BK, jb.cb * TC_BN);
      f(s++, wh, q * TC_BK, p.minv_lo, q * TC_BK, jb.cb * TC_BN);
      if (cd == CR_PREC_FP32) f(s++, wl, q * TC_BK, p.minv_hi, q * TC_BK, jb.cb * TC_BN);
    }
  } else {
    const int i = jb.i;
    for (int k = 0; k < i; ++k) {
      const int a = v.hi16[tidx(i, k)];
      for (int q = 0; q < nq; ++q) f(s++, a, q * TC_BK, -1, k * v.nb + q * TC_BK, jb.cb * TC_BN);
    }
    const int nqd = (jb.rb + 1) * (TC_BM / TC_BK);    // the diagonal factor is lower triangular
    const int dh = v.hi16[tidx(i, i)], dl = v.lo16[tidx(i, i)];
    for (int q = 0; q < nqd; ++q) {
      f(s++, dh, q * TC_BK, -1, i * v.nb + q * TC_BK, jb.cb * TC_BN);
      f(s++, dl, q * TC_BK, -1, i * v.nb + q * TC_BK, jb.cb * TC_BN);
    }
  }
  return s;
}

struct NoOp {
  __device__ void operator()(int, int, int, int, int, int) const {}
};

__device__ __forceinline__ void epilogue_store(const TcParams& p, const Job& jb, int r_local, int c0, const float* acc) {
  const TileView& v = p.v;
  const int nb = v.nb;
  const size_t nb2 = (size_t)nb * nb;
  if (p.mode == TC_TRMM) {
    const int row = jb.i * nb + jb.rb * TC_BM + r_local;
    if (row >= v.n) return;
    const bool f16 = (p.flags & CR_TRMM_FP16_DEST) != 0;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int col = jb.cb * TC_BN + c0 + q;
      if (col < p.M) {
        const float a = f16 ? __half2float(__float2half_rn(acc[q])) : acc[q];
        p.Y[(size_t)col * p.ldy + row] = (double)a;
      }
    }
    return;
  }
  const int i = jb.i, j = p.j;
  const int t = tidx(i, j);
  const int cd = v.cls[t];
  const size_t off = (size_t)(jb.rb * TC_BM + r_local) * nb + jb.cb * TC_BN + c0;
  if (p.mode == TC_UPD_OLD) {
    // older terms: class storage -> intermediate (FP64 in place / FP64 workspace / FP32 workspace)
    if (i == j || cd == CR_PREC_FP64) {
      const double* src = v.pool64 + (size_t)v.i64[t] * nb2 + off;
      double* dst = (i == j) ? const_cast<double*>(src) : p.ws64 + (size_t)i * nb2 + off;
#pragma unroll
      for (int q = 0; q < 16; q += 2) {
        const double2 a = *reinterpret_cast<const double2*>(src + q);
        *reinterpret_cast<double2*>(dst + q) = make_double2(a.x - (double)acc[q], a.y - (double)acc[q + 1]);
      }
    } else {
      float* dst = p.w32 + (size_t)i * nb2 + off;
      if (cd == CR_PREC_FP32) {
        const float* src = v.pool32 + (size_t)v.i32[t] * nb2 + off;
#pragma unroll
        for (int q = 0; q < 16; q += 4)
          *reinterpret_cast<float4*>(dst + q) =
              make_float4(src[q] - acc[q], src[q + 1] - acc[q + 1], src[q + 2] - acc[q + 2], src[q + 3] - acc[q + 3]);
      } else {
        const __half* src = v.pool16 + (size_t)v.hi16[t] * nb2 + off;
#pragma unroll
        for (int q = 0; q < 16; q += 4)
          *reinterpret_cast<float4*>(dst + q) =
              make_float4(__half2float(src[q]) - acc[q], __half2float(src[q + 1]) - acc[q + 1],
                          __half2float(src[q + 2]) - acc[q + 2], __half2float(src[q + 3]) - acc[q + 3]);
      }
    }
  } else if (p.mode == TC_UPD_NEW) {
    // newest term: intermediate -> solve inputs in the tile's precision
    if (i == j || cd == CR_PREC_FP64) {
      double* dst = (i == j) ? v.pool64 + (size_t)v.i64[t] * nb2 + off : p.ws64 + (size_t)i * nb2 + off;
#pragma unroll
      for (int q = 0; q < 16; q += 2) {
        const double2 a = *reinterpret_cast<const double2*>(dst + q);
        *reinterpret_cast<double2*>(dst + q) = make_double2(a.x - (double)acc[q], a.y - (double)acc[q + 1]);
      }
    } else if (cd == CR_PREC_FP32) {
      const float* src = p.w32 + (size_t)i * nb2 + off;
      __half* hi = v.pool16 + (size_t)(p.ws_hi0 + i) * nb2 + off;
      __half* lo = v.pool16 + (size_t)(p.ws_lo0 + i) * nb2 + off;
      const float sc = ldexpf(1.0f, -p.eA);
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float w = (src[q] - acc[q]) * sc;
        const __half h = __float2half_rn(w);
        hi[q] = h;
        lo[q] = __float2half_rn(w - __half2float(h));
      }
    } else {
      const float* src = p.w32 + (size_t)i * nb2 + off;
      __half* dst = v.pool16 + (size_t)(p.ws_hi0 + i) * nb2 + off;
#pragma unroll
      for (int q = 0; q < 16; ++q) dst[q] = __float2half_rn(src[q] - acc[q]);
    }
  } else {   // TC_TRSM
    const int eM = p.status[2];
    if (cd == CR_PREC_FP16) {
      const float sc = ldexpf(1.0f, -eM);
      __half* dst = v.pool16 + (size_t)v.hi16[t] * nb2 + off;
#pragma unroll
      for (int q = 0; q < 16; ++q) dst[q] = __float2half_rn(acc[q] * sc);
    } else {
      const float sc = ldexpf(1.0f, p.eA - eM);
      float* d32 = v.pool32 + (size_t)v.i32[t] * nb2 + off;
      __half* hi = v.pool16 + (size_t)v.hi16[t] * nb2 + off;
      __half* lo = v.pool16 + (size_t)v.lo16[t] * nb2 + off;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float x = acc[q] * sc;
        d32[q] = x;
        const __half h = __float2half_rn(x);
        hi[q] = h;
        lo[q] = __float2half_rn(x - __half2float(h));
      }
    }
  }
}

}  // namespace

__global__ void __launch_bounds__(TC_THREADS, 1)
    k_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const TcParams p) {
  const Job jb = decode(p);
  if (jb.skip) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + TC_STAGES * TC_STAGE_BYTES);
  uint64_t* empty = full + TC_STAGES;
  uint64_t* accb = empty + TC_STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accb + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < TC_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accb, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, TC_BN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int S = for_each_step(p, jb, NoOp());

  if (warp == 0) {
    if (lane == 0 && S > 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      for_each_step(p, jb, [&](int s, int aslot, int ak, int bslot, int bc0, int bc1) {
        if (*abort_flag) return;
        const int st = s % TC_STAGES;
        const uint32_t ph = (uint32_t)(s / TC_STAGES) & 1u;
        if (!mbar_wait(&empty[st], ph ^ 1u)) {
          *abort_flag = 1;
          atomicOr(p.err, DEV_ERR_TIMEOUT);
          return;
        }
        mbar_arrive_expect_tx(&full[st], TC_STAGE_BYTES);
        uint8_t* sa = smem + st * TC_STAGE_BYTES;
        uint8_t* sb = sa + TC_BM * TC_BK * 2;
        tma_load_3d(sa, &tmA, &full[st], ak, jb.rb * TC_BM, aslot);
        if (bslot >= 0) tma_load_3d(sb, &tmA, &full[st], bc0, bc1, bslot);
        else tma_load_2d(sb, &tmB, &full[st], bc0, bc1);
      });
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(TC_BM, TC_BN);
      for (int s = 0; s < S; ++s) {
        const int st = s % TC_STAGES;
        const uint32_t ph = (uint32_t)(s / TC_STAGES) & 1u;
        if (*abort_flag) break;
        if (!mbar_wait(&full[st], ph)) {
          *abort_flag = 1;
          atomicOr(p.err, DEV_ERR_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + st * TC_STAGE_BYTES);
        const uint32_t sb = sa + TC_BM * TC_BK * 2;
        const uint64_t da = desc_sw128(sa), db = desc_sw128(sb);
#pragma unroll
        for (int kk = 0; kk < TC_BK / 16; ++kk)
          mma_f16(tmem, da + (uint64_t)((kk * 32) >> 4), db + (uint64_t)((kk * 32) >> 4), idesc, (s | kk) != 0);
        mma_commit(&empty[st]);
      }
      if (S > 0) mma_commit(accb);
      else mbar_arrive(accb);
    }
  } else {
    // epilogue: warp w reads TMEM lanes of quadrant (w % 4)
    const int quad = warp & 3;
    const int r_local = quad * 32 + lane;
    bool ok = true;
    if (S > 0) {
      ok = mbar_wait(accb, 0);
      if (!ok && lane == 0) atomicOr(p.err, DEV_ERR_TIMEOUT);
      tc_fence_after();
    }
    for (int c0 = 0; c0 < TC_BN; c0 += 16) {
      float acc[16];
      if (S > 0) {
        tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)c0, acc);
      } else {
#pragma unroll
        for (int q = 0; q < 16; ++q) acc[q] = 0.0f;
      }
      if (ok) epilogue_store(p, jb, r_local, c0, acc);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    // all MMAs issued by this CTA are complete once accb has fired
    if (S > 0) mbar_wait(accb, 0);
    tc_fence_after();
    tmem_dealloc(tmem, TC_BN);
  }
}

cr_status tc_launch(const TcParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, int grid, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    CR_CUDA(cudaFuncSetAttribute(k_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TC_SMEM));
    CR_CUDA(cudaFuncSetAttribute(k_tc, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared));
    configured = true;
  }
  if (grid <= 0) return CR_OK;
  k_tc<<<grid, TC_THREADS, TC_SMEM, stream>>>(tmA, tmB, p);
  CR_CHECK_LAUNCH("k_tc");
  return CR_OK;
}

}  // namespace cr
