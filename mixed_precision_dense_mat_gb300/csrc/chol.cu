// Adaptive mixed-precision tile Cholesky driver (left-looking by tile column, with lookahead).
//
// "Mixed-Precision GPU Acceleration for Confidence Regions of Spatial Excursion Sets",
// Section IV-B and Alg.2 step 12: L_s = chol(s^2 V) with the tile precisions of the map;
// diagonal tiles FP64.  For tile column j the update A_ij -= sum_{k<j} L_ik L_jk^T is split:
//   OLD(j)  terms k < j-1, on a low-priority stream: FP64 products on the FP64 units, all
//           others on the tensor cores (FP16 MMAs, or FP16 high/low parts for FP32-class
//           accuracy) accumulated in FP32 into an intermediate;
//   NEW(j)  term k = j-1, on a high-priority stream, finishing the solve inputs;
// then, on the high-priority stream, the FP64 diagonal tile is factored together with its
// inverse by the on-device dataflow executor (diag.cu), and the off-diagonal tiles are
// solved, L_ij = A_ij L_jj^-T, as a product with that inverse in the tile's precision.
// OLD(j+1) needs only columns < j, so it runs on the tensor cores while column j's FP64
// diagonal factorisation (the critical path) runs on the FP64 units.  Work buffers are
// double-buffered by column parity.  The schedule depends only on the map: all job lists
// are built on the host and uploaded in one copy, then replayed with events between the
// two streams.  This replaces the paper's PaRSEC task runtime on one GPU.
#include <stdlib.h>

#include <algorithm>
#include <functional>

#include "common.cuh"
#include "diag.cuh"
#include "fp64.cuh"
#include "tc.cuh"

namespace cr {

// d_tiles: count tile codes (i << 16 | j), the first ndiag of them diagonal (FP64 class)
cr_status convert_tiles(cr_tilemat V, const int* d_tiles, int count, int ndiag, int nheavy, bool diag_df,
                        cudaStream_t stream);

namespace {

struct Exec {
  cudaStream_t hi, lo, mid, gen;
  const DJob* dj;
  const DPair* dp;
  // per column j: OLD(j) done (lo); diagonal factor and inverse split (hi); NEW(j) rows j+1..
  // done (mid); solve of row j+1 done (hi); solves of rows j+2.. done (mid)
  std::vector<cudaEvent_t> ev_old, ev_split, ev_newr, ev_crit, ev_rest;
  std::vector<cudaEvent_t> ev_gen;   // per column range: its tiles generated
  std::vector<cudaEvent_t> ev_gdiag; // per column range: its diagonal tiles generated
  cudaEvent_t start;                  // critical stream: status and executor flags cleared
  cudaEvent_t start0, start1;         // caller: before the prologue; after the job uploads
};

using Op = std::function<cr_status(Exec&)>;

struct Plan {
  std::vector<DJob> jobs;
  std::vector<DPair> pairs;
  std::vector<Op> ops;

  int add_pair(const double* A, const double* B, int sAm, int sAk, int sBn, int sBk, int K) {
    pairs.push_back(DPair{A, B, sAm, sAk, sBn, sBk, K});
    return (int)pairs.size() - 1;
  }
  void dgemm(int block, const std::vector<DJob>& js, bool on_lo, bool on_mid = false) {
    if (js.empty()) return;
    const int off = (int)jobs.size(), cnt = (int)js.size();
    jobs.insert(jobs.end(), js.begin(), js.end());
    ops.push_back([=](Exec& x) -> cr_status {
      return dgemm_launch(block, x.dj + off, x.dp, cnt, on_lo ? x.lo : (on_mid ? x.mid : x.hi));
    });
  }
};

DJob job(double* C, int sCm, int sCn, int m, int n, int pbeg, int pcnt, double alpha, double beta, int arow, int brow,
         int kmax) {
  DJob j;
  j.C = C; j.sCm = sCm; j.sCn = sCn; j.m = m; j.n = n; j.pbeg = pbeg; j.pcnt = pcnt;
  j.alpha = alpha; j.beta = beta; j.arow = arow; j.brow = brow; j.kmax = kmax;
  return j;
}

}  // namespace

cr_status build_and_run_cholesky(cr_tilemat V, cudaStream_t caller) {
  const int nt = V->nt, nb = V->nb;
  const size_t nb2 = (size_t)nb * nb;
  const auto& cls = V->h_cls;
  auto t64 = [&](int i, int j) { return V->pool64 + (size_t)V->h_i64[tidx(i, j)] * nb2; };
  auto ws64 = [&](int par, int i) { return V->ws64 + ((size_t)par * nt + i) * nb2; };
  Plan P;
  int* status = V->d_status;
  int* dflags = V->diag_flags;
  unsigned long long* damax = reinterpret_cast<unsigned long long*>(V->minv_part);
  const size_t dwords = 2 * (size_t)diag_flag_words(nb, V->diag_db);
  double* dpub = V->diag_pub;
  const size_t dpub_bytes = diag_pub_doubles(nb, V->diag_db) * sizeof(double);
  // arithmetic of the diagonal executor: double-float (FP64 emulated on the FP32 units) for
  // adaptive factorisations unless the caller asked otherwise
  const int arith = option_diag_arith();
  const bool use_df = arith == CR_DIAG_DF || (arith == CR_DIAG_AUTO && V->amp);
  const unsigned long long wait_ns = option_wait_ns();
  if (use_df && !V->diag_df) CR_CUDA(cudaMalloc(&V->diag_df, 2 * nb2 * sizeof(float2)));
  // Tile generation on its own stream, column by column in ranges of doubling width
  // ([0,1), [1,3), [3,7), [7,15), ...), diagonal tiles first in each range: the factorisation
  // of column j waits only for its range, so it starts after the first column's tiles
  // instead of after all of them.
  if (nt > 32767) return fail(CR_ERR_ARG, "cr_potrf_adaptive: more than 32767 tile rows");
  std::vector<int> gen_list, gen_off{0}, gen_ndiag, gen_nheavy, gen_range_of(nt, 0);
  for (int c0 = 0, w = 1; c0 < nt; c0 += w, w *= 2) {
    const int c1 = std::min(nt, c0 + w);
    gen_ndiag.push_back(c1 - c0);
    for (int c = c0; c < c1; ++c) {
      gen_list.push_back(c << 16 | c);
      gen_range_of[c] = (int)gen_off.size() - 1;
    }
    // the other tiles of the range by cost, heaviest first (FP64 evaluations, then
    // double-float, then single precision), so that a launch does not end on a few long CTAs
    for (int pass = 0; pass < 3; ++pass) {
      for (int c = c0; c < c1; ++c)
        for (int i = c + 1; i < nt; ++i) {
          const int k = cls[tidx(i, c)];
          const int rank = k == CR_PREC_FP64 ? 0 : (k == CR_PREC_FP32 ? 1 : 2);
          if (rank == pass) gen_list.push_back(i << 16 | c);
        }
      if (pass == 1) gen_nheavy.push_back((int)gen_list.size() - gen_off.back() - gen_ndiag.back());
    }
    gen_off.push_back((int)gen_list.size());
  }
  const int n_ranges = (int)gen_off.size() - 1;
  // rows solved on the tensor cores, per column
  std::vector<int> rows_flat;
  std::vector<int> rows_off(nt + 1, 0);
  for (int j = 0; j < nt; ++j) {
    rows_off[j] = (int)rows_flat.size();
    for (int i = j + 1; i < nt; ++i)
      if (cls[tidx(i, j)] != CR_PREC_FP64) rows_flat.push_back(i);
  }
  rows_off[nt] = (int)rows_flat.size();
  // both lists in one device buffer kept by the tile matrix (the previous call's kernels are
  // complete: every call ends by synchronising its streams)
  const size_t n_ints = rows_flat.size() + gen_list.size();
  if (n_ints > V->sched_ints_cap) {
    if (V->sched_ints) cudaFree(V->sched_ints);
    V->sched_ints = nullptr;
    V->sched_ints_cap = 0;
    CR_CUDA(cudaMalloc(&V->sched_ints, n_ints * sizeof(int)));
    V->sched_ints_cap = n_ints;
  }
  int* d_rows = V->sched_ints;
  int* d_gen = V->sched_ints + rows_flat.size();
  {
    std::vector<int> both(rows_flat);
    both.insert(both.end(), gen_list.begin(), gen_list.end());
    CR_CUDA(cudaMemcpyAsync(V->sched_ints, both.data(), n_ints * sizeof(int), cudaMemcpyHostToDevice, caller));
  }
  if (!V->s_hi) {
    int lo_prio = 0, hi_prio = 0;
    CR_CUDA(cudaDeviceGetStreamPriorityRange(&lo_prio, &hi_prio));
    CR_CUDA(cudaStreamCreateWithPriority(&V->s_hi, cudaStreamNonBlocking, hi_prio));
    CR_CUDA(cudaStreamCreateWithPriority(&V->s_mid, cudaStreamNonBlocking, hi_prio));
    // the bulk updates rank just above the tile generation, which runs ahead of them
    CR_CUDA(cudaStreamCreateWithPriority(&V->s_lo, cudaStreamNonBlocking, std::max(hi_prio, lo_prio - 1)));
    CR_CUDA(cudaStreamCreateWithPriority(&V->s_gen, cudaStreamNonBlocking, lo_prio));
  }
  Exec x;
  x.hi = V->s_hi;
  x.lo = V->s_lo;
  x.mid = V->s_mid;
  x.gen = V->s_gen;
  // events: created once per tile matrix (7 per column and three start events)
  if (V->sched_ev.size() != 7 * (size_t)nt + 3) {
    for (cudaEvent_t e : V->sched_ev) cudaEventDestroy(e);
    V->sched_ev.assign(7 * (size_t)nt + 3, nullptr);
    for (auto& e : V->sched_ev) CR_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
  }
  {
    size_t q = 0;
    for (auto* evs : {&x.ev_old, &x.ev_split, &x.ev_newr, &x.ev_crit, &x.ev_rest, &x.ev_gen, &x.ev_gdiag}) {
      evs->assign(V->sched_ev.begin() + q, V->sched_ev.begin() + q + nt);
      q += nt;
    }
    x.start = V->sched_ev[q];
    x.start0 = V->sched_ev[q + 1];
    x.start1 = V->sched_ev[q + 2];
  }
  // The prologue runs at once, so that the GPU generates the first tiles while the host
  // builds the rest of the schedule: after the caller's prior work and the list upload, the
  // critical stream clears the status and the executor's flags, and the generation stream
  // starts on the first column range.
  CR_CUDA(cudaEventRecord(x.start0, caller));
  CR_CUDA(cudaStreamWaitEvent(x.hi, x.start0, 0));
  CR_CUDA(cudaStreamWaitEvent(x.gen, x.start0, 0));
  CR_TRY(status_init_launch(status, x.hi));
  // both parities of the executor's flags and abs-max start cleared
  CR_CUDA(cudaMemsetAsync(dflags, 0, dwords * sizeof(int), x.hi));
  CR_CUDA(cudaMemsetAsync(damax, 0, 2 * sizeof(unsigned long long), x.hi));
  CR_CUDA(cudaMemsetAsync(dpub, 0xff, dpub_bytes, x.hi));   // every element unpublished
  CR_CUDA(cudaEventRecord(x.start, x.hi));   // the first two OLD steps wait for the status and flags
  for (int r = 0; r < n_ranges; ++r) {
    if (r <= gen_range_of[std::min(1, nt - 1)]) {
      // the ranges of columns 0 and 1: the diagonal tiles first, in a launch of their own (the
      // first two diagonal factorisations need nothing else)
      CR_TRY(convert_tiles(V, d_gen + gen_off[r], gen_ndiag[r], gen_ndiag[r], 0, use_df, x.gen));
      CR_CUDA(cudaEventRecord(x.ev_gdiag[r], x.gen));
      CR_TRY(convert_tiles(V, d_gen + gen_off[r] + gen_ndiag[r], gen_off[r + 1] - gen_off[r] - gen_ndiag[r], 0,
                           gen_nheavy[r], use_df, x.gen));
    } else {
      // later ranges in one launch, diagonal tiles issued first, so that their FP64 work
      // overlaps the other tiles' FP32 work
      CR_TRY(convert_tiles(V, d_gen + gen_off[r], gen_off[r + 1] - gen_off[r], gen_ndiag[r], gen_nheavy[r], use_df,
                           x.gen));
      CR_CUDA(cudaEventRecord(x.ev_gdiag[r], x.gen));
    }
    CR_CUDA(cudaEventRecord(x.ev_gen[r], x.gen));
  }

  TcParams base{};
  base.v = V->view();
  base.minv_hi = V->minv_hi;
  base.minv_lo = V->minv_lo;
  base.eA = V->eA;
  base.status = V->d_status;
  base.err = V->d_status;
  const CUtensorMap* tm = &V->tm_pool16;
  // grid caps: the persistent tensor-core CTAs hold their SMs for a whole launch, and a
  // higher stream priority does not preempt them, so the bulk and lookahead launches leave
  // SMs free for the few blocks the critical stream launches (at most 8 per launch)
  int sms = 0;
  CR_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, V->device));
  // lookahead launches of column j have about 8 (nt - j) output blocks of short inner length
  // that must finish within one diagonal factorisation: about 16 blocks per CTA
  // The critical stream's single-tile tensor-core launches (the last update of the diagonal
  // tile, the solve of the tile below it) spread each output block's epilogue over HI_ESPLIT
  // CTAs, and the bulk stream leaves HI_SMS SMs free for them.
  constexpr int HI_ESPLIT = 4, HI_SMS = 32;
  auto cap_mid_of = [&](int j) { return std::min(48, std::max(8, (8 * (nt - j) + 15) / 16)); };

  // FP64 products of the newest term k = j - 1 into rows [r0, r1) of column j
  auto new_dgemm = [&](int j, int r0, int r1, bool on_mid) {
    const int knew = j - 1, par = j & 1;
    if (knew < 0) return;
    std::vector<DJob> js;
    for (int i = r0; i < r1; ++i) {
      if (cls[tidx(i, j)] != CR_PREC_FP64) continue;
      if (!(cls[tidx(i, knew)] == CR_PREC_FP64 && cls[tidx(j, knew)] == CR_PREC_FP64)) continue;
      const int p = P.add_pair(t64(i, knew), t64(j, knew), nb, 1, nb, 1, nb);
      double* C = i == j ? t64(i, j) : ws64(par, i);
      for (int bi = 0; bi < nb / 64; ++bi)
        for (int bj = 0; bj < nb / 64; ++bj) {
          if (i == j && bj > bi) continue;
          js.push_back(job(C + (size_t)bi * 64 * nb + bj * 64, nb, 1, 64, 64, p, 1, -1.0, 1.0, bi * 64, bj * 64, nb));
        }
    }
    P.dgemm(64, js, false, on_mid);
  };
  // solves of rows [r0, r1) of column j: tensor cores for FP16/FP32-class tiles (rows list at
  // d_rows + off, cnt entries), FP64 products with the inverse for FP64-class tiles
  auto solves = [&](int j, int r0, int r1, const TcParams& tp, int off, int cnt, bool on_mid, int cap_mid) {
    const int par = j & 1;
    if (cnt > 0) {
      TcParams t = tp;
      t.mode = TC_TRSM;
      t.rows = d_rows + off;
      t.nrows = cnt;
      t.max_ctas = on_mid ? cap_mid : 0;
      t.esplit = on_mid ? 1 : HI_ESPLIT;
      P.ops.push_back([=](Exec& x) -> cr_status { return tc_launch(t, *tm, *tm, on_mid ? x.mid : x.hi); });
    }
    std::vector<DJob> js;
    std::vector<int> fp64_rows;
    double* Minv = V->minv + (size_t)par * nb2;
    for (int i = r0; i < r1; ++i) {
      if (cls[tidx(i, j)] != CR_PREC_FP64) continue;
      fp64_rows.push_back(i);
      const int p = P.add_pair(ws64(par, i), Minv, nb, 1, nb, 1, nb);
      double* C = t64(i, j);
      for (int bi = 0; bi < nb / 64; ++bi)
        for (int bj = 0; bj < nb / 64; ++bj)
          js.push_back(job(C + (size_t)bi * 64 * nb + bj * 64, nb, 1, 64, 64, p, 1, 1.0, 0.0, bi * 64, bj * 64, (bj + 1) * 64));
    }
    P.dgemm(64, js, false, on_mid);
    if (V->amp) {
      for (int i : fp64_rows) {
        const double* src = t64(i, j);
        __half* h = V->pool16 + (size_t)V->h_hi16[tidx(i, j)] * nb2;
        __half* l = V->pool16 + (size_t)V->h_lo16[tidx(i, j)] * nb2;
        P.ops.push_back([=](Exec& x) -> cr_status { return split_tile_launch(src, nb, h, l, 0, on_mid ? x.mid : x.hi); });
      }
    }
  };

  for (int j = 0; j < nt; ++j) {
    const int par = j & 1;
    const int knew = j - 1;                  // newest term (none for j = 0)
    const int kold_end = j > 0 ? j - 1 : 0;  // older terms [0, kold_end)
    TcParams tp = base;
    tp.j = j;
    tp.ws_hi0 = V->ws_hi0 + par * nt;
    tp.ws_lo0 = V->ws_lo0 + par * nt;
    tp.minv_hi = V->minv_hi + par;
    tp.minv_lo = V->minv_lo + par;
    tp.status = V->d_status + par;           // status[2 + par]: exponent of this column's scaled inverse
    tp.ws64 = V->ws64 ? ws64(par, 0) : nullptr;
    tp.w32 = V->w32 ? V->w32 + (size_t)par * nt * nb2 : nullptr;
    const int cap_mid = cap_mid_of(j), cap_lo = std::max(1, sms - cap_mid - HI_SMS);

    // ---------------- OLD(j) on the low-priority stream: needs columns <= j-2 complete
    const int grange = gen_range_of[j];
    P.ops.push_back([=](Exec& x) -> cr_status {
      if (j >= 2) {
        CR_CUDA(cudaStreamWaitEvent(x.lo, x.ev_crit[j - 2], 0));
        CR_CUDA(cudaStreamWaitEvent(x.lo, x.ev_rest[j - 2], 0));
      } else {
        CR_CUDA(cudaStreamWaitEvent(x.lo, x.start, 0));
      }
      // column j's tiles (every later use of them is ordered after OLD(j))
      CR_CUDA(cudaStreamWaitEvent(x.lo, x.ev_gen[grange], 0));
      return CR_OK;
    });
    {
      std::vector<DJob> js;
      for (int i = j; i < nt; ++i) {
        if (cls[tidx(i, j)] != CR_PREC_FP64) continue;
        const int pbeg = (int)P.pairs.size();
        for (int k = 0; k < kold_end; ++k)
          if (cls[tidx(i, k)] == CR_PREC_FP64 && cls[tidx(j, k)] == CR_PREC_FP64)
            P.add_pair(t64(i, k), t64(j, k), nb, 1, nb, 1, nb);
        const int pcnt = (int)P.pairs.size() - pbeg;
        if (pcnt == 0) continue;
        double* C = t64(i, j);
        for (int bi = 0; bi < nb / 64; ++bi)
          for (int bj = 0; bj < nb / 64; ++bj) {
            if (i == j && bj > bi) continue;
            js.push_back(job(C + (size_t)bi * 64 * nb + bj * 64, nb, 1, 64, 64, pbeg, pcnt, -1.0, 1.0, bi * 64, bj * 64, nb));
          }
      }
      P.dgemm(64, js, true);
    }
    if (V->amp) {
      TcParams t = tp;
      t.mode = TC_UPD_OLD;
      t.kbeg = 0;
      t.kend = kold_end;
      // without old terms the FP64 diagonal tile is already what its factorisation needs: it
      // is left out (the critical stream then waits only for its generation, below)
      t.row0 = kold_end == 0 ? j + 1 : j;
      t.nrows = nt - t.row0;
      t.max_ctas = cap_lo;
      if (t.nrows > 0) P.ops.push_back([=](Exec& x) -> cr_status { return tc_launch(t, *tm, *tm, x.lo); });
    } else {
      for (int i = j + 1; i < nt; ++i) {
        double* dst = ws64(par, i);
        const double* src = t64(i, j);
        P.ops.push_back([=](Exec& x) -> cr_status {
          CR_CUDA(cudaMemcpyAsync(dst, src, nb2 * sizeof(double), cudaMemcpyDeviceToDevice, x.lo));
          return CR_OK;
        });
      }
    }
    P.ops.push_back([=](Exec& x) -> cr_status { CR_CUDA(cudaEventRecord(x.ev_old[j], x.lo)); return CR_OK; });

    // ---------------- lookahead stream, part 1: NEW(j) for rows j+1.. (needs OLD(j) and the
    // solve of row j of column j-1, which is on the critical stream)
    P.ops.push_back([=](Exec& x) -> cr_status {
      CR_CUDA(cudaStreamWaitEvent(x.mid, x.ev_old[j], 0));
      if (j >= 1) CR_CUDA(cudaStreamWaitEvent(x.mid, x.ev_crit[j - 1], 0));
      return CR_OK;
    });
    new_dgemm(j, j + 1, nt, true);
    if (V->amp && j + 1 < nt) {
      TcParams t = tp;
      t.mode = TC_UPD_NEW;
      t.kbeg = knew >= 0 ? knew : 0;
      t.kend = knew >= 0 ? j : 0;
      t.row0 = j + 1;
      t.nrows = nt - j - 1;
      t.max_ctas = cap_mid;
      P.ops.push_back([=](Exec& x) -> cr_status { return tc_launch(t, *tm, *tm, x.mid); });
    }
    P.ops.push_back([=](Exec& x) -> cr_status { CR_CUDA(cudaEventRecord(x.ev_newr[j], x.mid)); return CR_OK; });

    // ---------------- critical stream: NEW(j) for the diagonal tile, its factor and inverse
    if (V->amp && kold_end == 0) {
      // the diagonal tile has no old terms: its generation is all the critical stream waits for
      P.ops.push_back([=](Exec& x) -> cr_status {
        CR_CUDA(cudaStreamWaitEvent(x.hi, x.ev_gdiag[grange], 0));
        CR_CUDA(cudaStreamWaitEvent(x.hi, x.start, 0));
        return CR_OK;
      });
    } else {
      P.ops.push_back([=](Exec& x) -> cr_status { CR_CUDA(cudaStreamWaitEvent(x.hi, x.ev_old[j], 0)); return CR_OK; });
    }
    new_dgemm(j, j, j + 1, false);
    if (V->amp) {
      TcParams t = tp;
      t.mode = TC_UPD_NEW;
      t.kbeg = knew >= 0 ? knew : 0;
      t.kend = knew >= 0 ? j : 0;
      t.row0 = j;
      t.nrows = 1;
      t.esplit = HI_ESPLIT;
      P.ops.push_back([=](Exec& x) -> cr_status { return tc_launch(t, *tm, *tm, x.hi); });
    }
    double* Ajj = t64(j, j);
    double* Minv = V->minv + (size_t)par * nb2;
    unsigned long long* amax = reinterpret_cast<unsigned long long*>(V->minv_part);
    double* W = V->scratch64;
    {
      const int db = V->diag_db, ntask = V->diag_ntasks, g = j * nb;
      // one executor CTA per SM: the chain CTA plus one worker per remaining SM
      int dgrid = 0;
      CR_CUDA(cudaDeviceGetAttribute(&dgrid, cudaDevAttrMultiProcessorCount, V->device));
      int* flags = V->diag_flags;
      const int4* tasks = V->diag_tasks;
      if (use_df) {
        // double-float executor, then one kernel writing the FP64 factor and inverse and their
        // FP16 high/low parts (amp only)
        float2* Ldf = V->diag_df;
        float2* Mdf = V->diag_df + nb2;
        float2* Wdf = reinterpret_cast<float2*>(W);
        __half *mh = nullptr, *ml = nullptr, *dh = nullptr, *dl = nullptr;
        if (V->amp) {
          mh = V->pool16 + (size_t)(V->minv_hi + par) * nb2;
          ml = V->pool16 + (size_t)(V->minv_lo + par) * nb2;
          dh = V->pool16 + (size_t)V->h_hi16[tidx(j, j)] * nb2;
          dl = V->pool16 + (size_t)V->h_lo16[tidx(j, j)] * nb2;
        }
        int* st_par = status + par;
        P.ops.push_back([=](Exec& x) -> cr_status {
          CR_TRY(diag_chol_df_launch(db, Ajj, Ldf, Mdf, Wdf, nb, g, status, flags, par, dpub, tasks, ntask, dgrid, amax,
                                     wait_ns, x.hi));
          return split_diag_df_launch(Mdf, Ldf, nb, amax + par, Minv, Ajj, mh, ml, dh, dl, st_par, x.hi);
        });
      } else {
        P.ops.push_back([=](Exec& x) -> cr_status {
          // the executor zeroes the upper parts of Ajj and Minv and clears the other parity's
          // flags and abs-max for the next column
          return diag_chol_launch(db, Ajj, Minv, W, nb, g, status, flags, par, dpub, tasks, ntask, dgrid, amax, wait_ns,
                                  x.hi);
        });
      }
      if (V->minv_all) {
        double* keep = V->minv_all + (size_t)j * nb2;
        P.ops.push_back([=](Exec& x) -> cr_status {
          CR_CUDA(cudaMemcpyAsync(keep, Minv, nb2 * sizeof(double), cudaMemcpyDeviceToDevice, x.hi));
          return CR_OK;
        });
      }
    }
    if (V->amp && !use_df) {
      __half* mh = V->pool16 + (size_t)(V->minv_hi + par) * nb2;
      __half* ml = V->pool16 + (size_t)(V->minv_lo + par) * nb2;
      __half* dh = V->pool16 + (size_t)V->h_hi16[tidx(j, j)] * nb2;
      __half* dl = V->pool16 + (size_t)V->h_lo16[tidx(j, j)] * nb2;
      int* st_par = status + par;
      P.ops.push_back([=](Exec& x) -> cr_status { return split_diag_launch(Minv, Ajj, nb, amax + par, mh, ml, dh, dl, st_par, x.hi); });
    }
    P.ops.push_back([=](Exec& x) -> cr_status { CR_CUDA(cudaEventRecord(x.ev_split[j], x.hi)); return CR_OK; });
    // the solve of row j+1 (its update is on the lookahead stream) feeds the next column
    P.ops.push_back([=](Exec& x) -> cr_status { CR_CUDA(cudaStreamWaitEvent(x.hi, x.ev_newr[j], 0)); return CR_OK; });
    {
      const int off = rows_off[j];
      const int cnt = (rows_off[j + 1] > off && j + 1 < nt && rows_flat[off] == j + 1) ? 1 : 0;
      solves(j, j + 1, std::min(nt, j + 2), tp, off, cnt, false, 0);
    }
    P.ops.push_back([=](Exec& x) -> cr_status { CR_CUDA(cudaEventRecord(x.ev_crit[j], x.hi)); return CR_OK; });

    // ---------------- lookahead stream, part 2: solves of rows j+2.. once the inverse is split
    P.ops.push_back([=](Exec& x) -> cr_status { CR_CUDA(cudaStreamWaitEvent(x.mid, x.ev_split[j], 0)); return CR_OK; });
    {
      int off = rows_off[j];
      if (rows_off[j + 1] > off && rows_flat[off] == j + 1) ++off;
      solves(j, j + 2, nt, tp, off, rows_off[j + 1] - off, true, cap_mid);
    }
    P.ops.push_back([=](Exec& x) -> cr_status { CR_CUDA(cudaEventRecord(x.ev_rest[j], x.mid)); return CR_OK; });
  }

  // streams, events, job upload, replay
  cr_status st = CR_OK;
  // job and pair lists in one device buffer kept by the tile matrix
  const size_t jobs_bytes = (P.jobs.size() * sizeof(DJob) + 255) & ~(size_t)255;
  const size_t need = jobs_bytes + P.pairs.size() * sizeof(DPair);
  if (need > V->sched_jobs_cap) {
    if (V->sched_jobs) cudaFree(V->sched_jobs);
    V->sched_jobs = nullptr;
    V->sched_jobs_cap = 0;
    if (cudaMalloc(&V->sched_jobs, need) != cudaSuccess) {
      V->sched_jobs = nullptr;
      st = fail(CR_ERR_NOMEM, "job list");
    } else {
      V->sched_jobs_cap = need;
    }
  }
  DJob* d_jobs = P.jobs.empty() || !V->sched_jobs ? nullptr : reinterpret_cast<DJob*>(V->sched_jobs);
  DPair* d_pairs = P.pairs.empty() || !V->sched_jobs
                       ? nullptr
                       : reinterpret_cast<DPair*>(reinterpret_cast<char*>(V->sched_jobs) + jobs_bytes);
  if (st == CR_OK && d_jobs)
    if (cudaMemcpyAsync(d_jobs, P.jobs.data(), P.jobs.size() * sizeof(DJob), cudaMemcpyHostToDevice, caller) != cudaSuccess)
      st = fail(CR_ERR_CUDA, "job upload");
  if (st == CR_OK && d_pairs)
    if (cudaMemcpyAsync(d_pairs, P.pairs.data(), P.pairs.size() * sizeof(DPair), cudaMemcpyHostToDevice, caller) != cudaSuccess)
      st = fail(CR_ERR_CUDA, "pair upload");
  x.dj = d_jobs;
  x.dp = d_pairs;
  if (st == CR_OK) {
    // the schedule's streams start after the job and pair uploads
    cudaEventRecord(x.start1, caller);
    cudaStreamWaitEvent(x.hi, x.start1, 0);
    cudaStreamWaitEvent(x.lo, x.start1, 0);
    cudaStreamWaitEvent(x.mid, x.start1, 0);
  }
  for (size_t q = 0; st == CR_OK && q < P.ops.size(); ++q) st = P.ops[q](x);
  cudaError_t e1 = cudaStreamSynchronize(x.hi);
  cudaError_t e2 = cudaStreamSynchronize(x.lo);
  cudaError_t e3 = cudaStreamSynchronize(x.mid);
  cudaError_t e4 = cudaStreamSynchronize(x.gen);
  if (st == CR_OK && e4 != cudaSuccess) st = cuda_fail(e4, "tile generation");
  if (st == CR_OK && e1 != cudaSuccess) st = cuda_fail(e1, "cholesky (critical stream)");
  if (st == CR_OK && e2 != cudaSuccess) st = cuda_fail(e2, "cholesky (bulk stream)");
  if (st == CR_OK && e3 != cudaSuccess) st = cuda_fail(e3, "cholesky (lookahead stream)");
  return st;
}

}  // namespace cr

using namespace cr;

extern "C" cr_status cr_potrf_adaptive(cr_tilemat V, cr_stream stream, int* info) {
  if (!V) return fail(CR_ERR_ARG, "cr_potrf_adaptive: NULL handle");
  if (info) *info = 0;
  if (!V->mapped) return fail(CR_ERR_STATE, "cr_potrf_adaptive: call cr_precision_map first");
  CR_CUDA(cudaSetDevice(V->device));
  // block size of the diagonal-tile dataflow factorisation
  const int db = 16;
  if (db != V->diag_db) {
    if (V->diag_tasks) cudaFree(V->diag_tasks);
    if (V->diag_flags) cudaFree(V->diag_flags);
    if (V->diag_pub) cudaFree(V->diag_pub);
    V->diag_pub = nullptr;
    V->diag_tasks = nullptr;
    V->diag_flags = nullptr;
    std::vector<int4> tasks;
    if (!diag_task_list(V->nb / db, tasks)) return fail(CR_ERR_STATE, "cr_potrf_adaptive: diagonal task list failed its progress check");
    CR_CUDA(cudaMalloc(&V->diag_tasks, tasks.size() * sizeof(int4)));
    CR_CUDA(cudaMemcpy(V->diag_tasks, tasks.data(), tasks.size() * sizeof(int4), cudaMemcpyHostToDevice));
    CR_CUDA(cudaMalloc(&V->diag_flags, 2 * (size_t)diag_flag_words(V->nb, db) * sizeof(int)));
    CR_CUDA(cudaMalloc(&V->diag_pub, diag_pub_doubles(V->nb, db) * sizeof(double)));
    V->diag_ntasks = (int)tasks.size();
    V->diag_db = db;
  }
  if (!V->minv_part) CR_CUDA(cudaMalloc(&V->minv_part, 64 * sizeof(double)));
  CR_TRY(build_and_run_cholesky(V, stream));
  int h[4];
  CR_CUDA(cudaMemcpy(h, V->d_status, sizeof(h), cudaMemcpyDeviceToHost));
  V->info = h[1] == 0x7fffffff ? 0 : h[1];
  if (info) *info = V->info;
  if (h[0] & DEV_ERR_TIMEOUT) return fail(CR_ERR_TIMEOUT, "cr_potrf_adaptive: a device-side wait timed out");
  if (V->info) return fail(CR_ERR_NOT_SPD, "cr_potrf_adaptive: leading minor not positive definite at column " + std::to_string(V->info));
  V->factored = true;
  return CR_OK;
}
