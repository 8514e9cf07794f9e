"""The pages' coverage study at their own size ("Mixed-Precision GPU Acceleration for Confidence
Regions of Spatial Excursion Sets", Section VI-B.2 and Fig. 3): 1000 replicates per correlation
level, nsim = 80,000 conditional simulations each, adaptive mixed precision with the automatic
tolerance (A7: the map refined until the FP16 checks pass), or at a fixed tolerance
(CR_PAPER_COVERAGE_FIXEDACC).

Geometry of Section VI-B.1: 3200 uniform observations (one fixed seed) and a 120 x 120 grid of
prediction cells (n = 17,600), power-exponential covariance (sigma^2 = 1, nu = 0.5, range 0.033,
0.1 and 0.234), trend b = (0, 15, 10), threshold u = 10, level 0.90; the observation noise is
not stated on the pages, tau^2 = 0.01 is used (as in the paper-workload test).  The locations
are fixed, so the kriging weights, the MSPEs and both factors are computed once per level; each
replicate draws a new truth Z = X b + L eta (L the all-FP64 factor) and new simulations
(cr_rnorm inside the simulation multiply), and the correction runs as the Ozaki product.  The
test counts the inner event (C_in inside the truth's excursion set A, Fig. 3a), the outer one
(A inside C_out, Fig. 3b) and both together (the criterion of the text).

The study takes minutes of GPU time per level, so it runs only when CR_PAPER_COVERAGE names the
ranges to study (e.g. "0.033,0.1,0.234"); CR_PAPER_COVERAGE_R and CR_PAPER_COVERAGE_NSIM
override the replicate and simulation counts.  At fixedacc 1e-4 this geometry's map has no
FP16 tile (at range 0.1: 35 FP64, 595 FP32), so the default is the automatic tolerance, whose
maps do (the pages' Fig. 5 shares are for that mode)."""
import os
import time

import numpy as np
import pytest
import torch

import inputgen
import oracle

pytestmark = pytest.mark.gpu

RANGES = [float(x) for x in os.environ.get("CR_PAPER_COVERAGE", "").split(",") if x.strip()]
R_REPLICATES = int(os.environ.get("CR_PAPER_COVERAGE_R", "1000"))
NSIM = int(os.environ.get("CR_PAPER_COVERAGE_NSIM", "80000"))
FIXEDACC = os.environ.get("CR_PAPER_COVERAGE_FIXEDACC", "")


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def colmajor(a):
    return torch.from_numpy(np.asfortranarray(a).T.copy()).cuda().T


@pytest.mark.skipif(not RANGES, reason="the full coverage study runs only with CR_PAPER_COVERAGE set")
@pytest.mark.parametrize("beta", RANGES or [0.1])
def test_paper_coverage_study(lib, beta):
    m, n_o, nb = 120, 3200, 512
    nu, tau2, u, level = 0.5, 0.01, 10.0, 0.90
    b = np.array([0.0, 15.0, 10.0])
    pred = inputgen.morton_sorted(inputgen.grid_cell_centres(m))
    obs = inputgen.morton_sorted(inputgen.uniform_locations(n_o, 51))
    xy = np.ascontiguousarray(np.concatenate([pred, obs]))
    n_p, n = len(pred), len(xy)
    X = np.column_stack([np.ones(n), xy[:, 0], xy[:, 1]])

    def build():
        G = lib.TileMat(n, nb)
        lib.cov_build(G, dev(xy), "powexp", 1.0, beta, nu, nugget=0.0, n_pred=n_p, tau2=tau2)
        return G

    old = lib.get_option(lib.CR_OPT_FP64_GEMM)
    lib.set_option(lib.CR_OPT_FP64_GEMM, lib.CR_GEMM_OZAKI)
    try:
        G64 = build()
        W, _, v = lib.krige(G64, colmajor(X[n_p:]), colmajor(X[:n_p]), dev(np.zeros(n_o)))
        lib.precision_map(G64, amp=False)
        assert lib.potrf_adaptive(G64) == 0
        G16 = build()
        if FIXEDACC:
            pmap, info = lib.precision_map(G16, amp=True, fixedacc=float(FIXEDACC))
        else:
            pmap, info = lib.precision_map(G16, amp=True, auto=True)
        assert lib.potrf_adaptive(G16) == 0
        # every replicate's truth at once: Z = X b + L eta (FP64 factor, FP64 multiply)
        truths = lib.trmm_sim(G64, lib.rnorm(n, R_REPLICATES, 1000), R_REPLICATES)
        truths += dev(X @ b)[:, None]
        zero_col = colmajor(np.zeros((n, 1)))
        Y = lib.colmajor_empty(n, NSIM, torch.float64)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        hits = inner = outer = 0
        for r in range(R_REPLICATES):
            y = truths[n_p:, r].contiguous()
            z = lib.krige_correct(W, y, zero_col, n_p, n_o)[:, 0].contiguous()
            lib.trmm_sim(G16, None, NSIM, seed=5000 + r, out=Y, flags=lib.CR_TRMM_GENERATE)
            out = lib.correct_calibrate(W, y, Y, n_p, n_o, z, v, u, level)
            t_p, c_in, c_out = truths[:n_p, r].cpu().numpy(), out["c_in"].cpu().numpy(), out["c_out"].cpu().numpy()
            hits += oracle.coverage_event(t_p, c_in, c_out, u)
            inner += oracle.inner_event(t_p, c_in, u)
            outer += oracle.outer_event(t_p, c_out, u)
        torch.cuda.synchronize()
        secs = time.perf_counter() - t0
    finally:
        lib.set_option(lib.CR_OPT_FP64_GEMM, old)
    G64.close()
    G16.close()
    def rate(k):
        p = k / R_REPLICATES
        h = 1.96 * np.sqrt(p * (1.0 - p) / R_REPLICATES)
        return p, f"{p:.3f} [{p - h:.3f}, {p + h:.3f}]"

    (pi, si), (po, so), (pj, sj) = rate(inner), rate(outer), rate(hits)
    mode = "fixed" if FIXEDACC else "automatic"
    msg = (f"range {beta}: inner {si}, outer {so}, both {sj} over {R_REPLICATES} replicates of {NSIM} "
           f"simulations, {mode} tolerance {info['fixedacc']:g}, tiles fp64/32/16 "
           f"{info['n_fp64']}/{info['n_fp32']}/{info['n_fp16']}, {secs / R_REPLICATES:.3f} s per replicate")
    print(msg)
    # the pages' Fig. 3 shows inner and outer rates of about 0.83-0.91 for this study; the
    # bounds leave three binomial standard errors on either side at 1000 replicates
    if R_REPLICATES >= 1000:
        assert 0.80 <= pi <= 0.97 and 0.80 <= po <= 0.97, msg
        assert 0.75 <= pj <= 0.95, msg
