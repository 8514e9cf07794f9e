"""The pages' own synthetic workload end to end on the GPU, mixed precision (automatic
tolerance) against the all-FP64 chain ("Mixed-Precision GPU Acceleration for Confidence
Regions of Spatial Excursion Sets", Section VI-B and the region-inclusion differences it
reports between the DP and MP runs).

Geometry of Section VI-B.1: 3200 uniform observations and a 120 x 120 grid of prediction
cells (n = 17,600), power-exponential covariance (sigma^2 = 1, nu = 0.5, range 0.033, 0.1
and 0.234: the weak, medium and strong correlation levels), trend b = (0, 15, 10), threshold
u = 10, level 0.90.  The measurement noise of the observations is not stated on the pages;
tau^2 = 0.01 is used.
Both chains share the kriging weights, the truths (drawn with the FP64 factor) and the
N(0,1) draws; they differ only in the factor and the simulation multiply."""
import numpy as np
import pytest
import torch

import inputgen
import oracle

pytestmark = pytest.mark.gpu


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def colmajor(a):
    return torch.from_numpy(np.asfortranarray(a).T.copy()).cuda().T


@pytest.mark.parametrize("beta", [0.033, 0.1, 0.234])
def test_paper_workload_auto_mixed_precision_against_fp64(lib, beta):
    m, n_o, nb, M, R = 120, 3200, 512, 1024, 8
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

    # kriging weights and MSPEs (FP64, from the covariance) before either factorisation
    G64 = build()
    W, _, v = lib.krige(G64, colmajor(X[n_p:]), colmajor(X[:n_p]), dev(np.zeros(n_o)))
    lib.precision_map(G64, amp=False)
    assert lib.potrf_adaptive(G64) == 0
    G16 = build()
    pmap, info = lib.precision_map(G16, amp=True, auto=True)
    # automatic tolerance: refined until both FP16 checks pass or no FP16 tile is left
    assert info["iters"] >= 1 and ((info["check1"] and info["check2"]) or info["n_fp16"] == 0), info
    assert lib.potrf_adaptive(G16) == 0
    zero_col = colmajor(np.zeros((n, 1)))
    mean = X @ b

    diffs, hits64, hits16 = [], 0, 0
    for r in range(R):
        eta = lib.rnorm(n, 1, 1000 + r)
        truth = mean + lib.trmm_sim(G64, eta, 1)[:, 0].cpu().numpy()
        y = dev(truth[n_p:])
        Z = lib.rnorm(n, M, 5000 + r)
        z = lib.krige_correct(W, y, zero_col, n_p, n_o)[:, 0].contiguous()
        out = {}
        for name, G in (("fp64", G64), ("mp", G16)):
            S = lib.krige_correct(W, y, lib.trmm_sim(G, Z, M), n_p, n_o)
            res = lib.calibrate(S, z, v, u, level)
            out[name] = (res["c_in"].cpu().numpy(), res["c_out"].cpu().numpy())
        diffs.append((np.mean(out["fp64"][0] != out["mp"][0]), np.mean(out["fp64"][1] != out["mp"][1])))
        hits64 += oracle.coverage_event(truth[:n_p], *out["fp64"], u)
        hits16 += oracle.coverage_event(truth[:n_p], *out["mp"], u)
    G64.close()
    G16.close()
    d = np.array(diffs)
    msg = (f"range {beta}: auto fixedacc {info['fixedacc']:.3g} after {info['iters']} steps, tiles fp64/32/16 "
           f"{info['n_fp64']}/{info['n_fp32']}/{info['n_fp16']}; region differences MP vs FP64: inner mean "
           f"{100 * d[:, 0].mean():.3f} % max {100 * d[:, 0].max():.3f} %, outer mean {100 * d[:, 1].mean():.3f} % "
           f"max {100 * d[:, 1].max():.3f} %; coverage over {R} replicates fp64 {hits64 / R:.3f} mp {hits16 / R:.3f}")
    print(msg)
    # the pages report 0.03-0.54 % of the sites changing region between the DP and MP runs
    assert d.max() <= 0.01, msg
    assert abs(hits64 - hits16) <= 1, msg


def test_paper_workload_fixedacc_against_oracle_fp64_chain(lib):
    """The weak-correlation level of the pages' workload (range 0.033, the one with FP16-class
    tiles) at the pages' user tolerance fixedacc = 1e-4, the GPU's mixed-precision chain against
    the oracle's own FP64 chain: the oracle's covariance, unblocked Cholesky, kriging (Eq.5-6),
    simulation, correction (Eq.7) and calibration.  Both chains see the same truths (drawn with
    the oracle's factor) and the same N(0,1) draws.  North-star gate: region membership differs
    at <= 1 % of the sites (the pages report 0.03-0.54 % between their DP and MP runs)."""
    m, n_o, nb, M, R = 120, 3200, 512, 512, 2
    beta, nu, tau2, u, level, fixedacc = 0.033, 0.5, 0.01, 10.0, 0.90, 1e-4
    b = np.array([0.0, 15.0, 10.0])
    pred = inputgen.morton_sorted(inputgen.grid_cell_centres(m))
    obs = inputgen.morton_sorted(inputgen.uniform_locations(n_o, 51))
    xy = np.ascontiguousarray(np.concatenate([pred, obs]))
    n_p, n = len(pred), len(xy)
    X = np.column_stack([np.ones(n), xy[:, 0], xy[:, 1]])
    mean = X @ b
    # the oracle's FP64 chain pieces
    Vo = oracle.covariance_matrix(xy, "powexp", 1.0, beta, nu, 0.0, n_p, tau2)
    Lo = oracle.cholesky_lower(Vo)
    # the GPU's mixed-precision chain at the user tolerance
    G = lib.TileMat(n, nb)
    lib.cov_build(G, dev(xy), "powexp", 1.0, beta, nu, nugget=0.0, n_pred=n_p, tau2=tau2)
    W, _, v = lib.krige(G, colmajor(X[n_p:]), colmajor(X[:n_p]), dev(np.zeros(n_o)))
    pmap, info = lib.precision_map(G, amp=True, fixedacc=fixedacc)
    assert info["n_fp16"] > 0, info
    assert lib.potrf_adaptive(G) == 0
    zero_col = colmajor(np.zeros((n, 1)))
    diffs = []
    for r in range(R):
        truth = mean + Lo @ inputgen.standard_normals(n, 1, 1000 + r)[:, 0]
        yo = truth[n_p:]
        Z = inputgen.standard_normals(n, M, 5000 + r)
        # GPU chain
        y = dev(yo)
        z = lib.krige_correct(W, y, zero_col, n_p, n_o)[:, 0].contiguous()
        S = lib.krige_correct(W, y, lib.trmm_sim(G, colmajor(Z), M), n_p, n_o)
        got = lib.calibrate(S, z, v, u, level)
        # oracle chain
        Wo, zo, vo = oracle.universal_kriging(Vo[n_p:, n_p:], Vo[n_p:, :n_p], X[n_p:], X[:n_p], yo, 1.0)
        Yo = oracle.simulate(Lo, Z)
        So = oracle.conditional_correction(Wo, yo, Yo[:n_p], Yo[n_p:])
        ref = oracle.calibrate(So, zo, vo, u, level)
        diffs.append((np.mean(got["c_in"].cpu().numpy() != ref["c_in"]), np.mean(got["c_out"].cpu().numpy() != ref["c_out"])))
    G.close()
    d = np.array(diffs)
    msg = (f"fixedacc {fixedacc}: tiles fp64/32/16 {info['n_fp64']}/{info['n_fp32']}/{info['n_fp16']}, checks "
           f"{info['check1']}/{info['check2']}; sites changing region, GPU mixed precision vs oracle FP64: inner "
           f"{100 * d[:, 0].mean():.3f} % (max {100 * d[:, 0].max():.3f} %), outer {100 * d[:, 1].mean():.3f} % "
           f"(max {100 * d[:, 1].max():.3f} %) over {R} replicates")
    print(msg)
    assert d.max() <= 0.01, msg
