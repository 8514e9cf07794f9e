"""Universal kriging and the conditional pipeline on the GPU against the oracle
("Mixed-Precision GPU Acceleration for Confidence Regions of Spatial Excursion Sets",
Section V-A Eq.5-6, Section V-B Eq.7, Section V-C)."""
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


def relf(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


def _case(n_o, m, seed, nu=1.0, beta=0.1, tau2=0.01):
    pred = inputgen.morton_sorted(inputgen.grid_cell_centres(m))
    obs = inputgen.morton_sorted(inputgen.uniform_locations(n_o, seed))
    xy = np.ascontiguousarray(np.concatenate([pred, obs]))
    n_p = len(pred)
    X = np.column_stack([np.ones(len(xy)), xy[:, 0], xy[:, 1]])
    y = inputgen.observation_values(obs, (1.0, 0.5, -0.3), 0.3, seed + 1)
    V = oracle.covariance_matrix(xy, "matern", 1.0, beta, nu, 0.0, n_p, tau2)
    return xy, n_p, X, y, V


@pytest.mark.parametrize("n_o,m,nb", [(1024, 32, 128), (1000, 24, 128), (4096, 64, 512)])
def test_kriging_matches_oracle(lib, n_o, m, nb):
    xy, n_p, X, y, V = _case(n_o, m, 5)
    G = lib.TileMat(len(xy), nb)
    lib.cov_build(G, dev(xy), "matern", 1.0, 0.1, 1.0, nugget=0.0, n_pred=n_p, tau2=0.01)
    W, z, v = lib.krige(G, colmajor(X[n_p:]), colmajor(X[:n_p]), dev(y))
    Wo, zo, vo = oracle.universal_kriging(V[n_p:, n_p:], V[n_p:, :n_p], X[n_p:], X[:n_p], y, 1.0)
    # two FP64 orderings of the same solves; the bordered-system solve gives the noise scale
    K = np.block([[V[n_p:, n_p:], X[n_p:]], [X[n_p:].T, np.zeros((3, 3))]])
    Wl = np.linalg.solve(K, np.vstack([V[n_p:, :n_p], X[:n_p].T]))[:n_o]
    tol = max(1e-10, 20 * relf(Wl, Wo))
    Wg = W.cpu().numpy()
    assert relf(Wg, Wo) <= tol, (relf(Wg, Wo), tol)
    assert relf(z.cpu().numpy(), zo) <= tol
    assert np.max(np.abs(v.cpu().numpy() - vo)) <= 1e-9
    np.testing.assert_allclose(X[n_p:].T @ Wg, X[:n_p].T, atol=1e-8)      # unbiasedness X_o^T W = X_p^T
    G.close()


def test_conditional_pipeline_regions_match_oracle(lib):
    """Kriging, FP64 simulation of the joint field, correction and calibration, end to end."""
    n_o, m, nb, M, u, level = 512, 24, 128, 400, 1.3, 0.9
    xy, n_p, X, y, V = _case(n_o, m, 7)
    n = len(xy)
    G = lib.TileMat(n, nb)
    lib.cov_build(G, dev(xy), "matern", 1.0, 0.1, 1.0, nugget=0.0, n_pred=n_p, tau2=0.01)
    W, z, v = lib.krige(G, colmajor(X[n_p:]), colmajor(X[:n_p]), dev(y))
    lib.precision_map(G, amp=False)
    assert lib.potrf_adaptive(G) == 0
    Z = inputgen.standard_normals(n, M, 11)
    Yg = lib.trmm_sim(G, colmajor(Z), M)
    S = lib.krige_correct(W, dev(y), Yg, n_p, n_o)
    out = lib.calibrate(S, z, v, u, level, counts=True)
    # oracle on the GPU's own kriging outputs and simulations: the calibration is exact
    Sg = S.cpu().numpy()
    ref = oracle.calibrate(Sg, z.cpu().numpy(), v.cpu().numpy(), u, level)
    assert out["q_in"] == ref["q_in"] and out["q_out"] == ref["q_out"]
    np.testing.assert_array_equal(out["c_in"].cpu().numpy(), ref["c_in"])
    np.testing.assert_array_equal(out["c_out"].cpu().numpy(), ref["c_out"])
    np.testing.assert_array_equal(out["count"].cpu().numpy(), ref["count"])
    # and the whole chain against the oracle's own FP64 chain
    Wo, zo, vo = oracle.universal_kriging(V[n_p:, n_p:], V[n_p:, :n_p], X[n_p:], X[:n_p], y, 1.0)
    Yo = oracle.simulate(oracle.cholesky_lower(V), Z)
    So = oracle.conditional_correction(Wo, y, Yo[:n_p], Yo[n_p:])
    assert relf(Sg, So) <= 1e-9
    full = oracle.calibrate(So, zo, vo, u, level)
    diff_in = np.mean(out["c_in"].cpu().numpy() != full["c_in"])
    diff_out = np.mean(out["c_out"].cpu().numpy() != full["c_out"])
    assert diff_in <= 0.01 and diff_out <= 0.01
    G.close()
