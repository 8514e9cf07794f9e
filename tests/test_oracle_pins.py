"""Pins of the oracle against things other than itself (CPU only).

Each test ties one oracle function to a closed form, a library routine on a special case,
brute force on a tiny input, or an invariant printed in "Mixed-Precision GPU Acceleration
for Confidence Regions of Spatial Excursion Sets".  A plausible mistake (dropped term,
wrong sign or index, transposed operand) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.linalg
import scipy.stats

import inputgen
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- covariance
@pytest.mark.parametrize("sigma2,beta", [(1.0, 0.1), (2.5, 0.03)])
def test_matern_half_integer_closed_forms(sigma2, beta):
    h = np.linspace(0.0, 1.0, 257)
    x = h / beta
    np.testing.assert_allclose(oracle.matern(h, sigma2, beta, 0.5), sigma2 * np.exp(-x), rtol=1e-13, atol=1e-300)
    np.testing.assert_allclose(oracle.matern(h, sigma2, beta, 1.5), sigma2 * (1 + x) * np.exp(-x), rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(oracle.matern(h, sigma2, beta, 2.5), sigma2 * (1 + x + x * x / 3) * np.exp(-x),
                               rtol=1e-12, atol=1e-300)


def test_matern_nu1_small_distance_limit_and_monotone():
    h = np.array([0.0, 1e-12, 1e-8, 1e-4, 0.01, 0.1, 1.0])
    c = oracle.matern(h, 1.0, 0.1, 1.0)
    assert c[0] == 1.0
    assert abs(c[1] - 1.0) < 1e-9 and abs(c[2] - 1.0) < 1e-6
    assert np.all(np.diff(c) < 0)
    # K_1(x) x -> 1 as x -> 0: C(h) = x K_1(x) for nu = 1, sigma2 = 1; at x = 1: K_1(1) = 0.6019072302
    np.testing.assert_allclose(oracle.matern(np.array([0.1]), 1.0, 0.1, 1.0), [0.6019072301972346], rtol=1e-12)


def test_powexp_definition_points():
    b = 0.234
    np.testing.assert_allclose(oracle.powexp(np.array([0.0, b, 2 * b]), 1.0, b, 0.5),
                               [1.0, math.exp(-1.0), math.exp(-math.sqrt(2.0))], rtol=1e-15)
    h = np.linspace(0, 1, 33)
    np.testing.assert_allclose(oracle.powexp(h, 1.3, 0.1, 1.0), oracle.matern(h, 1.3, 0.1, 0.5), rtol=1e-13)


def test_joint_covariance_hand_example():
    # 3-4-5 triangle: distances 3, 4, 5; exponential kernel with beta = 5
    xy = np.array([[0.0, 0.0], [3.0, 0.0], [0.0, 4.0]])
    V = oracle.covariance_matrix(xy, "matern", 2.0, 5.0, 0.5, nugget=0.1, n_pred=2, tau2=0.5)
    e = lambda d: 2.0 * math.exp(-d / 5.0)
    want = np.array([[2.1, e(3), e(4)], [e(3), 2.1, e(5)], [e(4), e(5), 2.6]])
    np.testing.assert_allclose(V, want, rtol=1e-15)
    # block extraction and entry sampling agree with the full matrix
    np.testing.assert_array_equal(oracle.covariance_matrix(xy, "matern", 2.0, 5.0, 0.5, 0.1, 2, 0.5,
                                                           rows=slice(1, 3), cols=slice(0, 2)), V[1:3, 0:2])
    r, c = np.array([0, 2, 1, 2]), np.array([0, 2, 2, 0])
    np.testing.assert_array_equal(oracle.covariance_entries(xy, r, c, "matern", 2.0, 5.0, 0.5, 0.1, 2, 0.5), V[r, c])


# ----------------------------------------------------------------------------- linear algebra
def test_cholesky_textbook_3x3():
    A = np.array([[4.0, 12.0, -16.0], [12.0, 37.0, -43.0], [-16.0, -43.0, 98.0]])
    np.testing.assert_array_equal(oracle.cholesky_lower(A), [[2, 0, 0], [6, 1, 0], [-8, 5, 3]])


def test_cholesky_matches_lapack_and_residual():
    xy = inputgen.morton_sorted(inputgen.uniform_locations(300, 7))
    V = oracle.covariance_matrix(xy, "matern", 1.0, 0.1, 0.5, nugget=1e-6)
    L = oracle.cholesky_lower(V)
    Lref = np.linalg.cholesky(V)
    assert np.linalg.norm(L - Lref) / np.linalg.norm(Lref) < 1e-13
    assert np.linalg.norm(L @ L.T - V) / np.linalg.norm(V) <= 1e-13
    assert np.all(np.triu(L, 1) == 0)


def test_cholesky_not_spd_column():
    A = np.eye(4)
    A[2, 2] = -1.0
    with pytest.raises(oracle.NotSPD) as ei:
        oracle.cholesky_lower(A)
    assert ei.value.column == 3


def test_triangular_solves_match_scipy():
    rng = np.random.default_rng(3)
    L = np.tril(rng.standard_normal((40, 40))) + 8 * np.eye(40)
    B = rng.standard_normal((40, 7))
    np.testing.assert_allclose(oracle.solve_lower(L, B), scipy.linalg.solve_triangular(L, B, lower=True), rtol=1e-12)
    np.testing.assert_allclose(oracle.solve_lower_transpose(L, B),
                               scipy.linalg.solve_triangular(L, B, lower=True, trans="T"), rtol=1e-12)
    np.testing.assert_allclose(oracle.solve_lower(L, B[:, 0]), scipy.linalg.solve_triangular(L, B[:, 0], lower=True),
                               rtol=1e-12)


# ----------------------------------------------------------------------------- simulation
def test_simulate_brute_force_and_compensation():
    rng = np.random.default_rng(5)
    L = np.tril(rng.standard_normal((5, 5)))
    Z = rng.standard_normal((5, 3))
    Y = oracle.simulate(L, Z)
    for i in range(5):
        for j in range(3):
            assert abs(Y[i, j] - sum(L[i, k] * Z[k, j] for k in range(i + 1))) < 1e-13
    s = 681.0  # compensation of Section V-E: (s L)(Z / s) = L Z
    np.testing.assert_allclose(oracle.simulate(s * L, Z / s), Y, rtol=1e-13, atol=1e-13)


def test_sample_covariance_converges_to_sigma():
    xy = inputgen.morton_sorted(inputgen.uniform_locations(40, 11))
    V = oracle.covariance_matrix(xy, "matern", 1.0, 0.2, 0.5, nugget=1e-4)
    L = oracle.cholesky_lower(V)
    errs = []
    for M in (1000, 10000, 100000):
        Y = oracle.simulate(L, inputgen.standard_normals(40, M, 99))
        errs.append(np.linalg.norm(Y @ Y.T / M - V) / np.linalg.norm(V))
    # error ~ M^-1/2: each tenfold increase cuts it by about sqrt(10)
    assert errs[1] < errs[0] / 2 and errs[2] < errs[1] / 2 and errs[2] < 0.02


def test_rng_splitmix64_reference_and_distribution():
    # SplitMix64 (Steele, Lea, Flood 2014) started from state 0: first output
    assert int(oracle.splitmix64(0, np.array([0], dtype=np.uint64))[0]) == 0xE220A8397B1DCDAF
    z = oracle.rnorm(1000, 100, seed=2024)
    assert z.shape == (1000, 100) and z.flags.f_contiguous
    flat = z.ravel(order="F")
    assert abs(flat.mean()) < 0.02 and abs(flat.var() - 1.0) < 0.02
    assert scipy.stats.kstest(flat, "norm").pvalue > 1e-3
    # the two members of a Box-Muller pair are uncorrelated
    assert abs(np.corrcoef(flat[0::2], flat[1::2])[0, 1]) < 0.02
    # offsets address the same stream
    np.testing.assert_array_equal(oracle.rnorm(10, 1, 2024, offset=1000).ravel(), flat[1000:1010])


# ----------------------------------------------------------------------------- kriging
def _krige_case(n_o=60, m=6, tau2=0.0, seed=3):
    obs = inputgen.uniform_locations(n_o, seed)
    pred = inputgen.grid_cell_centres(m)
    xy = np.concatenate([pred, obs])
    n_p = len(pred)
    V = oracle.covariance_matrix(xy, "matern", 1.0, 0.3, 1.0, nugget=0.0, n_pred=n_p, tau2=tau2)
    X = np.column_stack([np.ones(len(xy)), xy[:, 0], xy[:, 1]])
    return xy, n_p, V, X


def test_kriging_matches_bordered_system_and_is_unbiased():
    xy, n_p, V, X = _krige_case(tau2=0.01)
    Sy, Vop = V[n_p:, n_p:], V[n_p:, :n_p]
    Xo, Xp = X[n_p:], X[:n_p]
    y = inputgen.observation_values(xy[n_p:], (1.0, 0.5, -0.3), 0.3, 8)
    W, z, v = oracle.universal_kriging(Sy, Vop, Xo, Xp, y, 1.0)
    # universal kriging = the bordered (Lagrange) system solved by a library routine
    K = np.block([[Sy, Xo], [Xo.T, np.zeros((3, 3))]])
    sol = np.linalg.solve(K, np.vstack([Vop, Xp.T]))
    np.testing.assert_allclose(W, sol[:len(y)], rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(Xo.T @ W, Xp.T, atol=1e-10)          # X_o^T W = X_p^T (Section V-A)
    np.testing.assert_allclose(z, W.T @ y, rtol=1e-14)
    # MSPE = diagonal of the prediction-error covariance, by brute force per site
    for i in range(0, n_p, 7):
        w = W[:, i]
        want = V[i, i] + w @ Sy @ w - 2 * w @ Vop[:, i]
        assert abs(v[i] - want) < 1e-12


def test_kriging_interpolates_noise_free_data():
    obs = inputgen.uniform_locations(50, 4)
    pred = obs[:10].copy()              # predict exactly at observed sites
    xy = np.concatenate([pred, obs])
    V = oracle.covariance_matrix(xy, "matern", 1.0, 0.2, 0.5, n_pred=10, tau2=0.0)
    X = np.column_stack([np.ones(len(xy)), xy[:, 0], xy[:, 1]])
    y = inputgen.observation_values(obs, (1.0, 0.5, -0.3), 0.5, 1)
    W, z, v = oracle.universal_kriging(V[10:, 10:], V[10:, :10], X[10:], X[:10], y, 1.0)
    np.testing.assert_allclose(z, y[:10], atol=1e-9)
    np.testing.assert_allclose(v, 0.0, atol=1e-9)


def test_conditional_simulation_mean_and_variance_match_kriging():
    """Section V-B: in exact arithmetic E[S] = W^T y_o and diag Cov(S) = v."""
    xy, n_p, V, X = _krige_case(n_o=40, m=4, tau2=0.05, seed=21)
    Sy, Vop = V[n_p:, n_p:], V[n_p:, :n_p]
    y = inputgen.observation_values(xy[n_p:], (1.0, 0.5, -0.3), 0.3, 2)
    W, z, v = oracle.universal_kriging(Sy, Vop, X[n_p:], X[:n_p], y, 1.0)
    L = oracle.cholesky_lower(V)
    M = 200000
    Y = oracle.simulate(L, inputgen.standard_normals(len(xy), M, 77))
    S = oracle.conditional_correction(W, y, Y[:n_p], Y[n_p:])
    se = np.sqrt(v / M)
    assert np.all(np.abs(S.mean(axis=1) - z) < 5 * se + 1e-12)
    np.testing.assert_allclose(S.var(axis=1), v, rtol=0.02)


# ----------------------------------------------------------------------------- calibration
def test_calibration_brute_force_small():
    rng = np.random.default_rng(9)
    n_p, M, u = 7, 12, 0.3
    S = rng.standard_normal((n_p, M))
    z = rng.standard_normal(n_p)
    v = rng.uniform(0.5, 2.0, n_p)
    out = oracle.calibrate(S, z, v, u, 0.9)
    t = [(z[i] - u) / math.sqrt(v[i]) for i in range(n_p)]
    for j in range(M):
        up = [t[i] for i in range(n_p) if S[i, j] >= u]
        lo = [t[i] for i in range(n_p) if S[i, j] <= u]
        assert out["psi"][j] == (min(up) if up else math.inf)
        assert out["phi"][j] == (max(lo) if lo else -math.inf)
    for i in range(n_p):
        assert out["count"][i] == sum(1 for j in range(M) if S[i, j] >= u)
    psi = sorted(x for x in out["psi"] if x != math.inf)
    phi = sorted(x for x in out["phi"] if x != -math.inf)
    kq = lambda p, N: max(1, min(N, math.ceil(round(p * N, 9))))
    assert out["q_out"] == psi[kq(0.1, len(psi)) - 1]
    assert out["q_in"] == phi[kq(0.9, len(phi)) - 1]
    for i in range(n_p):
        assert out["c_out"][i] == (t[i] >= out["q_out"])
        assert out["c_in"][i] == (t[i] > out["q_in"])


def test_negative_excursion_hand_case():
    """Section III's sign reversal, worked by hand on 3 sites x 4 simulations (u = 0, level 0.5):
    t = (0.2, -0.15, 0.1), so the reversed t' = (-0.2, 0.15, -0.1); psi'_j takes the sites with
    S_ij <= 0, phi'_j those with S_ij >= 0; Q_0.5 of 4 values is the 2nd smallest."""
    S = np.array([[1.0, -1.0, 2.0, -2.0], [-1.0, 1.0, -1.0, 1.0], [0.5, 0.5, -0.5, -0.5]])
    z = np.array([0.2, -0.3, 0.1])
    v = np.array([1.0, 4.0, 1.0])
    out = oracle.calibrate_negative(S, z, v, 0.0, 0.5)
    np.testing.assert_array_equal(out["t"], [-0.2, 0.15, -0.1])
    np.testing.assert_array_equal(out["psi"], [0.15, -0.2, -0.1, -0.2])
    np.testing.assert_array_equal(out["phi"], [-0.1, 0.15, -0.2, 0.15])
    np.testing.assert_array_equal(out["count"], [2, 2, 2])
    assert out["q_out"] == -0.2 and out["q_in"] == -0.1
    np.testing.assert_array_equal(out["c_out"], [1, 1, 1])
    np.testing.assert_array_equal(out["c_in"], [0, 1, 0])
    # the negative set of a field is the positive set of the reversed field (Section III)
    assert list(oracle.excursion_set(np.array([-1.0, 0.0, 1.0]), 0.0, negative=True)) == [True, True, False]


def test_negative_excursion_brute_force():
    """Negative regions against a direct brute-force statement: psi'_j = min{-t_i : S_ij <= u},
    phi'_j = max{-t_i : S_ij >= u}, counts #{j : S_ij <= u}."""
    rng = np.random.default_rng(19)
    n_p, M, u = 9, 15, -0.2
    S = rng.standard_normal((n_p, M))
    z = rng.standard_normal(n_p)
    v = rng.uniform(0.5, 2.0, n_p)
    out = oracle.calibrate_negative(S, z, v, u, 0.8)
    t = [-(z[i] - u) / math.sqrt(v[i]) for i in range(n_p)]
    for j in range(M):
        a = [t[i] for i in range(n_p) if S[i, j] <= u]
        b = [t[i] for i in range(n_p) if S[i, j] >= u]
        assert out["psi"][j] == (min(a) if a else math.inf)
        assert out["phi"][j] == (max(b) if b else -math.inf)
    for i in range(n_p):
        assert out["count"][i] == sum(1 for j in range(M) if S[i, j] <= u)


def test_quantile_index_eq9():
    a = np.arange(1.0, 21.0)
    assert oracle.empirical_quantile(a, 0.05) == 1.0
    assert oracle.empirical_quantile(a, 1.0 - 0.95) == 1.0   # 0.0500000000000000444 * 20 is 1 up to rounding
    assert oracle.empirical_quantile(a, 0.051) == 2.0
    assert oracle.empirical_quantile(a, 0.95) == 19.0
    assert oracle.empirical_quantile(a, 1.0) == 20.0
    assert oracle.empirical_quantile(a, 0.0) == 1.0
    assert oracle.empirical_quantile(np.array([3.0]), 0.9) == 3.0


def test_regions_strictness_and_empty_sample():
    t = np.array([-1.0, 0.0, 0.5, 1.0])
    c_in, c_out = oracle.confidence_regions(t, 0.5, 0.5)
    assert list(c_in) == [0, 0, 0, 1] and list(c_out) == [0, 0, 1, 1]
    S = np.full((3, 4), 5.0)                       # every value above u: the phi sample is empty
    with pytest.raises(oracle.EmptySample):
        oracle.calibrate(S, np.zeros(3), np.ones(3), 1.0, 0.9)
    with pytest.raises(ValueError):
        oracle.standardized_statistic(np.zeros(2), np.array([1.0, 0.0]), 0.0)


# ----------------------------------------------------------------------------- policy
def _toy_stats():
    # NT = 3; hand-chosen tile norms and extrema (lower tiles)
    frob = np.array([[10.0, 0, 0], [1e-3, 10.0, 0], [1e-7, 2.0, 10.0]])
    vmin = np.array([[0.5, 0, 0], [1e-6, 0.5, 0], [1e-9, 0.01, 0.5]])
    vmax = np.array([[1.0, 0, 0], [1e-4, 1.0, 0], [1e-8, 0.1, 1.0]])
    return frob, vmin, vmax


def test_precision_map_hand_example():
    frob, vmin, vmax = _toy_stats()
    g = math.sqrt(3 * 100 + 2 * (1e-6 + 1e-14 + 4.0))
    # ratio_ij = frob * NT / g; FP16 iff ratio <= fixedacc * 2^10, FP32 iff <= fixedacc * 2^23
    fixedacc = 1e-4
    pm = oracle.precision_map(frob, fixedacc)
    r = lambda f: f * 3 / g
    assert r(1e-3) <= fixedacc * 1024 and r(1e-7) <= fixedacc * 1024
    assert fixedacc * 1024 < r(2.0) <= fixedacc * 2 ** 23
    assert pm.tolist() == [[0, -1, -1], [2, 0, -1], [2, 1, 0]]
    pm2 = oracle.precision_map(frob, 1e-9)          # 1e-9 * 2^23 = 0.0084 > r(1e-3) = 1.7e-4
    assert pm2.tolist() == [[0, -1, -1], [1, 0, -1], [2, 0, 0]]


def test_checks_and_scale_hand_example():
    frob, vmin, vmax = _toy_stats()
    pm = np.array([[0, -1, -1], [2, 0, -1], [2, 1, 0]], dtype=np.int8)
    c = oracle.fp16_checks(pm, frob, vmin, vmax)
    assert c["n_fp16"] == 2
    assert c["R_hp"] == pytest.approx(1e-4 / 1e-9)
    assert c["rho1"] == pytest.approx(1e-4) and c["rho2"] == pytest.approx(1e-4)
    assert c["check1"] and c["check2"]
    sc = oracle.covariance_scale(pm, vmin, vmax)
    # u_16 = sqrt(65504 / 1e-4) = 25593.75..., u_32 = sqrt(FLT_MAX / 0.1) huge, so s = 25593 - 1
    assert sc["s"] == 25592.0
    assert sc["ell"] == pytest.approx(math.sqrt(2.0 ** -14 / 1e-9))
    # check 1 fails when the FP16 extrema span more than 65504 / 2^-24
    vmin2 = vmin.copy(); vmin2[2, 0] = 1e-17
    assert not oracle.fp16_checks(pm, frob, vmin2, vmax)["check1"]
    # no reduced-precision tile: no scaling
    assert oracle.covariance_scale(np.zeros((3, 3), dtype=np.int8), vmin, vmax)["s"] == 1.0
    # FP32 tiles only: the FP32 bound sqrt(FLT_MAX / 0.1) is far above the FP16 range, so the
    # FP16 cast of the factor (largest entry sqrt(max V_ii) = 2) bounds s: u_s = 65504 / 2
    pm32 = np.array([[0, -1, -1], [1, 0, -1], [1, 1, 0]], dtype=np.int8)
    vmax4 = vmax.copy(); vmax4[1, 1] = 4.0
    sc32 = oracle.covariance_scale(pm32, vmin, vmax4)
    assert sc32["u_s"] == 32752.0 and sc32["s"] == 32751.0 and sc32["s"] * 2.0 < 65504.0


def test_auto_refinement_steps():
    # one off-diagonal tile that is FP16 at 1e-4 but fails check 2 through rho1 = 0.5 > 0.1024
    NT = 2
    frob = np.array([[10.0, 0.0], [0.5, 10.0]])
    vmin = np.array([[0.5, 0.0], [0.01, 0.5]])
    vmax = np.array([[1.0, 0.0], [0.5, 1.0]])
    g = math.sqrt(2 * 100.0 + 2 * 0.25)
    ratio = 0.5 * NT / g                                  # 0.0705 <= 0.1024: FP16 at the start
    assert ratio <= 1e-4 * 1024
    out = oracle.select_precision(frob, vmin, vmax, fixedacc=123.0, auto=True)
    # FP16 while ratio <= 1e-4 * 0.9^k * 1024; the loop stops at the first k where it is not
    k = 0
    fa = 1e-4
    while ratio <= fa * 1024:
        k += 1
        fa = fa * 0.9
    assert k == 4
    assert out["fixedacc"] == fa and out["iters"] == k + 1
    assert out["map"][1, 0] == oracle.PREC_FP32 and out["n_fp16"] == 0
    # user tolerance: failures are reported, the map is kept
    user = oracle.select_precision(frob, vmin, vmax, fixedacc=1e-4, auto=False)
    assert user["map"][1, 0] == oracle.PREC_FP16 and not user["check2"] and user["iters"] == 1
    assert user["rho1"] == 0.5


def test_page_constants():
    g = json.load(open(os.path.join(GOLDEN, "page_constants.json")))
    from oracle.policy import FP16_MAX, FP16_MIN_SUBNORMAL, EPS, PREC_FP16
    assert FP16_MAX / FP16_MIN_SUBNORMAL == pytest.approx(g["eq10_limit"]["value"], rel=g["eq10_limit"]["rel_tol"])
    assert EPS[PREC_FP16] == g["eps_fp16"]["value"]
    assert 1e-4 / EPS[PREC_FP16] == pytest.approx(g["eq11_limit"]["value"])
    sh = g["fp16_tile_shares"]
    assert sh["grid"] * (sh["grid"] + 1) // 2 == sh["tiles"]
    for cnt, pct in zip(sh["fp16"], sh["percent"]):
        assert round(100 * cnt / sh["tiles"], 2) == pct
    gs = g["grid_spacing"]
    assert gs["m"] ** 2 == gs["n_pred"] and gs["n_pred"] + gs["n_obs"] == gs["n"]
    b, u = g["trend_contour"]["b"], g["trend_contour"]["u"]
    for x in (0.0, 0.3, 0.6):        # m(s) = b1 x + b2 y equals u on y = 1 - 1.5 x
        assert b[1] * x + b[2] * (1 - 1.5 * x) == pytest.approx(u)


def test_tile_stats_ragged_and_lower_only():
    xy = inputgen.uniform_locations(70, 1)
    V = oracle.covariance_matrix(xy, "matern", 1.0, 0.1, 0.5, nugget=1e-3)
    fr, mn, mx = oracle.tile_stats(V, 32)           # NT = 3, last tile 6 wide
    assert fr.shape == (3, 3)
    T = V[64:70, 32:64]
    assert fr[2, 1] == pytest.approx(np.linalg.norm(T)) and mn[2, 1] == T.min() and mx[2, 1] == T.max()
    fr2, mn2, mx2 = oracle.tile_stats_from_locations(xy, 32, "matern", 1.0, 0.1, 0.5, nugget=1e-3)
    np.testing.assert_allclose(fr2, fr, rtol=1e-14)
    np.testing.assert_array_equal(mn2, mn)
    np.testing.assert_array_equal(mx2, mx)


def test_inputgen_morton_and_grid():
    g = inputgen.grid_cell_centres(4)
    assert g[0].tolist() == [0.125, 0.125] and g[1].tolist() == [0.375, 0.125] and g[4].tolist() == [0.125, 0.375]
    p = inputgen.morton_permutation(g)
    # Z-order of the 4x4 grid: (0,0),(1,0),(0,1),(1,1),(2,0),...
    assert p[:4].tolist() == [0, 1, 4, 5] and p[4:8].tolist() == [2, 3, 6, 7]


def test_coverage_event_hand_cases_and_set_semantics():
    # truth over four prediction sites, u = 1.6: A = {0, 2}
    truth = np.array([2.0, 0.5, 1.6, 1.59])
    assert oracle.excursion_set(truth, 1.6).tolist() == [True, False, True, False]
    assert oracle.coverage_event(truth, [1, 0, 0, 0], [1, 0, 1, 1], 1.6)        # {0} in A in {0,2,3}
    assert not oracle.coverage_event(truth, [1, 1, 0, 0], [1, 1, 1, 1], 1.6)    # site 1 in C_in, not in A
    assert not oracle.coverage_event(truth, [0, 0, 0, 0], [1, 1, 0, 1], 1.6)    # site 2 in A, not in C_out
    assert oracle.coverage_event(truth, [0, 0, 0, 0], [1, 0, 1, 0], 1.6)        # C_out = A exactly
    # against plain set inclusion on random masks
    rng = np.random.default_rng(4)
    for _ in range(300):
        t = rng.standard_normal(9)
        ci, co = rng.random(9) < 0.2, rng.random(9) < 0.7
        A = {i for i in range(9) if t[i] >= 0.3}
        want = {i for i in range(9) if ci[i]} <= A <= {i for i in range(9) if co[i]}
        assert oracle.coverage_event(t, ci, co, 0.3) == want
        # the separate inner and outer events of Fig. 3a/3b, and their conjunction
        inner = {i for i in range(9) if ci[i]} <= A
        outer = A <= {i for i in range(9) if co[i]}
        assert oracle.inner_event(t, ci, 0.3) == inner and oracle.outer_event(t, co, 0.3) == outer
        assert (inner and outer) == want
    assert oracle.inner_event(truth, [1, 0, 1, 0], 1.6) and not oracle.inner_event(truth, [0, 1, 0, 0], 1.6)
    assert oracle.outer_event(truth, [1, 0, 1, 0], 1.6) and not oracle.outer_event(truth, [1, 1, 0, 1], 1.6)


def test_truth_field_mean_and_covariance():
    # Z = X b + L eta has mean X b and covariance L L^T = V: Monte Carlo on three sites
    V = np.array([[2.0, 0.6, 0.2], [0.6, 1.0, 0.3], [0.2, 0.3, 1.5]])
    L = oracle.cholesky_lower(V)
    X = np.array([[1.0, 0.2], [1.0, 0.5], [1.0, 0.9]])
    b = np.array([1.0, -2.0])
    eta = np.random.default_rng(8).standard_normal((3, 200000))
    Z = oracle.truth_field(L, X, b, eta)
    R = eta.shape[1]
    np.testing.assert_allclose(Z.mean(axis=1), X @ b, atol=5 * np.sqrt(np.diag(V).max() / R))
    C = np.cov(Z)
    assert np.max(np.abs(C - V)) < 5 * np.sqrt(2.0 * 2.0 / R) * 2
    # one draw as a vector gives the same column
    np.testing.assert_array_equal(oracle.truth_field(L, X, b, eta[:, 0]), Z[:, 0])


def test_fp16_per_product_simulation_pins():
    """The task-by-task FP16 destination (Alg.1 with §V-F's FP16 storage): a hand-computed case
    where the order of roundings decides the result, the single-tile case (one rounding of the
    exact product), exactness when every partial sum is an FP16 integer, and FP16-representable
    outputs."""
    # n = 3, nb = 1: row 2 is fp16(1.0), then + 0.75 2^-11 twice; each addition is below half
    # an FP16 ulp of 1.0 (2^-11), so the per-product result stays 1.0, while the exact sum
    # 1 + 0.75 2^-10 rounds once to 1 + 2^-10
    t = 0.75 * 2.0 ** -11
    L = np.array([[1.0, 0.0, 0.0], [0.0, 1.0, 0.0], [t, t, 1.0]])
    B = np.ones((3, 1))
    Y = oracle.simulate_fp16_per_product(L, B, 1)
    assert Y[2, 0] == 1.0
    assert np.float16(L[2] @ B[:, 0]) == np.float16(1.0 + 2.0 ** -10)
    rng = np.random.default_rng(0)
    # one tile row: a single rounding of the exact product
    L1 = np.tril(rng.standard_normal((6, 6)))
    B1 = rng.standard_normal((6, 4))
    np.testing.assert_array_equal(oracle.simulate_fp16_per_product(L1, B1, 8),
                                  (L1 @ B1).astype(np.float16).astype(np.float64))
    # small integers: every partial sum is exact in FP16, so the result is the exact product
    Li = np.tril(rng.integers(-3, 4, (10, 10))).astype(np.float64)
    Bi = rng.integers(-3, 4, (10, 5)).astype(np.float64)
    np.testing.assert_array_equal(oracle.simulate_fp16_per_product(Li, Bi, 3), Li @ Bi)
    # outputs are FP16 values
    L2 = np.tril(rng.standard_normal((9, 9)))
    Y2 = oracle.simulate_fp16_per_product(L2, rng.standard_normal((9, 3)), 4)
    np.testing.assert_array_equal(Y2, Y2.astype(np.float16).astype(np.float64))
