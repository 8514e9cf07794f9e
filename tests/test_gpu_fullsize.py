"""Parity at the benchmark sizes, in the configuration bench.py runs, on outputs the oracle
can compute piece by piece and on properties that hold at any size:
  * tile statistics of sampled tiles against the oracle's;
  * the precision map, checks and scale recomputed by the oracle's policy from the GPU's
    statistics (host logic, bit-exact);
  * the leading principal block of the factor and of the simulations: the Cholesky factor
    of a leading block of V is the leading block of the full factor, and Y = L Z is lower
    triangular, so the oracle computes both exactly on that block;
  * sampled rows of Y against the GPU's own factor (the simulation multiply at full K);
  * the calibration of the GPU's simulations, bit-exact against the oracle;
  * kriging at 16384 + 16384 sites: unbiasedness X_o^T W = X_p^T and positive MSPEs.
"""
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


def _sampled_stats_check(w, xy, f, mn, mx, rng, count=24):
    nt = f.shape[0]
    picks = {(0, 0), (nt - 1, nt - 1), (nt - 1, 0)}
    while len(picks) < count:
        i = int(rng.integers(0, nt))
        picks.add((i, int(rng.integers(0, i + 1))))
    n, nb = w.n, w.nb
    for (i, j) in picks:
        T = oracle.covariance_matrix(xy, w.family, w.sigma2, w.beta, w.nu, w.nugget, w.n_pred, w.tau2,
                                     rows=slice(i * nb, min(n, (i + 1) * nb)), cols=slice(j * nb, min(n, (j + 1) * nb)))
        assert f[i, j] == pytest.approx(np.linalg.norm(T), rel=1e-12)
        assert mn[i, j] == pytest.approx(T.min(), rel=1e-12, abs=1e-300)
        assert mx[i, j] == pytest.approx(T.max(), rel=1e-12)


def _policy_check(f, mn, mx, pmap, info, fixedacc):
    ref = oracle.select_precision(f, mn, mx, fixedacc, auto=False)
    low = np.tril(np.ones(pmap.shape, dtype=bool))
    np.testing.assert_array_equal(pmap[low], ref["map"][low])
    assert info["s"] == ref["s"]
    assert bool(info["check1"]) == ref["check1"] and bool(info["check2"]) == ref["check2"]


def _leading_block(lib, V, w, xy, Z, Y, s, n_s, tol_L, tol_Y):
    Vo = oracle.covariance_matrix(xy[:n_s], w.family, w.sigma2, w.beta, w.nu, w.nugget)
    Lo = oracle.cholesky_lower(Vo)
    Ld = lib.tilemat_to_dense(V, 1)
    Lg = Ld[:n_s, :n_s].cpu().numpy() / s
    eL = relf(Lg, Lo)
    eY = relf(Y[:n_s], oracle.simulate(Lo, Z[:n_s]))
    assert eL <= tol_L and eY <= tol_Y, (eL, eY)
    return Ld


def test_headline_workload_full_size(lib):
    w = inputgen.WORKLOADS["c"]
    rng = np.random.default_rng(0)
    xy = inputgen.workload_locations(w)
    V = lib.TileMat(w.n, w.nb)
    lib.cov_build(V, dev(xy), w.family, w.sigma2, w.beta, w.nu, nugget=w.nugget)
    f, mn, mx = lib.tile_stats(V)
    _sampled_stats_check(w, xy, f, mn, mx, rng)
    pmap, info = lib.precision_map(V, amp=True, fixedacc=w.fixedacc)
    _policy_check(f, mn, mx, pmap, info, w.fixedacc)
    assert info["n_fp16"] > info["n_fp32"] > 0           # majority FP16 tiles at this tolerance
    assert lib.potrf_adaptive(V) == 0
    Z = inputgen.standard_normals(w.n, w.M, 12345)
    Yt = lib.trmm_sim(V, colmajor(Z), w.M)
    Y = Yt.cpu().numpy()
    s = info["s"]
    Ld = _leading_block(lib, V, w, xy, Z, Y, s, 2048, 1e-2, 1e-2)
    # sampled rows at full K-chain length against the GPU's own factor
    rows = np.sort(rng.choice(w.n, 12, replace=False))
    Lr = Ld[torch.from_numpy(rows).cuda()].cpu().numpy() / s
    # far tiles of the factor against the oracle's covariance: (L_s L_s^T)_ij, formed on the
    # host from the stored factor's block rows, against s^2 V_ij.  Every product of the
    # factorisation is taken at least at FP16 precision (unit roundoff 2^-11) with FP32 or
    # FP64 accumulation and every stored tile is rounded at most to FP16, so the backward
    # error of a tile obeys ||E_ij||_F <= c 2^-10 sum_k ||L_ik||_F ||L_jk||_F
    # <= c 2^-10 s^2 sqrt(tr V_ii tr V_jj) (Cauchy-Schwarz; ||L_i,:||_F^2 = s^2 tr V_ii); c = 2
    nb, nt = w.nb, w.n // w.nb
    pairs = {(nt - 1, nt - 1), (nt - 1, 0), (nt - 1, nt - 2), (nt - 1, nt // 2), (nt // 2, nt // 2 - 1)}
    while len(pairs) < 16:
        i = int(rng.integers(1, nt))
        pairs.add((i, int(rng.integers(0, i + 1))))
    tr = nb * (w.sigma2 + w.nugget)
    worst = 0.0
    for (i, j) in sorted(pairs):
        Li = Ld[i * nb:(i + 1) * nb, :(j + 1) * nb].cpu().numpy()
        Lj = Ld[j * nb:(j + 1) * nb, :(j + 1) * nb].cpu().numpy()
        P = Li @ Lj.T
        if i == j:
            P = np.tril(P)
        T = oracle.covariance_matrix(xy, w.family, w.sigma2, w.beta, w.nu, w.nugget,
                                     rows=slice(i * nb, (i + 1) * nb), cols=slice(j * nb, (j + 1) * nb))
        T = s * s * (np.tril(T) if i == j else T)
        ratio = np.linalg.norm(P - T) / (2.0 * 2.0 ** -10 * s * s * tr)
        worst = max(worst, ratio)
        assert ratio <= 1.0, (i, j, ratio)
    print(f"far tiles: worst backward error {worst:.3e} of the bound")
    del Ld
    torch.cuda.empty_cache()
    assert relf(Y[rows], Lr @ Z) <= 2e-3
    # calibration of these simulations (no observations: zhat = 0, v = V_ii), bit-exact
    v = np.full(w.n, w.sigma2 + w.nugget)
    out = lib.calibrate(Yt, dev(np.zeros(w.n)), dev(v), w.u, w.level, counts=True)
    ref = oracle.calibrate(Y, np.zeros(w.n), v, w.u, w.level)
    assert out["q_in"] == ref["q_in"] and out["q_out"] == ref["q_out"]
    np.testing.assert_array_equal(out["count"].cpu().numpy(), ref["count"])
    np.testing.assert_array_equal(out["c_in"].cpu().numpy(), ref["c_in"])
    np.testing.assert_array_equal(out["c_out"].cpu().numpy(), ref["c_out"])
    V.close()


def test_headline_fast_statistics_full_size(lib):
    """At the benchmark size and in the bench's call sequence (no cr_tile_stats before the
    map): the FP32 statistics records hold their stated bounds against the oracle on sampled
    off-diagonal tiles, and the map, checks and scale taken on them (with the policy's exact
    recomputations) equal those taken after making every record exact."""
    w = inputgen.WORKLOADS["c"]
    rng = np.random.default_rng(2)
    xy = inputgen.workload_locations(w)
    n, nb = w.n, w.nb
    V = lib.TileMat(n, nb)
    lib.cov_build(V, dev(xy), w.family, w.sigma2, w.beta, w.nu, nugget=w.nugget)
    f, mn, mx, err = lib.tile_stats_records(V)
    nt = f.shape[0]
    off = np.tril(np.ones((nt, nt), dtype=bool), -1)
    assert np.all(err[off] > 0) and np.all(err[off] < 1e-3)
    for _ in range(16):
        i = int(rng.integers(1, nt))
        j = int(rng.integers(0, i))
        T = oracle.covariance_matrix(xy, w.family, w.sigma2, w.beta, w.nu, w.nugget, w.n_pred, w.tau2,
                                     rows=slice(i * nb, min(n, (i + 1) * nb)), cols=slice(j * nb, min(n, (j + 1) * nb)))
        for got, ref in ((f[i, j], np.linalg.norm(T)), (mn[i, j], T.min()), (mx[i, j], T.max())):
            assert abs(got - ref) <= err[i, j] * abs(ref), (i, j, got, ref, err[i, j])
    pm_fast, info_fast = lib.precision_map(V, amp=True, fixedacc=w.fixedacc)
    V.close()
    torch.cuda.empty_cache()
    V = lib.TileMat(n, nb)
    lib.cov_build(V, dev(xy), w.family, w.sigma2, w.beta, w.nu, nugget=w.nugget)
    lib.tile_stats(V)   # every record exact
    pm_exact, info_exact = lib.precision_map(V, amp=True, fixedacc=w.fixedacc)
    V.close()
    np.testing.assert_array_equal(pm_fast, pm_exact)
    for k in info_fast:
        a, b = info_fast[k], info_exact[k]
        assert (a == b) or (np.isnan(a) and np.isnan(b)), (k, a, b)


def test_strong_correlation_workload_full_size(lib):
    w = inputgen.WORKLOADS["b"]
    rng = np.random.default_rng(1)
    xy = inputgen.workload_locations(w)
    V = lib.TileMat(w.n, w.nb)
    lib.cov_build(V, dev(xy), w.family, w.sigma2, w.beta, w.nu, nugget=w.nugget)
    f, mn, mx = lib.tile_stats(V)
    _sampled_stats_check(w, xy, f, mn, mx, rng)
    pmap, info = lib.precision_map(V, amp=True, fixedacc=w.fixedacc)
    _policy_check(f, mn, mx, pmap, info, w.fixedacc)
    assert lib.potrf_adaptive(V) == 0
    Z = inputgen.standard_normals(w.n, w.M, 7)
    Y = lib.trmm_sim(V, colmajor(Z), w.M).cpu().numpy()
    lead = 2048 // w.nb
    all64 = bool(np.all(pmap[:lead, :lead][np.tril(np.ones((lead, lead), dtype=bool))] == 0))
    # leading tiles in FP64 keep FP64 accuracy of the factor; the simulation multiply runs
    # on FP16 operands in the adaptive mode (Alg.1)
    _leading_block(lib, V, w, xy, Z, Y, info["s"], 2048, 1e-9 if all64 else 1e-2, 1e-2)
    V.close()


_ORACLE_FACTOR = {}


def _oracle_factor_b512():
    """The oracle's V and L for config b's geometry (computed once per session)."""
    if not _ORACLE_FACTOR:
        w = inputgen.WORKLOADS["b"]
        xy = inputgen.workload_locations(w)
        Vo = oracle.covariance_matrix(xy, w.family, w.sigma2, w.beta, w.nu, w.nugget)
        Lo = oracle.cholesky_lower(Vo)
        scale = max(1.0, relf(np.linalg.cholesky(Vo), Lo) / 1e-14)
        _ORACLE_FACTOR.update(xy=xy, Lo=Lo, scale=scale)
    return _ORACLE_FACTOR


@pytest.mark.parametrize("arith", ["fp64", "df"])
def test_all_fp64_factor_at_product_tile_size(lib, arith):
    """The all-FP64 mode at the tile size the product runs (nb = 512: 16 x 16 tiles, 32 x 32
    blocks in each diagonal executor launch), on config b's geometry (8192 jittered grid sites,
    Matern nu = 1.5, range 0.3, nugget 1e-4): the whole factor and the whole simulation
    Y = L Z (M = 512) against the oracle at the FP64 gate, 1e-11 relative Frobenius (scaled by
    the measured FP64 ordering noise between the oracle and LAPACK), with the diagonal tiles in
    FP64 and in double-float arithmetic."""
    w = inputgen.WORKLOADS["b"]
    ref = _oracle_factor_b512()
    xy, Lo, scale = ref["xy"], ref["Lo"], ref["scale"]
    nb = 512
    V = lib.TileMat(w.n, nb)
    lib.cov_build(V, dev(xy), w.family, w.sigma2, w.beta, w.nu, nugget=w.nugget)
    lib.precision_map(V, amp=False)
    mode = lib.CR_DIAG_FP64 if arith == "fp64" else lib.CR_DIAG_DF
    old = lib.get_option(lib.CR_OPT_DIAG_ARITH)
    lib.set_option(lib.CR_OPT_DIAG_ARITH, mode)
    try:
        assert lib.potrf_adaptive(V) == 0
    finally:
        lib.set_option(lib.CR_OPT_DIAG_ARITH, old)
    L = lib.tilemat_to_dense(V, 1).cpu().numpy()
    Z = inputgen.standard_normals(w.n, w.M, 7)
    Y = lib.trmm_sim(V, colmajor(Z), w.M).cpu().numpy()
    V.close()
    eL = relf(L, Lo)
    eY = relf(Y, oracle.simulate(Lo, Z))
    assert eL <= 1e-11 * scale and eY <= 1e-11 * scale, (arith, eL, eY, scale)


def test_scale_sweep_workload_full_size(lib):
    """The largest scale-sweep configuration (n = 65536, range 0.1, tolerance 1e-6, M = 4096)
    in the bench's call sequence: the map taken on the fast statistics equals the one taken on
    exact statistics, and the factor and the simulations agree with the oracle on the leading
    2048 x 2048 block."""
    w = inputgen.WORKLOADS["e2"]
    rng = np.random.default_rng(3)
    xy = inputgen.workload_locations(w)
    V = lib.TileMat(w.n, w.nb)
    lib.cov_build(V, dev(xy), w.family, w.sigma2, w.beta, w.nu, nugget=w.nugget)
    f, mn, mx = lib.tile_stats(V)
    _sampled_stats_check(w, xy, f, mn, mx, rng, count=12)
    pm_exact, info_exact = lib.precision_map(V, amp=True, fixedacc=w.fixedacc)
    _policy_check(f, mn, mx, pm_exact, info_exact, w.fixedacc)
    V.close()
    torch.cuda.empty_cache()
    V = lib.TileMat(w.n, w.nb)
    lib.cov_build(V, dev(xy), w.family, w.sigma2, w.beta, w.nu, nugget=w.nugget)
    pmap, info = lib.precision_map(V, amp=True, fixedacc=w.fixedacc)
    np.testing.assert_array_equal(pmap, pm_exact)
    assert info["s"] == info_exact["s"]
    assert lib.potrf_adaptive(V) == 0
    s = info["s"]
    Z = inputgen.standard_normals(2048, w.M, 31)
    # n x M column-major, zero below the leading rows: the leading rows of L Z depend on the
    # leading rows of Z only
    Zd = torch.zeros((w.M, w.n), dtype=torch.float64, device="cuda").T
    Zd[:2048] = torch.from_numpy(Z).cuda()
    Yt = lib.trmm_sim(V, Zd, w.M)
    del Zd
    Y = Yt[:2048].cpu().numpy()
    del Yt
    torch.cuda.empty_cache()
    Vo = oracle.covariance_matrix(xy[:2048], w.family, w.sigma2, w.beta, w.nu, w.nugget)
    Lo = oracle.cholesky_lower(Vo)
    Ld = lib.tilemat_to_dense(V, 1)
    eL = relf(Ld[:2048, :2048].cpu().numpy() / s, Lo)
    del Ld
    torch.cuda.empty_cache()
    eY = relf(Y, oracle.simulate(Lo, Z))
    assert eL <= 1e-2 and eY <= 1e-2, (eL, eY, info)
    V.close()


def test_kriging_workload_full_size(lib):
    w = inputgen.WORKLOADS["k"]
    xy = inputgen.workload_locations(w)
    n_p, n_o = w.n_pred, w.n_obs
    X = np.column_stack([np.ones(w.n), xy[:, 0], xy[:, 1]])
    y = inputgen.observation_values(xy[n_p:], (1.0, 0.5, -0.3), 0.1, 3)
    V = lib.TileMat(w.n, w.nb)
    lib.cov_build(V, dev(xy), w.family, w.sigma2, w.beta, w.nu, nugget=w.nugget, n_pred=n_p, tau2=w.tau2)
    W, z, v = lib.krige(V, colmajor(X[n_p:]), colmajor(X[:n_p]), dev(y))
    Wt = W
    # unbiasedness, evaluated on the device in FP64
    XoT_W = (torch.from_numpy(X[n_p:]).cuda().T @ Wt).cpu().numpy()
    assert np.max(np.abs(XoT_W - X[:n_p].T)) <= 1e-6 * np.max(np.abs(X[:n_p]))
    vv = v.cpu().numpy()
    assert np.all(vv > 0) and np.all(vv < 2 * w.sigma2)
    zz = z.cpu().numpy()
    assert np.all(np.isfinite(zz))
    # prediction at a grid site next to an observation is close to the trend plus noise scale
    assert abs(np.mean(zz) - np.mean(1.0 + 0.5 * xy[:n_p, 0] - 0.3 * xy[:n_p, 1])) < 0.1
    V.close()
