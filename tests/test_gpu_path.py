"""Parity of the CUDA path with the oracle (GPU).  Inputs come from inputgen only; expected
values come from oracle/ only.  Tolerances: FP64 paths 1e-11 relative Frobenius (tighter
where the arithmetic allows), adaptive simulation 1e-2 relative Frobenius on Y, integer and
index outputs bit-exact."""
import contextlib

import numpy as np
import pytest
import torch

import inputgen
import oracle

pytestmark = pytest.mark.gpu


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def colmajor(a):
    """numpy (n, m) -> CUDA column-major tensor"""
    return torch.from_numpy(np.asfortranarray(a).T.copy()).cuda().T


def relf(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


COV_CASES = {
    "a_exp": dict(n=1024, nb=128, family="matern", beta=0.1, nu=0.5, nugget=1e-6, n_pred=None, tau2=0.0),
    "ragged_nu15": dict(n=1000, nb=128, family="matern", beta=0.3, nu=1.5, nugget=1e-4, n_pred=None, tau2=0.0),
    "nu1_krige": dict(n=600, nb=128, family="matern", beta=0.1, nu=1.0, nugget=0.0, n_pred=300, tau2=0.01),
    "nu07": dict(n=500, nb=128, family="matern", beta=0.2, nu=0.7, nugget=1e-5, n_pred=None, tau2=0.0),
    "nu25": dict(n=384, nb=128, family="matern", beta=0.2, nu=2.5, nugget=1e-3, n_pred=None, tau2=0.0),
    "powexp": dict(n=512, nb=128, family="powexp", beta=0.033, nu=0.5, nugget=1e-6, n_pred=None, tau2=0.0),
    # scaled distances up to ~70: the far end of the fast statistics' error bound
    "exp_short": dict(n=1024, nb=128, family="matern", beta=0.02, nu=0.5, nugget=1e-4, n_pred=None, tau2=0.0),
    # the product's tile size: 32 x 32 blocks per diagonal tile in the executor
    "nb512": dict(n=2048, nb=512, family="matern", beta=0.03, nu=0.5, nugget=1e-4, n_pred=None, tau2=0.0),
}


@contextlib.contextmanager
def diag_arith(lib, mode):
    """Runs the block with the diagonal executor's arithmetic set to `mode` (CR_DIAG_*)."""
    old = lib.get_option(lib.CR_OPT_DIAG_ARITH)
    lib.set_option(lib.CR_OPT_DIAG_ARITH, mode)
    try:
        yield
    finally:
        lib.set_option(lib.CR_OPT_DIAG_ARITH, old)


def _build(lib, c, seed=1):
    xy = inputgen.morton_sorted(inputgen.uniform_locations(c["n"], seed))
    V = lib.TileMat(c["n"], c["nb"])
    lib.cov_build(V, dev(xy), c["family"], 1.0, c["beta"], c["nu"], nugget=c["nugget"], n_pred=c["n_pred"],
                  tau2=c["tau2"])
    Vo = oracle.covariance_matrix(xy, c["family"], 1.0, c["beta"], c["nu"], c["nugget"], c["n_pred"], c["tau2"])
    return xy, V, Vo


@pytest.mark.parametrize("case", list(COV_CASES))
def test_covariance_and_stats(lib, case):
    c = COV_CASES[case]
    xy, V, Vo = _build(lib, c)
    G = lib.tilemat_to_dense(V, 0).cpu().numpy()
    Lo = np.tril(Vo)
    err = np.max(np.abs(G - Lo))
    assert err <= 2e-14, f"max abs covariance error {err:.3e}"
    f, mn, mx = lib.tile_stats(V)
    fo, mno, mxo = oracle.tile_stats(Vo, c["nb"])
    low = np.tril(np.ones_like(f, dtype=bool))
    # double-float statistics: the scaled distance x carries ~2^-48 relative error, which
    # the exponential turns into ~x 2^-48 relative on the entry (x up to 80 before the FP64
    # fallback): 1e-13 covers x < ~28, 5e-13 the whole range
    x_max = np.sqrt(2.0) / c["beta"]
    rt = 1e-13 if x_max < 28 else 5e-13
    np.testing.assert_allclose(f[low], fo[low], rtol=rt)
    np.testing.assert_allclose(mn[low], mno[low], rtol=rt, atol=1e-300)
    np.testing.assert_allclose(mx[low], mxo[low], rtol=rt)
    V.close()


@pytest.mark.parametrize("case", ["a_exp", "ragged_nu15", "nu25", "nu07", "exp_short"])
def test_fast_statistics_records_within_their_bounds(lib, case):
    """The FP32 statistics pass of the closed-form Matern orders: each off-diagonal record is
    within its stated relative bound of the oracle's exact statistics, the bound is small
    enough to decide on, and the diagonal tiles' records (and every record of the other
    orders) are exact."""
    c = COV_CASES[case]
    xy, V, Vo = _build(lib, c)
    f, mn, mx, err = lib.tile_stats_records(V)
    fo, mno, mxo = oracle.tile_stats(Vo, c["nb"])
    nt = V.nt
    off = np.tril(np.ones((nt, nt), dtype=bool), -1)
    diag = np.eye(nt, dtype=bool)
    closed = c["family"] == "matern" and c["nu"] in (0.5, 1.5, 2.5)
    if closed:
        assert np.all(err[off] > 0) and np.all(err[off] < 1e-3), err[off].max()
    else:
        assert np.all(err[off] == 0)
    assert np.all(err[diag] == 0)
    for got, ref in ((f, fo), (mn, mno), (mx, mxo)):
        fast = off & (err > 0)
        assert np.all(np.abs(got[fast] - ref[fast]) <= err[fast] * np.abs(ref[fast]))
        exact = (diag | off) & (err == 0)
        np.testing.assert_allclose(got[exact], ref[exact], rtol=5e-13, atol=1e-300)
    # cr_tile_stats recomputes every fast record exactly (double-float: rtol as in
    # test_covariance_and_stats)
    rt = 1e-13 if np.sqrt(2.0) / c["beta"] < 28 else 5e-13
    f2, mn2, mx2 = lib.tile_stats(V)
    low = diag | off
    np.testing.assert_allclose(f2[low], fo[low], rtol=rt)
    np.testing.assert_allclose(mn2[low], mno[low], rtol=rt, atol=1e-300)
    np.testing.assert_allclose(mx2[low], mxo[low], rtol=rt)
    assert np.all(lib.tile_stats_records(V)[3][low] == 0)
    V.close()


@pytest.mark.parametrize("fixedacc,auto", [(1e-6, False), (1e-3, False), (1e-4, True), (3e-5, False)])
def test_precision_map_on_fast_statistics_equals_exact(lib, fixedacc, auto):
    """The map, checks and scale taken on the fast statistics (with the exact recomputation of
    the tiles the decisions depend on) equal those taken on exact statistics of every tile."""
    c = COV_CASES["a_exp"]
    xy, V1, _ = _build(lib, c)
    m1, i1 = lib.precision_map(V1, amp=True, fixedacc=fixedacc, auto=auto)
    xy, V2, _ = _build(lib, c)
    lib.tile_stats(V2)   # every record exact first
    m2, i2 = lib.precision_map(V2, amp=True, fixedacc=fixedacc, auto=auto)
    np.testing.assert_array_equal(m1, m2)
    for k in i1:
        a, b = i1[k], i2[k]
        assert (a == b) or (np.isnan(a) and np.isnan(b)), (k, a, b)
    V1.close()
    V2.close()


@pytest.mark.parametrize("fixedacc,auto", [(1e-6, False), (1e-3, False), (1e-4, True)])
def test_precision_map_matches_oracle(lib, fixedacc, auto):
    c = COV_CASES["a_exp"]
    xy, V, Vo = _build(lib, c)
    m, info = lib.precision_map(V, amp=True, fixedacc=fixedacc, auto=auto)
    fo, mno, mxo = oracle.tile_stats(Vo, c["nb"])
    ref = oracle.select_precision(fo, mno, mxo, fixedacc, auto)
    low = np.tril(np.ones(m.shape, dtype=bool))
    np.testing.assert_array_equal(m[low], ref["map"][low])
    assert info["s"] == ref["s"]
    assert info["iters"] == ref["iters"] and info["fixedacc"] == ref["fixedacc"]
    assert bool(info["check1"]) == ref["check1"] and bool(info["check2"]) == ref["check2"]
    assert info["n_fp16"] == ref["n_fp16"]
    for k in ("R_hp", "rho1", "rho2", "ell", "u_s"):
        if k in ref and not (np.isnan(info[k]) and np.isnan(ref[k])):
            assert info[k] == pytest.approx(ref[k], rel=1e-12), k
    V.close()


@pytest.mark.parametrize("case", ["a_exp", "ragged_nu15"])
def test_fp64_cholesky_and_simulation(lib, case):
    c = COV_CASES[case]
    xy, V, Vo = _build(lib, c)
    lib.precision_map(V, amp=False)
    assert lib.potrf_adaptive(V) == 0
    L = lib.tilemat_to_dense(V, 1).cpu().numpy()
    Lo = oracle.cholesky_lower(Vo)
    # FP64 rounding differences between two Cholesky orderings, measured against LAPACK
    scale = max(1.0, relf(np.linalg.cholesky(Vo), Lo) / 1e-14)
    eL = relf(L, Lo)
    assert eL <= 1e-11 * scale, f"L error {eL:.3e} (ordering noise x{scale:.1f})"
    M = 64
    Z = inputgen.standard_normals(c["n"], M, 3)
    Y = lib.trmm_sim(V, colmajor(Z), M).cpu().numpy()
    eY = relf(Y, oracle.simulate(Lo, Z))
    assert eY <= 1e-11 * scale, f"Y error {eY:.3e}"
    V.close()


@pytest.mark.parametrize("case", ["a_exp", "ragged_nu15", "nb512"])
def test_double_float_executor_in_fp64_mode(lib, case):
    """The diagonal executor in double-float arithmetic (FP64 emulated on the FP32 units, the
    default of adaptive factorisations) forced into the all-FP64 mode: the factor and the
    simulations meet the FP64 gate against the oracle, 1e-11 relative Frobenius (scaled by the
    FP64 ordering noise as in test_fp64_cholesky_and_simulation), and the factor agrees with
    the FP64 executor's to within the double-float precision."""
    c = COV_CASES[case]
    xy, V, Vo = _build(lib, c)
    lib.precision_map(V, amp=False)
    with diag_arith(lib, lib.CR_DIAG_DF):
        assert lib.potrf_adaptive(V) == 0
    Ldf = lib.tilemat_to_dense(V, 1).cpu().numpy()
    M = 64
    Z = inputgen.standard_normals(c["n"], M, 3)
    Ydf = lib.trmm_sim(V, colmajor(Z), M).cpu().numpy()
    V.close()
    xy, V, _ = _build(lib, c)
    lib.precision_map(V, amp=False)
    with diag_arith(lib, lib.CR_DIAG_FP64):
        assert lib.potrf_adaptive(V) == 0
    L64 = lib.tilemat_to_dense(V, 1).cpu().numpy()
    V.close()
    Lo = oracle.cholesky_lower(Vo)
    scale = max(1.0, relf(np.linalg.cholesky(Vo), Lo) / 1e-14)
    eL, eY, e64 = relf(Ldf, Lo), relf(Ydf, oracle.simulate(Lo, Z)), relf(Ldf, L64)
    msg = f"double-float: L {eL:.2e}, Y {eY:.2e}, against the FP64 executor {e64:.2e} (noise x{scale:.1f})"
    assert eL <= 1e-11 * scale and eY <= 1e-11 * scale, msg
    assert e64 <= 1e-11 * scale, msg


@pytest.mark.parametrize("mode", ["fp64", "df"])
def test_not_spd_at_the_last_pivot_of_a_block(lib, mode):
    """A zero pivot at the 16th column of the first diagonal block (the last column of the
    executor's first 16 x 16 block) is reported as column 16 in both arithmetics.  Sites 14
    and 15 coincide and are far from sites 0-13 (their covariances underflow to exactly 0),
    with no nugget: rows 14 and 15 stay equal, with unit entries, through the first 14 steps,
    so the 16th pivot is 1 - 1 * 1 = 0 exactly."""
    rng = np.random.default_rng(5)
    xy = np.vstack([rng.uniform(0.0, 0.3, (14, 2)), [[0.99, 0.99], [0.99, 0.99]], rng.uniform(0.0, 0.3, (240, 2))])
    V = lib.TileMat(256, 128)
    lib.cov_build(V, dev(xy), "matern", 1.0, 0.001, 0.5, nugget=0.0)
    lib.precision_map(V, amp=False)
    with diag_arith(lib, lib.CR_DIAG_FP64 if mode == "fp64" else lib.CR_DIAG_DF):
        info = lib.potrf_adaptive(V)
    assert info == 16
    V.close()


@pytest.mark.parametrize("case,fixedacc", [("a_exp", 1e-6), ("a_exp", 1e-3), ("ragged_nu15", 1e-6), ("nu07", 1e-2),
                                           ("powexp", 1e-3), ("nb512", 1e-4)])
def test_adaptive_cholesky_and_simulation(lib, case, fixedacc):
    c = COV_CASES[case]
    xy, V, Vo = _build(lib, c)
    m, info = lib.precision_map(V, amp=True, fixedacc=fixedacc)
    assert lib.potrf_adaptive(V) == 0
    s = info["s"]
    L = lib.tilemat_to_dense(V, 1).cpu().numpy() / s
    Lo = oracle.cholesky_lower(Vo)
    eL = relf(L, Lo)
    M = 200
    Z = inputgen.standard_normals(c["n"], M, 4)
    Y = lib.trmm_sim(V, colmajor(Z), M).cpu().numpy()
    Yo = oracle.simulate(Lo, Z)
    eY = relf(Y, Yo)
    Y16 = lib.trmm_sim(V, colmajor(Z), M, flags=lib.CR_TRMM_FP16_DEST).cpu().numpy()
    eY16 = relf(Y16, Yo)
    msg = (f"fp64/32/16 tiles {info['n_fp64']}/{info['n_fp32']}/{info['n_fp16']} s={s} "
           f"eL={eL:.2e} eY={eY:.2e} eY16={eY16:.2e}")
    if case == "powexp":
        assert info["n_fp16"] > 0, msg   # the single-precision power-exponential tiles are exercised
    assert eY <= 1e-2 and eY16 <= 1e-2, msg
    assert eL <= 1e-2, msg
    V.close()


@pytest.mark.parametrize("case,fixedacc", [("a_exp", 1e-6), ("ragged_nu15", 1e-5)])
def test_trmm_split_factor_tiles(lib, case, fixedacc):
    """CR_TRMM_SPLIT_L: FP32/FP64-class factor tiles enter the simulation multiply as FP16
    high/low pairs.  Against the exact product of the GPU's own stored factor with the FP16
    right-hand side B = fp16(Z / s) (so that only the multiply's treatment of L and its FP32
    accumulation remain), the split multiply is accurate to the FP32 level, and the default
    one (FP16 casts, Alg.1 step 15) to the FP16 cast level."""
    c = COV_CASES[case]
    xy, V, Vo = _build(lib, c)
    m, info = lib.precision_map(V, amp=True, fixedacc=fixedacc)
    assert info["n_fp32"] > 0, info
    assert lib.potrf_adaptive(V) == 0
    s = info["s"]
    Ls = lib.tilemat_to_dense(V, 1).cpu().numpy()   # L_s = s L as stored, lower part
    M = 96
    Z = inputgen.standard_normals(c["n"], M, 11)
    B = (Z / s).astype(np.float16).astype(np.float64)
    Yref = np.tril(Ls) @ B
    Yc = lib.trmm_sim(V, colmajor(Z), M).cpu().numpy()
    Ysp = lib.trmm_sim(V, colmajor(Z), M, flags=lib.CR_TRMM_SPLIT_L).cpu().numpy()
    e_cast, e_split = relf(Yc, Yref), relf(Ysp, Yref)
    msg = f"tiles {info['n_fp64']}/{info['n_fp32']}/{info['n_fp16']}: cast {e_cast:.2e} split {e_split:.2e}"
    assert e_split <= 2e-6, msg
    assert e_cast >= 20 * e_split, msg
    # the split multiply is still the simulation: against the oracle within the adaptive bound
    assert relf(Ysp, oracle.simulate(oracle.cholesky_lower(Vo), Z)) <= 1e-2, msg
    V.close()


def test_trmm_fp16_destination_per_product(lib):
    """CR_TRMM_FP16_PER_GEMM: each block row's products (the diagonal one, then k = i-1 down
    to 0) are rounded to the FP16 destination one at a time.  Compared with the oracle's
    statement of that task sequence on the GPU's own factor (off-diagonal tiles as their FP16
    casts, FP64 products, FP16 rounding after each), and with the single final rounding of
    CR_TRMM_FP16_DEST, which it must differ from."""
    c = COV_CASES["a_exp"]
    xy, V, Vo = _build(lib, c)
    m, info = lib.precision_map(V, amp=True, fixedacc=1e-4)
    assert lib.potrf_adaptive(V) == 0
    s, n, nb = info["s"], c["n"], c["nb"]
    Ls = np.tril(lib.tilemat_to_dense(V, 1).cpu().numpy())
    M = 80
    Z = inputgen.standard_normals(n, M, 21)
    B = (Z / s).astype(np.float16).astype(np.float64)
    Yp = lib.trmm_sim(V, colmajor(Z), M, flags=lib.CR_TRMM_FP16_PER_GEMM).cpu().numpy()
    Yd = lib.trmm_sim(V, colmajor(Z), M, flags=lib.CR_TRMM_FP16_DEST).cpu().numpy()
    # the factor as the multiply uses it: off-diagonal tiles as their FP16 casts (Alg.1 step 15)
    nt = (n + nb - 1) // nb
    Lc = Ls.astype(np.float16).astype(np.float64)
    for i in range(nt):
        r = slice(i * nb, min(n, (i + 1) * nb))
        Lc[r, r] = Ls[r, r]
    Ye = oracle.simulate_fp16_per_product(Lc, B, nb)
    e_emul, e_once = relf(Yp, Ye), relf(Yp, Yd)
    msg = f"per-product vs emulation {e_emul:.2e}, vs single rounding {e_once:.2e}"
    assert e_emul <= 2e-4 and e_emul <= 0.25 * e_once, msg
    # still the simulation: within the adaptive bound of the oracle's FP64 chain
    assert relf(Yp, oracle.simulate(oracle.cholesky_lower(Vo), Z)) <= 1e-2, msg
    V.close()


def test_rnorm_stream_matches_oracle(lib):
    n, M, seed, off = 777, 33, 42, 5
    Z = lib.rnorm(n, M, seed, off).cpu().numpy()
    Zo = oracle.rnorm(n, M, seed, off)
    assert np.max(np.abs(Z - Zo)) <= 1e-13


def test_generated_simulation_matches_oracle_stream(lib):
    c = COV_CASES["a_exp"]
    xy, V, Vo = _build(lib, c)
    _, info = lib.precision_map(V, amp=True, fixedacc=1e-6)
    assert lib.potrf_adaptive(V) == 0
    s = info["s"]
    M, seed = 100, 9
    Y, bn = lib.trmm_sim(V, None, M, seed=seed, flags=lib.CR_TRMM_GENERATE, want_bnorm=True)
    Zo = oracle.rnorm(c["n"], M, seed)
    Yo = oracle.simulate(oracle.cholesky_lower(Vo), Zo)
    assert relf(Y.cpu().numpy(), Yo) <= 1e-2
    # ||B||_F of B = M_rand / s before rounding (Alg.1 step 6): the fused path draws the same
    # stream in FP32 (about 1e-7 relative per draw) ...
    assert bn == pytest.approx(np.linalg.norm(Zo) / s, rel=1e-6)
    # ... and a given FP64 right-hand side is divided as it stands
    _, bn2 = lib.trmm_sim(V, colmajor(Zo), M, want_bnorm=True)
    assert bn2 == pytest.approx(np.linalg.norm(Zo) / s, rel=1e-12)
    V.close()


def test_calibration_bit_exact(lib):
    rng = np.random.default_rng(17)
    n_p, M, u = 3000, 257, 0.25
    S = rng.standard_normal((n_p, M))
    z = rng.standard_normal(n_p) * 0.5
    v = rng.uniform(0.3, 2.0, n_p)
    out = lib.calibrate(colmajor(S), dev(z), dev(v), u, 0.9, counts=True, extrema=True)
    ref = oracle.calibrate(S, z, v, u, 0.9)
    np.testing.assert_array_equal(out["psi"].cpu().numpy(), ref["psi"])
    np.testing.assert_array_equal(out["phi"].cpu().numpy(), ref["phi"])
    np.testing.assert_array_equal(out["count"].cpu().numpy(), ref["count"])
    assert out["q_in"] == ref["q_in"] and out["q_out"] == ref["q_out"]
    assert out["n_psi"] == ref["n_psi"] and out["n_phi"] == ref["n_phi"]
    np.testing.assert_array_equal(out["c_in"].cpu().numpy(), ref["c_in"])
    np.testing.assert_array_equal(out["c_out"].cpu().numpy(), ref["c_out"])


@pytest.mark.parametrize("u", [0.25, 0.0, -1.5])
def test_calibration_bit_exact_edge_values(lib, u):
    # elements equal to u, one ulp either side, sharing u's high 32 bits, +-0, subnormals,
    # +-inf and NaN, and rows with equal t: the scan decides most elements on 32-bit words
    # and must agree exactly with the oracle's double comparisons on all of these
    rng = np.random.default_rng(23)
    n_p, M = 2500, 70
    S = rng.standard_normal((n_p, M))
    ub = np.float64(u).view(np.uint64)
    special = np.array([u, np.nextafter(u, np.inf), np.nextafter(u, -np.inf), 0.0, -0.0, 5e-324, -5e-324,
                        np.inf, -np.inf, np.nan, 2.2250738585072014e-308,
                        (ub ^ np.uint64(0x5A5A5A5A)).view(np.float64), (ub ^ np.uint64(0xFFFFFFFF)).view(np.float64)])
    mask = rng.random((n_p, M)) < 0.3
    S[mask] = rng.choice(special, size=int(mask.sum()))
    z = rng.standard_normal(n_p) * 0.5
    v = rng.uniform(0.3, 2.0, n_p)
    z[100:140] = z[99]      # equal t values on several rows
    v[100:140] = v[99]
    out = lib.calibrate(colmajor(S), dev(z), dev(v), u, 0.9, counts=True, extrema=True)
    ref = oracle.calibrate(S, z, v, u, 0.9)
    np.testing.assert_array_equal(out["psi"].cpu().numpy(), ref["psi"])
    np.testing.assert_array_equal(out["phi"].cpu().numpy(), ref["phi"])
    np.testing.assert_array_equal(out["count"].cpu().numpy(), ref["count"])
    assert out["q_in"] == ref["q_in"] and out["q_out"] == ref["q_out"]
    np.testing.assert_array_equal(out["c_in"].cpu().numpy(), ref["c_in"])
    np.testing.assert_array_equal(out["c_out"].cpu().numpy(), ref["c_out"])


@pytest.mark.parametrize("u", [0.25, 0.0, -1.5])
def test_negative_excursion_calibration_bit_exact(lib, u):
    """The negative excursion set (Section III's sign reversal) against the oracle, bit-exact,
    including elements equal to u, +-0, infinities and NaN."""
    rng = np.random.default_rng(41)
    n_p, M = 2300, 90
    S = rng.standard_normal((n_p, M))
    mask = rng.random((n_p, M)) < 0.2
    S[mask] = rng.choice(np.array([u, np.nextafter(u, np.inf), 0.0, -0.0, np.inf, -np.inf, np.nan]), size=int(mask.sum()))
    z = rng.standard_normal(n_p) * 0.5
    v = rng.uniform(0.3, 2.0, n_p)
    out = lib.calibrate(colmajor(S), dev(z), dev(v), u, 0.9, counts=True, extrema=True, negative=True)
    ref = oracle.calibrate_negative(S, z, v, u, 0.9)
    np.testing.assert_array_equal(out["psi"].cpu().numpy(), ref["psi"])
    np.testing.assert_array_equal(out["phi"].cpu().numpy(), ref["phi"])
    np.testing.assert_array_equal(out["count"].cpu().numpy(), ref["count"])
    assert out["q_in"] == ref["q_in"] and out["q_out"] == ref["q_out"]
    np.testing.assert_array_equal(out["c_in"].cpu().numpy(), ref["c_in"])
    np.testing.assert_array_equal(out["c_out"].cpu().numpy(), ref["c_out"])


def test_calibration_errors(lib):
    n_p, M = 100, 10
    S = np.full((n_p, M), 5.0)
    with pytest.raises(lib.CrError) as ei:
        lib.calibrate(colmajor(S), dev(np.zeros(n_p)), dev(np.ones(n_p)), 1.0, 0.9)
    assert ei.value.name == "CR_ERR_EMPTY_SAMPLE"
    v = np.ones(n_p)
    v[7] = 0.0
    with pytest.raises(lib.CrError) as ei:
        lib.calibrate(colmajor(np.zeros((n_p, M))), dev(np.zeros(n_p)), dev(v), 1.0, 0.9)
    assert ei.value.name == "CR_ERR_NONPOS_MSPE"


def test_krige_correct_matches_oracle(lib):
    """Eq.7 in double-float arithmetic (48 significant bits) against the oracle's FP64, element
    by element within the product's error bound (n_o + 8) 2^-46 (|W|^T |R|) + 2^-52 |S|, which
    also covers the oracle's own FP64 rounding (n_o 2^-53 (|W|^T |R|))."""
    rng = np.random.default_rng(2)
    for n_p, n_o, M in ((300, 200, 70), (129, 1000, 65)):
        W = rng.standard_normal((n_o, n_p))
        y = rng.standard_normal(n_o)
        Y = rng.standard_normal((n_p + n_o, M))
        S = lib.krige_correct(colmajor(W), dev(y), colmajor(Y), n_p, n_o).cpu().numpy()
        So = oracle.conditional_correction(W, y, Y[:n_p], Y[n_p:])
        R = y[:, None] - Y[n_p:]
        bound = (n_o + 8) * 2.0 ** -46 * (np.abs(W).T @ np.abs(R)) + 2.0 ** -52 * np.abs(So)
        assert np.all(np.abs(S - So) <= bound), np.max(np.abs(S - So) / bound)
        assert np.linalg.norm(S - So) <= np.linalg.norm(bound)


@pytest.mark.parametrize("negative", [False, True])
def test_fused_correction_calibration_matches_unfused(lib, negative):
    """cr_correct_calibrate (S never written) against cr_krige_correct followed by cr_calibrate
    on the same inputs, bit-exact, on ragged sizes (not multiples of the 64 x 64 blocks or of the
    16-wide inner chunks); and against the oracle's calibration of the GPU's own S."""
    rng = np.random.default_rng(31)
    n_p, n_o, M, u, level = 1000, 777, 300, 0.4, 0.9
    W = rng.standard_normal((n_o, n_p)) * 0.05
    y = rng.standard_normal(n_o)
    Y = rng.standard_normal((n_p + n_o, M))
    z = rng.standard_normal(n_p) * 0.5
    v = rng.uniform(0.3, 2.0, n_p)
    Wd, yd, Yd, zd, vd = colmajor(W), dev(y), colmajor(Y), dev(z), dev(v)
    S = lib.krige_correct(Wd, yd, Yd, n_p, n_o)
    a = lib.calibrate(S, zd, vd, u, level, counts=True, extrema=True, negative=negative)
    b = lib.correct_calibrate(Wd, yd, Yd, n_p, n_o, zd, vd, u, level, counts=True, extrema=True, negative=negative)
    for k in ("psi", "phi", "count", "c_in", "c_out"):
        np.testing.assert_array_equal(a[k].cpu().numpy(), b[k].cpu().numpy(), err_msg=k)
    for k in ("q_in", "q_out", "n_psi", "n_phi"):
        assert a[k] == b[k], k
    Sg = S.cpu().numpy()
    ref = (oracle.calibrate_negative if negative else oracle.calibrate)(Sg, z, v, u, level)
    assert b["q_in"] == ref["q_in"] and b["q_out"] == ref["q_out"]
    np.testing.assert_array_equal(b["c_in"].cpu().numpy(), ref["c_in"])
    np.testing.assert_array_equal(b["c_out"].cpu().numpy(), ref["c_out"])
    np.testing.assert_array_equal(b["count"].cpu().numpy(), ref["count"])


def test_not_spd_reports_column(lib):
    # points 0 and 1 coincide and there is no nugget: V_00 = V_01 = V_11 = 1 exactly, so the
    # second pivot is 1 - 1 * 1 = 0 exactly and column 2 (1-based) is reported
    xy = inputgen.morton_sorted(inputgen.uniform_locations(256, 3))
    xy[1] = xy[0]
    V = lib.TileMat(256, 128)
    lib.cov_build(V, dev(xy), "matern", 1.0, 0.1, 0.5, nugget=0.0)
    lib.precision_map(V, amp=False)
    info = lib.potrf_adaptive(V)
    assert info == 2
    V.close()
