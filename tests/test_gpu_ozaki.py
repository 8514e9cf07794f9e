"""The conditioning correction (Eq.7 of "Mixed-Precision GPU Acceleration for Confidence Regions
of Spatial Excursion Sets", Section V-B) with its FP64 product emulated on the FP16 tensor cores
by the Ozaki scheme (CR_OPT_FP64_GEMM = CR_GEMM_OZAKI), against the oracle's FP64.

Error bound of the emulated product C = W^T R, entry (i, j), with Ea_i the exponent of column i
of W (max_k |W_ki| < 2^Ea_i) and Eb_j that of column j of R:
  - slicing: each entry is cut into 8 slices of 6 bits below 2^Ea (truncation), so
    W_ki = sum_s a_s 2^(Ea - 6 s) + d with |d| < 2^(Ea - 48), |a_s| <= 63 (same for R);
  - per term k, the two truncations are below 2 2^(Ea + Eb - 48), and the dropped slice
    products (s + t >= 10: 17 - L of them at level L) below
    sum_L (17 - L) 63^2 2^(Ea + Eb - 6 L) < 6.9 2^(Ea + Eb - 48), together < 8.95 2^(Ea + Eb - 48);
  - the kept products are exact integers (FP16 x FP16 summed over at most 4096 terms, below
    2^24, in FP32; a level's chunk sums exact in 32-bit integers); the 8 levels' power-of-two-
    scaled sums are added in double-float pairs, each addition within 2^-47 of the running
    magnitude, itself below (|W|^T |R|)_ij: at most 16 2^-47 (|W|^T |R|)_ij with margin;
  - S = M_p + C rounds once in FP64, and the oracle's own FP64 product errs by up to
    n_o 2^-53 (|W|^T |R|)_ij.
So |S - S_oracle| <= n_o 9 2^-48 2^(Ea_i + Eb_j) + (16 2^-47 + n_o 2^-53) (|W|^T |R|)_ij
+ 2^-52 |S_ij|."""
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
    return torch.from_numpy(np.asfortranarray(a).T.copy()).cuda().T


@contextlib.contextmanager
def gemm_mode(lib, mode):
    old = lib.get_option(lib.CR_OPT_FP64_GEMM)
    lib.set_option(lib.CR_OPT_FP64_GEMM, mode)
    try:
        yield
    finally:
        lib.set_option(lib.CR_OPT_FP64_GEMM, old)


def _exp_above(X):
    """E per column with max |X| < 2^E (0 for a zero column)."""
    m = np.max(np.abs(X), axis=0)
    e = np.zeros(X.shape[1], dtype=np.int64)
    nz = m > 0
    e[nz] = np.floor(np.log2(m[nz])).astype(np.int64) + 1
    return e


def _bound(W, R, S, n_o):
    Ea, Eb = _exp_above(W), _exp_above(R)
    WR = np.abs(W).T @ np.abs(R)
    return (n_o * 9.0 * 2.0 ** -48 * np.exp2((Ea[:, None] + Eb[None, :]).astype(float))
            + (16 * 2.0 ** -47 + n_o * 2.0 ** -53) * WR + 2.0 ** -52 * np.abs(S))


@pytest.mark.parametrize("n_p,n_o,M,scale", [(300, 200, 70, 1.0), (129, 1000, 65, 1.0), (257, 2100, 130, 1e-3),
                                             (64, 4000, 33, 1.0), (100, 6000, 40, 1.0)])
def test_ozaki_correction_matches_oracle(lib, n_p, n_o, M, scale):
    """Element by element within the bound above, on ragged sizes (n_o not a multiple of the
    128-row padding of the chunks: the padding slices are zero; n_o = 2100 is one chunk of 2176
    rows per slice, 4000 one of 4096, 6000 two of 3072, so each level's product spans several
    chunks and slices) and with columns of W spanning several orders
    of magnitude (as kriging weights do)."""
    rng = np.random.default_rng(n_p + n_o)
    W = rng.standard_normal((n_o, n_p)) * scale * np.exp(rng.uniform(-8, 2, n_p))[None, :]
    W[rng.random((n_o, n_p)) < 0.2] *= 1e-6
    y = rng.standard_normal(n_o)
    Y = rng.standard_normal((n_p + n_o, M))
    with gemm_mode(lib, lib.CR_GEMM_OZAKI):
        S = lib.krige_correct(colmajor(W), dev(y), colmajor(Y), n_p, n_o).cpu().numpy()
    So = oracle.conditional_correction(W, y, Y[:n_p], Y[n_p:])
    R = y[:, None] - Y[n_p:]
    b = _bound(W, R, So, n_o)
    err = np.abs(S - So)
    assert np.all(err <= b), float(np.max(err / b))
    assert np.linalg.norm(err) <= np.linalg.norm(b)
    assert np.linalg.norm(S - So) <= 1e-11 * np.linalg.norm(So)


@pytest.mark.parametrize("n_p,n_o,M", [(1, 1, 1), (3, 1, 5), (1, 4097, 1), (7, 129, 2), (2, 8193, 3)])
def test_ozaki_correction_degenerate_sizes(lib, n_p, n_o, M):
    """One output, an inner dimension of 1, and inner dimensions just past a 128-row padding step
    (129) and past one and two 4096-row chunks (4097: two chunks of 2176 rows; 8193: three of
    2816), within the bound above."""
    rng = np.random.default_rng(n_p * 100000 + n_o * 10 + M)
    W = rng.standard_normal((n_o, n_p))
    y = rng.standard_normal(n_o)
    Y = rng.standard_normal((n_p + n_o, M))
    with gemm_mode(lib, lib.CR_GEMM_OZAKI):
        S = lib.krige_correct(colmajor(W), dev(y), colmajor(Y), n_p, n_o).cpu().numpy()
    So = oracle.conditional_correction(W, y, Y[:n_p], Y[n_p:])
    R = y[:, None] - Y[n_p:]
    assert np.all(np.abs(S - So) <= _bound(W, R, So, n_o))


@pytest.mark.parametrize("sw,sy", [(1e30, 1e20), (1e-30, 1e-20), (1e150, 1e-160)])
def test_ozaki_correction_beyond_fp32_range(lib, sw, sy):
    """Operands whose products lie far outside FP32's range (about 1e50, 1e-50, 1e-10 from
    1e150 x 1e-160): the accumulation runs in units of each output's column exponents, so the
    result keeps FP64's range and the bound above."""
    rng = np.random.default_rng(3)
    n_p, n_o, M = 90, 1300, 33
    W = rng.standard_normal((n_o, n_p)) * sw
    y = rng.standard_normal(n_o) * sy
    Y = rng.standard_normal((n_p + n_o, M)) * sy
    with gemm_mode(lib, lib.CR_GEMM_OZAKI):
        S = lib.krige_correct(colmajor(W), dev(y), colmajor(Y), n_p, n_o).cpu().numpy()
    So = oracle.conditional_correction(W, y, Y[:n_p], Y[n_p:])
    R = y[:, None] - Y[n_p:]
    assert np.all(np.isfinite(S))
    assert np.all(np.abs(S - So) <= _bound(W, R, So, n_o))


def test_ozaki_slices_exact_on_integers(lib):
    """Entries that are small integers times powers of two are represented exactly by their
    slices and every slice product is exact, so the product equals the exact integer result."""
    rng = np.random.default_rng(5)
    n_p, n_o, M = 200, 3000, 40
    W = rng.integers(-1000, 1000, (n_o, n_p)).astype(np.float64) * 2.0 ** -20
    y = rng.integers(-50, 50, n_o).astype(np.float64)
    Y = np.zeros((n_p + n_o, M))
    Y[n_p:] = rng.integers(-50, 50, (n_o, M)).astype(np.float64)
    with gemm_mode(lib, lib.CR_GEMM_OZAKI):
        S = lib.krige_correct(colmajor(W), dev(y), colmajor(Y), n_p, n_o).cpu().numpy()
    Wi = (W * 2.0 ** 20).astype(np.int64)
    Ri = (y[:, None] - Y[n_p:]).astype(np.int64)
    exact = (Wi.T @ Ri).astype(np.float64) * 2.0 ** -20
    np.testing.assert_array_equal(S, exact)


@pytest.mark.parametrize("negative", [False, True])
def test_ozaki_correct_calibrate_matches_unfused(lib, negative):
    """cr_correct_calibrate with the Ozaki product against cr_krige_correct (Ozaki) followed by
    cr_calibrate: bit-exact (the same S), and the oracle's calibration of that S."""
    rng = np.random.default_rng(41)
    n_p, n_o, M, u, level = 1000, 1500, 300, 0.4, 0.9
    W = rng.standard_normal((n_o, n_p)) * 0.05
    y = rng.standard_normal(n_o)
    Y = rng.standard_normal((n_p + n_o, M))
    z = rng.standard_normal(n_p) * 0.5
    v = rng.uniform(0.3, 2.0, n_p)
    Wd, yd, Yd, zd, vd = colmajor(W), dev(y), colmajor(Y), dev(z), dev(v)
    with gemm_mode(lib, lib.CR_GEMM_OZAKI):
        S = lib.krige_correct(Wd, yd, Yd, n_p, n_o)
        a = lib.calibrate(S, zd, vd, u, level, counts=True, extrema=True, negative=negative)
        b = lib.correct_calibrate(Wd, yd, Yd, n_p, n_o, zd, vd, u, level, counts=True, extrema=True,
                                  negative=negative)
    for k in ("psi", "phi", "count", "c_in", "c_out"):
        np.testing.assert_array_equal(a[k].cpu().numpy(), b[k].cpu().numpy(), err_msg=k)
    for k in ("q_in", "q_out", "n_psi", "n_phi"):
        assert a[k] == b[k], k
    Sg = S.cpu().numpy()
    ref = (oracle.calibrate_negative if negative else oracle.calibrate)(Sg, z, v, u, level)
    assert b["q_in"] == ref["q_in"] and b["q_out"] == ref["q_out"]
    np.testing.assert_array_equal(b["c_in"].cpu().numpy(), ref["c_in"])
    np.testing.assert_array_equal(b["c_out"].cpu().numpy(), ref["c_out"])


def test_ozaki_nonfinite_operands_give_nan(lib):
    """A NaN or an infinity in W (or in R = y_o 1^T - M_o) reaches, in an FP64 product, every
    output of its column of W (row of S) or of R (column of S): the Ozaki product makes exactly
    those outputs NaN and leaves the others as they are without the bad entry's column."""
    rng = np.random.default_rng(13)
    n_p, n_o, M = 150, 700, 40
    W = rng.standard_normal((n_o, n_p)) * 0.1
    y = rng.standard_normal(n_o)
    Y = rng.standard_normal((n_p + n_o, M))
    W[17, 5] = np.nan
    W[300, 80] = np.inf
    Y[n_p + 9, 33] = -np.inf
    with gemm_mode(lib, lib.CR_GEMM_OZAKI):
        S = lib.krige_correct(colmajor(W), dev(y), colmajor(Y), n_p, n_o).cpu().numpy()
    bad = np.zeros((n_p, M), dtype=bool)
    bad[[5, 80], :] = True
    bad[:, 33] = True
    assert np.all(np.isnan(S[bad]))
    Wc, Yc = W.copy(), Y.copy()
    Wc[:, [5, 80]] = 0.0
    Yc[:, 33] = 0.0
    So = oracle.conditional_correction(Wc, y, Yc[:n_p], Yc[n_p:])
    R = y[:, None] - Yc[n_p:]
    b = _bound(Wc, R, So, n_o)
    assert np.all(np.abs(S[~bad] - So[~bad]) <= b[~bad])


@pytest.mark.parametrize("negative", [False, True])
def test_prepared_weights_bit_exact(lib, negative):
    """cr_weights_prepare then cr_krige_correct_prepared / cr_correct_calibrate_prepared give
    the bits of cr_krige_correct / cr_correct_calibrate with CR_GEMM_OZAKI on the same W, over
    several simulation batches, with W overwritten after the handle was made (the handle does
    not read W again) and whatever CR_OPT_FP64_GEMM says."""
    rng = np.random.default_rng(23)
    n_p, n_o, u, level = 700, 2300, 0.3, 0.9
    W = rng.standard_normal((n_o, n_p)) * 0.05
    y = rng.standard_normal(n_o)
    z = rng.standard_normal(n_p) * 0.5
    v = rng.uniform(0.3, 2.0, n_p)
    Wd, yd, zd, vd = colmajor(W), dev(y), dev(z), dev(v)
    Wp = lib.Weights(Wd)
    torch.cuda.synchronize()
    Wkeep = Wd.clone()
    Wd.fill_(7.0)
    for batch, M in enumerate((64, 129)):
        Y = colmajor(np.random.default_rng(100 + batch).standard_normal((n_p + n_o, M)))
        with gemm_mode(lib, lib.CR_GEMM_OZAKI):
            S = lib.krige_correct(Wkeep, yd, Y, n_p, n_o).cpu().numpy()
            a = lib.correct_calibrate(Wkeep, yd, Y, n_p, n_o, zd, vd, u, level, extrema=True, negative=negative)
        with gemm_mode(lib, lib.CR_GEMM_DF):
            Sp = lib.krige_correct_prepared(Wp, yd, Y).cpu().numpy()
            b = lib.correct_calibrate_prepared(Wp, yd, Y, zd, vd, u, level, extrema=True, negative=negative)
        np.testing.assert_array_equal(S, Sp)
        for k in ("psi", "phi", "count", "c_in", "c_out"):
            np.testing.assert_array_equal(a[k].cpu().numpy(), b[k].cpu().numpy(), err_msg=k)
        assert (a["q_in"], a["q_out"]) == (b["q_in"], b["q_out"])
    Wp.close()


def test_pooled_scratch_reused_and_trimmed(lib):
    """The correction's scratch comes from the library pool: repeated calls, and a call after
    cr_workspace_trim has returned the pool's memory, give the same bits."""
    rng = np.random.default_rng(9)
    n_p, n_o, M = 500, 2500, 96
    W = colmajor(rng.standard_normal((n_o, n_p)) * 0.1)
    y = dev(rng.standard_normal(n_o))
    Y = colmajor(rng.standard_normal((n_p + n_o, M)))
    with gemm_mode(lib, lib.CR_GEMM_OZAKI):
        a = lib.krige_correct(W, y, Y, n_p, n_o).cpu().numpy()
        b = lib.krige_correct(W, y, Y, n_p, n_o).cpu().numpy()
        torch.cuda.synchronize()
        lib.workspace_trim()
        c = lib.krige_correct(W, y, Y, n_p, n_o).cpu().numpy()
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(a, c)


def test_ozaki_full_size_sampled_rows(lib):
    """The kriging workload's shape (16384 observations, 16384 prediction sites) with 1100
    simulations: 4096-row chunks, and the chunk products of a level for all 1100 columns no
    longer fit the 2 GiB budget, so the product runs in two blocks of columns (1024 and 76).
    Sampled rows of S against the oracle within the bound."""
    rng = np.random.default_rng(77)
    n_p, n_o, M = 16384, 16384, 1100
    W = rng.standard_normal((n_o, n_p)) * np.exp(rng.uniform(-6, 1, n_p))[None, :]
    y = rng.standard_normal(n_o)
    Y = rng.standard_normal((n_p + n_o, M))
    with gemm_mode(lib, lib.CR_GEMM_OZAKI):
        S = lib.krige_correct(colmajor(W), dev(y), colmajor(Y), n_p, n_o)
    rows = np.sort(rng.choice(n_p, 48, replace=False))
    rows[0], rows[-1] = 0, n_p - 1
    Sg = S[torch.from_numpy(rows).cuda()].cpu().numpy()
    del S
    So = oracle.conditional_correction(W[:, rows], y, Y[rows], Y[n_p:])
    R = y[:, None] - Y[n_p:]
    b = _bound(W[:, rows], R, So, n_o)
    err = np.abs(Sg - So)
    assert np.all(err <= b), float(np.max(err / b))


def relf(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


def _krige_case(n_o, m, seed, nu=1.0, beta=0.1, tau2=0.01):
    pred = inputgen.morton_sorted(inputgen.grid_cell_centres(m))
    obs = inputgen.morton_sorted(inputgen.uniform_locations(n_o, seed))
    xy = np.ascontiguousarray(np.concatenate([pred, obs]))
    n_p = len(pred)
    X = np.column_stack([np.ones(len(xy)), xy[:, 0], xy[:, 1]])
    y = inputgen.observation_values(obs, (1.0, 0.5, -0.3), 0.3, seed + 1)
    V = oracle.covariance_matrix(xy, "matern", 1.0, beta, nu, 0.0, n_p, tau2)
    return xy, n_p, X, y, V


@pytest.mark.parametrize("n_o,m,nb", [(1024, 32, 128), (1000, 24, 128), (4096, 64, 512), (2600, 40, 512),
                                      (100, 8, 128)])
def test_ozaki_kriging_matches_oracle(lib, n_o, m, nb):
    """cr_krige with its many-right-hand-side triangular solves as Ozaki products (Section V-A
    Eq.5-6; Alg.2 steps 2-6) against the oracle, with the FP64 path's tolerance: W and z_hat
    within max(1e-10, 20 x the distance between two FP64 orderings of the same solves) in
    relative Frobenius norm, v within 1e-9, and X_o^T W = X_p^T.  Ragged cases: n_o = 1000 and
    2600 leave a partial last tile row; n_o = 100 is a single partial tile (no off-diagonal
    update, only the diagonal steps)."""
    xy, n_p, X, y, V = _krige_case(n_o, m, 5)
    G = lib.TileMat(len(xy), nb)
    lib.cov_build(G, dev(xy), "matern", 1.0, 0.1, 1.0, nugget=0.0, n_pred=n_p, tau2=0.01)
    with gemm_mode(lib, lib.CR_GEMM_OZAKI):
        W, z, v = lib.krige(G, colmajor(X[n_p:]), colmajor(X[:n_p]), dev(y))
    Wo, zo, vo = oracle.universal_kriging(V[n_p:, n_p:], V[n_p:, :n_p], X[n_p:], X[:n_p], y, 1.0)
    K = np.block([[V[n_p:, n_p:], X[n_p:]], [X[n_p:].T, np.zeros((3, 3))]])
    Wl = np.linalg.solve(K, np.vstack([V[n_p:, :n_p], X[:n_p].T]))[:n_o]
    tol = max(1e-10, 20 * relf(Wl, Wo))
    Wg = W.cpu().numpy()
    assert relf(Wg, Wo) <= tol, (relf(Wg, Wo), tol)
    assert relf(z.cpu().numpy(), zo) <= tol
    assert np.max(np.abs(v.cpu().numpy() - vo)) <= 1e-9
    np.testing.assert_allclose(X[n_p:].T @ Wg, X[:n_p].T, atol=1e-8)
    G.close()


def test_ozaki_kriging_full_size_against_fp64_solves(lib):
    """The kriging workload (16384 observations, 128 x 128 grid, tile 512): W, z_hat and v from
    the Ozaki solves against those of the FP64 solves on the same factor, within the oracle
    tests' 1e-10 floor (relative Frobenius; v within 1e-9), and X_o^T W = X_p^T."""
    w = inputgen.WORKLOADS["k"]
    xy = inputgen.workload_locations(w)
    n_p, n_o = w.n_pred, w.n_obs
    X = np.column_stack([np.ones(w.n), xy[:, 0], xy[:, 1]])
    y = inputgen.observation_values(xy[n_p:], (1.0, 0.5, -0.3), 0.1, 3)
    V = lib.TileMat(w.n, w.nb)
    lib.cov_build(V, dev(xy), w.family, w.sigma2, w.beta, w.nu, nugget=w.nugget, n_pred=n_p, tau2=w.tau2)
    Xo, Xp, yd = colmajor(X[n_p:]), colmajor(X[:n_p]), dev(y)
    with gemm_mode(lib, lib.CR_GEMM_DF):
        W64, z64, v64 = lib.krige(V, Xo, Xp, yd)
    with gemm_mode(lib, lib.CR_GEMM_OZAKI):
        W, z, v = lib.krige(V, Xo, Xp, yd)
    e = (torch.linalg.norm(W - W64) / torch.linalg.norm(W64)).item()
    assert e <= 1e-10, e
    assert (torch.linalg.norm(z - z64) / torch.linalg.norm(z64)).item() <= 1e-10
    assert torch.max(torch.abs(v - v64)).item() <= 1e-9
    XoT_W = (torch.from_numpy(X[n_p:]).cuda().T @ W).cpu().numpy()
    assert np.max(np.abs(XoT_W - X[:n_p].T)) <= 1e-6 * np.max(np.abs(X[:n_p]))
    V.close()
