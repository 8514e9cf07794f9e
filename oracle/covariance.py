"""Covariance models and the joint covariance (oracle; test infrastructure only).

"Mixed-Precision GPU Acceleration for Confidence Regions of Spatial Excursion Sets":
  * §VI-B.2: stationary power-exponential model with parameters (sigma^2 : beta : nu).
  * §VI-C:   Matern model.  The page gives no formula; the reading taken here is
             C(h) = sigma^2 2^(1-nu)/Gamma(nu) (h/beta)^nu K_nu(h/beta), C(0) = sigma^2,
             with beta the range as given.
  * §V Eq.4: joint covariance over prediction sites (first) and observation sites; the
             measurement-error variance tau^2 is added to the observation block only.
Reading for workloads without observations: a nugget is added to every diagonal entry.
K_nu and Gamma come from scipy.special (library primitives).
"""
from __future__ import annotations

import numpy as np
from scipy import special


def matern(h, sigma2: float, beta: float, nu: float) -> np.ndarray:
    """Matern covariance at distances h (§VI-C, reading above)."""
    h = np.asarray(h, dtype=np.float64)
    out = np.full(h.shape, float(sigma2))
    pos = h > 0
    x = h[pos] / beta
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        val = sigma2 * (2.0 ** (1.0 - nu) / special.gamma(nu)) * np.power(x, nu) * special.kv(nu, x)
    # K_nu underflows to 0 for very large x; x^nu * 0 = 0 there, which is the limit.
    val = np.where(np.isfinite(val), val, 0.0)
    out[pos] = val
    return out


def powexp(h, sigma2: float, beta: float, nu: float) -> np.ndarray:
    """Power-exponential covariance sigma^2 exp(-(h/beta)^nu) (§VI-B.2)."""
    h = np.asarray(h, dtype=np.float64)
    return sigma2 * np.exp(-np.power(h / beta, nu))


def covariance_fn(family: str):
    if family == "matern":
        return matern
    if family == "powexp":
        return powexp
    raise ValueError(family)


def _distances(xa: np.ndarray, xb: np.ndarray) -> np.ndarray:
    dx = xa[:, None, 0] - xb[None, :, 0]
    dy = xa[:, None, 1] - xb[None, :, 1]
    return np.sqrt(dx * dx + dy * dy)


def covariance_entries(xy: np.ndarray, rows: np.ndarray, cols: np.ndarray, family: str,
                       sigma2: float, beta: float, nu: float, nugget: float = 0.0,
                       n_pred: int | None = None, tau2: float = 0.0) -> np.ndarray:
    """V[rows[q], cols[q]] of the joint covariance (Eq.4) for index pairs q."""
    xy = np.asarray(xy, dtype=np.float64)
    rows = np.asarray(rows)
    cols = np.asarray(cols)
    dx = xy[rows, 0] - xy[cols, 0]
    dy = xy[rows, 1] - xy[cols, 1]
    h = np.sqrt(dx * dx + dy * dy)
    v = covariance_fn(family)(h, sigma2, beta, nu)
    diag = rows == cols
    v = np.where(diag, float(sigma2) + nugget, v)
    if n_pred is not None and tau2 != 0.0:
        v = np.where(diag & (rows >= n_pred), v + tau2, v)
    return v


def covariance_matrix(xy: np.ndarray, family: str, sigma2: float, beta: float, nu: float,
                      nugget: float = 0.0, n_pred: int | None = None, tau2: float = 0.0,
                      rows: slice | None = None, cols: slice | None = None) -> np.ndarray:
    """Dense block V[rows, cols] of the joint covariance (§V Eq.4).

    V_ij = C(|x_i - x_j|); the diagonal is C(0) = sigma^2, plus ``nugget`` everywhere
    and plus ``tau2`` on observation rows (index >= n_pred), Sigma_y = V_o + tau^2 I.
    """
    xy = np.asarray(xy, dtype=np.float64)
    n = xy.shape[0]
    rows = rows if rows is not None else slice(0, n)
    cols = cols if cols is not None else slice(0, n)
    ri = np.arange(n)[rows]
    ci = np.arange(n)[cols]
    V = covariance_fn(family)(_distances(xy[ri], xy[ci]), sigma2, beta, nu)
    same = ri[:, None] == ci[None, :]
    V[same] = float(sigma2) + nugget
    if n_pred is not None and tau2 != 0.0:
        V[same & (ri[:, None] >= n_pred)] += tau2
    return V
