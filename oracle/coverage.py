"""Coverage of the confidence regions (oracle; test infrastructure).

"Mixed-Precision GPU Acceleration for Confidence Regions of Spatial Excursion Sets":
  * §VI-B.1: the true field of a replicate is Z = X b + L eta, with L L^T the joint
    covariance V of all sites (prediction and observation) and eta i.i.d. N(0, 1).  The
    observations are the true field at the observation sites; their measurement noise is
    the tau^2 already on V's observation block (the reading taken for the noise).
  * §VI-B.2 / Fig. 3: the excursion set of the truth over the prediction sites is
    A = {i in D_p : Z_i >= u}; a replicate succeeds when C_in is inside A and A is inside
    C_out.  The empirical coverage is the fraction of successful replicates.  Fig. 3 plots
    an inner coverage rate (panel a) and an outer one (panel b): the fractions of replicates
    with C_in inside A, and with A inside C_out, each on its own.
  * §III: for a negative excursion set the truth's set is {i : Z_i <= u} (the positive set
    of the sign-reversed field at -u).
"""
from __future__ import annotations

import numpy as np


def truth_field(L: np.ndarray, X: np.ndarray, b, eta: np.ndarray) -> np.ndarray:
    """Z = X b + L eta for a lower-triangular L with L L^T = V (§VI-B.1); eta may hold one
    draw per column."""
    mean = np.asarray(X, dtype=np.float64) @ np.asarray(b, dtype=np.float64)
    eta = np.asarray(eta, dtype=np.float64)
    return (mean[:, None] if eta.ndim == 2 else mean) + np.asarray(L) @ eta


def excursion_set(z_p: np.ndarray, u: float, negative: bool = False) -> np.ndarray:
    """A = {i : z_i >= u} as a boolean mask (§VI-B.2); {i : z_i <= u} for a negative set (§III)."""
    return np.asarray(z_p) <= u if negative else np.asarray(z_p) >= u


def coverage_event(truth_p: np.ndarray, c_in, c_out, u: float, negative: bool = False) -> bool:
    """True when C_in is a subset of A and A is a subset of C_out (§VI-B.2)."""
    A = excursion_set(truth_p, u, negative)
    inner = np.asarray(c_in).astype(bool)
    outer = np.asarray(c_out).astype(bool)
    return bool(np.all(A[inner]) and np.all(outer[A]))


def inner_event(truth_p: np.ndarray, c_in, u: float, negative: bool = False) -> bool:
    """True when C_in is a subset of A (the inner region's event of Fig. 3a)."""
    A = excursion_set(truth_p, u, negative)
    return bool(np.all(A[np.asarray(c_in).astype(bool)]))


def outer_event(truth_p: np.ndarray, c_out, u: float, negative: bool = False) -> bool:
    """True when A is a subset of C_out (the outer region's event of Fig. 3b)."""
    A = excursion_set(truth_p, u, negative)
    return bool(np.all(np.asarray(c_out).astype(bool)[A]))
