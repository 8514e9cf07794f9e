"""Calibration of the inner and outer confidence regions (oracle; test infrastructure).

"Mixed-Precision GPU Acceleration for Confidence Regions of Spatial Excursion Sets":
  * §III Eq.1 / Alg.2 step 18: t = (z_hat - u 1) / sqrt(v); positive MSPEs are required.
  * §V-C Eq.8 / Alg.2 step 19: A+_j = {i : S_ij >= u}, A-_j = {i : S_ij <= u};
    psi_j = min_{i in A+_j} t_i, phi_j = max_{i in A-_j} t_i.  An empty set leaves a
    sentinel (+inf for psi, -inf for phi) that is left out of the sample (§V-C), so the
    two samples may differ in size; both must be non-empty.
  * §V-C Eq.9: Q_p(a) = a_(max{1, min{N, ceil(p N)}}) on the sorted sample (1-based).
    Reading for the ceiling under floating point: k = ceil(p N - 1e-9), so a p N that is
    an integer up to representation error is not pushed to the next index.
  * §V-C and Alg.2 steps 21-22: with c = 1 - alpha, q_out = Q_alpha(psi),
    q_in = Q_{1-alpha}(phi); C_out = {t_i >= q_out} (non-strict), C_in = {t_i > q_in}.
  * Per-location exceedance counts count_i = #{j : S_ij >= u} (the exceedance idea of §I).
  * §III: negative excursion sets {Z <= u} are handled by reversing the sign of the process
    and of the threshold: calibrate_negative(S, z_hat, v, u) = calibrate(-S, -z_hat, v, -u).
"""
from __future__ import annotations

import math
import numpy as np


class EmptySample(ValueError):
    pass


def standardized_statistic(z_hat: np.ndarray, v: np.ndarray, u: float) -> np.ndarray:
    v = np.asarray(v, dtype=np.float64)
    if not np.all(v > 0):
        raise ValueError("non-positive MSPE")
    return (np.asarray(z_hat, dtype=np.float64) - u) / np.sqrt(v)


def extrema_scan(S: np.ndarray, t: np.ndarray, u: float):
    """psi_j, phi_j of Eq.8 with +inf / -inf sentinels for empty sets."""
    S = np.asarray(S, dtype=np.float64)
    tt = np.asarray(t, dtype=np.float64)[:, None]
    psi = np.min(np.where(S >= u, tt, np.inf), axis=0)
    phi = np.max(np.where(S <= u, tt, -np.inf), axis=0)
    return psi, phi


def exceedance_counts(S: np.ndarray, u: float) -> np.ndarray:
    return np.sum(np.asarray(S) >= u, axis=1).astype(np.int32)


def sample_without_sentinels(a: np.ndarray, sentinel: float) -> np.ndarray:
    a = np.asarray(a, dtype=np.float64)
    return np.sort(a[a != sentinel])


def empirical_quantile(sorted_a: np.ndarray, p: float) -> float:
    """Q_p of Eq.9 on an already sorted, non-empty sample."""
    N = len(sorted_a)
    if N == 0:
        raise EmptySample("empty sample")
    k = math.ceil(p * N - 1e-9)
    k = max(1, min(N, k))
    return float(sorted_a[k - 1])


def confidence_regions(t: np.ndarray, q_in: float, q_out: float):
    t = np.asarray(t, dtype=np.float64)
    return (t > q_in).astype(np.uint8), (t >= q_out).astype(np.uint8)


def calibrate(S: np.ndarray, z_hat: np.ndarray, v: np.ndarray, u: float, level: float) -> dict:
    """Alg.2 steps 18-22 plus per-location exceedance counts."""
    t = standardized_statistic(z_hat, v, u)
    psi, phi = extrema_scan(S, t, u)
    a_psi = sample_without_sentinels(psi, np.inf)
    a_phi = sample_without_sentinels(phi, -np.inf)
    if len(a_psi) == 0 or len(a_phi) == 0:
        raise EmptySample(f"n_psi={len(a_psi)} n_phi={len(a_phi)}")
    alpha = 1.0 - level
    q_out = empirical_quantile(a_psi, alpha)
    q_in = empirical_quantile(a_phi, 1.0 - alpha)
    c_in, c_out = confidence_regions(t, q_in, q_out)
    return {"t": t, "psi": psi, "phi": phi, "q_in": q_in, "q_out": q_out, "c_in": c_in,
            "c_out": c_out, "count": exceedance_counts(S, u), "n_psi": len(a_psi),
            "n_phi": len(a_phi)}


def calibrate_negative(S: np.ndarray, z_hat: np.ndarray, v: np.ndarray, u: float, level: float) -> dict:
    """Confidence regions of the negative excursion set {Z <= u} (§III: the method applied to the
    sign-reversed field -Z and threshold -u).  t, psi, phi, q_in, q_out and the regions are
    those of the reversed problem; count_i = #{j : -S_ij >= -u} = #{j : S_ij <= u}."""
    return calibrate(-np.asarray(S, dtype=np.float64), -np.asarray(z_hat, dtype=np.float64), v, -u, level)
