"""Universal kriging, pointwise MSPE and the conditioning correction (oracle; test infra).

"Mixed-Precision GPU Acceleration for Confidence Regions of Spatial Excursion Sets":
  * §V-A Eq.5:  W = Sigma_y^-1 [V_op - X_o (X_o^T Sigma_y^-1 X_o)^-1 (X_o^T Sigma_y^-1 V_op - X_p^T)],
    evaluated as in Alg.2 steps 2-4: factor Sigma_y = L_o L_o^T and solve Sigma_y F = X_o;
    G = X_o^T F; solve G H = F^T V_op - X_p^T; solve L_o Y = V_op - X_o H, then L_o^T W = Y.
  * §V-A: z_hat = W^T y_o (Alg.2 step 5); U = Sigma_y W with the unfactored Sigma_y.
  * §V-A Eq.6:  v = theta0 1 + colsum(W .* U) - 2 colsum(V_op .* W), theta0 = sigma^2
    ("initialized from theta[0]").
  * §V-B Eq.7:  S = M_p + W^T (y_o 1^T - M_o).
V_op is the n_o x n_p lower-left block of the joint covariance of Eq.4.
"""
from __future__ import annotations

import numpy as np

from .linalg import cholesky_lower, solve_lower, solve_lower_transpose


def universal_kriging(Sigma_y: np.ndarray, V_op: np.ndarray, X_o: np.ndarray, X_p: np.ndarray,
                      y_o: np.ndarray, theta0: float):
    """Returns (W, z_hat, v) following Alg.2 steps 2-6."""
    L_o = cholesky_lower(Sigma_y)                                   # step 2
    F = solve_lower_transpose(L_o, solve_lower(L_o, X_o))           # Sigma_y F = X_o
    G = X_o.T @ F                                                   # step 3
    Lg = cholesky_lower(G)
    H = solve_lower_transpose(Lg, solve_lower(Lg, F.T @ V_op - X_p.T))
    Yk = solve_lower(L_o, V_op - X_o @ H)                           # step 4
    W = solve_lower_transpose(L_o, Yk)
    z_hat = W.T @ y_o                                               # step 5
    U = Sigma_y @ W
    v = theta0 * np.ones(W.shape[1]) + np.sum(W * U, axis=0) - 2.0 * np.sum(V_op * W, axis=0)
    return W, z_hat, v


def conditional_correction(W: np.ndarray, y_o: np.ndarray, M_p: np.ndarray, M_o: np.ndarray) -> np.ndarray:
    """S = M_p + W^T (y_o 1^T - M_o) (Eq.7)."""
    R = y_o[:, None] - M_o
    return M_p + W.T @ R
