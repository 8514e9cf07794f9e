"""Unblocked FP64 Cholesky and triangular solves (oracle; test infrastructure only).

"Mixed-Precision GPU Acceleration for Confidence Regions of Spatial Excursion Sets",
Alg.2 steps 2-4 and 12 factor covariance matrices and solve with the factor.  The oracle
states the textbook definitions directly, with no blocking:
  l_jj = sqrt(a_jj - sum_{k<j} l_jk^2),  l_ij = (a_ij - sum_{k<j} l_ik l_jk) / l_jj.
Each inner sum is one library dot/matrix-vector product.
"""
from __future__ import annotations

import math
import numpy as np


class NotSPD(ArithmeticError):
    """Raised when a pivot is not positive; ``column`` is 1-based (LAPACK info)."""

    def __init__(self, column: int):
        super().__init__(f"matrix is not positive definite at column {column}")
        self.column = column


def cholesky_lower(A: np.ndarray) -> np.ndarray:
    """Lower Cholesky factor L, A = L L^T, column by column (definition above)."""
    A = np.asarray(A, dtype=np.float64)
    n = A.shape[0]
    L = np.zeros((n, n), dtype=np.float64, order="C")
    for j in range(n):
        lj = L[j, :j]
        d = A[j, j] - float(lj @ lj)
        if not d > 0.0:
            raise NotSPD(j + 1)
        ljj = math.sqrt(d)
        L[j, j] = ljj
        if j + 1 < n:
            L[j + 1:, j] = (A[j + 1:, j] - L[j + 1:, :j] @ lj) / ljj
    return L


def solve_lower(L: np.ndarray, B: np.ndarray) -> np.ndarray:
    """X with L X = B by forward substitution, row by row."""
    L = np.asarray(L, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    vec = B.ndim == 1
    B2 = B[:, None] if vec else B
    n = L.shape[0]
    X = np.zeros_like(B2, dtype=np.float64)
    for i in range(n):
        X[i] = (B2[i] - L[i, :i] @ X[:i]) / L[i, i]
    return X[:, 0] if vec else X


def solve_lower_transpose(L: np.ndarray, B: np.ndarray) -> np.ndarray:
    """X with L^T X = B by backward substitution, row by row."""
    L = np.asarray(L, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    vec = B.ndim == 1
    B2 = B[:, None] if vec else B
    n = L.shape[0]
    X = np.zeros_like(B2, dtype=np.float64)
    for i in range(n - 1, -1, -1):
        X[i] = (B2[i] - L[i + 1:, i] @ X[i + 1:]) / L[i, i]
    return X[:, 0] if vec else X
