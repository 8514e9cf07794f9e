"""Unconditional simulation and the standard-normal generator (oracle; test infrastructure).

"Mixed-Precision GPU Acceleration for Confidence Regions of Spatial Excursion Sets":
  * §IV-C Eq.3 / Alg.1: the simulations are M = L_s B with B = M_rand / s; in exact
    arithmetic L_s (M_rand / s) = (s L)(M_rand / s) = L M_rand (§V-E: the compensation
    preserves the simulation covariance), so the FP64 oracle is Y = L Z with L = chol(V).
  * Alg.1 / §V-F, FP16 destination task by task: simulate_fp16_per_product.
  * §V-B: M_rand has i.i.d. N(0,1) entries drawn on the GPU from a seeded stream with a
    Box-Muller draw ordering.  The page's stream (LAPACK's) is not reproduced; the
    library defines its own counter-based stream, restated here from its published
    pieces so that the two sides can be compared element by element:
      - SplitMix64 output function (Steele, Lea, Flood, "Fast splittable pseudorandom
        number generators", OOPSLA 2014), applied to seed + (c + 1) * golden_gamma;
      - uniform u = (top 53 bits + 1/2) * 2^-53, strictly inside (0, 1);
      - Box-Muller (1958): r = sqrt(-2 ln u1), z_even = r cos(2 pi u2), z_odd = r sin(2 pi u2).
    Element (i, j) of an n x M column-major matrix has logical index e = offset + j n + i,
    belongs to pair p = floor(e / 2), and draws u1, u2 from counters 2p and 2p + 1.
"""
from __future__ import annotations

import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def simulate(L: np.ndarray, Z: np.ndarray) -> np.ndarray:
    """Y = L Z in FP64 (Alg.1 with AMP = 0; equal in exact arithmetic to L_s (Z/s))."""
    return np.asarray(L, dtype=np.float64) @ np.asarray(Z, dtype=np.float64)


def simulate_fp16_per_product(Ls: np.ndarray, B: np.ndarray, nb: int) -> np.ndarray:
    """Alg.1's task sequence with the FP16 destination of §V-F, one product at a time.

    For each block row i of nb rows: Y_i = fp16(L_ii B_i) (the diagonal TRMM task), then for
    k = i-1 down to 0 (the descending order of Alg.1's GEMM tasks) Y_i = fp16(Y_i + L_ik B_k),
    each product in FP64 and the destination rounded to FP16 after it ("FP32 accumulation
    disabled" read as: no higher-precision buffer between tasks).  Ls is the factor as the
    multiply uses it (lower part; any FP16 casts already applied), B the right-hand side."""
    Ls = np.asarray(Ls, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    n = Ls.shape[0]
    nt = (n + nb - 1) // nb
    f16 = lambda a: a.astype(np.float16).astype(np.float64)
    Y = np.zeros((n, B.shape[1]))
    for i in range(nt):
        r = slice(i * nb, min(n, (i + 1) * nb))
        y = f16(np.tril(Ls[r, r]) @ B[r])
        for k in range(i - 1, -1, -1):
            q = slice(k * nb, (k + 1) * nb)
            y = f16(y + Ls[r, q] @ B[q])
        Y[r] = y
    return Y


def splitmix64(seed: int, counters: np.ndarray) -> np.ndarray:
    """SplitMix64 output for state seed + (c + 1) * gamma (mod 2^64), vectorised."""
    c = np.asarray(counters, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (c + np.uint64(1)) * GOLDEN_GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform53(seed: int, counters: np.ndarray) -> np.ndarray:
    z = splitmix64(seed, counters)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def rnorm(n: int, M: int, seed: int, offset: int = 0) -> np.ndarray:
    """n x M column-major standard normals of the library's counter-based stream."""
    e = np.uint64(offset) + np.arange(n * M, dtype=np.uint64)
    p = e >> np.uint64(1)
    u1 = uniform53(seed, np.uint64(2) * p)
    u2 = uniform53(seed, np.uint64(2) * p + np.uint64(1))
    r = np.sqrt(-2.0 * np.log(u1))
    theta = 2.0 * np.pi * u2
    z = np.where((e & np.uint64(1)) == 0, r * np.cos(theta), r * np.sin(theta))
    return np.asfortranarray(z.reshape(M, n).T)
