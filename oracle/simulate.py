"""Unconditional simulation and the standard-normal generator (oracle; test infrastructure).

"Mixed-Precision GPU Acceleration for Confidence Regions of Spatial Excursion Sets":
  * §IV-C Eq.3 / Alg.1: the simulations are M = L_s B with B = M_rand / s; in exact
    arithmetic L_s (M_rand / s) = (s L)(M_rand / s) = L M_rand (§V-E: the compensation
    preserves the simulation covariance), so the FP64 oracle is Y = L Z with L = chol(V).
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
