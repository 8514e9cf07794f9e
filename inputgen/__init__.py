"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the benchmark.

This module only produces inputs: locations, their spatial ordering, standard-normal
draws and observation vectors.  It holds none of the method's arithmetic (no covariance,
no factorisation, no kriging, no calibration), so the oracle and the CUDA path can both
consume it without sharing any computational code.

Recipes follow "Mixed-Precision GPU Acceleration for Confidence Regions of Spatial
Excursion Sets", §VI-B.1 (observation locations i.i.d. uniform on [0,1]^2 with a fixed
seed, prediction sites at the centres of an m x m grid, predictions ordered first).
"""
from __future__ import annotations

import dataclasses
import numpy as np

__all__ = [
    "uniform_locations", "grid_cell_centres", "jittered_grid", "morton_permutation",
    "morton_sorted", "standard_normals", "observation_values", "Workload", "WORKLOADS",
    "workload_locations",
]


def uniform_locations(n: int, seed: int) -> np.ndarray:
    """n points i.i.d. uniform on [0,1)^2, shape (n, 2), float64."""
    rng = np.random.default_rng(seed)
    return rng.random((n, 2))


def grid_cell_centres(m: int) -> np.ndarray:
    """Centres ((2j+1)h/2, (2i+1)h/2), h = 1/m, i, j = 0..m-1 (§VI-B.1); row i outer."""
    h = 1.0 / m
    c = (2.0 * np.arange(m) + 1.0) * h / 2.0
    yy, xx = np.meshgrid(c, c, indexing="ij")
    return np.stack([xx.ravel(), yy.ravel()], axis=1)


def jittered_grid(mx: int, my: int, jitter: float, seed: int) -> np.ndarray:
    """Cell centres of an mx x my grid on [0,1]^2, each moved uniformly within
    +-jitter cell widths (seeded)."""
    rng = np.random.default_rng(seed)
    hx, hy = 1.0 / mx, 1.0 / my
    cx = (2.0 * np.arange(mx) + 1.0) * hx / 2.0
    cy = (2.0 * np.arange(my) + 1.0) * hy / 2.0
    yy, xx = np.meshgrid(cy, cx, indexing="ij")
    pts = np.stack([xx.ravel(), yy.ravel()], axis=1)
    d = rng.uniform(-jitter, jitter, size=pts.shape)
    pts[:, 0] += d[:, 0] * hx
    pts[:, 1] += d[:, 1] * hy
    return np.clip(pts, 0.0, 1.0)


def _spread_bits16(v: np.ndarray) -> np.ndarray:
    v = v.astype(np.uint64) & np.uint64(0xFFFF)
    v = (v | (v << np.uint64(8))) & np.uint64(0x00FF00FF)
    v = (v | (v << np.uint64(4))) & np.uint64(0x0F0F0F0F)
    v = (v | (v << np.uint64(2))) & np.uint64(0x33333333)
    v = (v | (v << np.uint64(1))) & np.uint64(0x55555555)
    return v


def morton_permutation(xy: np.ndarray) -> np.ndarray:
    """Stable Z-order permutation of points in [0,1]^2 (coordinates quantised to 2^16
    levels per axis, x bits in the even positions)."""
    q = np.clip(np.floor(np.asarray(xy, dtype=np.float64) * 65536.0), 0, 65535).astype(np.uint64)
    key = _spread_bits16(q[:, 0]) | (_spread_bits16(q[:, 1]) << np.uint64(1))
    return np.argsort(key, kind="stable")


def morton_sorted(xy: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(xy[morton_permutation(xy)])


def standard_normals(n: int, M: int, seed: int) -> np.ndarray:
    """n x M matrix of i.i.d. N(0,1) draws, column-major (Fortran order), float64."""
    rng = np.random.default_rng(seed)
    return np.asfortranarray(rng.standard_normal((M, n)).T)


def observation_values(xy_obs: np.ndarray, beta_trend, noise_sd: float, seed: int) -> np.ndarray:
    """Synthetic observation vector: linear trend beta0 + beta1 x + beta2 y plus i.i.d.
    N(0, noise_sd^2) noise.  Used where a test needs any seeded y_o; the coverage study
    draws its truth from the model instead."""
    rng = np.random.default_rng(seed)
    b = np.asarray(beta_trend, dtype=np.float64)
    return b[0] + b[1] * xy_obs[:, 0] + b[2] * xy_obs[:, 1] + noise_sd * rng.standard_normal(len(xy_obs))


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n_pred: int            # prediction sites (ordered first)
    n_obs: int             # observation sites
    layout: str            # "uniform", "jittered", "krige"
    family: str            # "matern" or "powexp"
    sigma2: float
    beta: float            # range parameter
    nu: float
    nugget: float          # added to every diagonal entry
    tau2: float            # added to the observation diagonal only
    nb: int
    M: int
    fixedacc: float
    u: float
    level: float
    loc_seed: int = 1
    jitter_seed: int = 2
    z_seed: int = 12345

    @property
    def n(self) -> int:
        return self.n_pred + self.n_obs


# The workloads of the benchmark configurations.  Without observations every location is
# a "prediction" site (n_obs = 0).
WORKLOADS = {
    "a": Workload("a: n=1024 uniform, exponential Matern, nb=128, M=64", 1024, 0, "uniform",
                  "matern", 1.0, 0.1, 0.5, 1e-6, 0.0, 128, 64, 1e-6, 0.5, 0.90),
    "b": Workload("b: n=8192 jittered grid, Matern nu=1.5, nb=256, M=512", 8192, 0, "jittered",
                  "matern", 1.0, 0.3, 1.5, 1e-4, 0.0, 256, 512, 1e-8, 0.5, 0.90),
    "c": Workload("c: n=32768 uniform, exponential Matern range 0.03, nb=512, M=2048", 32768, 0,
                  "uniform", "matern", 1.0, 0.03, 0.5, 1e-4, 0.0, 512, 2048, 1e-4, 0.5, 0.90),
    "k": Workload("krige: 16384 noisy obs + 128x128 grid, Matern nu=1, nb=512, M=1024", 16384, 16384,
                  "krige", "matern", 1.0, 0.1, 1.0, 0.0, 0.01, 512, 1024, 1e-6, 1.6, 0.90),
    "e1": Workload("e: n=49152 uniform, exponential Matern range 0.1, nb=512, M=4096", 49152, 0,
                   "uniform", "matern", 1.0, 0.1, 0.5, 1e-4, 0.0, 512, 4096, 1e-6, 0.5, 0.90),
    "e2": Workload("e: n=65536 uniform, exponential Matern range 0.1, nb=512, M=4096", 65536, 0,
                   "uniform", "matern", 1.0, 0.1, 0.5, 1e-4, 0.0, 512, 4096, 1e-6, 0.5, 0.90),
}


def workload_locations(w: Workload) -> np.ndarray:
    """Locations of a workload, predictions first, each block in Morton order."""
    if w.layout == "uniform":
        return morton_sorted(uniform_locations(w.n_pred, w.loc_seed))
    if w.layout == "jittered":
        # 128 x 64 cell-centre grid, each point jittered within +-0.4 cell.
        assert w.n_pred == 8192
        return morton_sorted(jittered_grid(128, 64, 0.4, w.jitter_seed))
    if w.layout == "krige":
        m = int(round(np.sqrt(w.n_pred)))
        assert m * m == w.n_pred
        pred = morton_sorted(grid_cell_centres(m))
        obs = morton_sorted(uniform_locations(w.n_obs, w.loc_seed))
        return np.ascontiguousarray(np.concatenate([pred, obs], axis=0))
    raise ValueError(w.layout)
