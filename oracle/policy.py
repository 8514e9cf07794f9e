"""Tile statistics and the adaptive precision policy (oracle; test infrastructure only).

"Mixed-Precision GPU Acceleration for Confidence Regions of Spatial Excursion Sets":
  * §IV-B and §VI-D: each tile gets FP64, FP32 or FP16; diagonal tiles stay FP64; the
    rule "compares the norm of each tile with the global matrix norm" (the exact rule is
    in the page's ref. [13]).  Reading taken: an off-diagonal tile (i, j) takes the
    lowest p in {FP16, FP32} with ||V_ij||_F * NT <= (fixedacc / eps_p) * ||V||_F,
    else FP64; eps_FP16 = 2^-10 (as in Eq.11), eps_FP32 = 2^-23 by analogy; ||V||_F is
    over the full symmetric matrix (off-diagonal tiles counted twice).
  * §V-D: automatic mode starts at fixedacc = 1e-4 and multiplies it by 0.9 while either
    check fails, stopping when both pass or no FP16 tile is left.
  * §V-D.1 Eq.10: R_HP = v_max^HP / v_min^HP < 65504 / 2^-24 (strict; extrema over the
    FP16 tiles' entries, no absolute values, zeros kept).
  * §V-D.2 Eq.11: max(rho1, rho2) < 1e-4 / eps_FP16 with rho1 = v_max^HP / v_max and
    rho2 = max_{FP16 tiles} ||V_ij||_F / max_{all tiles} ||V_ij||_F.
  * §V-E Eq.12: l_f = sqrt(x_min,norm^(f) / v_min^(f)), u_f = sqrt(x_max^(f) / v_max^(f))
    for each present f in {FP32, FP16}; u_s = min(65504, min_f u_f); s = floor(u_s) - 1
    when that exceeds 1, else 1.  Reading: with no reduced-precision tile present s = 1.
Statistics are taken over the lower tiles (i >= j) and over valid entries only.
"""
from __future__ import annotations

import math
import numpy as np

from .covariance import covariance_matrix

PREC_FP64, PREC_FP32, PREC_FP16 = 0, 1, 2
EPS = {PREC_FP16: 2.0 ** -10, PREC_FP32: 2.0 ** -23}
FP16_MAX = 65504.0
FP16_MIN_NORMAL = 2.0 ** -14
FP16_MIN_SUBNORMAL = 2.0 ** -24
FP32_MAX = float(np.finfo(np.float32).max)
FP32_MIN_NORMAL = 2.0 ** -126


def _ntiles(n: int, nb: int) -> int:
    return (n + nb - 1) // nb


def tile_stats(V: np.ndarray, nb: int):
    """Per lower tile (i >= j): Frobenius norm, min entry, max entry (valid entries)."""
    n = V.shape[0]
    NT = _ntiles(n, nb)
    frob = np.zeros((NT, NT))
    vmin = np.zeros((NT, NT))
    vmax = np.zeros((NT, NT))
    for i in range(NT):
        for j in range(i + 1):
            T = V[i * nb:min(n, (i + 1) * nb), j * nb:min(n, (j + 1) * nb)]
            frob[i, j] = math.sqrt(float(np.sum(T * T)))
            vmin[i, j] = float(T.min())
            vmax[i, j] = float(T.max())
    return frob, vmin, vmax


def tile_stats_from_locations(xy: np.ndarray, nb: int, family: str, sigma2: float, beta: float,
                              nu: float, nugget: float = 0.0, n_pred: int | None = None,
                              tau2: float = 0.0):
    """Same as tile_stats, building one tile of V at a time (for large n)."""
    n = xy.shape[0]
    NT = _ntiles(n, nb)
    frob = np.zeros((NT, NT))
    vmin = np.zeros((NT, NT))
    vmax = np.zeros((NT, NT))
    for i in range(NT):
        for j in range(i + 1):
            T = covariance_matrix(xy, family, sigma2, beta, nu, nugget, n_pred, tau2,
                                  rows=slice(i * nb, min(n, (i + 1) * nb)),
                                  cols=slice(j * nb, min(n, (j + 1) * nb)))
            frob[i, j] = math.sqrt(float(np.sum(T * T)))
            vmin[i, j] = float(T.min())
            vmax[i, j] = float(T.max())
    return frob, vmin, vmax


def global_norm(frob: np.ndarray) -> float:
    """||V||_F of the symmetric matrix from its lower-tile norms."""
    NT = frob.shape[0]
    s = 0.0
    for i in range(NT):
        s += frob[i, i] ** 2
        for j in range(i):
            s += 2.0 * frob[i, j] ** 2
    return math.sqrt(s)


def precision_map(frob: np.ndarray, fixedacc: float) -> np.ndarray:
    """Tile precision map (reading of §IV-B / §VI-D given in the module docstring)."""
    NT = frob.shape[0]
    g = global_norm(frob)
    pmap = np.full((NT, NT), -1, dtype=np.int8)
    for i in range(NT):
        pmap[i, i] = PREC_FP64
        for j in range(i):
            lhs = frob[i, j] * NT
            if lhs <= (fixedacc / EPS[PREC_FP16]) * g:
                pmap[i, j] = PREC_FP16
            elif lhs <= (fixedacc / EPS[PREC_FP32]) * g:
                pmap[i, j] = PREC_FP32
            else:
                pmap[i, j] = PREC_FP64
    return pmap


def _lower(NT):
    return [(i, j) for i in range(NT) for j in range(i + 1)]


def fp16_checks(pmap, frob, vmin, vmax) -> dict:
    """Eq.10 (FP16 representability range) and Eq.11 (relative magnitude)."""
    NT = pmap.shape[0]
    hp = [(i, j) for (i, j) in _lower(NT) if pmap[i, j] == PREC_FP16]
    out = {"n_fp16": len(hp)}
    if not hp:
        out.update(R_hp=float("nan"), rho1=float("nan"), rho2=float("nan"),
                   check1=True, check2=True)
        return out
    vmax_hp = max(vmax[i, j] for (i, j) in hp)
    vmin_hp = min(vmin[i, j] for (i, j) in hp)
    vmax_all = max(vmax[i, j] for (i, j) in _lower(NT))
    fmax_hp = max(frob[i, j] for (i, j) in hp)
    fmax_all = max(frob[i, j] for (i, j) in _lower(NT))
    with np.errstate(divide="ignore", invalid="ignore"):
        R = np.float64(vmax_hp) / np.float64(vmin_hp)
    rho1 = vmax_hp / vmax_all
    rho2 = fmax_hp / fmax_all
    out.update(R_hp=float(R), rho1=rho1, rho2=rho2,
               check1=bool(R < FP16_MAX / FP16_MIN_SUBNORMAL),
               check2=bool(max(rho1, rho2) < 1e-4 / EPS[PREC_FP16]))
    return out


def covariance_scale(pmap, vmin, vmax) -> dict:
    """Applied scale s of §V-E Eq.12.

    Alg.1 (step 15) casts every off-diagonal factor tile of L_s = s L to FP16, and the
    largest factor entry is sqrt(max V_ii) (|L_ij| <= sqrt(V_ii)), so the upper bound u_s
    also keeps s sqrt(max V_ii) inside FP16; it binds only when no FP16-class tile bounds s
    more tightly (for instance when none is left)."""
    NT = pmap.shape[0]
    consts = {PREC_FP32: (FP32_MIN_NORMAL, FP32_MAX), PREC_FP16: (FP16_MIN_NORMAL, FP16_MAX)}
    vmax_all = max(vmax[i, j] for (i, j) in _lower(NT))
    ell, us = -math.inf, FP16_MAX
    if vmax_all > 0:
        us = min(us, FP16_MAX / math.sqrt(vmax_all))
    present = False
    for f, (xmin, xmax) in consts.items():
        tiles = [(i, j) for (i, j) in _lower(NT) if i != j and pmap[i, j] == f]
        if not tiles:
            continue
        present = True
        vmn = min(vmin[i, j] for (i, j) in tiles)
        vmx = max(vmax[i, j] for (i, j) in tiles)
        ell_f = math.sqrt(xmin / vmn) if vmn > 0 else math.inf
        u_f = math.sqrt(xmax / vmx) if vmx > 0 else math.inf
        ell = max(ell, ell_f)
        us = min(us, u_f)
    if not present:
        return {"s": 1.0, "ell": float("nan"), "u_s": float("nan"), "range_ok": True}
    s_cand = math.floor(us) - 1
    s = float(s_cand) if s_cand > 1 else 1.0
    return {"s": s, "ell": ell, "u_s": us, "range_ok": bool(ell <= us)}


def select_precision(frob, vmin, vmax, fixedacc: float, auto: bool, amp: bool = True,
                     max_iter: int = 100000) -> dict:
    """Precision map, tolerance, checks and scale (Alg.2 steps 7 and 9-10, §V-D, §V-E)."""
    NT = frob.shape[0]
    if not amp:
        pmap = np.full((NT, NT), -1, dtype=np.int8)
        for (i, j) in _lower(NT):
            pmap[i, j] = PREC_FP64
        chk = fp16_checks(pmap, frob, vmin, vmax)
        return {"map": pmap, "fixedacc": fixedacc, "iters": 0, "s": 1.0, **chk,
                "ell": float("nan"), "u_s": float("nan"), "range_ok": True}
    it = 0
    if auto:
        fixedacc = 1e-4
    while True:
        pmap = precision_map(frob, fixedacc)
        chk = fp16_checks(pmap, frob, vmin, vmax)
        it += 1
        if not auto or chk["n_fp16"] == 0 or (chk["check1"] and chk["check2"]) or it >= max_iter:
            break
        fixedacc = fixedacc * 0.9
    sc = covariance_scale(pmap, vmin, vmax)
    return {"map": pmap, "fixedacc": fixedacc, "iters": it, **chk, **sc}
