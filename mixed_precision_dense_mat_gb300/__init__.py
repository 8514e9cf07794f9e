"""Python binding of libcr.so (the GB300 conditional-simulation library).

Argument marshalling only: every computation runs in the library's CUDA kernels.  PyTorch
supplies device memory and streams.  Matrices are column-major like the C ABI: a column-major
n x m matrix is a torch tensor whose transpose is contiguous (stride (1, ld)); the helpers
``colmajor_empty`` / ``as_colmajor`` build such tensors.

The functions mirror include/cr.h:
  TileMat(n, nb)                         cr_tilemat_create / destroy
  cov_build(V, xy, ...)                  cr_cov_build
  tile_stats(V)                          cr_tile_stats
  tile_stats_records(V)                  cr_tile_stats_records
  precision_map(V, amp, fixedacc, auto)  cr_precision_map
  potrf_adaptive(V)                      cr_potrf_adaptive
  tilemat_to_dense(V, what)              cr_tilemat_to_dense
  rnorm(n, M, seed, offset)              cr_rnorm
  trmm_sim(V, Z, M, ...)                 cr_trmm_sim
  krige(V, Xo, Xp, yo)                   cr_krige
  krige_correct(W, yo, Y, n_p, n_o)      cr_krige_correct
  correct_calibrate(W, yo, Y, ...)       cr_correct_calibrate (correction fused with calibration)
  Weights(W)                             cr_weights_prepare / cr_weights_release
  krige_correct_prepared(Wp, yo, Y)      cr_krige_correct_prepared
  correct_calibrate_prepared(Wp, ...)    cr_correct_calibrate_prepared
  calibrate(S, zhat, v, u, level)        cr_calibrate (negative=True: cr_calibrate_negative)
  morton_order(xy)                       cr_morton_order (host only)
The library is never replaced by a fallback: if libcr.so is missing or fails to load, every
call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libcr.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "cr.h")

CR_PREC_FP64, CR_PREC_FP32, CR_PREC_FP16 = 0, 1, 2
CR_COV_MATERN, CR_COV_POWEXP = 0, 1
CR_TRMM_FP16_DEST, CR_TRMM_GENERATE, CR_TRMM_SPLIT_L, CR_TRMM_FP16_PER_GEMM = 1, 2, 4, 8
CR_OPT_WAIT_LIMIT_US, CR_OPT_DIAG_ARITH, CR_OPT_FP64_GEMM = 1, 2, 4
CR_DIAG_AUTO, CR_DIAG_FP64, CR_DIAG_DF = 0, 1, 2
CR_GEMM_DF, CR_GEMM_OZAKI = 0, 1
CR_PEAK_DFMA, CR_PEAK_FFMA, CR_PEAK_DF_MAC, CR_PEAK_DMMA = 1, 2, 3, 4
STATUS = {0: "CR_OK", 1: "CR_ERR_ARG", 2: "CR_ERR_CUDA", 3: "CR_ERR_NOMEM", 4: "CR_ERR_NOT_SPD",
          5: "CR_ERR_EMPTY_SAMPLE", 6: "CR_ERR_NONPOS_MSPE", 7: "CR_ERR_TIMEOUT", 8: "CR_ERR_STATE",
          9: "CR_ERR_NOT_IMPLEMENTED", 10: "CR_ERR_RANGE"}


class CrError(RuntimeError):
    def __init__(self, code: int, detail: str):
        self.code = code
        self.name = STATUS.get(code, f"CR_ERR_{code}")
        self.detail = detail
        super().__init__(f"{self.name}: {detail}")


class CovParams(ctypes.Structure):
    _fields_ = [("family", ctypes.c_int), ("sigma2", ctypes.c_double), ("range", ctypes.c_double),
                ("nu", ctypes.c_double), ("nugget", ctypes.c_double), ("n_pred", ctypes.c_int),
                ("tau2", ctypes.c_double)]


class PmapInfo(ctypes.Structure):
    _fields_ = [("fixedacc", ctypes.c_double), ("iters", ctypes.c_int), ("n_fp64", ctypes.c_int),
                ("n_fp32", ctypes.c_int), ("n_fp16", ctypes.c_int), ("R_hp", ctypes.c_double),
                ("rho1", ctypes.c_double), ("rho2", ctypes.c_double), ("check1", ctypes.c_int),
                ("check2", ctypes.c_int), ("ell", ctypes.c_double), ("u_s", ctypes.c_double),
                ("s", ctypes.c_double), ("range_ok", ctypes.c_int)]


class CalibInfo(ctypes.Structure):
    _fields_ = [("q_in", ctypes.c_double), ("q_out", ctypes.c_double), ("n_psi", ctypes.c_int),
                ("n_phi", ctypes.c_int)]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_D = ctypes.c_double
_U64 = ctypes.c_uint64

_SIGNATURES = {
    "cr_status_str": (ctypes.c_char_p, [_I]),
    "cr_last_error_detail": (ctypes.c_char_p, []),
    "cr_version": (_I, [ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "cr_kernel_launches": (_I, [ctypes.POINTER(_U64)]),
    "cr_workspace_trim": (_I, []),
    "cr_set_option": (_I, [_I, ctypes.c_longlong]),
    "cr_peak_probe": (_I, [_I, _I, ctypes.POINTER(_D), _P]),
    "cr_get_option": (_I, [_I, ctypes.POINTER(ctypes.c_longlong)]),
    "cr_timing_enable": (_I, [_I]),
    "cr_timing_read": (_I, [ctypes.c_char_p, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_U64)]),
    "cr_timing_reset": (_I, []),
    "cr_tilemat_create": (_I, [_I, _I, ctypes.POINTER(_P)]),
    "cr_tilemat_destroy": (_I, [_P]),
    "cr_tilemat_info": (_I, [_P, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "cr_cov_build": (_I, [_P, _P, ctypes.POINTER(CovParams), _P]),
    "cr_tile_stats": (_I, [_P, _P, _P, _P]),
    "cr_tile_stats_records": (_I, [_P, _P, _P, _P, _P]),
    "cr_precision_map": (_I, [_P, _I, _D, _I, _P, ctypes.POINTER(PmapInfo)]),
    "cr_potrf_adaptive": (_I, [_P, _P, ctypes.POINTER(_I)]),
    "cr_tilemat_to_dense": (_I, [_P, _I, _P, _I, _P]),
    "cr_rnorm": (_I, [_P, _I, _I, _I, _U64, _U64, _P]),
    "cr_trmm_sim": (_I, [_P, _P, _I, _I, _U64, _U64, _P, _I, _I, ctypes.POINTER(_D), _P]),
    "cr_krige": (_I, [_P, _P, _P, _P, _P, _I, _P, _P, _P, ctypes.POINTER(_I)]),
    "cr_krige_correct": (_I, [_P, _I, _P, _P, _I, _I, _I, _I, _P, _I, _P]),
    "cr_morton_order": (_I, [_P, _I, _P]),
    "cr_calibrate": (_I, [_P, _I, _I, _I, _P, _P, _D, _D, _P, _P, _P, _P, _P, ctypes.POINTER(CalibInfo), _P]),
    "cr_correct_calibrate": (_I, [_P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _D, _D, _I, _P, _P, _P, _P, _P,
                                  ctypes.POINTER(CalibInfo), _P]),
    "cr_calibrate_negative": (_I, [_P, _I, _I, _I, _P, _P, _D, _D, _P, _P, _P, _P, _P, ctypes.POINTER(CalibInfo),
                                   _P]),
    "cr_calibrate_noalloc": (_I, [_P, _I, _I, _I, _P, _P, _D, _D, _P, _P, _P, _P, _P, ctypes.POINTER(CalibInfo),
                                  _P]),
    "cr_weights_prepare": (_I, [_P, _I, _I, _I, _P, ctypes.POINTER(_P)]),
    "cr_weights_release": (_I, [_P]),
    "cr_krige_correct_prepared": (_I, [_P, _P, _P, _I, _I, _P, _I, _P]),
    "cr_correct_calibrate_prepared": (_I, [_P, _P, _P, _I, _I, _P, _P, _D, _D, _I, _P, _P, _P, _P, _P,
                                           ctypes.POINTER(CalibInfo), _P]),
}


def header_functions() -> list[str]:
    """Names of the entry points declared in include/cr.h."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(cr_[a-z0-9_]+)\s*\(", src)))


def load(path: str | None = None):
    """Loads libcr.so (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(code: int):
    if code != 0:
        raise CrError(code, (_lib.cr_last_error_detail() or b"").decode())


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> int | None:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def colmajor_empty(n: int, m: int, dtype, device="cuda"):
    """Uninitialised n x m column-major tensor (leading dimension n)."""
    import torch
    return torch.empty((m, n), dtype=dtype, device=device).T


def as_colmajor(t):
    """t as a column-major tensor (copies if needed); returns (tensor, ld)."""
    if t.dim() == 1:
        return t.contiguous(), t.shape[0]
    if t.stride(0) != 1:
        t = t.T.contiguous().T
    return t, max(1, t.stride(1))


def kernel_launches() -> int:
    """cr_kernel_launches: kernels launched by the library in this process so far."""
    load()
    c = _U64(0)
    _check(_lib.cr_kernel_launches(ctypes.byref(c)))
    return c.value


def workspace_trim() -> None:
    """cr_workspace_trim: return the library's pooled scratch memory to the driver."""
    load()
    _check(_lib.cr_workspace_trim())


def set_option(option: int, value: int) -> None:
    """cr_set_option: CR_OPT_WAIT_LIMIT_US (microseconds), CR_OPT_DIAG_ARITH (CR_DIAG_*) or
    CR_OPT_FP64_GEMM (CR_GEMM_*)."""
    load()
    _check(_lib.cr_set_option(option, int(value)))


def peak_probe(kind: int, iters: int = 4096, stream=None) -> float:
    """cr_peak_probe: measured TFLOP/s of one arithmetic unit (CR_PEAK_*)."""
    load()
    v = _D(0.0)
    _check(_lib.cr_peak_probe(kind, iters, ctypes.byref(v), _stream(stream)))
    return v.value


def get_option(option: int) -> int:
    load()
    v = ctypes.c_longlong(0)
    _check(_lib.cr_get_option(option, ctypes.byref(v)))
    return v.value


def timing_enable(on: bool) -> None:
    """cr_timing_enable: bracket launches of the timed kernels with CUDA events."""
    load()
    _check(_lib.cr_timing_enable(1 if on else 0))


def timing_read(kernel: str) -> tuple[float, int]:
    """cr_timing_read: (total milliseconds, launches) of a timed kernel; synchronises."""
    load()
    ms = ctypes.c_double(0.0)
    n = _U64(0)
    _check(_lib.cr_timing_read(kernel.encode(), ctypes.byref(ms), ctypes.byref(n)))
    return ms.value, n.value


def timing_reset() -> None:
    """cr_timing_reset: clear the accumulated kernel times."""
    load()
    _check(_lib.cr_timing_reset())


class TileMat:
    """Opaque lower-tile storage of a symmetric n x n matrix (cr_tilemat)."""

    def __init__(self, n: int, nb: int):
        load()
        h = _P()
        _check(_lib.cr_tilemat_create(n, nb, ctypes.byref(h)))
        self._h = h
        self.n, self.nb = n, nb
        self.nt = (n + nb - 1) // nb

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None):
            _lib.cr_tilemat_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def morton_order(xy) -> np.ndarray:
    """cr_morton_order: the stable Z-order permutation of the (n, 2) FP64 host array xy."""
    load()
    xy = np.ascontiguousarray(xy, dtype=np.float64)
    assert xy.ndim == 2 and xy.shape[1] == 2
    n = xy.shape[0]
    perm = np.empty(n, dtype=np.int32)
    _check(_lib.cr_morton_order(xy.ctypes.data if n else None, n, perm.ctypes.data if n else None))
    return perm


def cov_build(V: TileMat, xy, family: str = "matern", sigma2: float = 1.0, range: float = 0.1, nu: float = 0.5,
              nugget: float = 0.0, n_pred: int | None = None, tau2: float = 0.0, stream=None):
    """cr_cov_build: xy is an (n, 2) float64 CUDA tensor (row-major pairs)."""
    assert xy.is_cuda and xy.dtype.is_floating_point and xy.shape == (V.n, 2) and xy.is_contiguous()
    p = CovParams(CR_COV_MATERN if family == "matern" else CR_COV_POWEXP, sigma2, range, nu, nugget,
                  V.n if n_pred is None else n_pred, tau2)
    _check(_lib.cr_cov_build(V.handle, _ptr(xy), ctypes.byref(p), _stream(stream)))


def tile_stats(V: TileMat):
    nt = V.nt
    f, a, b = (np.zeros((nt, nt)) for _ in range(3))
    _check(_lib.cr_tile_stats(V.handle, f.ctypes.data, a.ctypes.data, b.ctypes.data))
    return f, a, b


def tile_stats_records(V: TileMat):
    """cr_tile_stats_records: (frob, vmin, vmax, err) as NT x NT arrays, nothing recomputed."""
    nt = V.nt
    f, a, b, e = (np.zeros((nt, nt)) for _ in range(4))
    _check(_lib.cr_tile_stats_records(V.handle, f.ctypes.data, a.ctypes.data, b.ctypes.data, e.ctypes.data))
    return f, a, b, e


def precision_map(V: TileMat, amp: bool = True, fixedacc: float = 1e-4, auto: bool = False):
    m = np.zeros((V.nt, V.nt), dtype=np.int8)
    info = PmapInfo()
    _check(_lib.cr_precision_map(V.handle, 1 if amp else 0, fixedacc, 1 if auto else 0, m.ctypes.data,
                                 ctypes.byref(info)))
    d = {k: getattr(info, k) for k, _ in PmapInfo._fields_}
    return m, d


def potrf_adaptive(V: TileMat, stream=None) -> int:
    info = _I(0)
    code = _lib.cr_potrf_adaptive(V.handle, _stream(stream), ctypes.byref(info))
    if code == 4:   # CR_ERR_NOT_SPD: report through info like LAPACK
        return info.value
    _check(code)
    return info.value


def tilemat_to_dense(V: TileMat, what: int = 1, stream=None):
    import torch
    out = colmajor_empty(V.n, V.n, torch.float64)
    _check(_lib.cr_tilemat_to_dense(V.handle, what, _ptr(out), V.n, _stream(stream)))
    return out


def rnorm(n: int, M: int, seed: int, offset: int = 0, out=None, stream=None):
    import torch
    load()
    if out is None:
        out = colmajor_empty(n, M, torch.float64)
    out, ld = as_colmajor(out)
    _check(_lib.cr_rnorm(_ptr(out), ld, n, M, seed, offset, _stream(stream)))
    return out


def trmm_sim(V: TileMat, Z, M: int, seed: int = 0, offset: int = 0, out=None, flags: int = 0,
             want_bnorm: bool = False, stream=None):
    """cr_trmm_sim: Z is n x M column-major FP64 (or None with CR_TRMM_GENERATE)."""
    import torch
    if out is None:
        out = colmajor_empty(V.n, M, torch.float64)
    out, ldy = as_colmajor(out)
    zp, ldz = (None, V.n)
    if Z is not None:
        Z, ldz = as_colmajor(Z)
        zp = _ptr(Z)
    bn = _D(0.0)
    _check(_lib.cr_trmm_sim(V.handle, zp, ldz, M, seed, offset, _ptr(out), ldy, flags,
                            ctypes.byref(bn) if want_bnorm else None, _stream(stream)))
    return (out, bn.value) if want_bnorm else out


def krige(V: TileMat, Xo, Xp, yo, stream=None):
    import torch
    n_o, n_p = Xo.shape[0], Xp.shape[0]
    Xo, _ = as_colmajor(Xo)
    Xp, _ = as_colmajor(Xp)
    W = colmajor_empty(n_o, n_p, torch.float64)
    zhat = torch.empty(n_p, dtype=torch.float64, device="cuda")
    v = torch.empty(n_p, dtype=torch.float64, device="cuda")
    info = _I(0)
    _check(_lib.cr_krige(V.handle, _ptr(Xo), _ptr(Xp), _ptr(yo.contiguous()), _ptr(W), n_o, _ptr(zhat), _ptr(v),
                         _stream(stream), ctypes.byref(info)))
    return W, zhat, v


def krige_correct(W, yo, Y, n_p: int, n_o: int, out=None, stream=None):
    import torch
    W, ldw = as_colmajor(W)
    Y, ldy = as_colmajor(Y)
    M = Y.shape[1]
    if out is None:
        out = colmajor_empty(n_p, M, torch.float64)
    out, lds = as_colmajor(out)
    _check(_lib.cr_krige_correct(_ptr(W), ldw, _ptr(yo.contiguous()), _ptr(Y), ldy, n_p, n_o, M, _ptr(out), lds,
                                 _stream(stream)))
    return out


def _calib_outputs(n_p: int, M: int, counts: bool, extrema: bool):
    import torch
    cin = torch.empty(n_p, dtype=torch.uint8, device="cuda")
    cout = torch.empty(n_p, dtype=torch.uint8, device="cuda")
    cnt = torch.empty(n_p, dtype=torch.int32, device="cuda") if counts else None
    psi = torch.empty(M, dtype=torch.float64, device="cuda") if extrema else None
    phi = torch.empty(M, dtype=torch.float64, device="cuda") if extrema else None
    return cin, cout, cnt, psi, phi, CalibInfo()


def _calib_dict(cin, cout, cnt, psi, phi, info, counts: bool, extrema: bool):
    out = {"q_in": info.q_in, "q_out": info.q_out, "n_psi": info.n_psi, "n_phi": info.n_phi, "c_in": cin,
           "c_out": cout}
    if counts:
        out["count"] = cnt
    if extrema:
        out["psi"], out["phi"] = psi, phi
    return out


def correct_calibrate(W, yo, Y, n_p: int, n_o: int, zhat, v, u: float, level: float, counts: bool = True,
                      extrema: bool = False, negative: bool = False, stream=None):
    """cr_correct_calibrate: the correction S = M_p + W^T (y_o 1^T - M_o) fused with the
    calibration (S is never formed); returns the dict of calibrate()."""
    W, ldw = as_colmajor(W)
    Y, ldy = as_colmajor(Y)
    M = Y.shape[1]
    cin, cout, cnt, psi, phi, info = _calib_outputs(n_p, M, counts, extrema)
    _check(_lib.cr_correct_calibrate(_ptr(W), ldw, _ptr(yo.contiguous()), _ptr(Y), ldy, n_p, n_o, M,
                                     _ptr(zhat.contiguous()), _ptr(v.contiguous()), u, level, 1 if negative else 0,
                                     _ptr(cin), _ptr(cout), _ptr(cnt), _ptr(psi), _ptr(phi), ctypes.byref(info),
                                     _stream(stream)))
    return _calib_dict(cin, cout, cnt, psi, phi, info, counts, extrema)


class Weights:
    """cr_weights: kriging weights W (n_o x n_p) prepared for repeated Ozaki corrections."""

    def __init__(self, W, stream=None):
        load()
        W, ldw = as_colmajor(W)
        self.n_o, self.n_p = W.shape
        h = _P()
        _check(_lib.cr_weights_prepare(_ptr(W), ldw, self.n_o, self.n_p, _stream(stream), ctypes.byref(h)))
        self.handle = h

    def close(self):
        if self.handle:
            _check(_lib.cr_weights_release(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def krige_correct_prepared(Wp: Weights, yo, Y, out=None, stream=None):
    """cr_krige_correct_prepared: the Ozaki correction with prepared weights; returns S."""
    import torch
    Y, ldy = as_colmajor(Y)
    M = Y.shape[1]
    if out is None:
        out = colmajor_empty(Wp.n_p, M, torch.float64)
    out, lds = as_colmajor(out)
    _check(_lib.cr_krige_correct_prepared(Wp.handle, _ptr(yo.contiguous()), _ptr(Y), ldy, M, _ptr(out), lds,
                                          _stream(stream)))
    return out


def correct_calibrate_prepared(Wp: Weights, yo, Y, zhat, v, u: float, level: float, counts: bool = True,
                               extrema: bool = False, negative: bool = False, stream=None):
    """cr_correct_calibrate_prepared: the Ozaki correction with prepared weights, then the
    calibration; returns the dict of calibrate()."""
    Y, ldy = as_colmajor(Y)
    M = Y.shape[1]
    cin, cout, cnt, psi, phi, info = _calib_outputs(Wp.n_p, M, counts, extrema)
    _check(_lib.cr_correct_calibrate_prepared(Wp.handle, _ptr(yo.contiguous()), _ptr(Y), ldy, M,
                                              _ptr(zhat.contiguous()), _ptr(v.contiguous()), u, level,
                                              1 if negative else 0, _ptr(cin), _ptr(cout), _ptr(cnt), _ptr(psi),
                                              _ptr(phi), ctypes.byref(info), _stream(stream)))
    return _calib_dict(cin, cout, cnt, psi, phi, info, counts, extrema)


def calibrate(S, zhat, v, u: float, level: float, counts: bool = True, extrema: bool = False, negative: bool = False,
              stream=None):
    """cr_calibrate (cr_calibrate_negative with negative=True: the negative excursion set);
    returns a dict with q_in, q_out, n_psi, n_phi, c_in, c_out and optionally count, psi, phi
    (CUDA tensors)."""
    import torch
    S, lds = as_colmajor(S)
    n_p, M = S.shape
    cin = torch.empty(n_p, dtype=torch.uint8, device="cuda")
    cout = torch.empty(n_p, dtype=torch.uint8, device="cuda")
    cnt = torch.empty(n_p, dtype=torch.int32, device="cuda") if counts else None
    psi = torch.empty(M, dtype=torch.float64, device="cuda") if extrema else None
    phi = torch.empty(M, dtype=torch.float64, device="cuda") if extrema else None
    info = CalibInfo()
    fn = _lib.cr_calibrate_negative if negative else _lib.cr_calibrate
    _check(fn(_ptr(S), lds, n_p, M, _ptr(zhat.contiguous()), _ptr(v.contiguous()), u, level,
                             _ptr(cin), _ptr(cout), _ptr(cnt), _ptr(psi), _ptr(phi), ctypes.byref(info),
                             _stream(stream)))
    out = {"q_in": info.q_in, "q_out": info.q_out, "n_psi": info.n_psi, "n_phi": info.n_phi, "c_in": cin,
           "c_out": cout}
    if counts:
        out["count"] = cnt
    if extrema:
        out["psi"], out["phi"] = psi, phi
    return out
