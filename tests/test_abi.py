"""The C-ABI library loads and exports every entry point declared in include/cr.h (CPU only:
no call here touches a GPU; argument checks return before any device work)."""
import ctypes
import os

import pytest

import mixed_precision_dense_mat_gb300 as cr
from mixed_precision_dense_mat_gb300 import build_lib


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(build_lib.LIB):
        build_lib.build()
    return ctypes.CDLL(build_lib.LIB)


def test_every_declared_symbol_is_exported(lib):
    names = cr.header_functions()
    assert len(names) >= 16
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert set(cr._SIGNATURES) == set(names)


def test_status_strings_and_version(lib):
    cr.load()
    assert cr._lib.cr_status_str(0) == b"CR_OK"
    assert cr._lib.cr_status_str(4) == b"CR_ERR_NOT_SPD"
    for code, name in cr.STATUS.items():
        assert cr._lib.cr_status_str(code).decode() == name
    a, b = ctypes.c_int(), ctypes.c_int()
    assert cr._lib.cr_version(ctypes.byref(a), ctypes.byref(b)) == 0


def test_argument_errors_without_gpu(lib):
    cr.load()
    h = ctypes.c_void_p()
    assert cr._lib.cr_tilemat_create(100, 100, ctypes.byref(h)) == 1      # nb must be a multiple of 128
    assert b"nb" in cr._lib.cr_last_error_detail()
    assert cr._lib.cr_tilemat_create(-5, 128, ctypes.byref(h)) == 1
    assert cr._lib.cr_tilemat_create(10, 128, None) == 1
    assert cr._lib.cr_cov_build(None, None, None, None) == 1
    assert cr._lib.cr_potrf_adaptive(None, None, None) == 1
    assert cr._lib.cr_rnorm(None, 1, 1, 1, 0, 0, None) == 1
    assert cr._lib.cr_calibrate(None, 1, 1, 1, None, None, 0.0, 0.9, None, None, None, None, None, None, None) == 1
    assert cr._lib.cr_krige_correct(None, 1, None, None, 1, 1, 1, 1, None, 1, None) == 1
    assert cr._lib.cr_tilemat_destroy(None) == 0
    w = ctypes.c_void_p(1)
    assert cr._lib.cr_weights_prepare(None, 10, 10, 10, None, ctypes.byref(w)) == 1 and w.value is None
    assert cr._lib.cr_weights_prepare(None, 10, 10, 10, None, None) == 1
    assert cr._lib.cr_weights_release(None) == 0
    assert cr._lib.cr_krige_correct_prepared(None, None, None, 1, 1, None, 1, None) == 1
    assert cr._lib.cr_correct_calibrate_prepared(None, None, None, 1, 1, None, None, 0.0, 0.9, 0, None, None, None,
                                                 None, None, None, None) == 1


def test_header_declares_documented_path():
    names = cr.header_functions()
    for n in ("cr_cov_build", "cr_precision_map", "cr_potrf_adaptive", "cr_trmm_sim", "cr_krige", "cr_calibrate"):
        assert n in names


def test_binding_constants_match_the_header():
    """The enum values the binding passes (precision classes, covariance families, simulation
    flags, status codes) are the ones include/cr.h declares."""
    import re
    text = open(cr.HEADER).read()
    declared = {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(CR_[A-Z0-9_]+)\s*=\s*(\d+)", text)}
    for name in ("CR_PREC_FP64", "CR_PREC_FP32", "CR_PREC_FP16", "CR_COV_MATERN", "CR_COV_POWEXP",
                 "CR_TRMM_FP16_DEST", "CR_TRMM_GENERATE", "CR_TRMM_SPLIT_L", "CR_TRMM_FP16_PER_GEMM",
                 "CR_OPT_WAIT_LIMIT_US", "CR_OPT_DIAG_ARITH", "CR_OPT_FP64_GEMM", "CR_DIAG_AUTO", "CR_DIAG_FP64",
                 "CR_DIAG_DF", "CR_GEMM_DF", "CR_GEMM_OZAKI",
                 "CR_PEAK_DFMA", "CR_PEAK_FFMA", "CR_PEAK_DF_MAC", "CR_PEAK_DMMA"):
        assert name in declared, name
        assert getattr(cr, name) == declared[name], name
    for code, name in cr.STATUS.items():
        assert declared.get(name, code if name == "CR_OK" else None) == code, name


def test_morton_order_matches_the_input_generator(lib):
    """cr_morton_order (host-only entry point) gives the same permutation, element for element,
    as the input generator's Z-order on uniform, gridded, jittered and ragged site sets,
    including points on the unit square's edges and duplicated sites (stable order)."""
    import numpy as np
    import inputgen
    cr.load()
    cases = [
        inputgen.uniform_locations(4096, 1),
        inputgen.uniform_locations(1000, 7),              # ragged size
        inputgen.grid_cell_centres(64),
        inputgen.jittered_grid(128, 64, 0.4, 2),
        np.array([[0.0, 0.0], [1.0, 1.0], [1.0, 0.0], [0.0, 1.0], [0.5, 0.5], [0.5, 0.5],
                  [-0.25, 2.0], [0.999999999, 0.0000001], [0.5, 0.5]]),
        np.repeat(inputgen.uniform_locations(37, 3), 3, axis=0),   # triples of equal keys
    ]
    for xy in cases:
        perm = cr.morton_order(xy)
        ref = inputgen.morton_permutation(xy)
        np.testing.assert_array_equal(perm, ref.astype(np.int32))
    assert cr.morton_order(np.zeros((0, 2))).shape == (0,)
    bad = np.array([[0.1, 0.2], [np.nan, 0.3]])
    with pytest.raises(cr.CrError) as e:
        cr.morton_order(bad)
    assert e.value.code == 1


def test_options_host_side(lib):
    """cr_set_option / cr_get_option: round trip, range checks and unknown options (host only);
    cr_peak_probe rejects bad arguments before any device work."""
    cr.load()
    v = ctypes.c_longlong()
    assert cr._lib.cr_get_option(cr.CR_OPT_WAIT_LIMIT_US, ctypes.byref(v)) == 0 and v.value == 2000000
    assert cr._lib.cr_get_option(cr.CR_OPT_DIAG_ARITH, ctypes.byref(v)) == 0 and v.value == cr.CR_DIAG_AUTO
    assert cr._lib.cr_set_option(cr.CR_OPT_WAIT_LIMIT_US, 5000) == 0
    assert cr._lib.cr_get_option(cr.CR_OPT_WAIT_LIMIT_US, ctypes.byref(v)) == 0 and v.value == 5000
    assert cr._lib.cr_set_option(cr.CR_OPT_WAIT_LIMIT_US, -1) == 1
    assert cr._lib.cr_set_option(cr.CR_OPT_WAIT_LIMIT_US, 2000000) == 0
    assert cr._lib.cr_set_option(cr.CR_OPT_DIAG_ARITH, 7) == 1
    assert cr._lib.cr_get_option(cr.CR_OPT_FP64_GEMM, ctypes.byref(v)) == 0 and v.value == cr.CR_GEMM_DF
    assert cr._lib.cr_set_option(cr.CR_OPT_FP64_GEMM, 2) == 1
    assert cr._lib.cr_set_option(cr.CR_OPT_FP64_GEMM, cr.CR_GEMM_OZAKI) == 0
    assert cr._lib.cr_get_option(cr.CR_OPT_FP64_GEMM, ctypes.byref(v)) == 0 and v.value == cr.CR_GEMM_OZAKI
    assert cr._lib.cr_set_option(cr.CR_OPT_FP64_GEMM, cr.CR_GEMM_DF) == 0
    assert cr._lib.cr_set_option(99, 0) == 1 and cr._lib.cr_get_option(99, ctypes.byref(v)) == 1
    assert cr._lib.cr_get_option(cr.CR_OPT_DIAG_ARITH, None) == 1
    assert cr._lib.cr_workspace_trim() == 0   # no pool yet: nothing to return, no device call
    d = ctypes.c_double()
    assert cr._lib.cr_peak_probe(cr.CR_PEAK_DFMA, 100, None, None) == 1
    assert cr._lib.cr_peak_probe(cr.CR_PEAK_DFMA, 0, ctypes.byref(d), None) == 1
