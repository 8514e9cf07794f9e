"""Failure reporting of the library (GPU), made on the host or by a short device-side wait
limit; nothing here faults, traps or hangs the GPU:
  * a NaN site coordinate is reported as CR_ERR_ARG by the precision map (from the
    statistics pass), before any factorisation;
  * a zero wait limit (CR_OPT_WAIT_LIMIT_US) makes the diagonal executor's bounded waits give
    up: the factorisation returns CR_ERR_TIMEOUT, and the same tile matrix factored again with
    the default limit matches the oracle, which shows the executor's flags and buffers start
    clean on the next call;
  * a covariance whose factor cannot be held in FP16 (sqrt(V_ii) above 65504 with no room to
    scale) is reported as CR_ERR_RANGE by the precision map."""
import contextlib

import numpy as np
import pytest
import torch

import inputgen
import oracle

pytestmark = pytest.mark.gpu


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def colmajor(a):
    return torch.from_numpy(np.asfortranarray(a).T.copy()).cuda().T


def relf(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


@contextlib.contextmanager
def option(lib, opt, value):
    old = lib.get_option(opt)
    lib.set_option(opt, value)
    try:
        yield
    finally:
        lib.set_option(opt, old)


def test_nan_coordinate_is_an_argument_error(lib):
    xy = inputgen.morton_sorted(inputgen.uniform_locations(600, 2))
    xy[437, 1] = np.nan
    V = lib.TileMat(600, 128)
    lib.cov_build(V, dev(xy), "matern", 1.0, 0.1, 0.5, nugget=1e-4)
    with pytest.raises(lib.CrError) as e:
        lib.precision_map(V, amp=True, fixedacc=1e-4)
    assert e.value.name == "CR_ERR_ARG" and "NaN" in e.value.detail
    with pytest.raises(lib.CrError) as e:
        lib.potrf_adaptive(V)            # no map was taken: the factorisation is refused
    assert e.value.name == "CR_ERR_STATE"
    V.close()


@pytest.mark.parametrize("arith", ["fp64", "df"])
def test_wait_limit_runs_out_then_next_call_is_clean(lib, arith):
    n, nb = 1024, 512
    xy = inputgen.morton_sorted(inputgen.uniform_locations(n, 4))
    V = lib.TileMat(n, nb)
    lib.cov_build(V, dev(xy), "matern", 1.0, 0.05, 0.5, nugget=1e-4)
    lib.precision_map(V, amp=False)
    mode = lib.CR_DIAG_FP64 if arith == "fp64" else lib.CR_DIAG_DF
    with option(lib, lib.CR_OPT_DIAG_ARITH, mode):
        with option(lib, lib.CR_OPT_WAIT_LIMIT_US, 0):
            with pytest.raises(lib.CrError) as e:
                lib.potrf_adaptive(V)
            assert e.value.name == "CR_ERR_TIMEOUT"
        assert lib.get_option(lib.CR_OPT_WAIT_LIMIT_US) == 2000000
        assert lib.potrf_adaptive(V) == 0
    L = lib.tilemat_to_dense(V, 1).cpu().numpy()
    Vo = oracle.covariance_matrix(xy, "matern", 1.0, 0.05, 0.5, 1e-4)
    Lo = oracle.cholesky_lower(Vo)
    scale = max(1.0, relf(np.linalg.cholesky(Vo), Lo) / 1e-14)
    assert relf(L, Lo) <= 1e-11 * scale
    V.close()


def test_factor_out_of_fp16_range(lib):
    xy = inputgen.morton_sorted(inputgen.uniform_locations(512, 6))
    V = lib.TileMat(512, 128)
    lib.cov_build(V, dev(xy), "matern", 1e10, 0.05, 0.5, nugget=1e-4)   # sqrt(V_ii) = 1e5
    with pytest.raises(lib.CrError) as e:
        lib.precision_map(V, amp=True, fixedacc=1e-3)
    assert e.value.name == "CR_ERR_RANGE"
    # the all-FP64 mode has no FP16 operand and accepts it
    lib.precision_map(V, amp=False)
    assert lib.potrf_adaptive(V) == 0
    V.close()
