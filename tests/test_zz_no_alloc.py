"""The allocation-free calibration entry point (cr_calibrate_noalloc).

It serves callers that cannot allocate device memory (a pool or capture regime that forbids
cudaMalloc/cudaFree, or an embedder whose device footprint must not grow after start-up).
Its scratch is a fixed array inside the library, shared by every call, so these tests call
it twice in a row on different inputs and compare both results with cr_calibrate, which
uses library-managed scratch.  The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import mixed_precision_dense_mat_gb300 as cr

pytestmark = pytest.mark.gpu


def _colmajor(a):
    return torch.from_numpy(np.asfortranarray(a).T.copy()).cuda().T


def _call(name, S, z, v, u, level):
    n_p, M = S.shape
    lds = S.stride(1)
    cin = torch.empty(n_p, dtype=torch.uint8, device="cuda")
    cout = torch.empty(n_p, dtype=torch.uint8, device="cuda")
    cnt = torch.full((n_p,), -7, dtype=torch.int32, device="cuda")   # must be cleared by the call
    psi = torch.empty(M, dtype=torch.float64, device="cuda")
    phi = torch.empty(M, dtype=torch.float64, device="cuda")
    info = cr.CalibInfo()
    code = getattr(cr._lib, name)(S.data_ptr(), lds, n_p, M, z.data_ptr(), v.data_ptr(), u, level, cin.data_ptr(),
                                  cout.data_ptr(), cnt.data_ptr(), psi.data_ptr(), phi.data_ptr(), ctypes.byref(info),
                                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert code == 0, (name, code, cr._lib.cr_last_error_detail())
    return {"q_in": info.q_in, "q_out": info.q_out, "n_psi": info.n_psi, "n_phi": info.n_phi,
            "c_in": cin.cpu().numpy(), "c_out": cout.cpu().numpy(), "count": cnt.cpu().numpy(),
            "psi": psi.cpu().numpy(), "phi": phi.cpu().numpy()}


def _case(seed, n_p, M, u):
    rng = np.random.default_rng(seed)
    S = _colmajor(rng.standard_normal((n_p, M)))
    z = torch.from_numpy(rng.standard_normal(n_p) * 0.5).cuda()
    v = torch.from_numpy(rng.uniform(0.3, 2.0, n_p)).cuda()
    return S, z, v, u


def test_noalloc_matches_calibrate_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cr.load()
    # the second call is smaller than the first, so stale scratch from the first would show
    for seed, n_p, M, u in ((5, 5000, 300, 0.2), (6, 2100, 77, -0.1)):
        S, z, v, u = _case(seed, n_p, M, u)
        a = _call("cr_calibrate_noalloc", S, z, v, u, 0.9)
        b = _call("cr_calibrate", S, z, v, u, 0.9)
        # identical kernels and reduction order: the results agree exactly (tolerance 0)
        for k in ("psi", "phi", "count", "c_in", "c_out"):
            np.testing.assert_array_equal(a[k], b[k], err_msg=k)
        for k in ("q_in", "q_out", "n_psi", "n_phi"):
            assert a[k] == b[k], k


def test_noalloc_rejects_oversized_problem():
    cr.load()
    info = cr.CalibInfo()
    # M above the documented limit is refused before any device work
    code = cr._lib.cr_calibrate_noalloc(1, 100, 100, 70000, 1, 1, 0.0, 0.9, 1, 1, None, None, None,
                                        ctypes.byref(info), None)
    assert code == 1 and b"CR_NOALLOC_MAX_M" in cr._lib.cr_last_error_detail()
    # scratch needed for n_p = 10^6 sites and M = 4096 exceeds the fixed array
    code = cr._lib.cr_calibrate_noalloc(1, 1000000, 1000000, 4096, 1, 1, 0.0, 0.9, 1, 1, None, None, None,
                                        ctypes.byref(info), None)
    assert code == 1 and b"CR_NOALLOC_SCRATCH_BYTES" in cr._lib.cr_last_error_detail()
