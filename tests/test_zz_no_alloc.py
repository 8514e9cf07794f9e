"""The allocation-free calibration entry point (cr_calibrate_noalloc).

It serves callers that cannot allocate device memory (code under a memory pool that owns
every device allocation, or an embedder whose device footprint must not grow after
start-up).  Its scratch is a fixed array inside the library, shared by every call, so these
tests call it twice in a row on different inputs and compare both results with
cr_calibrate, which uses library-managed scratch; they also issue two calls on two
different streams with nothing between them, and take the two error paths that reuse the
array's flag and the host buffer.  The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import mixed_precision_dense_mat_gb300 as cr

pytestmark = pytest.mark.gpu


def _colmajor(a):
    return torch.from_numpy(np.asfortranarray(a).T.copy()).cuda().T


def _issue(name, S, z, v, u, level, stream=None):
    """One call through the C ABI on `stream` (default: the current stream), without any
    synchronisation around it; returns (status, info, output tensors)."""
    n_p, M = S.shape
    lds = S.stride(1)
    stream = stream or torch.cuda.current_stream()
    with torch.cuda.stream(stream):
        cin = torch.empty(n_p, dtype=torch.uint8, device="cuda")
        cout = torch.empty(n_p, dtype=torch.uint8, device="cuda")
        cnt = torch.full((n_p,), -7, dtype=torch.int32, device="cuda")   # must be cleared by the call
        psi = torch.empty(M, dtype=torch.float64, device="cuda")
        phi = torch.empty(M, dtype=torch.float64, device="cuda")
    info = cr.CalibInfo()
    code = getattr(cr._lib, name)(S.data_ptr(), lds, n_p, M, z.data_ptr(), v.data_ptr(), u, level, cin.data_ptr(),
                                  cout.data_ptr(), cnt.data_ptr(), psi.data_ptr(), phi.data_ptr(), ctypes.byref(info),
                                  stream.cuda_stream)
    return code, info, (cin, cout, cnt, psi, phi)


def _result(info, outs):
    cin, cout, cnt, psi, phi = outs
    return {"q_in": info.q_in, "q_out": info.q_out, "n_psi": info.n_psi, "n_phi": info.n_phi,
            "c_in": cin.cpu().numpy(), "c_out": cout.cpu().numpy(), "count": cnt.cpu().numpy(),
            "psi": psi.cpu().numpy(), "phi": phi.cpu().numpy()}


def _call(name, S, z, v, u, level):
    code, info, outs = _issue(name, S, z, v, u, level)
    torch.cuda.synchronize()
    assert code == 0, (name, code, cr._lib.cr_last_error_detail())
    return _result(info, outs)


def _same(a, b):
    # identical kernels and reduction order: the results agree exactly (tolerance 0)
    for k in ("psi", "phi", "count", "c_in", "c_out"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    for k in ("q_in", "q_out", "n_psi", "n_phi"):
        assert a[k] == b[k], k


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
        _same(a, b)


def test_noalloc_back_to_back_on_two_streams():
    """Two calls on two different streams, nothing between them: the second may start its
    kernels only after the first call's last read of the shared array (the call returns after
    it), so both results equal cr_calibrate's.  The second problem is the smaller one, so a
    first call still reading t while the second overwrites it would change the first's
    regions."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cr.load()
    cases = [_case(11, 6000, 257, 0.15), _case(12, 1500, 64, -0.2)]
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    r = []
    for (S, z, v, u), st in zip(cases, (s1, s2)):
        code, info, outs = _issue("cr_calibrate_noalloc", S, z, v, u, 0.9, stream=st)
        assert code == 0, (code, cr._lib.cr_last_error_detail())
        r.append((info, outs))
    torch.cuda.synchronize()
    got = [_result(info, outs) for info, outs in r]
    for (S, z, v, u), g in zip(cases, got):
        _same(g, _call("cr_calibrate", S, z, v, u, 0.9))
    # the library-managed entry point under the same pattern
    r = []
    for (S, z, v, u), st in zip(cases, (s1, s2)):
        code, info, outs = _issue("cr_calibrate", S, z, v, u, 0.9, stream=st)
        assert code == 0, (code, cr._lib.cr_last_error_detail())
        r.append((info, outs))
    torch.cuda.synchronize()
    for g, (info, outs) in zip(got, r):
        _same(g, _result(info, outs))


def test_noalloc_error_paths_then_normal_call():
    """A non-positive MSPE and an empty sample give the same codes as cr_calibrate (they use the
    array's flag and compact the host buffer in place); a normal call right after them still
    matches cr_calibrate exactly."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cr.load()
    S, z, v, u = _case(21, 3000, 128, 0.1)
    v_bad = v.clone()
    v_bad[1234] = 0.0
    codes = []
    for name in ("cr_calibrate_noalloc", "cr_calibrate"):
        code, _, _ = _issue(name, S, z, v_bad, u, 0.9)
        torch.cuda.synchronize()
        codes.append(code)
    assert codes == [6, 6], codes   # CR_ERR_NONPOS_MSPE
    u_high = float(S.max().item()) + 1.0   # no S_ij >= u: every psi set is empty
    codes, infos = [], []
    for name in ("cr_calibrate_noalloc", "cr_calibrate"):
        code, info, _ = _issue(name, S, z, v, u_high, 0.9)
        torch.cuda.synchronize()
        codes.append(code)
        infos.append((info.n_psi, info.n_phi))
    assert codes == [5, 5], codes   # CR_ERR_EMPTY_SAMPLE
    assert infos[0] == infos[1] == (0, 128), infos
    a = _call("cr_calibrate_noalloc", S, z, v, u, 0.9)
    b = _call("cr_calibrate", S, z, v, u, 0.9)
    _same(a, b)


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
