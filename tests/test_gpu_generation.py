"""The generated working tiles against round_p(s^2 V) ("Mixed-Precision GPU Acceleration for
Confidence Regions of Spatial Excursion Sets", Alg.2 step 12 with Section IV-C's scale s: the
tiles of s^2 V in their precision classes).

cr_tilemat_to_dense(what = 2) runs the factorisation's generation step alone.  The oracle's
FP64 covariance, times s^2 and rounded to each tile's class (round to nearest even), is the
reference:
  - FP64-class (diagonal) tiles: within 1e-12 relative (FP64, or double-float when the
    double-float executor factors them);
  - FP32-class tiles: within one FP32 ulp of the rounded value (the evaluation is accurate to
    about 2^-39, so only values within that of a rounding midpoint can round the other way),
    and equal to it at all but 0.1 % of the entries;
  - FP16-class tiles: within one FP16 ulp (FP32 evaluation, about 2^-21), equal at all but 1 %.
A factorisation after the export gives the same bits as one without it."""
import numpy as np
import pytest
import torch

import inputgen
import oracle

pytestmark = pytest.mark.gpu


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("family,nu", [("matern", 0.5), ("matern", 1.5), ("matern", 2.5), ("powexp", 0.5),
                                       ("matern", 1.0)])
def test_generated_tiles_are_the_rounded_scaled_covariance(lib, family, nu):
    n, nb, beta, fixedacc = 1500, 128, 0.03, 1e-4
    xy = np.ascontiguousarray(inputgen.morton_sorted(inputgen.uniform_locations(n, 71)))

    def build():
        G = lib.TileMat(n, nb)
        lib.cov_build(G, dev(xy), family, 1.0, beta, nu, nugget=0.0, n_pred=0, tau2=0.0)
        pmap, info = lib.precision_map(G, amp=True, fixedacc=fixedacc)
        return G, pmap, info

    G, pmap, info = build()
    assert info["n_fp16"] + info["n_fp32"] > 0, info
    T = lib.tilemat_to_dense(G, 2).cpu().numpy()
    ref = info["s"] ** 2 * oracle.covariance_matrix(xy, family, 1.0, beta, nu, 0.0, 0, 0.0)
    nt = (n + nb - 1) // nb
    mism32 = mism16 = cnt32 = cnt16 = 0
    for I in range(nt):
        for J in range(I + 1):
            rs, cs = slice(I * nb, min(n, (I + 1) * nb)), slice(J * nb, min(n, (J + 1) * nb))
            t, r = T[rs, cs], ref[rs, cs]
            if I == J:
                t, r = np.tril(t), np.tril(r)
            cls = pmap[I, J]
            if cls == lib.CR_PREC_FP64:
                assert np.all(np.abs(t - r) <= 1e-12 * np.abs(r) + 1e-300), (I, J)
            elif cls == lib.CR_PREC_FP32:
                r32 = r.astype(np.float32)
                assert np.all(np.abs(t - r32.astype(np.float64)) <= np.spacing(np.abs(r32)).astype(np.float64)), (I, J)
                mism32 += int(np.sum(t != r32.astype(np.float64)))
                cnt32 += t.size
            else:
                r16 = r.astype(np.float16)
                assert np.all(np.abs(t - r16.astype(np.float64)) <= np.spacing(np.abs(r16)).astype(np.float64)), (I, J)
                mism16 += int(np.sum(t != r16.astype(np.float64)))
                cnt16 += t.size
    assert mism32 <= 1e-3 * cnt32, (mism32, cnt32)
    assert mism16 <= 1e-2 * cnt16, (mism16, cnt16)
    # a factorisation after the export equals one without it
    assert lib.potrf_adaptive(G) == 0
    L1 = lib.tilemat_to_dense(G, 1).cpu().numpy()
    G2, _, _ = build()
    assert lib.potrf_adaptive(G2) == 0
    np.testing.assert_array_equal(L1, lib.tilemat_to_dense(G2, 1).cpu().numpy())
    G.close()
    G2.close()
