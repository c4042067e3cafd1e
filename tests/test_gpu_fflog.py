"""The tree build's float-float logarithm, checked directly against double-precision
ln over [1e-30, 1e30] (it gives the draft rows' log-normaliser ln Z, from which the
dynamic tree's cumulative scores ln q are formed).  Method: range reduction
z = 2^k w with w in [1/sqrt 2, sqrt 2) and the atanh series of ln w, on the fp32 pipe
in float-float arithmetic (about 48 significant bits)."""
import numpy as np
import pytest
import torch

from eagle_speculative_decoding_tree_gb300 import binding as B

pytestmark = pytest.mark.gpu


def test_ff_log_against_double():
    g = np.random.default_rng(20261202)
    e = g.uniform(np.log(1e-30), np.log(1e30), 200_000)
    z = np.exp(e)
    z = np.concatenate([z, 2.0 ** np.arange(-99, 100), [1.0, 1.0 + 2 ** -23, 1.0 - 2 ** -24, 0.70710678, 1.41421356,
                                                         3.4e38, 1.2e-38]])
    hi = z.astype(np.float32)
    lo = (z - hi.astype(np.float64)).astype(np.float32)
    lo[: 1000] = 0.0  # some inputs with no low part
    zz = hi.astype(np.float64) + lo.astype(np.float64)  # exactly the float-float input
    oh, ol = B.selftest_ff_log(torch.from_numpy(hi).cuda(), torch.from_numpy(lo).cuda())
    got = oh.cpu().numpy().astype(np.float64) + ol.cpu().numpy().astype(np.float64)
    ref = np.log(zz)
    err = np.abs(got - ref)
    bound = 1e-12 * np.maximum(1.0, np.abs(ref))
    worst = int(np.argmax(err / bound))
    assert (err <= bound).all(), f"z={zz[worst]!r}: ln {ref[worst]!r}, got {got[worst]!r} (err {err[worst]:.3e})"
    # the fp32 logarithm is far coarser: the float-float one must beat it everywhere
    assert err.max() < 1e-9
