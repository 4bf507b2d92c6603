"""The oracle against closed forms, invariants, library routines and brute
force (CPU only).  See tests/oracle_pins.py for what each check pins."""
import math

import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(oracle.forward)


def _brute_linear(a, W):
    """sum_k a[t][k] * W[n][k] by plain Python loops."""
    T, K = a.shape
    N = W.shape[0]
    return np.array([[math.fsum(float(a[t, k]) * float(W[n, k]) for k in range(K)) for n in range(N)]
                     for t in range(T)])


def test_in_proj_selector_weights_copy_columns():
    """A 0/1 selector weight (row i picks input column perm[i]) copies columns exactly: fixes the
    [out][in] weight layout and the absence of any scaling or bias."""
    r = np.random.default_rng(5)
    T, H = 7, 16
    hid = r.standard_normal((T, H)).astype(np.float32)
    sel = lambda perm: np.eye(H, dtype=np.float32)[perm]
    pq, pz, pa, pb = (r.integers(0, H, n) for n in (24, 12, 3, 3))
    x, z, a, b = oracle.in_proj(hid, sel(pq), sel(pz), sel(pa), sel(pb))
    for out, perm in ((x, pq), (z, pz), (a, pa), (b, pb)):
        assert np.array_equal(out, hid[:, perm].astype(np.float64))


def test_projections_brute_force():
    r = np.random.default_rng(6)
    T, H, HvD = 3, 8, 5
    hid = r.standard_normal((T, H)).astype(np.float32)
    Ws = [r.standard_normal((n, H)).astype(np.float32) for n in (6, 5, 2, 2)]
    for got, W in zip(oracle.in_proj(hid, *Ws), Ws):
        np.testing.assert_allclose(got, _brute_linear(hid, W), rtol=0, atol=1e-12)
    y = r.standard_normal((T, HvD)).astype(np.float32)
    Wo = r.standard_normal((H, HvD)).astype(np.float32)
    np.testing.assert_allclose(oracle.out_proj(y, Wo), _brute_linear(y, Wo), rtol=0, atol=1e-12)
