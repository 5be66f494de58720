"""Pins for the dt-projection oracle (rustytorch commit log, "MambaBlock" S6
forward commit: "delta=softplus(dt.dt_proj+dt_bias)"): numpy's matrix
product for the pre-activation, softplus identities, and finite differences
for the backward -- nothing here re-types the oracle's loops."""
import math

import numpy as np
import pytest

import oracle


def rnd(seed, M=37, D=24, R=16):
    r = np.random.default_rng(seed)
    return r.standard_normal((M, R)), r.standard_normal((D, R)) / np.sqrt(R), r.standard_normal(D) - 2.0


def test_pre_activation_is_the_matrix_product():
    a, w, b = rnd(1)
    pre = oracle.dtproj_fwd(a, w, b, softplus=False)
    np.testing.assert_allclose(pre, a @ w.T + b, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(oracle.dtproj_fwd(a, w, None, softplus=False), a @ w.T, rtol=1e-13, atol=1e-13)


def test_softplus_values_and_identities():
    a, w, b = rnd(2)
    pre = a @ w.T + b
    got = oracle.dtproj_fwd(a, w, b)
    np.testing.assert_allclose(got, np.logaddexp(0.0, pre), rtol=1e-13, atol=1e-15)
    # softplus(v) - softplus(-v) = v, softplus(0) = ln 2, softplus(v) -> v for large v
    neg = oracle.dtproj_fwd(-a, w, -b)
    np.testing.assert_allclose(got - neg, pre, rtol=1e-12, atol=1e-12)
    zero = oracle.dtproj_fwd(np.zeros((3, 4)), np.ones((5, 4)), np.zeros(5))
    np.testing.assert_allclose(zero, math.log(2.0), rtol=1e-15)
    big = oracle.dtproj_fwd(np.zeros((1, 4)), np.ones((1, 4)), np.array([60.0]))
    assert big[0, 0] == 60.0


def test_backward_matches_finite_differences():
    a, w, b = rnd(3, M=9, D=7, R=8)
    g = np.random.default_rng(4).standard_normal((9, 7))
    out = oracle.dtproj_bwd(a, w, g, b)

    def loss(aa, bb):
        return float(np.sum(g * oracle.dtproj_fwd(aa, w, bb)))

    h = 1e-6
    # dbias = sum_m dpre
    fd_b = np.array([(loss(a, b + h * e) - loss(a, b - h * e)) / (2 * h) for e in np.eye(7)])
    np.testing.assert_allclose(out["dbias"], fd_b, rtol=1e-7, atol=1e-9)
    # dL/da = dpre @ w (a plain product of the oracle's dpre with w)
    fd_a = np.zeros_like(a)
    for idx in np.ndindex(a.shape):
        up, dn = a.copy(), a.copy()
        up[idx] += h
        dn[idx] -= h
        fd_a[idx] = (loss(up, b) - loss(dn, b)) / (2 * h)
    np.testing.assert_allclose(out["dpre"] @ w, fd_a, rtol=1e-7, atol=1e-9)


def test_without_softplus_the_gradient_passes_through():
    a, w, b = rnd(5)
    g = np.random.default_rng(6).standard_normal((37, 24))
    out = oracle.dtproj_bwd(a, w, g, b, softplus=False)
    np.testing.assert_array_equal(out["dpre"], g)
    np.testing.assert_allclose(out["dbias"], g.sum(0), rtol=1e-13)


@pytest.mark.parametrize("dtype", ["f32"])
def test_float_instantiation_is_close(dtype):
    a, w, b = rnd(7)
    np.testing.assert_allclose(oracle.dtproj_fwd(a, w, b, dtype=dtype), oracle.dtproj_fwd(a, w, b), rtol=2e-6, atol=1e-6)
