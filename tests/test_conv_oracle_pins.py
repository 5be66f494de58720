"""Pins for the conv1d + SiLU oracle (rustytorch commit log, "MambaBlock" S6
forward commit: "in_proj -> causal depthwise conv1d -> SiLU -> x_proj";
MambaRecurrence commit: the conv-ring state carried between steps), checked
against numpy's convolution, special kernels, causality, state chaining,
the step form and finite differences -- nothing here re-types the oracle's
own loops."""
import numpy as np
import pytest

import oracle


def sig(v):
    return 1.0 / (1.0 + np.exp(-v))


def rnd(seed, B=2, L=13, D=3, K=4, state=True):
    r = np.random.default_rng(seed)
    xin = r.standard_normal((B, L, D))
    w = r.standard_normal((D, K)) * 0.7
    b = r.standard_normal(D) * 0.3
    st = r.standard_normal((B, D, K - 1)) if state and K > 1 else None
    return xin, w, b, st


def numpy_conv(xin, w, b, st):
    B, L, D = xin.shape
    K = w.shape[1]
    pre = np.zeros((B, L, D))
    for bb in range(B):
        for d in range(D):
            head = st[bb, d] if st is not None else np.zeros(K - 1)
            pad = np.concatenate([head, xin[bb, :, d]])
            pre[bb, :, d] = np.convolve(pad, w[d][::-1], mode="valid") + b[d]
    return pre


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_matches_numpy_convolve(K):
    xin, w, b, st = rnd(K, K=K)
    pre = numpy_conv(xin, w, b, st)
    got = oracle.conv_fwd(xin, w, b, st)
    np.testing.assert_allclose(got["x"], pre * sig(pre), rtol=1e-12, atol=1e-13)
    if K > 1:
        pad = np.concatenate([st, xin.transpose(0, 2, 1)], axis=2)
        np.testing.assert_array_equal(got["state_out"], pad[:, :, -(K - 1):])


def test_special_kernels():
    xin, _, b, st = rnd(7, K=4)
    B, L, D = xin.shape
    ident = np.zeros((D, 4)); ident[:, 3] = 1.0           # newest tap only: pre = xin + b
    shift = np.zeros((D, 4)); shift[:, 0] = 1.0           # oldest tap only: pre_t = xin[t-3]
    pre = xin + b
    np.testing.assert_allclose(oracle.conv_fwd(xin, ident, b, st)["x"], pre * sig(pre), rtol=1e-14)
    got = oracle.conv_fwd(xin, shift, np.zeros(D), st)["x"]
    src = np.concatenate([st.transpose(0, 2, 1), xin], axis=1)[:, :L]
    np.testing.assert_allclose(got, src * sig(src), rtol=1e-14)
    w1 = np.full((D, 1), 0.5)                              # K = 1: pointwise, no state
    np.testing.assert_allclose(oracle.conv_fwd(xin, w1, b)["x"], (0.5 * xin + b) * sig(0.5 * xin + b), rtol=1e-14)


def test_causal():
    xin, w, b, st = rnd(11, L=20)
    base = oracle.conv_fwd(xin, w, b, st)["x"]
    x2 = xin.copy()
    x2[:, 12] += 1.0
    moved = oracle.conv_fwd(x2, w, b, st)["x"]
    np.testing.assert_array_equal(moved[:, :12], base[:, :12])
    assert np.all(np.abs(moved[:, 12] - base[:, 12]) > 0)


def test_state_chains_and_steps_reproduce_the_sequence():
    xin, w, b, st = rnd(13, L=17)
    full = oracle.conv_fwd(xin, w, b, st)
    a = oracle.conv_fwd(xin[:, :9], w, b, st)
    c = oracle.conv_fwd(xin[:, 9:], w, b, a["state_out"])
    np.testing.assert_array_equal(np.concatenate([a["x"], c["x"]], axis=1), full["x"])
    np.testing.assert_array_equal(c["state_out"], full["state_out"])
    # float32: one token at a time through the ring state is bitwise the sequence
    f = {k: None if v is None else v.astype(np.float32) for k, v in dict(xin=xin, w=w, b=b, st=st).items()}
    seq = oracle.conv_fwd(f["xin"], f["w"], f["b"], f["st"], dtype="f32")
    ring = f["st"].copy()
    for t in range(xin.shape[1]):
        o = oracle.conv_fwd(f["xin"][:, t:t + 1], f["w"], f["b"], ring, dtype="f32")
        np.testing.assert_array_equal(o["x"][:, 0], seq["x"][:, t])
        ring = o["state_out"]
    np.testing.assert_array_equal(ring, seq["state_out"])


def test_gradients_match_finite_differences():
    xin, w, b, st = rnd(17, B=2, L=7, D=2, K=4)
    dx = np.random.default_rng(3).standard_normal(xin.shape)
    g = oracle.conv_bwd(xin, w, dx, b, st)

    def loss(xi, ww, bb, ss):
        return float(np.sum(oracle.conv_fwd(xi, ww, bb, ss)["x"] * dx))

    h = 1e-6
    for name, arr, pos in (("dxin", xin, 0), ("dw", w, 1), ("dbias", b, 2), ("dstate", st, 3)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            args = [xin, w, b, st]
            up, dn = arr.copy(), arr.copy()
            up[idx] += h
            dn[idx] -= h
            args[pos] = up
            lp = loss(*args)
            args[pos] = dn
            lm = loss(*args)
            fd[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g[name], fd, rtol=1e-6, atol=1e-8, err_msg=name)


def test_zero_bias_and_zero_state_defaults():
    xin, w, _, _ = rnd(19)
    D, K = w.shape
    a = oracle.conv_fwd(xin, w)
    b = oracle.conv_fwd(xin, w, np.zeros(D), np.zeros((xin.shape[0], D, K - 1)))
    np.testing.assert_array_equal(a["x"], b["x"])
