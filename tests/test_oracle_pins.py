"""Pins of the CPU oracle against facts that do not come from the oracle
itself: closed forms, a brute-force non-recurrent formula, special cases
that reduce to library routines, causality, linearity, the step identity,
finite differences and the adjoint identity.

The scan being pinned is the S6 recurrence of the rustytorch "MambaBlock"
commits: Delta = softplus(dt + dt_bias), h_t = exp(Delta*A) * h_{t-1} +
Delta*B_t*x_t, y_t = (sum_n C_t h_t + D*x_t) * silu(z_t)."""
import math
import os
from dataclasses import replace

import numpy as np
import pytest

import gen
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def expit(z):
    # logistic function written as tanh: an independent route from the
    # oracle's exp-based sigmoid
    return 0.5 * (1.0 + np.tanh(0.5 * z))


def small(B=2, L=7, D=3, N=4, seed=0, **kw):
    return gen.make_inputs(B, L, D, N, seed=seed, dt_std=0.5, delta_target=0.2, **kw)


def random_A(D, N, seed):
    u = gen.uniform53(seed, D * N).reshape(D, N)
    return -(0.1 + 3.0 * u)  # negative, not structured by n


def ema_inputs(L, D, deltas, x):
    """N = 1, B = C = 1, no skip, no gate, Delta given directly."""
    deltas = np.asarray(deltas, np.float64)
    inp = gen.make_inputs(1, L, D, 1, seed=1, gate=False, skip=False, bias=False)
    inp.delta_softplus = 0
    inp.dt = np.broadcast_to(deltas, (1, L, D)).copy()
    inp.A = (np.log1p(-deltas) / deltas).reshape(D, 1)
    inp.Bm = np.ones((1, L, 1))
    inp.Cm = np.ones((1, L, 1))
    inp.x = np.asarray(x, np.float64).reshape(1, L, D)
    return inp


# ---------------------------------------------------------------- forward

def test_ema_golden_fixture():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "ema_half.txt"))
            if l.strip() and not l.startswith("#")]
    L = len(rows)
    y = oracle.fwd(ema_inputs(L, 1, [0.5], np.ones(L)))["y"][0, :, 0]
    for t, num, den in rows:
        assert abs(y[int(t)] - int(num) / int(den)) < 1e-14


def test_ema_constant_input_closed_form():
    L, deltas, c = 300, [0.3, 0.05, 0.001], 1.7
    y = oracle.fwd(ema_inputs(L, 3, deltas, np.full((L, 3), c)))["y"][0]
    t = np.arange(L)[:, None]
    ref = c * (1.0 - (1.0 - np.asarray(deltas)) ** (t + 1))
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-14)


def test_ema_general_input_closed_form():
    L, deltas = 120, [0.25, 0.02]
    x = gen.normal_f32(4, L * 2).reshape(L, 2).astype(np.float64)
    y = oracle.fwd(ema_inputs(L, 2, deltas, x))["y"][0]
    for d, dl in enumerate(deltas):
        for t in range(L):
            ref = dl * sum((1 - dl) ** (t - s) * x[s, d] for s in range(t + 1))
            assert abs(y[t, d] - ref) <= 1e-12 * max(1.0, abs(ref))


def quadratic_form(inp, delta):
    """y_t = [sum_{s<=t} sum_n C_tn exp(A_n sum_{r=s+1}^t Delta_r) Delta_s B_sn x_s
              + sum_n C_tn exp(A_n sum_{r=0}^t Delta_r) h0_n + D x_t] * silu(z_t),
    evaluated directly from its definition (no recurrence)."""
    B, L, D, N = inp.B, inp.L, inp.D, inp.N
    y = np.zeros((B, L, D))
    h0 = inp.h0 if inp.h0 is not None else np.zeros((B, D, N))
    for b in range(B):
        for d in range(D):
            for t in range(L):
                acc = 0.0
                for n in range(N):
                    A = float(inp.A[d, n])
                    C = float(inp.Cm[b, t, n])
                    for s in range(t + 1):
                        seg = sum(float(delta[b, r, d]) for r in range(s + 1, t + 1))
                        acc += C * math.exp(A * seg) * float(delta[b, s, d]) * \
                            float(inp.Bm[b, s, n]) * float(inp.x[b, s, d])
                    seg0 = sum(float(delta[b, r, d]) for r in range(0, t + 1))
                    acc += C * math.exp(A * seg0) * float(h0[b, d, n])
                acc += float(inp.Dskip[d]) * float(inp.x[b, t, d])
                zt = float(inp.z[b, t, d])
                y[b, t, d] = acc * zt * float(expit(zt))
    return y


def test_quadratic_form_bruteforce_with_h0():
    inp = small(with_h0=True)
    inp.A = random_A(inp.D, inp.N, 77)
    inp.Dskip = gen.normal_f32(78, inp.D)
    inp.delta_softplus = 0
    inp.dt = 0.05 + 0.8 * gen.uniform53(79, inp.B * inp.L * inp.D).reshape(inp.B, inp.L, inp.D)
    inp.dt_bias = np.full(inp.D, 0.01)
    delta = inp.dt + inp.dt_bias
    got = oracle.fwd(inp)["y"]
    np.testing.assert_allclose(got, quadratic_form(inp, delta), rtol=1e-11, atol=1e-13)


def test_softplus_applies_to_dt_plus_bias():
    inp = small()
    ref_in = replace(inp, delta_softplus=0, dt_bias=None,
                     dt=np.logaddexp(0.0, inp.dt.astype(np.float64) + inp.dt_bias))
    np.testing.assert_allclose(oracle.fwd(inp)["y"], oracle.fwd(ref_in)["y"],
                               rtol=1e-13, atol=1e-15)


def test_gate_is_silu_of_z():
    inp = small()
    ungated = oracle.fwd(replace(inp, z=None))["y"]
    z = inp.z.astype(np.float64)
    np.testing.assert_allclose(oracle.fwd(inp)["y"], ungated * z * expit(z), rtol=1e-12,
                               atol=1e-15)


def test_tiny_delta_leaves_only_the_skip_term():
    inp = small()
    inp.dt = np.full_like(inp.dt, -40.0)  # softplus(-40) ~ 4e-18
    z = inp.z.astype(np.float64)
    ref = inp.Dskip[None, None, :] * inp.x * z * expit(z)
    np.testing.assert_allclose(oracle.fwd(inp)["y"], ref, rtol=1e-12, atol=1e-15)


def test_infinitely_fast_decay_is_memoryless():
    inp = small()
    inp.A = np.full_like(inp.A, -1e6)
    delta = np.logaddexp(0.0, inp.dt.astype(np.float64) + inp.dt_bias)
    h = delta[..., None] * inp.Bm[:, :, None, :] * inp.x[..., None]  # [B,L,D,N]
    p = np.einsum("bldn,bln->bld", h, inp.Cm.astype(np.float64)) + inp.Dskip * inp.x
    z = inp.z.astype(np.float64)
    np.testing.assert_allclose(oracle.fwd(inp)["y"], p * z * expit(z), rtol=1e-12, atol=1e-14)


def test_zero_A_is_cumulative_sum():
    inp = gen.make_inputs(2, 50, 3, 1, seed=5, skip=True, bias=False)
    inp.delta_softplus = 0
    inp.dt = np.ones_like(inp.dt)
    inp.A = np.zeros((3, 1))
    inp.Bm = np.ones((2, 50, 1))
    inp.Cm = np.ones((2, 50, 1))
    z = inp.z.astype(np.float64)
    ref = (np.cumsum(inp.x.astype(np.float64), axis=1) + inp.x) * z * expit(z)
    np.testing.assert_allclose(oracle.fwd(inp)["y"], ref, rtol=1e-12, atol=1e-12)


def test_causality():
    inp = small(L=12)
    y0 = oracle.fwd(inp)["y"]
    tstar = 5
    x = inp.x.astype(np.float64).copy()
    x[:, tstar, :] += 0.75
    y1 = oracle.fwd(replace(inp, x=x))["y"]
    assert np.array_equal(y0[:, :tstar], y1[:, :tstar])
    assert np.all(np.abs(y0[:, tstar] - y1[:, tstar]) > 0)


def test_linearity_in_x():
    inp = small(L=20)
    x1 = inp.x.astype(np.float64)
    x2 = gen.normal_f32(91, x1.size).reshape(x1.shape).astype(np.float64)
    al, be = 0.7, -1.3
    y1 = oracle.fwd(replace(inp, x=x1))["y"]
    y2 = oracle.fwd(replace(inp, x=x2))["y"]
    y12 = oracle.fwd(replace(inp, x=al * x1 + be * x2))["y"]
    np.testing.assert_allclose(y12, al * y1 + be * y2, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("dtype", ["f32", "f64"])
@pytest.mark.parametrize("with_h0", [False, True])
def test_step_reproduces_forward_bitwise(dtype, with_h0):
    # Stepping token by token from the starting state reproduces the
    # sequence forward exactly (max_abs_diff = 0.0), on the active block.
    inp = gen.workload_inputs("s6-tiny-active-f32", with_h0=with_h0)
    t = np.float32 if dtype == "f32" else np.float64
    ref = oracle.fwd(inp, dtype)
    state = (inp.h0 if with_h0 else np.zeros((inp.B, inp.D, inp.N))).astype(t).copy()
    ys = []
    for s in range(inp.L):
        ys.append(oracle.step(state, inp.x[:, s], inp.dt[:, s], inp.z[:, s], inp.Bm[:, s],
                              inp.Cm[:, s], inp.A, inp.Dskip, inp.dt_bias, 1, dtype))
    y = np.stack(ys, axis=1)
    assert np.max(np.abs(y - ref["y"])) == 0.0
    assert np.array_equal(state, ref["h_last"])


def test_forward_composes_over_split_sequence():
    inp = small(L=30, with_h0=True)
    full = oracle.fwd(inp, "f32")
    k = 13
    first = replace(inp, L=k, x=inp.x[:, :k], dt=inp.dt[:, :k], z=inp.z[:, :k],
                    Bm=inp.Bm[:, :k], Cm=inp.Cm[:, :k])
    a = oracle.fwd(first, "f32")
    second = replace(inp, L=30 - k, x=inp.x[:, k:], dt=inp.dt[:, k:], z=inp.z[:, k:],
                     Bm=inp.Bm[:, k:], Cm=inp.Cm[:, k:], h0=a["h_last"])
    b = oracle.fwd(second, "f32")
    assert np.array_equal(np.concatenate([a["y"], b["y"]], axis=1), full["y"])
    assert np.array_equal(b["h_last"], full["h_last"])


def test_threads_do_not_change_results():
    inp = small(B=3, L=40, D=5, with_h0=True, with_dh_last=True)
    f1, f4 = oracle.fwd(inp, threads=1), oracle.fwd(inp, threads=4)
    assert np.array_equal(f1["y"], f4["y"])
    b1, b4 = oracle.bwd(inp, threads=1), oracle.bwd(inp, threads=4)
    for k in ("dx", "ddt", "dz", "dh0"):
        assert np.array_equal(b1[k], b4[k])
    for k in ("dA", "dD", "ddt_bias", "dB", "dC"):
        np.testing.assert_allclose(b1[k], b4[k], rtol=1e-12, atol=1e-14)


def test_float_oracle_tracks_double_oracle():
    inp = gen.workload_inputs("s6-tiny-active-f32")
    a, b = oracle.fwd(inp, "f32")["y"], oracle.fwd(inp, "f64")["y"]
    assert np.max(np.abs(a - b)) / np.max(np.abs(b)) < 1e-5


# ---------------------------------------------------------------- backward

def loss(inp):
    out = oracle.fwd(inp)
    val = float(np.sum(inp.dy.astype(np.float64) * out["y"]))
    if inp.dh_last is not None:
        val += float(np.sum(inp.dh_last.astype(np.float64) * out["h_last"]))
    return val


GRAD_OF = {"x": "dx", "dt": "ddt", "z": "dz", "Bm": "dB", "Cm": "dC", "A": "dA",
           "Dskip": "dD", "dt_bias": "ddt_bias", "h0": "dh0"}


def fd_grad(inp, name, idx, rel=1e-6):
    base = getattr(inp, name).astype(np.float64)
    step = rel * max(1.0, abs(base[idx]))
    vals = []
    for sgn in (+1, -1):
        arr = base.copy()
        arr[idx] += sgn * step
        vals.append(loss(replace(inp, **{name: arr})))
    return (vals[0] - vals[1]) / (2 * step)


def fd_problem():
    inp = small(B=2, L=6, D=3, N=4, seed=21, with_h0=True, with_dh_last=True)
    inp.A = random_A(3, 4, 22)
    inp.Dskip = gen.normal_f32(23, 3)
    inp.dt_bias = 0.3 * gen.normal_f32(24, 3)
    for k in ("x", "dt", "z", "Bm", "Cm", "A", "Dskip", "dt_bias", "h0", "dy", "dh_last"):
        setattr(inp, k, getattr(inp, k).astype(np.float64))
    return inp


@pytest.mark.parametrize("name", list(GRAD_OF))
def test_backward_matches_central_differences_everywhere(name):
    inp = fd_problem()
    g = oracle.bwd(inp)[GRAD_OF[name]]
    base = getattr(inp, name)
    for idx in np.ndindex(base.shape):
        fd = fd_grad(inp, name, idx)
        assert abs(g[idx] - fd) <= 1e-7 + 1e-6 * abs(fd), (name, idx, g[idx], fd)


def test_backward_without_softplus_gate_or_skip():
    inp = fd_problem()
    inp = replace(inp, z=None, Dskip=None, delta_softplus=0,
                  dt=0.05 + np.abs(inp.dt) * 0.3)
    g = oracle.bwd(inp)
    assert g["dz"] is None
    for name in ("x", "dt", "A", "Bm", "Cm", "h0", "dt_bias"):
        base = getattr(inp, name)
        for idx in list(np.ndindex(base.shape))[::3]:
            fd = fd_grad(inp, name, idx)
            assert abs(g[GRAD_OF[name]][idx] - fd) <= 1e-7 + 1e-6 * abs(fd), (name, idx)


def test_float_backward_meets_the_pages_fd_tolerance():
    # >= 30 sampled gradient elements within 5e-3 + 5e-2*|fd| (central FD),
    # the gradcheck bound of the analytic-VJP commit; here the float oracle
    # is checked against double-precision differences.
    inp = fd_problem()
    g32 = oracle.bwd(inp, "f32")
    count = 0
    for name, gname in GRAD_OF.items():
        base = getattr(inp, name)
        for idx in list(np.ndindex(base.shape))[::4]:
            fd = fd_grad(inp, name, idx)
            assert abs(float(g32[gname][idx]) - fd) <= 5e-3 + 5e-2 * abs(fd)
            count += 1
    assert count >= 30


def test_ema_gradient_closed_form():
    L, dl = 60, 0.15
    inp = ema_inputs(L, 1, [dl], gen.normal_f32(31, L))
    inp.dy = gen.normal_f32(32, L).astype(np.float64).reshape(1, L, 1)
    dx = oracle.bwd(inp)["dx"][0, :, 0]
    dy = inp.dy[0, :, 0]
    for s in range(L):
        ref = dl * sum((1 - dl) ** (t - s) * dy[t] for t in range(s, L))
        assert abs(dx[s] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_adjoint_identity_in_x():
    inp = small(B=2, L=25, D=4, N=6, seed=41)
    dx = oracle.bwd(inp)["dx"]
    dxi = gen.normal_f32(42, inp.x.size).reshape(inp.x.shape).astype(np.float64)
    jvp = oracle.fwd(replace(inp, x=dxi))["y"]  # y is linear in x when h0 = 0
    lhs = float(np.sum(inp.dy * jvp))
    rhs = float(np.sum(dx * dxi))
    assert abs(lhs - rhs) <= 1e-11 * max(1.0, abs(lhs))


def test_dA_log_chain_rule():
    # A = -exp(A_log)  =>  dLoss/dA_log = dA * A
    inp = fd_problem()
    A_log = np.log(-inp.A)
    dA = oracle.bwd(inp)["dA"]
    for idx in np.ndindex(A_log.shape):
        h = 1e-6
        lp = A_log.copy(); lp[idx] += h
        lm = A_log.copy(); lm[idx] -= h
        fd = (loss(replace(inp, A=-np.exp(lp))) - loss(replace(inp, A=-np.exp(lm)))) / (2 * h)
        assert abs(dA[idx] * inp.A[idx] - fd) <= 1e-7 + 1e-6 * abs(fd)


def test_canonical_init_stays_finite_and_blowup_is_visible():
    # Canonical S6 init: A = -(1..N), softplus(dt_bias) = 0.01, D = 1.
    inp = gen.make_inputs(1, 4096, 8, 16, seed=3, dt_std=1.0, delta_target=0.01)
    f = oracle.fwd(inp, "f32")
    g = oracle.bwd(inp, "f32")
    assert np.all(np.isfinite(f["y"])) and np.all(np.isfinite(f["h_last"]))
    for k, v in g.items():
        if v is not None:
            assert np.all(np.isfinite(v)), k
    # Contrast: a negative Delta (no softplus) turns exp(Delta*A) into growth
    # and the trajectory overflows -- the oracle does not hide it.
    bad = replace(inp, delta_softplus=0, dt_bias=None, dt=np.full_like(inp.dt, -3.0))
    assert not np.all(np.isfinite(oracle.fwd(bad, "f32")["y"]))
