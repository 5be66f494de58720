"""Pins of the mLSTM oracle (oracle/mlstm_oracle.py) against what the page
fixes and against mathematics, not against itself:

* the parallel form equals the recurrent step (the page's equivalence,
  checked there for sequence lengths 1-12);
* the chunked evaluation equals the recurrent step for every chunk size,
  from a nonzero stabilized state, with a ragged last chunk;
* both equal the unstabilized definition (no m, no exponent differences),
  and their final states are the plain ones times exp(-m);
* the stabilizer's start value changes no output (the page's m_state fix);
* closed forms: one token; f = 1 and i = 1 (cumulative sums); a closed
  input gate (the state only decays);
* input gates far beyond exp's range keep the stabilized forms finite and
  in agreement;
* a run split at a chunk boundary, the state carried over, equals one run;
  outputs are causal;
* the head-wise layer norm: zero mean and unit variance per row with unit
  weights, invariance to a positive scale of its input, weights per
  channel.
Each of these fails for a dropped term, a wrong sign, a transposed operand,
an off-by-one in the causal mask or a misplaced stabilizer."""
import numpy as np
import pytest

import gen
from oracle import mlstm_oracle as M


def rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def make(B, H, T, K, V, seed, **kw):
    return gen.make_mlstm_inputs(B, H, T, K, V, seed=seed, io="f32", **kw)


@pytest.mark.parametrize("T", list(range(1, 13)))
def test_parallel_form_equals_the_recurrent_step(T):
    x = make(2, 2, T, 8, 6, seed=T, with_state=False)
    h_par = M.parallel(x.q, x.k, x.v, x.igate, x.fgate)
    h_rec, _, _, _ = M.recurrent(x.q, x.k, x.v, x.igate, x.fgate)
    assert rel(h_par, h_rec) < 1e-12


@pytest.mark.parametrize("chunk", [1, 3, 8, 16, 64])
def test_chunked_evaluation_equals_the_recurrent_step(chunk):
    x = make(2, 3, 45, 8, 5, seed=11)
    st = (x.C0, x.n0, x.m0)
    h1, C1, n1, m1 = M.chunkwise(x.q, x.k, x.v, x.igate, x.fgate, *st, chunk=chunk)
    h2, C2, n2, m2 = M.recurrent(x.q, x.k, x.v, x.igate, x.fgate, *st)
    assert rel(h1, h2) < 1e-12 and rel(C1, C2) < 1e-12 and rel(n1, n2) < 1e-12
    assert np.allclose(m1, m2, rtol=0, atol=1e-12)


def test_stabilized_forms_equal_the_plain_definition():
    x = make(1, 2, 30, 6, 4, seed=5)
    e0 = np.exp(x.m0.astype(np.float64))
    hp, Cp, npl = M.plain(x.q, x.k, x.v, x.igate, x.fgate, x.C0 * e0[..., None, None], x.n0 * e0[..., None])
    for h, C, n, m in (M.recurrent(x.q, x.k, x.v, x.igate, x.fgate, x.C0, x.n0, x.m0),
                       M.chunkwise(x.q, x.k, x.v, x.igate, x.fgate, x.C0, x.n0, x.m0, chunk=8)):
        assert rel(h, hp) < 1e-12
        em = np.exp(m)
        assert rel(C * em[..., None, None], Cp) < 1e-12 and rel(n * em[..., None], npl) < 1e-12


@pytest.mark.parametrize("m0", [-30.0, 5.0])
def test_the_stabilizer_start_changes_no_output(m0):
    # section 3 of the page moves m's start from -30 to 0: with a zero state
    # the outputs agree, and the final states agree as C * exp(m)
    x = make(2, 2, 25, 6, 4, seed=9, with_state=False)
    h0, C0, n0, mm0 = M.recurrent(x.q, x.k, x.v, x.igate, x.fgate)
    h1, C1, n1, mm1 = M.recurrent(x.q, x.k, x.v, x.igate, x.fgate, m0=np.full((2, 2), m0))
    assert rel(h1, h0) < 1e-12
    assert rel(C1 * np.exp(mm1)[..., None, None], C0 * np.exp(mm0)[..., None, None]) < 1e-12


def test_single_token_closed_form():
    x = make(1, 1, 1, 5, 3, seed=2, with_state=False)
    q, k, v = (a[0, 0, 0].astype(np.float64) for a in (x.q, x.k, x.v))
    i = np.exp(np.float64(x.igate[0, 0, 0]))
    s = float(q @ k) * x.scale
    want = i * s * v / max(abs(i * s), 1.0)
    for h in (M.recurrent(x.q, x.k, x.v, x.igate, x.fgate)[0], M.parallel(x.q, x.k, x.v, x.igate, x.fgate),
              M.chunkwise(x.q, x.k, x.v, x.igate, x.fgate)[0]):
        assert rel(h[0, 0, 0], want) < 1e-13


def test_open_forget_and_unit_input_gates_give_cumulative_sums():
    # f = 1 (log sigmoid(60) = -9e-27), i = 1: C_t = sum_{s<=t} k_s v_s^T, n_t = sum k_s
    x = make(1, 2, 20, 6, 4, seed=4, with_state=False)
    x.fgate[:] = 60.0
    x.igate[:] = 0.0
    q, k, v = (a.astype(np.float64) for a in (x.q, x.k, x.v))
    Cs = np.cumsum(k[..., :, None] * v[..., None, :], axis=2)
    ns = np.cumsum(k, axis=2)
    qs = q * x.scale
    want = np.einsum("bhtk,bhtkv->bhtv", qs, Cs) / np.maximum(np.abs(np.einsum("bhtk,bhtk->bht", qs, ns)), 1.0)[..., None]
    for h in (M.recurrent(x.q, x.k, x.v, x.igate, x.fgate)[0], M.parallel(x.q, x.k, x.v, x.igate, x.fgate),
              M.chunkwise(x.q, x.k, x.v, x.igate, x.fgate, chunk=7)[0]):
        assert rel(h, want) < 1e-12


def test_a_closed_input_gate_only_decays_the_state():
    x = make(1, 2, 16, 6, 4, seed=6)
    x.igate[:] = -1e4  # i = 0
    e0 = np.exp(x.m0.astype(np.float64))
    C0, n0 = x.C0 * e0[..., None, None], x.n0 * e0[..., None]
    f = 1.0 / (1.0 + np.exp(-x.fgate.astype(np.float64)))
    Fc = np.cumprod(f, axis=2)
    qs = x.q.astype(np.float64) * x.scale
    num = Fc[..., None] * np.einsum("bhtk,bhkv->bhtv", qs, C0)
    den = Fc * np.einsum("bhtk,bhk->bht", qs, n0)
    want = num / np.maximum(np.abs(den), 1.0)[..., None]
    for h in (M.recurrent(x.q, x.k, x.v, x.igate, x.fgate, x.C0, x.n0, x.m0)[0],
              M.chunkwise(x.q, x.k, x.v, x.igate, x.fgate, x.C0, x.n0, x.m0, chunk=5)[0]):
        assert rel(h, want) < 1e-12


def test_input_gates_beyond_the_exponential_range_stay_finite():
    # exp(800) overflows float64: only the stabilized forms can evaluate these
    x = make(1, 2, 40, 6, 4, seed=8, with_state=False, igate_mean=800.0)
    h_rec, C, n, m = M.recurrent(x.q, x.k, x.v, x.igate, x.fgate)
    h_par = M.parallel(x.q, x.k, x.v, x.igate, x.fgate)
    h_chk = M.chunkwise(x.q, x.k, x.v, x.igate, x.fgate, chunk=16)[0]
    assert np.isfinite(h_rec).all() and np.isfinite(C).all() and np.isfinite(n).all()
    # exponent differences of values near 800 carry ~800 * 2^-52 absolute error
    assert rel(h_par, h_rec) < 1e-10 and rel(h_chk, h_rec) < 1e-10
    # with |q . n| far above 1 (i ~ e^10 here) the output does not depend on
    # a common factor of the input gates: the same gates shifted by -790
    # give it through the plain definition
    hp, _, _ = M.plain(x.q, x.k, x.v, x.igate.astype(np.float64) - 790.0, x.fgate)
    assert rel(h_rec, hp) < 1e-9


def test_a_split_run_chains_through_the_state():
    x = make(1, 2, 150, 6, 4, seed=10)
    h, C, n, m = M.chunkwise(x.q, x.k, x.v, x.igate, x.fgate, x.C0, x.n0, x.m0, chunk=16)
    cut = 64
    a = lambda t, lo, hi: t[:, :, lo:hi]  # noqa: E731
    ha, Ca, na, ma = M.chunkwise(a(x.q, 0, cut), a(x.k, 0, cut), a(x.v, 0, cut), a(x.igate, 0, cut),
                                 a(x.fgate, 0, cut), x.C0, x.n0, x.m0, chunk=16)
    hb, Cb, nb, mb = M.chunkwise(a(x.q, cut, 150), a(x.k, cut, 150), a(x.v, cut, 150), a(x.igate, cut, 150),
                                 a(x.fgate, cut, 150), Ca, na, ma, chunk=16)
    assert rel(np.concatenate([ha, hb], axis=2), h) < 1e-12 and rel(Cb, C) < 1e-12 and rel(nb, n) < 1e-12


def test_outputs_are_causal():
    x = make(1, 1, 30, 5, 3, seed=12)
    h1 = M.chunkwise(x.q, x.k, x.v, x.igate, x.fgate, x.C0, x.n0, x.m0, chunk=8)[0]
    for a in (x.q, x.k, x.v):
        a[:, :, 20:] += 1.0
    x.igate[:, :, 20:] += 3.0
    x.fgate[:, :, 20:] -= 2.0
    h2 = M.chunkwise(x.q, x.k, x.v, x.igate, x.fgate, x.C0, x.n0, x.m0, chunk=8)[0]
    assert np.array_equal(h1[:, :, :20], h2[:, :, :20]) and not np.allclose(h1[:, :, 20:], h2[:, :, 20:])


def test_head_layer_norm():
    rng = np.random.default_rng(3)
    h = rng.normal(size=(2, 3, 7, 16)) * 4.0 + 1.5
    ones = np.ones((3, 16))
    y = M.head_layer_norm(h, ones, eps=0.0)
    assert np.allclose(y.mean(axis=-1), 0.0, atol=1e-12) and np.allclose(y.var(axis=-1), 1.0, rtol=1e-12)
    assert np.allclose(M.head_layer_norm(3.7 * h, ones, eps=0.0), y, rtol=1e-12, atol=1e-12)
    w = rng.normal(size=(3, 16))
    assert np.allclose(M.head_layer_norm(h, w, eps=0.0), y * w[None, :, None, :], rtol=1e-12, atol=1e-12)
    # eps shrinks every row by sqrt(var / (var + eps))
    ye = M.head_layer_norm(h, ones, eps=0.5)
    var = h.var(axis=-1, keepdims=True)
    assert np.allclose(ye, y * np.sqrt(var / (var + 0.5)), rtol=1e-12, atol=1e-12)
