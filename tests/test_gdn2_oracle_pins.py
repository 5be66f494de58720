"""Pins of the Gated DeltaNet-2 chunkwise-forward oracle (oracle/gdn2_oracle.py)
against what the page's method fixes and against mathematics, not against
itself:

* chunks of one token reduce the chunked steps to the per-token form
  (derived from the steps, evaluated by a separate loop);
* with key-uniform gates, or a single key channel, the intra-chunk key-mean
  of the decays is exact, so every chunk size gives the per-token result;
* with no erase (b = 0) and no decay (g = 0) the mixer is linear
  attention: o_t = scale * q_t (S0 + sum_{s<=t} k_s (w_s v_s)^T);
* a run split at a chunk boundary, the state carried over, equals one run;
* permuting key channels (q, k, g, b together) leaves the output unchanged,
  and permuting value channels (v, w, state columns) permutes it;
* the scale enters the output linearly when the initial state is zero.
Each of these fails for a dropped term, a wrong sign, a transposed operand
or an off-by-one in the masks or the substitution order."""
import numpy as np
import pytest

import gen
from oracle import gdn2_oracle as G


def args(x):
    return (x.q, x.k, x.v, x.g, x.b, x.w, x.state, x.scale)


def rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


@pytest.mark.parametrize("T", [1, 7, 20])
def test_chunks_of_one_token_are_the_per_token_form(T):
    x = gen.make_gdn2_inputs(2, 2, T, 6, 5, seed=T, io="f32")
    o1, s1 = G.chunk_wy_forward(*args(x), chunk=1)
    o2, s2 = G.recurrent(*args(x))
    assert rel(o1, o2) < 1e-12 and rel(s1, s2) < 1e-12


@pytest.mark.parametrize("chunk", [2, 3, 8, 16, 40])
def test_key_uniform_gates_give_the_per_token_result_for_every_chunk_size(chunk):
    x = gen.make_gdn2_inputs(1, 3, 40, 8, 6, seed=3, io="f32", key_uniform_gates=True)
    o1, s1 = G.chunk_wy_forward(*args(x), chunk=chunk)
    o2, s2 = G.recurrent(*args(x))
    assert rel(o1, o2) < 1e-10 and rel(s1, s2) < 1e-10


@pytest.mark.parametrize("chunk", [4, 16])
def test_a_single_key_channel_gives_the_per_token_result(chunk):
    x = gen.make_gdn2_inputs(2, 1, 33, 1, 4, seed=5, io="f32")
    o1, s1 = G.chunk_wy_forward(*args(x), chunk=chunk)
    o2, s2 = G.recurrent(*args(x))
    assert rel(o1, o2) < 1e-10 and rel(s1, s2) < 1e-10


def test_no_erase_and_no_decay_is_linear_attention():
    x = gen.make_gdn2_inputs(1, 2, 30, 5, 4, seed=7, io="f32")
    x.b[:] = 0.0
    x.g[:] = 0.0
    o, s = G.chunk_wy_forward(*args(x), chunk=8)
    q, k, v, w = (a.astype(np.float64) for a in (x.q, x.k, x.v, x.w))
    S = x.state.astype(np.float64).copy()
    for t in range(x.T):
        S = S + k[:, :, t, :, None] * (w[:, :, t] * v[:, :, t])[:, :, None, :]
        ref = x.scale * np.einsum("bhk,bhkv->bhv", q[:, :, t], S)
        assert rel(o[:, :, t], ref) < 1e-12
    assert rel(s, S) < 1e-12


def test_a_run_split_at_a_chunk_boundary_chains_through_the_state():
    x = gen.make_gdn2_inputs(1, 2, 48, 6, 5, seed=9, io="f32")
    o, s = G.chunk_wy_forward(*args(x), chunk=16)
    cut = 32
    sl = lambda a, lo, hi: a[:, :, lo:hi]  # noqa: E731
    oa, sa = G.chunk_wy_forward(sl(x.q, 0, cut), sl(x.k, 0, cut), sl(x.v, 0, cut), sl(x.g, 0, cut), sl(x.b, 0, cut),
                                sl(x.w, 0, cut), x.state, x.scale, chunk=16)
    ob, sb = G.chunk_wy_forward(sl(x.q, cut, 48), sl(x.k, cut, 48), sl(x.v, cut, 48), sl(x.g, cut, 48),
                                sl(x.b, cut, 48), sl(x.w, cut, 48), sa, x.scale, chunk=16)
    assert rel(np.concatenate([oa, ob], axis=2), o) < 1e-13 and rel(sb, s) < 1e-13


def test_channel_permutations():
    x = gen.make_gdn2_inputs(1, 2, 25, 7, 5, seed=13, io="f32")
    o, s = G.chunk_wy_forward(*args(x), chunk=8)
    pk = np.random.default_rng(1).permutation(x.K)
    pv = np.random.default_rng(2).permutation(x.V)
    op, sp = G.chunk_wy_forward(x.q[..., pk], x.k[..., pk], x.v[..., pv], x.g[..., pk], x.b[..., pk], x.w[..., pv],
                                x.state[:, :, pk][:, :, :, pv], x.scale, chunk=8)
    assert rel(op, o[..., pv]) < 1e-12
    assert rel(sp, s[:, :, pk][:, :, :, pv]) < 1e-12


def test_scale_is_linear_from_a_zero_state():
    x = gen.make_gdn2_inputs(1, 1, 20, 4, 3, seed=15, io="f32", with_state=False)
    o1, _ = G.chunk_wy_forward(*args(x), chunk=8)
    a = list(args(x))
    a[-1] = 2.5 * x.scale
    o2, _ = G.chunk_wy_forward(*a, chunk=8)
    assert rel(o2, 2.5 * o1) < 1e-13


def test_channel_varying_gates_make_the_result_depend_on_the_chunk_size():
    # the key-mean of step 2 is an approximation of the per-channel decays:
    # with channel-varying gates chunk sizes disagree (slightly), while with
    # key-uniform gates they do not (above) -- the oracle does not hide it
    x = gen.make_gdn2_inputs(1, 2, 32, 8, 4, seed=17, io="f32")
    o1, _ = G.chunk_wy_forward(*args(x), chunk=1)
    o16, _ = G.chunk_wy_forward(*args(x), chunk=16)
    d = rel(o16, o1)
    assert 1e-6 < d < 0.5
