"""ssm_step against the sequence forward: stepping token by token from the
state the forward started from (or from any checkpoint it saved)
reproduces the forward's outputs bit for bit ("max_abs_diff = 0.0", the
MambaRecurrence commit), for every lane split of either side."""
import numpy as np
import pytest

import gen
import oracle
from _util import TOL, rel_err, run_fwd, to_dev, to_np

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def ssm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import selective_state_space_07_gb300 as m
    m.build()
    return m


def step_through(ssm, dv, state, t0, t1, nsplit):
    ys = []
    for t in range(t0, t1):
        ys.append(ssm.step(state, dv["x"][:, t].contiguous(), dv["dt"][:, t].contiguous(), dv["A"],
                           dv["Bm"][:, t].contiguous(), dv["Cm"][:, t].contiguous(),
                           None if dv["z"] is None else dv["z"][:, t].contiguous(), dv["Dskip"], dv["dt_bias"],
                           nsplit=nsplit))
    return torch.stack(ys, dim=1)


@pytest.mark.parametrize("fwd_split,step_split", [(1, 1), (2, 4), (4, 1), (4, 2)])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_step_from_zero_is_bitwise_the_forward(ssm, fwd_split, step_split, io):
    w = gen.WORKLOADS["s6-tiny-active-f32"]
    inp = gen.make_inputs(w.B, w.L, w.D, w.N, io=io, seed=w.seed, dt_std=w.dt_std, delta_target=w.delta_target)
    dv = to_dev(inp)
    y, h_last, _, _ = run_fwd(ssm, dv, inp, nsplit=fwd_split, groups=1)
    state = torch.zeros(inp.B, inp.D, 16, device="cuda")
    ys = step_through(ssm, dv, state, 0, inp.L, step_split)
    torch.cuda.synchronize()
    assert torch.equal(ys, y), float((ys.float() - y.float()).abs().max())
    assert torch.equal(state, h_last)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_step_from_zero_is_bitwise_a_wide_single_group_forward(ssm, io):
    # one L-group over 2 x 7656 channels (240 forward CTAs, the last of each
    # batch row ragged): the step form reproduces it bit for bit
    inp = gen.make_inputs(2, 24, 7656, 16, io=io, seed=78)
    dv = to_dev(inp)
    y, h_last, _, _ = run_fwd(ssm, dv, inp, groups=1)
    state = torch.zeros(inp.B, inp.D, 16, device="cuda")
    ys = step_through(ssm, dv, state, 0, inp.L, 1)
    torch.cuda.synchronize()
    assert torch.equal(ys, y), float((ys.float() - y.float()).abs().max())
    assert torch.equal(state, h_last)


def test_step_from_every_checkpoint_is_bitwise_the_forward(ssm):
    # A forward split into 3 L-groups of 32 tokens: stepping from any saved
    # checkpoint (one every 8 tokens; ckpt_states gives them as [B, L/8, D, N])
    # reproduces those tokens' outputs exactly, and the state it reaches
    # equals the next checkpoint exactly inside a group. A group's first
    # checkpoint comes from the carry scan over groups, which re-associates
    # the products, so there it agrees to rounding only.
    K = ssm.CKPT_INTERVAL
    inp = gen.make_inputs(2, 96, 64, 16, io="bf16", seed=17, with_h0=True)
    dv = to_dev(inp)
    y, h_last, ckpt, _ = run_fwd(ssm, dv, inp, nsplit=2, groups=3)
    nck = 96 // K
    ck = ssm.ckpt_states(ckpt, 2, 96, 64)  # -> [B, nck, D, N]
    group_starts = {0, 32 // K, 64 // K}
    for c in range(nck):
        state = ck[:, c].contiguous().clone()
        ys = step_through(ssm, dv, state, K * c, K * c + K, 4)
        assert torch.equal(ys, y[:, K * c:K * c + K])
        nxt = ck[:, c + 1] if c < nck - 1 else h_last
        if c + 1 in group_starts:
            assert rel_err(to_np(state), to_np(nxt)) < 1e-5
        else:
            assert torch.equal(state, nxt), c
    assert torch.equal(ck[:, 0], dv["h0"])


def test_step_matches_the_oracle_step(ssm):
    inp = gen.workload_inputs("s6-small-f32", with_h0=True)
    dv = to_dev(inp)
    state = dv["h0"].clone()
    ref_state = inp.h0.astype(np.float64).copy()
    for t in range(3):
        y = ssm.step(state, dv["x"][:, t].contiguous(), dv["dt"][:, t].contiguous(), dv["A"],
                     dv["Bm"][:, t].contiguous(), dv["Cm"][:, t].contiguous(), dv["z"][:, t].contiguous(),
                     dv["Dskip"], dv["dt_bias"])
        ry = oracle.step(ref_state, inp.x[:, t], inp.dt[:, t], inp.z[:, t], inp.Bm[:, t], inp.Cm[:, t], inp.A,
                         inp.Dskip, inp.dt_bias)
        assert rel_err(to_np(y), ry) < TOL[("f32", "fwd")]
    assert rel_err(to_np(state), ref_state) < TOL[("f32", "fwd")]


def test_forward_is_deterministic(ssm):
    inp = gen.make_inputs(2, 200, 128, 16, io="bf16", seed=23)
    dv = to_dev(inp)
    a = run_fwd(ssm, dv, inp)[0].clone()
    b = run_fwd(ssm, dv, inp)[0].clone()
    assert torch.equal(a, b)
