"""Edge cases on the GPU: empty and ragged shapes, optional inputs absent,
Delta without softplus, in-place gradients, the non-finite status flag,
the A_log chain rule, canonical-init finiteness, and argument errors."""
import numpy as np
import pytest

import gen
import oracle
from _util import GRAD_KEYS, TOL, rel_err, run_bwd, run_fwd, to_dev, to_np

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def ssm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import selective_state_space_07_gb300 as m
    m.build()
    return m


def compare(ssm, inp, io, fwd_kw=None, bwd_kw=None):
    dv = to_dev(inp)
    y, h_last, ckpt, ws = run_fwd(ssm, dv, inp, **(fwd_kw or {}))
    g = run_bwd(ssm, dv, inp, ckpt, workspace=ws, **(bwd_kw or {}))
    rf, rb = oracle.fwd(inp), oracle.bwd(inp)
    assert rel_err(to_np(y), rf["y"]) <= TOL[(io, "fwd")]
    assert rel_err(to_np(h_last), rf["h_last"]) <= TOL[(io, "fwd")]
    for mine, theirs in GRAD_KEYS:
        if rb.get(theirs) is not None and g.get(mine) is not None:
            assert rel_err(to_np(g[mine]), rb[theirs]) <= TOL[(io, "bwd")], mine
    return dv, g


@pytest.mark.parametrize("L", [1, 2, 15, 16, 17, 31, 33, 100])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_ragged_lengths(ssm, L, io):
    inp = gen.make_inputs(2, L, 24, 16, io=io, seed=L, with_h0=True, with_dh_last=True)
    compare(ssm, inp, io, dict(groups=0), dict(groups=0))
    compare(ssm, inp, io, dict(groups=2, nsplit=1), dict(groups=2, nsplit=2))


@pytest.mark.parametrize("regime", ["no decay", "fast decay", "slow decay"])
@pytest.mark.parametrize("groups", [3, 5])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_carries_across_decay_regimes(ssm, regime, groups, io):
    # the L-group aggregates take the product of a group's decays as exp(A
    # times a running sum of Delta): states that never decay (A = 0, the
    # carries are plain sums over the group), decays that underflow within a
    # few tokens (Delta ~ 5) and decays that barely act (Delta ~ 1e-4), each
    # against the oracle's sequential recurrence, with ragged groups
    target = {"no decay": 0.05, "fast decay": 5.0, "slow decay": 1e-4}[regime]
    inp = gen.make_inputs(2, 300, 40, 16, io=io, seed=groups, dt_std=0.5, delta_target=target,
                          with_h0=True, with_dh_last=True)
    if regime == "no decay":
        inp.A[:, :5] = 0.0
    compare(ssm, inp, io, dict(groups=groups), dict(groups=groups))


@pytest.mark.parametrize("D", [8, 40, 136, 264])
def test_partial_channel_tiles(ssm, D):
    inp = gen.make_inputs(2, 40, D, 16, io="bf16", seed=D)
    for ns in (1, 2, 4):
        compare(ssm, inp, "bf16", dict(nsplit=ns), dict(nsplit=ns))


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_single_group_forward_over_a_wide_channel_grid(ssm, io):
    # 2 x 7656 channels: 240 forward CTAs of 64 channels in one L-group
    # (between one and two per SM on a 152-SM GB300), the last CTA of each
    # batch row ragged (40 of its 64 channels live)
    inp = gen.make_inputs(2, 40, 7656, 16, io=io, seed=77, with_h0=True, with_dh_last=True)
    compare(ssm, inp, io, dict(groups=0), dict(groups=0))


@pytest.mark.parametrize("gate,skip,bias", [(False, True, True), (True, False, True), (True, True, False),
                                            (False, False, False)])
def test_optional_inputs_absent(ssm, gate, skip, bias):
    inp = gen.make_inputs(2, 50, 32, 16, io="f32", seed=5, gate=gate, skip=skip, bias=bias)
    compare(ssm, inp, "f32")


def test_delta_without_softplus(ssm):
    inp = gen.make_inputs(2, 64, 32, 16, io="f32", seed=6, bias=False)
    inp.delta_softplus = 0
    inp.dt = (0.02 + 0.3 * gen.uniform53(61, inp.dt.size).reshape(inp.dt.shape)).astype(np.float32)
    compare(ssm, inp, "f32")


def test_in_place_gradients(ssm):
    inp = gen.make_inputs(2, 70, 48, 16, io="bf16", seed=8)
    dv = to_dev(inp)
    y, _, ckpt, ws = run_fwd(ssm, dv, inp)
    ref = run_bwd(ssm, dv, inp, ckpt, workspace=ws)
    ref = {k: v.clone() for k, v in ref.items() if isinstance(v, torch.Tensor)}
    dy, z, dt = dv["dy"].clone(), dv["z"].clone(), dv["dt"].clone()
    dvi = dict(dv, dy=dy, z=z, dt=dt)
    g = run_bwd(ssm, dvi, inp, ckpt, workspace=ws, inplace=True)
    assert g["dx"].data_ptr() == dy.data_ptr() and g["dz"].data_ptr() == z.data_ptr()
    assert g["d_dt"].data_ptr() == dt.data_ptr()
    for k in ("dx", "dz", "d_dt"):
        assert torch.equal(g[k], ref[k]), k
    for k in ("dA", "dD", "d_dt_bias", "dB", "dC"):
        assert rel_err(to_np(g[k]), to_np(ref[k])) < 1e-5, k


def test_empty_shapes(ssm):
    dev = "cuda"
    for B, L, D in ((0, 10, 16), (2, 0, 16), (2, 10, 0)):
        x = torch.zeros(B, L, D, device=dev)
        dt = torch.zeros(B, L, D, device=dev)
        A = -torch.ones(D, 16, device=dev)
        Bm = torch.zeros(B, L, 16, device=dev)
        h0 = torch.randn(B, D, 16, device=dev)
        y, h_last, ckpt, ws = ssm.scan_fwd(x, dt, A, Bm, Bm, h0=h0, return_last_state=True)
        assert y.shape == (B, L, D)
        if L == 0:
            assert torch.equal(h_last, h0)
        dh_last = torch.randn(B, D, 16, device=dev)
        g = ssm.scan_bwd(x, dt, A, Bm, Bm, x, ckpt, h0=h0, dh_last=dh_last, return_dh0=True, workspace=ws)
        torch.cuda.synchronize()
        assert float(g["dA"].abs().sum()) == 0.0 and float(g["dD"].abs().sum()) == 0.0
        if L == 0:
            assert torch.equal(g["dh0"], dh_last)


def test_nonfinite_outputs_are_flagged(ssm):
    # Delta < 0 without softplus turns exp(Delta*A) into growth: h overflows.
    inp = gen.make_inputs(1, 400, 16, 16, io="f32", seed=3, bias=False)
    inp.delta_softplus = 0
    inp.dt = np.full_like(inp.dt, -3.0)
    dv = to_dev(inp)
    _, _, _, ws = run_fwd(ssm, dv, inp)
    assert ssm.poll_status(ws) == -7
    assert ssm.poll_status(ws) == 0  # polling clears the word
    ok = gen.make_inputs(1, 400, 16, 16, io="f32", seed=3)
    dvo = to_dev(ok)
    _, _, _, ws2 = run_fwd(ssm, dvo, ok, workspace=ws)
    assert ssm.poll_status(ws2) == 0


@pytest.mark.parametrize("groups", [1, 3])
def test_bounded_wait_expiry_is_reported_and_the_context_stays_usable(ssm, groups):
    # The testing hook arms tile 1 of every warp of the next forward's main
    # kernel without issuing its copies and bounds the waits by 1 ms: the
    # waits run out, the warps drain the copies they have in flight and
    # leave, and the status word says so. The same workspace then serves a
    # normal call, whose results are exact again.
    inp = gen.make_inputs(2, 160, 64, 16, io="f32", seed=21, with_h0=True)
    dv = to_dev(inp)
    y_ref, h_ref, _, ws = run_fwd(ssm, dv, inp, groups=groups)
    assert ssm.poll_status(ws) == 0
    ssm.arm_wait_fault(1, 1_000_000)
    run_fwd(ssm, dv, inp, groups=groups, workspace=ws)
    assert ssm.poll_status(ws) == -6
    assert ssm.poll_status(ws) == 0  # polling clears the word
    y, h_last, _, ws = run_fwd(ssm, dv, inp, groups=groups, workspace=ws)  # the hook was one-shot
    assert ssm.poll_status(ws) == 0
    assert torch.equal(y, y_ref) and torch.equal(h_last, h_ref)


def test_canonical_init_is_finite_at_length_4096(ssm):
    inp = gen.make_inputs(1, 4096, 64, 16, io="bf16", seed=4, dt_std=1.0, delta_target=0.01)
    dv = to_dev(inp)
    y, h_last, ckpt, ws = run_fwd(ssm, dv, inp)
    g = run_bwd(ssm, dv, inp, ckpt, workspace=ws)
    assert ssm.poll_status(ws) == 0
    assert torch.isfinite(y.float()).all() and torch.isfinite(h_last).all()
    for k, v in g.items():
        if isinstance(v, torch.Tensor) and v.dtype != torch.uint8:
            assert torch.isfinite(v.float()).all(), k


def test_dA_log_chain_rule(ssm):
    # dA_log = dA * A (A = -exp(A_log)): the GPU's dA of a real backward,
    # taken through ssm_dA_log_grad, against the fp64 oracle's dA times A
    inp = gen.make_inputs(2, 200, 48, 16, io="f32", seed=9, with_h0=True, with_dh_last=True)
    dv = to_dev(inp)
    _, _, ckpt, ws = run_fwd(ssm, dv, inp)
    g = run_bwd(ssm, dv, inp, ckpt, workspace=ws)
    out = ssm.dA_log_grad(g["dA"], dv["A"])
    ref = oracle.bwd(inp)["dA"] * inp.A.astype(np.float64)
    assert rel_err(to_np(out), ref) <= TOL[("f32", "bwd")]
    # elementwise it is one rounded product, in place too
    dA = g["dA"].clone()
    assert torch.equal(ssm.dA_log_grad(dA, dv["A"], out=dA), g["dA"] * dv["A"])


def test_launch_counts(ssm):
    inp = gen.make_inputs(1, 64, 32, 16, io="f32", seed=1)
    dv = to_dev(inp)
    _, _, ckpt, ws = run_fwd(ssm, dv, inp, groups=1)
    assert ssm.last_launch_count() == 1
    _, _, ckpt, ws = run_fwd(ssm, dv, inp, groups=4)
    assert ssm.last_launch_count() == 3  # aggregate, carry scan, main
    run_bwd(ssm, dv, inp, ckpt, workspace=ws, groups=4)
    assert ssm.last_launch_count() == 3


def test_binding_argument_errors(ssm):
    x = torch.zeros(1, 8, 16, device="cuda")
    dt = torch.zeros(1, 8, 16, device="cuda")
    A = -torch.ones(16, 16, device="cuda")
    Bm = torch.zeros(1, 8, 16, device="cuda")
    with pytest.raises(TypeError):
        ssm.scan_fwd(x.double(), dt, A, Bm, Bm)
    with pytest.raises(ValueError):
        ssm.scan_fwd(x.transpose(1, 2).contiguous().transpose(1, 2), dt, A, Bm, Bm)
    with pytest.raises(ValueError):
        ssm.scan_fwd(x, dt, A, torch.zeros(1, 8, 8, device="cuda"), Bm)
    with pytest.raises(ssm.SsmError) as e:  # consistent shapes, but d_state 8
        ssm.scan_fwd(x, dt, -torch.ones(16, 8, device="cuda"), torch.zeros(1, 8, 8, device="cuda"),
                     torch.zeros(1, 8, 8, device="cuda"))
    assert e.value.code == -2
    x12 = torch.zeros(1, 8, 12, device="cuda")
    with pytest.raises(ssm.SsmError) as e:
        ssm.scan_fwd(x12, torch.zeros(1, 8, 12, device="cuda"), -torch.ones(12, 16, device="cuda"), Bm, Bm)
    assert e.value.code == -3
