"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs, element by element, for the forward (y, h_last)
and every gradient (dx, dz, d_dt, dA, dD, d_dt_bias, dB, dC, dh0).

Tolerance, per tensor, max|got - ref| / max|ref|: fp32 forward 1e-4, fp32
gradients 1e-3, bf16 2e-2 (oracle fed the same bf16-rounded inputs)."""
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


def check_all(ssm, inp, tol_io, fwd_kw=None, bwd_kw=None):
    dv = to_dev(inp)
    y, h_last, ckpt, ws = run_fwd(ssm, dv, inp, **(fwd_kw or {}))
    g = run_bwd(ssm, dv, inp, ckpt, workspace=ws, **(bwd_kw or {}))
    assert ssm.poll_status(ws) == 0
    rf, rb = oracle.fwd(inp), oracle.bwd(inp)
    errs = {"y": rel_err(to_np(y), rf["y"]), "h_last": rel_err(to_np(h_last), rf["h_last"])}
    for mine, theirs in GRAD_KEYS:
        if rb.get(theirs) is None:
            continue
        errs[mine] = rel_err(to_np(g[mine]), rb[theirs])
    tf, tb = TOL[(tol_io, "fwd")], TOL[(tol_io, "bwd")]
    bad = {k: v for k, v in errs.items() if v > (tf if k in ("y", "h_last") else tb)}
    assert not bad, f"over tolerance: {bad} (all: {errs})"
    return errs


SHAPES = [(1, 1), (2, 1), (4, 1), (1, 2), (2, 3), (4, 4), (1, 0), (4, 0)]


@pytest.mark.parametrize("nsplit,groups", SHAPES)
def test_tiny_active_block_every_launch_shape(ssm, nsplit, groups):
    inp = gen.workload_inputs("s6-tiny-active-f32", with_h0=True, with_dh_last=True)
    check_all(ssm, inp, "f32", dict(nsplit=nsplit, groups=groups), dict(nsplit=nsplit, groups=groups))


@pytest.mark.parametrize("nsplit,groups", [(0, 0), (1, 1), (2, 5), (4, 32)])
def test_small_fp32(ssm, nsplit, groups):
    inp = gen.workload_inputs("s6-small-f32")
    check_all(ssm, inp, "f32", dict(nsplit=nsplit, groups=groups), dict(nsplit=nsplit, groups=groups))


@pytest.mark.parametrize("nsplit,groups", [(0, 0), (1, 3), (2, 1), (4, 7)])
def test_small_bf16_ragged(ssm, nsplit, groups):
    # several channel tiles with a partial last tile, ragged L, random h0/dh_last
    inp = gen.make_inputs(3, 333, 104, 16, io="bf16", seed=9, with_h0=True, with_dh_last=True)
    check_all(ssm, inp, "bf16", dict(nsplit=nsplit, groups=groups), dict(nsplit=nsplit, groups=groups))


@pytest.mark.parametrize("name", ["mamba130m-bf16", "mamba1.4b-bf16", "long65k-bf16"])
def test_full_size_workloads(ssm, name):
    # full-size inputs, the automatic launch shape bench.py times, the
    # whole fp64 oracle (all channels, all tokens)
    inp = gen.workload_inputs(name)
    errs = check_all(ssm, inp, "bf16")
    print(name, {k: f"{v:.2e}" for k, v in errs.items()})


def test_float_oracle_within_fp32_bound_of_double_oracle(ssm):
    inp = gen.workload_inputs("s6-small-f32")
    assert rel_err(oracle.fwd(inp, "f32")["y"], oracle.fwd(inp, "f64")["y"]) < TOL[("f32", "fwd")]
