"""Host-buffer entry points: the one-shot call and the overlapped pipeline
give the device path's results for the inputs of each step."""
import pytest

import gen
from _util import to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

NAMES = ("x", "dt", "A", "Bm", "Cm", "z", "Dskip", "dt_bias", "dy")
EXACT = ("y", "dx", "dz", "d_dt")                     # no atomics: same bits every run
SUMMED = ("dA", "dD", "d_dt_bias", "dB", "dC")        # atomics: rounding order varies


@pytest.fixture(scope="module")
def ssm():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import selective_state_space_07_gb300 as m
    m.build()
    return m


def host_inputs(inp):
    dv = to_dev(inp)
    return {k: dv[k].cpu().pin_memory() for k in NAMES}, dv


def device_reference(ssm, dv):
    y, _, ckpt, ws = ssm.scan_fwd(dv["x"], dv["dt"], dv["A"], dv["Bm"], dv["Cm"], dv["z"], dv["Dskip"],
                                  dv["dt_bias"])
    g = ssm.scan_bwd(dv["x"], dv["dt"], dv["A"], dv["Bm"], dv["Cm"], dv["dy"], ckpt, dv["z"], dv["Dskip"],
                     dv["dt_bias"], workspace=ws)
    torch.cuda.synchronize()
    return {"y": y.cpu(), **{k: v.cpu() for k, v in g.items() if k != "workspace"}}


def check(res, ref):
    for k in EXACT:
        assert torch.equal(res[k], ref[k]), k
    for k in SUMMED:
        r, g = ref[k].double(), res[k].double()
        assert float((g - r).abs().max()) <= 1e-5 * max(1.0, float(r.abs().max())), k


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_one_shot_host_call(ssm, io):
    inp = gen.make_inputs(2, 300, 256, 16, io=io, seed=31)
    host, dv = host_inputs(inp)
    ref = device_reference(ssm, dv)
    res, _ = ssm.scan_fwd_bwd_host(host, torch.device("cuda"))
    torch.cuda.synchronize()
    check(res, ref)


def test_pipeline_steps_keep_their_own_inputs(ssm):
    # alternate two input sets over more steps than the pipeline has buffer
    # sets: each step's results must be those of its own inputs
    a, dva = host_inputs(gen.make_inputs(2, 512, 384, 16, io="bf16", seed=41))
    b, dvb = host_inputs(gen.make_inputs(2, 512, 384, 16, io="bf16", seed=42))
    refs = {"a": device_reference(ssm, dva), "b": device_reference(ssm, dvb)}
    pipe = ssm.HostPipeline(a, torch.device("cuda"))
    order = ["a", "b", "a", "a", "b", "b", "a"]
    outs = [pipe.step(a if k == "a" else b) for k in order]
    pipe.synchronize()
    for k, res in zip(order, outs):
        check(res, refs[k])
