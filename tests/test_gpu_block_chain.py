"""The widened path in the pages' block order ("MambaBlock" S6 forward
commit: in_proj -> causal depthwise conv1d -> SiLU -> x_proj ->
delta = softplus(dt.dt_proj + dt_bias) -> scan -> gate by SiLU(z)): the
conv, the dt projection read from the dt_rank columns of an x_proj-shaped
buffer, and the scan reading B_t / C_t in place from the same buffer with
the softplus already applied -- forward and backward -- against the same
chain of oracles fed the values the GPU passes between stages (bf16-rounded
where the GPU stores bf16)."""
from dataclasses import replace

import numpy as np
import pytest

import gen
import oracle
from _util import rel_err, to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-2  # bf16 I/O


@pytest.fixture(scope="module")
def ssm():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import selective_state_space_07_gb300 as m
    m.build()
    return m


def dev(a, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device="cuda", dtype=dtype)


@pytest.mark.parametrize("shape", [(2, 200, 256, 32), (1, 300, 520, 48)])
def test_conv_dtproj_scan_chain(ssm, shape):
    B, L, D, R = shape
    N, K, bf = 16, 4, torch.bfloat16
    c = gen.make_conv_inputs(B, L, D, K, io="bf16", seed=11)
    pj = gen.make_dtproj_inputs(B, L, D, R, seed=12)
    s = gen.make_inputs(B, L, D, N, io="bf16", seed=13)  # z, B_t, C_t, A, D, dy

    # the x_proj output: [dt_rank | B_t | C_t] per token, bf16
    xp = torch.zeros(B, L, R + 2 * N, dtype=bf, device="cuda")
    xp[..., :R] = dev(pj.a, bf)
    xp[..., R:R + N] = dev(s.Bm, bf)
    xp[..., R + N:] = dev(s.Cm, bf)
    a_v, b_v, c_v = xp[..., :R], xp[..., R:R + N], xp[..., R + N:]

    xin, cw, cb = dev(c.xin, bf), dev(c.w), dev(c.bias)
    W, dtb = dev(pj.w, bf), dev(pj.bias)
    A, Dk, z, dy = dev(s.A), dev(s.Dskip), dev(s.z, bf), dev(s.dy, bf)

    x, _ = ssm.conv1d_fwd(xin, cw, cb)
    delta = ssm.dtproj_fwd(a_v, W, dtb)
    y, _, ck, ws = ssm.scan_fwd(x, delta, A, b_v, c_v, z, Dk, None, delta_softplus=False)
    g = ssm.scan_bwd(x, delta, A, b_v, c_v, dy, ck, z, Dk, None, delta_softplus=False, workspace=ws)
    gc = ssm.conv1d_bwd(xin, cw, g["dx"], cb)
    gp = ssm.dtproj_bwd(a_v, W, g["d_dt"], dtb)
    torch.cuda.synchronize()

    # the oracle chain, stage by stage on what the GPU handed over
    x_o = to_np(x)  # the conv's bf16 output is the scan's input
    assert rel_err(x_o, oracle.conv_fwd(c.xin, c.w, c.bias)["x"]) <= TOL
    a2 = pj.a.reshape(-1, R)
    delta_o = oracle.dtproj_fwd(a2, pj.w, pj.bias).reshape(B, L, D)
    assert rel_err(to_np(delta), delta_o) <= 1e-4
    inp = replace(s, x=x_o, dt=to_np(delta), dt_bias=None, delta_softplus=0)
    assert rel_err(to_np(y), oracle.fwd(inp)["y"]) <= TOL
    rb = oracle.bwd(inp)
    assert rel_err(to_np(g["dx"]), rb["dx"]) <= TOL
    assert rel_err(to_np(g["d_dt"]), rb["ddt"]) <= TOL
    assert rel_err(to_np(g["dB"]), rb["dB"]) <= TOL and rel_err(to_np(g["dC"]), rb["dC"]) <= TOL

    rc = oracle.conv_bwd(c.xin, c.w, to_np(g["dx"]), c.bias)
    assert rel_err(to_np(gc["dxin"]), rc["dxin"]) <= TOL
    assert rel_err(to_np(gc["dw"]), rc["dw"]) <= TOL and rel_err(to_np(gc["dbias"]), rc["dbias"]) <= TOL
    rp = oracle.dtproj_bwd(a2, pj.w, to_np(g["d_dt"]).reshape(-1, D), pj.bias)
    assert rel_err(to_np(gp["dpre"]).reshape(-1, D), rp["dpre"]) <= 1e-3
    assert rel_err(to_np(gp["dbias"]), rp["dbias"]) <= 1e-3
