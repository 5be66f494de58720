"""The dt projection with its softplus on the tensor cores ("MambaBlock" S6
forward commit: "delta=softplus(dt.dt_proj+dt_bias)", dt the dt_rank columns
of the x_proj output): the tcgen05 path against the fp64 oracle fed the same
bf16 operands, with a read in place from an x_proj-shaped buffer."""
import numpy as np
import pytest

import gen
import oracle
from _util import rel_err, to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

# fp32 accumulation of bf16 products over R <= 256 terms: ~1e-6 relative;
# the fp32 tolerances of the scan apply
TOL_FWD, TOL_BWD = 1e-4, 1e-3


@pytest.fixture(scope="module")
def ssm():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import selective_state_space_07_gb300 as m
    m.build()
    return m


def xproj_buffer(a, extra=32):
    """a [B, L, R] as the first R columns of a [B, L, R + extra] bf16 buffer (the rest: B_t, C_t)."""
    B, L, R = a.shape
    buf = torch.randn(B, L, R + extra, device="cuda").to(torch.bfloat16)
    buf[..., :R] = torch.from_numpy(a).to(device="cuda", dtype=torch.bfloat16)
    return buf[..., :R]


def dev(x, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device="cuda", dtype=dtype)


@pytest.mark.parametrize("shape", [(2, 300, 1048, 64), (1, 129, 264, 16), (3, 50, 512, 48), (1, 200, 256, 128),
                                   (2, 77, 520, 256)])
@pytest.mark.parametrize("softplus", [True, False])
def test_parity_against_the_oracle(ssm, shape, softplus):
    B, L, D, R = shape
    c = gen.make_dtproj_inputs(B, L, D, R, seed=R + L)
    a = xproj_buffer(c.a)
    assert not a.is_contiguous()
    w, bias = dev(c.w, torch.bfloat16), dev(c.bias)
    delta = ssm.dtproj_fwd(a, w, bias, softplus)
    g = ssm.dtproj_bwd(a, w, dev(c.ddelta), bias, softplus)
    torch.cuda.synchronize()
    a2 = c.a.reshape(-1, R)
    ref = oracle.dtproj_fwd(a2, c.w, c.bias, softplus)
    rg = oracle.dtproj_bwd(a2, c.w, c.ddelta.reshape(-1, D), c.bias, softplus)
    assert delta.shape == (B, L, D)
    assert rel_err(to_np(delta).reshape(-1, D), ref) <= TOL_FWD
    assert rel_err(to_np(g["dpre"]).reshape(-1, D), rg["dpre"]) <= TOL_BWD
    assert rel_err(to_np(g["dbias"]), rg["dbias"]) <= TOL_BWD


@pytest.mark.parametrize("shape", [(1, 1, 264, 16), (1, 3, 8, 32), (3, 1, 4096, 128), (1, 129, 8, 256)])
def test_decode_and_narrow_shapes(ssm, shape):
    # one token (decoding), fewer tiles than SMs, a single 8-channel column,
    # the widest rank: every persistent CTA without a tile must still leave cleanly
    B, L, D, R = shape
    c = gen.make_dtproj_inputs(B, L, D, R, seed=B * 1000 + L + D + R)
    a = xproj_buffer(c.a)
    w, bias = dev(c.w, torch.bfloat16), dev(c.bias)
    delta = ssm.dtproj_fwd(a, w, bias)
    g = ssm.dtproj_bwd(a, w, dev(c.ddelta), bias)
    torch.cuda.synchronize()
    a2 = c.a.reshape(-1, R)
    assert rel_err(to_np(delta).reshape(-1, D), oracle.dtproj_fwd(a2, c.w, c.bias)) <= TOL_FWD
    rg = oracle.dtproj_bwd(a2, c.w, c.ddelta.reshape(-1, D), c.bias)
    assert rel_err(to_np(g["dpre"]).reshape(-1, D), rg["dpre"]) <= TOL_BWD
    assert rel_err(to_np(g["dbias"]), rg["dbias"]) <= TOL_BWD


def test_empty_rows(ssm):
    w = torch.zeros(256, 64, dtype=torch.bfloat16, device="cuda")
    a = torch.zeros(2, 0, 64, dtype=torch.bfloat16, device="cuda")
    assert ssm.dtproj_fwd(a, w).shape == (2, 0, 256)
    g = ssm.dtproj_bwd(a, w, torch.zeros(2, 0, 256, device="cuda"), torch.zeros(256, device="cuda"))
    torch.cuda.synchronize()
    assert not torch.any(g["dbias"])


def test_dense_a_without_bias_and_in_place_backward(ssm):
    c = gen.make_dtproj_inputs(2, 100, 256, 32, seed=5)
    a, w = dev(c.a, torch.bfloat16), dev(c.w, torch.bfloat16)
    delta = ssm.dtproj_fwd(a, w)
    dd = dev(c.ddelta)
    g = ssm.dtproj_bwd(a, w, dd, inplace=True)
    torch.cuda.synchronize()
    assert g["dpre"].data_ptr() == dd.data_ptr() and g["dbias"] is None
    a2 = c.a.reshape(-1, 32)
    assert rel_err(to_np(delta).reshape(-1, 256), oracle.dtproj_fwd(a2, c.w)) <= TOL_FWD
    assert rel_err(to_np(dd).reshape(-1, 256), oracle.dtproj_bwd(a2, c.w, c.ddelta.reshape(-1, 256))["dpre"]) <= TOL_BWD


def test_feeds_the_scan(ssm):
    # delta from the projection, given to the scan with softplus off, equals the
    # scan fusing the same softplus itself from the pre-activation (to rounding)
    B, L, D, R = 2, 256, 256, 64
    c = gen.make_dtproj_inputs(B, L, D, R, seed=9)
    a, w, bias = xproj_buffer(c.a), dev(c.w, torch.bfloat16), dev(c.bias)
    s = gen.make_inputs(B, L, D, 16, io="f32", seed=10)
    x, A, Bm, Cm = dev(s.x), dev(s.A), dev(s.Bm), dev(s.Cm)
    delta = ssm.dtproj_fwd(a, w, bias)
    pre = ssm.dtproj_fwd(a, w, None, softplus=False)
    y1 = ssm.scan_fwd(x, delta, A, Bm, Cm, delta_softplus=False)[0]
    y2 = ssm.scan_fwd(x, pre, A, Bm, Cm, dt_bias=bias, delta_softplus=True)[0]
    torch.cuda.synchronize()
    assert rel_err(to_np(y1), to_np(y2)) <= 1e-5


def test_nonfinite_is_latched(ssm):
    c = gen.make_dtproj_inputs(1, 130, 256, 16, seed=3)
    a = dev(c.a, torch.bfloat16)
    a[0, 17, 3] = float("inf")
    ws = ssm.Workspace(1, 1, 8, a.device)
    ssm.dtproj_fwd(a, dev(c.w, torch.bfloat16), dev(c.bias), workspace=ws)
    assert ssm.poll_status(ws) == -7
    ssm.dtproj_fwd(dev(c.a, torch.bfloat16), dev(c.w, torch.bfloat16), dev(c.bias), workspace=ws)
    assert ssm.poll_status(ws) == 0


def test_full_size_on_sampled_outputs(ssm):
    # the 1.4B layer (B=4, L=4096, D=4096, dt_rank=128) in the launch
    # configuration the bench times: sampled rows against the oracle
    # row by row, and dbias on sampled channels over every row
    B, L, D, R = 4, 4096, 4096, 128
    c = gen.make_dtproj_inputs(B, L, D, R, seed=2024)
    a, w, bias = xproj_buffer(c.a), dev(c.w, torch.bfloat16), dev(c.bias)
    delta = ssm.dtproj_fwd(a, w, bias)
    g = ssm.dtproj_bwd(a, w, dev(c.ddelta), bias)
    torch.cuda.synchronize()
    a2, dd2 = c.a.reshape(-1, R), c.ddelta.reshape(-1, D)
    rows = np.array([0, 1, 127, 128, 4095, 4096, 9000, 16255, 16383])
    ref = oracle.dtproj_fwd(a2[rows], c.w, c.bias)
    rt = torch.as_tensor(rows, device="cuda")
    assert rel_err(to_np(delta.reshape(-1, D)[rt]), ref) <= TOL_FWD
    rg = oracle.dtproj_bwd(a2[rows], c.w, dd2[rows], c.bias)
    assert rel_err(to_np(g["dpre"].reshape(-1, D)[rt]), rg["dpre"]) <= TOL_BWD
    cols = np.array([0, 5, 255, 256, 2047, 4095])
    rb = oracle.dtproj_bwd(a2, c.w[cols], dd2[:, cols], c.bias[cols])
    assert rel_err(to_np(g["dbias"][torch.as_tensor(cols, device="cuda")]), rb["dbias"]) <= TOL_BWD
