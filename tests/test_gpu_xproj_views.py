"""B_t and C_t read straight from the x_proj output ("MambaBlock" S6 forward
commit: x_proj emits dt_rank + 2*d_state values per token): Bm and Cm passed
as column slices of one [B, L, R + 2N] buffer give the dense call's results
-- the same bits where no atomic reduction is involved."""
import numpy as np
import pytest

import gen
from _util import to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

EXACT = ("dx", "dz", "d_dt")
SUMMED = ("dA", "dD", "d_dt_bias", "dB", "dC")


@pytest.fixture(scope="module")
def ssm():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import selective_state_space_07_gb300 as m
    m.build()
    return m


def xproj_views(Bm, Cm, R):
    """Lay Bm, Cm out as the last 2N columns of a [B, L, R + 2N] buffer (the
    first R columns, dt_rank, hold unrelated values) and return the views."""
    B, L, N = Bm.shape
    buf = torch.randn(B, L, R + 2 * N, device=Bm.device).to(Bm.dtype)
    buf[..., R:R + N] = Bm
    buf[..., R + N:] = Cm
    return buf[..., R:R + N], buf[..., R + N:]


@pytest.mark.parametrize("io,R,shape", [("bf16", 64, (2, 300, 256)), ("f32", 8, (2, 300, 256)),
                                        ("bf16", 128, (2, 1000, 512))])
def test_scan_reads_bc_from_xproj_columns(ssm, io, R, shape):
    B, L, D = shape
    dv = to_dev(gen.make_inputs(B, L, D, 16, io=io, seed=77))
    Bv, Cv = xproj_views(dv["Bm"], dv["Cm"], R)
    assert not Bv.is_contiguous() and Bv.stride(1) == R + 32
    outs = []
    for Bm, Cm in ((dv["Bm"], dv["Cm"]), (Bv, Cv)):
        y, hl, ck, ws = ssm.scan_fwd(dv["x"], dv["dt"], dv["A"], Bm, Cm, dv["z"], dv["Dskip"], dv["dt_bias"],
                                     return_last_state=True, groups=2)
        g = ssm.scan_bwd(dv["x"], dv["dt"], dv["A"], Bm, Cm, dv["dy"], ck, dv["z"], dv["Dskip"], dv["dt_bias"],
                         workspace=ws, groups=2)
        torch.cuda.synchronize()
        outs.append((y.clone(), hl.clone(), {k: v.clone() for k, v in g.items() if torch.is_tensor(v)}))
    (y0, h0, g0), (y1, h1, g1) = outs
    assert torch.equal(y0, y1) and torch.equal(h0, h1)
    for k in EXACT:
        assert torch.equal(g0[k], g1[k]), k
    for k in SUMMED:
        r, t = g0[k].double(), g1[k].double()
        assert float((t - r).abs().max()) <= 1e-5 * max(1.0, float(r.abs().max())), k


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_step_reads_bc_from_xproj_columns(ssm, io):
    B, D, R = 6, 264, 40 if io == "f32" else 48
    inp = gen.make_inputs(B, 1, D, 16, io=io, seed=91)
    dv = to_dev(inp)
    Bv, Cv = xproj_views(dv["Bm"], dv["Cm"], R)
    st0 = torch.randn(B, D, 16, device="cuda")
    ys = []
    for Bm, Cm in ((dv["Bm"][:, 0], dv["Cm"][:, 0]), (Bv[:, 0], Cv[:, 0])):
        st = st0.clone()
        y = ssm.step(st, dv["x"][:, 0].contiguous(), dv["dt"][:, 0].contiguous(), dv["A"], Bm, Cm,
                     dv["z"][:, 0].contiguous(), dv["Dskip"], dv["dt_bias"])
        torch.cuda.synchronize()
        ys.append((y, st))
    assert torch.equal(ys[0][0], ys[1][0]) and torch.equal(ys[0][1], ys[1][1])
