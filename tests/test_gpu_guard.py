"""Guard bands around every output: each output buffer of a ragged problem
(3 x 333 x 104, bf16, 5 L-groups) sits inside a NaN-filled allocation with
4 KiB of NaN before and after it. After the forward, the backward, the conv
(forward and backward) and the dt projection (forward and backward), every
byte of every guard band must still be NaN -- no kernel writes past the
ends of its outputs on ragged tiles -- and every output must have been
written (no NaN left inside it). Calls go through the C ABI."""
import ctypes

import numpy as np
import pytest

import gen
from _util import to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

GUARD_BYTES = 4096


@pytest.fixture(scope="module")
def ssm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import selective_state_space_07_gb300 as m
    m.build()
    return m


class Guarded:
    """An output tensor inside a NaN-filled buffer with GUARD_BYTES of NaN on both sides."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape)) if len(shape) else 1
        g = GUARD_BYTES // torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((g + n + g,), float("nan"), dtype=dtype, device="cuda")
        self.g, self.n = g, n
        self.t = self.buf[g:g + n].view(*shape)

    def ptr(self):
        return self.t.data_ptr()

    def guards_intact(self):
        return bool(torch.isnan(self.buf[:self.g].float()).all() and torch.isnan(self.buf[self.g + self.n:].float()).all())

    def written(self):
        return not bool(torch.isnan(self.t.float()).any())


def stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_scan_outputs_stay_inside_their_buffers(ssm):
    B, L, D = 3, 333, 104
    inp = gen.make_inputs(B, L, D, 16, io="bf16", seed=31, with_h0=True, with_dh_last=True)
    dv = to_dev(inp)
    io = torch.bfloat16
    f32 = torch.float32
    y, h_last = Guarded((B, L, D), io), Guarded((B, D, 16), f32)
    ckpt = Guarded((ssm.ckpt_elems(B, L, D),), f32)
    ws = ssm.Workspace(B, L, D, "cuda")
    p = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    fa = ssm.FwdArgs(B=B, L=L, D=D, N=16, io_dtype=1, delta_softplus=1, x=p(dv["x"]), z=p(dv["z"]),
                     Bm=p(dv["Bm"]), Cm=p(dv["Cm"]), dt=p(dv["dt"]), dt_bias=p(dv["dt_bias"]), A=p(dv["A"]),
                     Dskip=p(dv["Dskip"]), h0=p(dv["h0"]), y=y.ptr(), h_last=h_last.ptr(), ckpt=ckpt.ptr(),
                     workspace=ws.buf.data_ptr(), workspace_bytes=ws.nbytes, nsplit=0, groups=5)
    assert ssm.lib().ssm_scan_fwd(ctypes.byref(fa), stream()) == 0
    outs = {"dx": Guarded((B, L, D), io), "dz": Guarded((B, L, D), io), "d_dt": Guarded((B, L, D), f32),
            "dA": Guarded((D, 16), f32), "dD": Guarded((D,), f32), "d_dt_bias": Guarded((D,), f32),
            "dB": Guarded((B, L, 16), f32), "dC": Guarded((B, L, 16), f32), "dh0": Guarded((B, D, 16), f32)}
    ba = ssm.BwdArgs(f=fa, dy=p(dv["dy"]), dh_last=p(dv["dh_last"]), **{k: g.ptr() for k, g in outs.items()})
    assert ssm.lib().ssm_scan_bwd(ctypes.byref(ba), stream()) == 0
    assert ssm.poll_status(ws) == 0
    for name, g in [("y", y), ("h_last", h_last), ("ckpt", ckpt)] + list(outs.items()):
        assert g.guards_intact(), name
        assert g.written(), name


def test_conv_and_dtproj_outputs_stay_inside_their_buffers(ssm):
    B, L, D, K = 3, 333, 104, 4
    rng = np.random.default_rng(5)
    bf = torch.bfloat16
    f32 = torch.float32
    xin = torch.from_numpy(rng.standard_normal((B, L, D), dtype=np.float32)).to("cuda", bf)
    w = torch.from_numpy(rng.standard_normal((D, K), dtype=np.float32) * 0.5).cuda()
    bias = torch.from_numpy(rng.standard_normal(D, dtype=np.float32) * 0.1).cuda()
    st = torch.from_numpy(rng.standard_normal((B, D, K - 1), dtype=np.float32)).cuda()
    x, st_out = Guarded((B, L, D), bf), Guarded((B, D, K - 1), f32)
    ca = ssm.ConvArgs(B=B, L=L, D=D, K=K, io_dtype=1, xin=xin.data_ptr(), w=w.data_ptr(), bias=bias.data_ptr(),
                      state_in=st.data_ptr(), x=x.ptr(), state_out=st_out.ptr(), workspace=None)
    assert ssm.lib().ssm_conv1d_fwd(ctypes.byref(ca), stream()) == 0
    dx = torch.from_numpy(rng.standard_normal((B, L, D), dtype=np.float32)).to("cuda", bf)
    cb = {"dxin": Guarded((B, L, D), bf), "dw": Guarded((D, K), f32), "dbias": Guarded((D,), f32),
          "dstate_in": Guarded((B, D, K - 1), f32)}
    cba = ssm.ConvBwdArgs(f=ca, dx=dx.data_ptr(), **{k: g.ptr() for k, g in cb.items()})
    assert ssm.lib().ssm_conv1d_bwd(ctypes.byref(cba), stream()) == 0

    M, R = B * L, 32
    a = torch.from_numpy(rng.standard_normal((M, R), dtype=np.float32)).to("cuda", bf)
    wd = torch.from_numpy(rng.standard_normal((D, R), dtype=np.float32) / np.sqrt(R)).to("cuda", bf)
    bd = torch.from_numpy(rng.standard_normal(D, dtype=np.float32) - 4.6).cuda()
    delta = Guarded((M, D), f32)
    da = ssm.DtProjArgs(M=M, D=D, R=R, a_stride=0, softplus=1, a=a.data_ptr(), w=wd.data_ptr(), bias=bd.data_ptr(),
                        delta=delta.ptr(), workspace=None)
    assert ssm.lib().ssm_dtproj_fwd(ctypes.byref(da), stream()) == 0
    dd = torch.from_numpy(rng.standard_normal((M, D), dtype=np.float32)).cuda()
    dpre, dbias = Guarded((M, D), f32), Guarded((D,), f32)
    dba = ssm.DtProjBwdArgs(f=da, ddelta=dd.data_ptr(), dpre=dpre.ptr(), dbias=dbias.ptr())
    assert ssm.lib().ssm_dtproj_bwd(ctypes.byref(dba), stream()) == 0
    torch.cuda.synchronize()
    for name, g in [("x", x), ("state_out", st_out), ("delta", delta), ("dpre", dpre), ("dbias", dbias)] + \
            list(cb.items()):
        assert g.guards_intact(), name
        assert g.written(), name
