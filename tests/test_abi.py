"""The C ABI boundary without a GPU: the library builds for sm_103a, exports
every entry point include/ssm_scan.h declares, and rejects bad arguments on
the host with the documented codes before anything is launched."""
import ctypes
import importlib
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OK, INVALID, UNSUPPORTED, ALIGNMENT, WORKSPACE, CUDA, TIMEOUT, NONFINITE = 0, -1, -2, -3, -4, -5, -6, -7


@pytest.fixture(scope="module")
def ssm():
    import selective_state_space_07_gb300 as m
    m.build()
    return m


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"^[A-Za-z_][\w \*]*?\b((?:ssm|gdn2|mlstm)_\w+)\s*\(", text, flags=re.M))
    return names


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("ssm_scan_fwd", "ssm_scan_bwd", "ssm_step", "ssm_scan_workspace_bytes", "ssm_scan_ckpt_elems",
              "ssm_poll_status", "ssm_status_string", "ssm_dA_log_grad", "ssm_conv1d_fwd", "ssm_conv1d_bwd",
              "ssm_dtproj_fwd", "ssm_dtproj_bwd", "gdn2_chunk_fwd", "mlstm_chunk_fwd"):
        assert n in names


def test_library_exports_every_declared_symbol(ssm):
    lib = ctypes.CDLL(ssm.LIB_PATH)
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(ssm.EXPORTS) == declared_functions()


def test_library_is_built_for_sm_103a(ssm):
    b = importlib.import_module("selective_state_space_07_gb300._builder")
    assert "arch=compute_103a,code=sm_103a" in b.ARCH
    assert open(ssm.LIB_PATH, "rb").read().find(b"sm_103a") >= 0


def test_sizes(ssm):
    assert ssm.ckpt_elems(4, 4096, 4096) == 4 * 512 * 16 * 4096
    assert ssm.ckpt_elems(1, 17, 8) == 3 * 16 * 8
    assert ssm.ckpt_elems(2, 0, 8) == 0
    assert ssm.lib().ssm_scan_ckpt_interval() == ssm.CKPT_INTERVAL == 8
    assert ssm.workspace_bytes(1, 1, 8) >= 256
    # carries are bounded: B*D*groups <= 131072, fp32 [.., 16] x2 + sums
    assert ssm.workspace_bytes(4, 4096, 4096) <= 256 + 131072 * 33 * 4 + 512
    assert ssm.workspace_bytes(1, 65536, 2048) <= 256 + 131072 * 33 * 4 + 512


def test_status_strings(ssm):
    for code in (OK, INVALID, UNSUPPORTED, ALIGNMENT, WORKSPACE, CUDA, TIMEOUT, NONFINITE, 12345):
        assert isinstance(ssm.lib().ssm_status_string(code), bytes)
    assert b"wait" in ssm.lib().ssm_status_string(TIMEOUT)
    assert ssm.lib().ssm_status_string(TIMEOUT) != ssm.lib().ssm_status_string(12345)


FAKE = 1 << 20  # a 16-byte aligned address; never dereferenced: every case fails validation first


def fwd_args(ssm, **over):
    a = dict(B=2, L=32, D=16, N=16, io_dtype=1, delta_softplus=1, x=FAKE, z=FAKE, Bm=FAKE, Cm=FAKE, dt=FAKE,
             dt_bias=FAKE, A=FAKE, Dskip=FAKE, h0=None, y=FAKE, h_last=None, ckpt=FAKE, workspace=FAKE,
             workspace_bytes=1 << 30, nsplit=0, groups=0)
    a.update(over)
    return ssm.FwdArgs(**a)


@pytest.mark.parametrize("over,code", [
    (dict(N=8), UNSUPPORTED), (dict(io_dtype=7), UNSUPPORTED), (dict(D=12), ALIGNMENT),
    (dict(x=None), INVALID), (dict(y=None), INVALID), (dict(B=-1), INVALID), (dict(delta_softplus=2), INVALID),
    (dict(nsplit=3), INVALID), (dict(groups=-2), INVALID), (dict(x=FAKE + 4), ALIGNMENT),
    (dict(h0=FAKE + 8), ALIGNMENT), (dict(workspace=None), WORKSPACE), (dict(workspace_bytes=16), WORKSPACE),
    # Bm / Cm row stride: at least N, a multiple of 16 bytes (bf16: 8 elements)
    (dict(bc_stride=8), INVALID), (dict(bc_stride=20), ALIGNMENT), (dict(bc_stride=-16), INVALID),
    (dict(B=2, L=1 << 30), UNSUPPORTED),  # 2^31 token rows: past the 32-bit row coordinates of the copies
    (dict(B=1, L=(1 << 30) + 1), UNSUPPORTED),
    (dict(B=1 << 30, L=1 << 34), UNSUPPORTED),  # B*L would wrap past int64 (to 0) if multiplied unchecked
])
def test_fwd_rejects_bad_arguments(ssm, over, code):
    args = fwd_args(ssm, **over)
    assert ssm.lib().ssm_scan_fwd(ctypes.byref(args), None) == code


@pytest.mark.parametrize("over,code", [
    (dict(dy=None), INVALID), (dict(dx=None), INVALID), (dict(dz=None), INVALID), (dict(dA=None), INVALID),
    (dict(dB=None), INVALID), (dict(dC=FAKE + 2), ALIGNMENT), (dict(d_dt=None), INVALID),
])
def test_bwd_rejects_bad_arguments(ssm, over, code):
    g = dict(dy=FAKE, dh_last=None, dx=FAKE, dz=FAKE, d_dt=FAKE, dA=FAKE, dD=FAKE, d_dt_bias=FAKE, dB=FAKE,
             dC=FAKE, dh0=None)
    g.update(over)
    args = ssm.BwdArgs(f=fwd_args(ssm), **g)
    assert ssm.lib().ssm_scan_bwd(ctypes.byref(args), None) == code


def test_bwd_checks_the_bc_stride(ssm):
    g = dict(dy=FAKE, dx=FAKE, dz=FAKE, d_dt=FAKE, dA=FAKE, dD=FAKE, d_dt_bias=FAKE, dB=FAKE, dC=FAKE)
    args = ssm.BwdArgs(f=fwd_args(ssm, bc_stride=12), **g)
    assert ssm.lib().ssm_scan_bwd(ctypes.byref(args), None) == INVALID
    args = ssm.BwdArgs(f=fwd_args(ssm, bc_stride=36), **g)
    assert ssm.lib().ssm_scan_bwd(ctypes.byref(args), None) == ALIGNMENT


def test_bwd_needs_the_checkpoints(ssm):
    args = ssm.BwdArgs(f=fwd_args(ssm, ckpt=None), dy=FAKE, dx=FAKE, dz=FAKE, d_dt=FAKE, dA=FAKE, dD=FAKE,
                       d_dt_bias=FAKE, dB=FAKE, dC=FAKE)
    assert ssm.lib().ssm_scan_bwd(ctypes.byref(args), None) == INVALID


@pytest.mark.parametrize("over,code", [
    (dict(N=4), UNSUPPORTED), (dict(D=20), ALIGNMENT), (dict(state=None), INVALID), (dict(y_t=FAKE + 1), ALIGNMENT),
    (dict(io_dtype=-1), UNSUPPORTED), (dict(nsplit=8), INVALID), (dict(bc_stride=4), INVALID),
    (dict(bc_stride=18), ALIGNMENT),
])
def test_step_rejects_bad_arguments(ssm, over, code):
    a = dict(B=2, D=16, N=16, io_dtype=0, delta_softplus=1, x_t=FAKE, z_t=None, Bm_t=FAKE, Cm_t=FAKE, dt_t=FAKE,
             dt_bias=None, A=FAKE, Dskip=None, state=FAKE, y_t=FAKE, workspace=None, nsplit=0)
    a.update(over)
    args = ssm.StepArgs(**a)
    assert ssm.lib().ssm_step(ctypes.byref(args), None) == code


def conv_args(ssm, **over):
    a = dict(B=2, L=300, D=16, K=4, io_dtype=1, xin=FAKE, w=FAKE + 4096, bias=None, state_in=None,
             x=FAKE + 8192, state_out=None, workspace=None)
    a.update(over)
    return ssm.ConvArgs(**a)


@pytest.mark.parametrize("over,code", [
    (dict(K=5), UNSUPPORTED), (dict(K=0), UNSUPPORTED), (dict(io_dtype=3), UNSUPPORTED), (dict(D=12), ALIGNMENT),
    (dict(B=-1), INVALID), (dict(xin=None), INVALID), (dict(w=None), INVALID), (dict(x=None), INVALID),
    (dict(x=FAKE), INVALID), (dict(bias=FAKE + 4), ALIGNMENT), (dict(state_in=FAKE + 8), ALIGNMENT),
])
def test_conv_fwd_rejects_bad_arguments(ssm, over, code):
    args = conv_args(ssm, **over)
    assert ssm.lib().ssm_conv1d_fwd(ctypes.byref(args), None) == code


@pytest.mark.parametrize("over,code", [
    (dict(dx=None), INVALID), (dict(dxin=None), INVALID), (dict(dw=None), INVALID),
    (dict(dxin=FAKE + 16384), INVALID),  # dxin aliasing dx
    (dict(dxin=FAKE), INVALID),          # dxin aliasing xin
    (dict(dbias=FAKE + 2), ALIGNMENT), (dict(dstate_in=FAKE + 4), ALIGNMENT),
])
def test_conv_bwd_rejects_bad_arguments(ssm, over, code):
    g = dict(dx=FAKE + 16384, dxin=FAKE + 20480, dw=FAKE + 24576, dbias=None, dstate_in=None)
    g.update(over)
    args = ssm.ConvBwdArgs(f=conv_args(ssm), **g)
    assert ssm.lib().ssm_conv1d_bwd(ctypes.byref(args), None) == code


def dtproj_args(ssm, **over):
    a = dict(M=300, D=1048, R=64, a_stride=96, softplus=1, a=FAKE, w=FAKE + 4096, bias=None, delta=FAKE + 8192,
             workspace=None)
    a.update(over)
    return ssm.DtProjArgs(**a)


@pytest.mark.parametrize("over,code", [
    (dict(R=24), UNSUPPORTED), (dict(R=0), UNSUPPORTED), (dict(R=272), UNSUPPORTED), (dict(D=1044), ALIGNMENT),
    (dict(a_stride=60), INVALID), (dict(a_stride=100), ALIGNMENT), (dict(softplus=2), INVALID),
    (dict(a=None), INVALID), (dict(w=None), INVALID), (dict(delta=None), INVALID), (dict(bias=FAKE + 4), ALIGNMENT),
    (dict(M=-1), INVALID),
])
def test_dtproj_rejects_bad_arguments(ssm, over, code):
    args = dtproj_args(ssm, **over)
    assert ssm.lib().ssm_dtproj_fwd(ctypes.byref(args), None) == code


def test_dtproj_bwd_rejects_bad_arguments(ssm):
    for over, code in ((dict(ddelta=None), INVALID), (dict(dpre=None), INVALID), (dict(dbias=FAKE + 8), ALIGNMENT)):
        g = dict(ddelta=FAKE + 16384, dpre=FAKE + 20480, dbias=None)
        g.update(over)
        args = ssm.DtProjBwdArgs(f=dtproj_args(ssm), **g)
        assert ssm.lib().ssm_dtproj_bwd(ctypes.byref(args), None) == code
    args = ssm.DtProjBwdArgs(f=dtproj_args(ssm, R=8), ddelta=FAKE, dpre=FAKE)
    assert ssm.lib().ssm_dtproj_bwd(ctypes.byref(args), None) == UNSUPPORTED


def gdn2_args(ssm, **over):
    a = dict(B=2, H=3, T=100, K=128, V=128, chunk=64, scale=0.088, q=FAKE, k=FAKE + 4096, v=FAKE + 8192,
             g=FAKE + 12288, b=FAKE + 16384, w=FAKE + 20480, state_in=None, out=FAKE + 24576, state_out=None,
             workspace=None)
    a.update(over)
    return ssm.Gdn2Args(**a)


@pytest.mark.parametrize("over,code", [
    (dict(K=64), UNSUPPORTED), (dict(V=256), UNSUPPORTED), (dict(chunk=32), UNSUPPORTED), (dict(B=-1), INVALID),
    (dict(T=-5), INVALID), (dict(q=None), INVALID), (dict(g=None), INVALID), (dict(out=None), INVALID),
    (dict(w=FAKE + 2), ALIGNMENT), (dict(state_in=FAKE + 8), ALIGNMENT), (dict(state_out=FAKE + 4), ALIGNMENT),
    (dict(scale=float("nan")), INVALID), (dict(scale=float("inf")), INVALID),
    (dict(B=1, H=1, T=1 << 31), UNSUPPORTED), (dict(B=4, H=8, T=1 << 26), UNSUPPORTED),
    (dict(B=1 << 20, H=1 << 10, T=1 << 40), UNSUPPORTED),  # B*H*T beyond int64 if multiplied unchecked
])
def test_gdn2_rejects_bad_arguments(ssm, over, code):
    args = gdn2_args(ssm, **over)
    assert ssm.lib().gdn2_chunk_fwd(ctypes.byref(args), None) == code


def gdn2_step_args(ssm, **over):
    a = dict(B=2, H=3, K=128, V=128, scale=0.088, q=FAKE, k=FAKE + 4096, v=FAKE + 8192, g=FAKE + 12288,
             b=FAKE + 16384, w=FAKE + 20480, state=FAKE + 24576, out=FAKE + 28672, workspace=None)
    a.update(over)
    return ssm.Gdn2StepArgs(**a)


@pytest.mark.parametrize("over,code", [
    (dict(K=64), UNSUPPORTED), (dict(V=256), UNSUPPORTED), (dict(H=-1), INVALID), (dict(g=None), INVALID),
    (dict(state=None), INVALID), (dict(out=None), INVALID), (dict(state=FAKE + 8), ALIGNMENT),
    (dict(b=FAKE + 2), ALIGNMENT), (dict(scale=float("inf")), INVALID), (dict(B=0), OK),
])
def test_gdn2_step_rejects_bad_arguments(ssm, over, code):
    args = gdn2_step_args(ssm, **over)
    assert ssm.lib().gdn2_step(ctypes.byref(args), None) == code


def test_gdn2_fault_hook_arguments(ssm):
    assert ssm.lib().gdn2_debug_arm_wait_fault(0, 20_000_000_000) == INVALID
    assert ssm.lib().gdn2_debug_arm_wait_fault(-1, 0) == OK  # disarmed


def mlstm_args(ssm, **over):
    a = dict(B=2, H=3, T=100, K=128, V=128, chunk=64, scale=0.088, norm_eps=1e-5, q=FAKE, k=FAKE + 4096,
             v=FAKE + 8192, igate=FAKE + 12288, fgate=FAKE + 12292, C_in=None, n_in=None, m_in=None, norm_weight=None,
             h=FAKE + 24576, C_out=None, n_out=None, m_out=None, workspace=None)
    a.update(over)
    return ssm.MlstmArgs(**a)


@pytest.mark.parametrize("over,code", [
    (dict(K=64), UNSUPPORTED), (dict(V=256), UNSUPPORTED), (dict(chunk=32), UNSUPPORTED), (dict(B=-1), INVALID),
    (dict(T=-5), INVALID), (dict(q=None), INVALID), (dict(igate=None), INVALID), (dict(fgate=None), INVALID),
    (dict(h=None), INVALID), (dict(v=FAKE + 2), ALIGNMENT), (dict(igate=FAKE + 2), ALIGNMENT),
    (dict(norm_weight=FAKE + 1), ALIGNMENT), (dict(norm_weight=FAKE + 4), ALIGNMENT),
    (dict(C_in=FAKE + 8, n_in=FAKE, m_in=FAKE), ALIGNMENT), (dict(C_out=FAKE + 4, n_out=FAKE, m_out=FAKE), ALIGNMENT),
    (dict(C_in=FAKE), INVALID), (dict(n_out=FAKE, m_out=FAKE), INVALID),  # a partial state
    (dict(scale=float("nan")), INVALID), (dict(scale=float("inf")), INVALID),
    (dict(norm_eps=-1.0), INVALID), (dict(norm_eps=float("nan")), INVALID),
    (dict(B=1, H=1, T=1 << 31), UNSUPPORTED), (dict(B=4, H=8, T=1 << 26), UNSUPPORTED),
    (dict(B=1 << 20, H=1 << 10, T=1 << 40), UNSUPPORTED),  # B*H*T beyond int64 if multiplied unchecked
])
def test_mlstm_rejects_bad_arguments(ssm, over, code):
    args = mlstm_args(ssm, **over)
    assert ssm.lib().mlstm_chunk_fwd(ctypes.byref(args), None) == code


def mlstm_step_args(ssm, **over):
    a = dict(B=2, H=3, K=128, V=128, scale=0.088, norm_eps=1e-5, q=FAKE, k=FAKE + 4096, v=FAKE + 8192,
             igate=FAKE + 12288, fgate=FAKE + 12292, C=FAKE + 16384, n=FAKE + 20480, m=FAKE + 20484,
             norm_weight=None, h=FAKE + 24576, workspace=None)
    a.update(over)
    return ssm.MlstmStepArgs(**a)


@pytest.mark.parametrize("over,code", [
    (dict(K=64), UNSUPPORTED), (dict(V=256), UNSUPPORTED), (dict(B=-1), INVALID), (dict(q=None), INVALID),
    (dict(C=None), INVALID), (dict(m=None), INVALID), (dict(h=None), INVALID), (dict(C=FAKE + 8), ALIGNMENT),
    (dict(norm_weight=FAKE + 4), ALIGNMENT), (dict(n=FAKE + 2), ALIGNMENT), (dict(scale=float("nan")), INVALID),
    (dict(norm_eps=-1.0), INVALID), (dict(B=0), OK), (dict(B=0, q=None, C=None), OK),
])
def test_mlstm_step_rejects_bad_arguments(ssm, over, code):
    args = mlstm_step_args(ssm, **over)
    assert ssm.lib().mlstm_step(ctypes.byref(args), None) == code


def test_mlstm_fault_hook_arguments(ssm):
    assert ssm.lib().mlstm_debug_arm_wait_fault(0, 20_000_000_000) == INVALID
    assert ssm.lib().mlstm_debug_arm_wait_fault(-1, 0) == OK  # disarmed


def test_null_args_struct(ssm):
    assert ssm.lib().mlstm_chunk_fwd(None, None) == INVALID
    assert ssm.lib().mlstm_step(None, None) == INVALID
    assert ssm.lib().gdn2_step(None, None) == INVALID
    assert ssm.lib().gdn2_chunk_fwd(None, None) == INVALID
    assert ssm.lib().ssm_scan_fwd(None, None) == INVALID
    assert ssm.lib().ssm_scan_bwd(None, None) == INVALID
    assert ssm.lib().ssm_step(None, None) == INVALID
    assert ssm.lib().ssm_conv1d_fwd(None, None) == INVALID
    assert ssm.lib().ssm_conv1d_bwd(None, None) == INVALID
    assert ssm.lib().ssm_dtproj_fwd(None, None) == INVALID
    assert ssm.lib().ssm_dtproj_bwd(None, None) == INVALID


def test_dA_log_rejects_bad_arguments(ssm):
    assert ssm.lib().ssm_dA_log_grad(None, FAKE, FAKE, 4, None) == INVALID
    assert ssm.lib().ssm_dA_log_grad(FAKE, FAKE, FAKE, -1, None) == INVALID
    assert ssm.lib().ssm_dA_log_grad(None, None, None, 0, None) == OK


def test_binding_refuses_cpu_tensors(ssm):
    torch = pytest.importorskip("torch")
    x = torch.zeros(1, 4, 8)
    with pytest.raises(ValueError, match="CUDA"):
        ssm.scan_fwd(x, x, torch.zeros(8, 16), torch.zeros(1, 4, 16), torch.zeros(1, 4, 16))


def test_binding_fails_loudly_without_the_library(ssm, monkeypatch, tmp_path):
    monkeypatch.setattr(ssm, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(ssm, "_lib", None)
    with pytest.raises(ImportError):
        ssm.lib()
