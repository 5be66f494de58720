"""ssm_scan_fwd_noalloc, the forward for callers that cannot allocate
device memory (allocator callbacks, processes whose device memory is
planned by someone else, plug-ins handed only their tensors): its chunk
carries live in the library's built-in 8 MiB array instead of a caller
workspace. Checked through the C ABI, bit for bit against ssm_scan_fwd with
the same L-groups and within tolerance against the oracle, on two calls in a
row after a call that leaves Inf/NaN carries in the shared array, so
leftovers in the array cannot leak into the next result.

This file is collected last on purpose: if it fails, a run that stops at
the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest

import gen
import oracle
from _util import TOL, rel_err, to_dev, to_np

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def ssm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import selective_state_space_07_gb300 as m
    m.build()
    return m


def noalloc_fwd(ssm, dv, inp, groups, status_ws=None):
    B, L, D = dv["x"].shape
    y = torch.empty_like(dv["x"])
    h_last = torch.empty(B, D, 16, dtype=torch.float32, device="cuda")
    ckpt = torch.empty(ssm.ckpt_elems(B, L, D), dtype=torch.float32, device="cuda")
    p = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    args = ssm.FwdArgs(B=B, L=L, D=D, N=16, io_dtype=0 if dv["x"].dtype == torch.float32 else 1,
                       delta_softplus=int(inp.delta_softplus), x=p(dv["x"]), z=p(dv["z"]), Bm=p(dv["Bm"]),
                       Cm=p(dv["Cm"]), dt=p(dv["dt"]), dt_bias=p(dv["dt_bias"]), A=p(dv["A"]),
                       Dskip=p(dv["Dskip"]), h0=p(dv["h0"]), y=p(y), h_last=p(h_last), ckpt=p(ckpt),
                       workspace=None if status_ws is None else status_ws.buf.data_ptr(),
                       workspace_bytes=0 if status_ws is None else status_ws.nbytes, nsplit=0, groups=groups)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = ssm.lib().ssm_scan_fwd_noalloc(ctypes.byref(args), stream)
    return rc, y, h_last, ckpt


def reference_fwd(ssm, dv, inp, groups):
    y, h_last, ckpt, _ = ssm.scan_fwd(dv["x"], dv["dt"], dv["A"], dv["Bm"], dv["Cm"], dv["z"], dv["Dskip"],
                                      dv["dt_bias"], dv["h0"], bool(inp.delta_softplus), return_last_state=True,
                                      groups=groups)
    return y, h_last, ckpt


CASES = [
    # (B, L, D, io, groups): several L-groups, so the carries sit in the array
    (2, 333, 104, "bf16", 5),
    (1, 1000, 64, "f32", 4),
]


def poison_the_array(ssm, B, L, D, io, groups):
    # Delta < 0 without softplus: the states overflow, so every aggregate and
    # carry this call leaves in the shared array is Inf or NaN
    inp = gen.make_inputs(B, L, D, 16, io=io, seed=99, bias=False)
    inp.delta_softplus = 0
    inp.dt = np.full_like(inp.dt, -3.0)
    rc, y, _, _ = noalloc_fwd(ssm, to_dev(inp), inp, groups)
    assert rc == 0
    torch.cuda.synchronize()
    assert not torch.isfinite(y.float()).all()


def test_two_calls_in_a_row_match_ssm_scan_fwd_bitwise(ssm):
    # After a call that leaves Inf/NaN carries in the shared array, two calls
    # in a row (different shapes and dtypes) give exactly what ssm_scan_fwd
    # gives with the same L-groups (the same kernels and carries), and match
    # the oracle within tolerance: nothing left in the array leaks.
    poison_the_array(ssm, *CASES[0])
    for i, (B, L, D, io, groups) in enumerate(CASES):
        inp = gen.make_inputs(B, L, D, 16, io=io, seed=70 + i, with_h0=True)
        dv = to_dev(inp)
        rc, y, h_last, ckpt = noalloc_fwd(ssm, dv, inp, groups)
        assert rc == 0, ssm.lib().ssm_status_string(rc)
        assert ssm.last_launch_count() == 3  # aggregate pass, carry scan, main pass
        ry, rh, rck = reference_fwd(ssm, dv, inp, groups)
        torch.cuda.synchronize()
        n = ssm.ckpt_elems(B, L, D)
        assert torch.equal(y, ry) and torch.equal(h_last, rh) and torch.equal(ckpt[:n], rck[:n])
        rf = oracle.fwd(inp)
        assert rel_err(to_np(y), rf["y"]) <= TOL[(io, "fwd")]
        assert rel_err(to_np(h_last), rf["h_last"]) <= TOL[(io, "fwd")]


def test_automatic_groups_use_the_array(ssm):
    # groups = 0 on a long, narrow problem: the library picks several L-groups
    # (carries in the array), and the result matches the oracle
    poison_the_array(ssm, 1, 4096, 64, "f32", 8)
    inp = gen.make_inputs(1, 4096, 64, 16, io="f32", seed=75, with_h0=True)
    dv = to_dev(inp)
    rc, y, h_last, _ = noalloc_fwd(ssm, dv, inp, 0)
    assert rc == 0
    assert ssm.last_launch_count() == 3
    torch.cuda.synchronize()
    rf = oracle.fwd(inp)
    assert rel_err(to_np(y), rf["y"]) <= TOL[("f32", "fwd")]
    assert rel_err(to_np(h_last), rf["h_last"]) <= TOL[("f32", "fwd")]


def test_explicit_groups_beyond_the_array_are_rejected(ssm):
    # 4 x 4096 channels x 64 groups of carries is ~ 70 MB, past the 8 MiB array;
    # the check runs on the host before anything is touched
    fake = 1 << 20
    args = ssm.FwdArgs(B=4, L=4096, D=4096, N=16, io_dtype=1, delta_softplus=1, x=fake, z=fake, Bm=fake, Cm=fake,
                       dt=fake, dt_bias=fake, A=fake, Dskip=fake, h0=None, y=fake, h_last=None, ckpt=fake,
                       workspace=None, workspace_bytes=0, nsplit=0, groups=64)
    rc = ssm.lib().ssm_scan_fwd_noalloc(ctypes.byref(args), None)
    assert rc == -8
    assert b"8 MiB" in ssm.lib().ssm_status_string(rc)


def test_status_word_goes_to_a_caller_buffer_when_given(ssm):
    inp = gen.make_inputs(1, 200, 16, 16, io="f32", seed=3, bias=False)
    inp.delta_softplus = 0
    inp.dt = np.full_like(inp.dt, -3.0)  # growth: the state overflows
    dv = to_dev(inp)
    ws = ssm.Workspace(1, 1, 8, "cuda")
    rc, y, _, _ = noalloc_fwd(ssm, dv, inp, 2, status_ws=ws)
    assert rc == 0
    assert ssm.poll_status(ws) == -7
