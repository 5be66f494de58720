"""GB300-native Mamba S6 selective scan.

Python binding of ``libssmscan.so`` (C ABI in ``include/ssm_scan.h``). This
module only marshals arguments: it checks dtypes, shapes, contiguity,
devices and alignment, allocates outputs with PyTorch and passes raw device
pointers and the current CUDA stream to the library. Every step of the scan
runs in the library's CUDA kernels; there is no other implementation here,
and calls fail loudly when the library is missing.

The operation (rustytorch commit log, "MambaBlock" S6 forward commit):
    Delta = softplus(dt + dt_bias);  h_t = exp(Delta*A) * h_{t-1} + Delta*B_t*x_t
    y_t = (C_t . h_t + D*x_t) * silu(z_t)
Layouts: x, z, dt, y [B, L, D]; Bm, Cm [B, L, 16]; A [D, 16]; Dskip,
dt_bias [D]; states [B, D, 16]. x, z, Bm, Cm, y, dy, dx, dz are fp32 or bf16
(one dtype per call); everything else is fp32.

Also bound here: the conv1d + SiLU in front of the scan (``conv1d_fwd``,
``conv1d_bwd``, ``conv1d_step``), the dt projection with its softplus on the
tensor cores (``dtproj_fwd``, ``dtproj_bwd``), and the Gated DeltaNet-2
chunkwise forward (``gdn2_fwd``; C ABI in ``include/gdn2.h``; docs.rs,
burn-gdn2 0.1.4, src/forward.rs, chunk_wy_forward): q, k, b, g [B, H, T,
128], v, w [B, H, T, 128], state [B, H, 128, 128], chunks of 64 tokens; and
the mLSTM stabilized chunkwise forward (``mlstm_fwd``; C ABI in
``include/mlstm.h``; Evil-Inference-Code, README_FIX_RUST.md, "mLSTM
Equivalence Fixes (Rust vs Python)"): q, k, v [B, H, T, 128] bf16, gate
pre-activations [B, H, T] fp32, stabilized state C [B, H, 128, 128], n [B, H,
128], m [B, H], an optional head-wise norm, chunks of 64 tokens.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Dict, Optional

import torch

__all__ = [
    "SsmError", "build", "lib", "scan_fwd", "scan_bwd", "step", "dA_log_grad", "poll_status",
    "clear_status", "workspace_bytes", "ckpt_elems", "ckpt_states", "CKPT_INTERVAL", "Workspace",
    "scan_fwd_bwd_host", "arm_wait_fault",
    "last_launch_count", "HostPipeline", "conv1d_fwd", "conv1d_bwd", "conv1d_step", "dtproj_fwd", "dtproj_bwd",
    "gdn2_fwd", "GDN2_CHUNK", "gdn2_arm_wait_fault", "gdn2_step", "mlstm_fwd", "MLSTM_CHUNK", "mlstm_arm_wait_fault", "mlstm_step", "exp2_fma",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssmscan.so")
CKPT_INTERVAL = 8
_lock = threading.Lock()
_lib = None

SSM_F32, SSM_BF16 = 0, 1
_IO = {torch.float32: SSM_F32, torch.bfloat16: SSM_BF16}


class SsmError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = lib().ssm_status_string(code).decode()
        super().__init__(f"{where}: {msg} (code {code})")
        self.code = code


class FwdArgs(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("L", ctypes.c_int64), ("D", ctypes.c_int64), ("N", ctypes.c_int64),
                ("io_dtype", ctypes.c_int32), ("delta_softplus", ctypes.c_int32)] + [
        (n, ctypes.c_void_p) for n in ("x", "z", "Bm", "Cm", "dt", "dt_bias", "A", "Dskip", "h0", "y",
                                       "h_last", "ckpt", "workspace")] + [
        ("workspace_bytes", ctypes.c_size_t), ("nsplit", ctypes.c_int32), ("groups", ctypes.c_int32),
        ("bc_stride", ctypes.c_int64)]


class BwdArgs(ctypes.Structure):
    _fields_ = [("f", FwdArgs)] + [
        (n, ctypes.c_void_p) for n in ("dy", "dh_last", "dx", "dz", "d_dt", "dA", "dD", "d_dt_bias", "dB",
                                       "dC", "dh0")]


class StepArgs(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("D", ctypes.c_int64), ("N", ctypes.c_int64),
                ("io_dtype", ctypes.c_int32), ("delta_softplus", ctypes.c_int32)] + [
        (n, ctypes.c_void_p) for n in ("x_t", "z_t", "Bm_t", "Cm_t", "dt_t", "dt_bias", "A", "Dskip", "state",
                                       "y_t", "workspace")] + [
        ("nsplit", ctypes.c_int32), ("pad_", ctypes.c_int32), ("bc_stride", ctypes.c_int64)]


class ConvArgs(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("L", ctypes.c_int64), ("D", ctypes.c_int64), ("K", ctypes.c_int64),
                ("io_dtype", ctypes.c_int32), ("pad_", ctypes.c_int32)] + [
        (n, ctypes.c_void_p) for n in ("xin", "w", "bias", "state_in", "x", "state_out", "workspace")]


class ConvBwdArgs(ctypes.Structure):
    _fields_ = [("f", ConvArgs)] + [(n, ctypes.c_void_p) for n in ("dx", "dxin", "dw", "dbias", "dstate_in")]


class DtProjArgs(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("D", ctypes.c_int64), ("R", ctypes.c_int64), ("a_stride", ctypes.c_int64),
                ("softplus", ctypes.c_int32), ("pad_", ctypes.c_int32)] + [
        (n, ctypes.c_void_p) for n in ("a", "w", "bias", "delta", "workspace")]


class DtProjBwdArgs(ctypes.Structure):
    _fields_ = [("f", DtProjArgs)] + [(n, ctypes.c_void_p) for n in ("ddelta", "dpre", "dbias")]


class Gdn2Args(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("H", ctypes.c_int64), ("T", ctypes.c_int64), ("K", ctypes.c_int64),
                ("V", ctypes.c_int64), ("chunk", ctypes.c_int32), ("scale", ctypes.c_float)] + [
        (n, ctypes.c_void_p) for n in ("q", "k", "v", "g", "b", "w", "state_in", "out", "state_out", "workspace")]


GDN2_CHUNK = 64


class Gdn2StepArgs(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("H", ctypes.c_int64), ("K", ctypes.c_int64), ("V", ctypes.c_int64),
                ("scale", ctypes.c_float)] + [
        (n, ctypes.c_void_p) for n in ("q", "k", "v", "g", "b", "w", "state", "out", "workspace")]


class MlstmArgs(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("H", ctypes.c_int64), ("T", ctypes.c_int64), ("K", ctypes.c_int64),
                ("V", ctypes.c_int64), ("chunk", ctypes.c_int32), ("scale", ctypes.c_float),
                ("norm_eps", ctypes.c_float)] + [
        (n, ctypes.c_void_p) for n in ("q", "k", "v", "igate", "fgate", "C_in", "n_in", "m_in", "norm_weight", "h",
                                       "C_out", "n_out", "m_out", "workspace")]


MLSTM_CHUNK = 64


class MlstmStepArgs(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("H", ctypes.c_int64), ("K", ctypes.c_int64), ("V", ctypes.c_int64),
                ("scale", ctypes.c_float), ("norm_eps", ctypes.c_float)] + [
        (n, ctypes.c_void_p) for n in ("q", "k", "v", "igate", "fgate", "C", "n", "m", "norm_weight", "h", "workspace")]

EXPORTS = {
    "ssm_scan_fwd": ([ctypes.POINTER(FwdArgs), ctypes.c_void_p], ctypes.c_int),
    "ssm_scan_bwd": ([ctypes.POINTER(BwdArgs), ctypes.c_void_p], ctypes.c_int),
    "ssm_scan_fwd_noalloc": ([ctypes.POINTER(FwdArgs), ctypes.c_void_p], ctypes.c_int),
    "ssm_step": ([ctypes.POINTER(StepArgs), ctypes.c_void_p], ctypes.c_int),
    "ssm_scan_workspace_bytes": ([ctypes.c_int64] * 4, ctypes.c_size_t),
    "ssm_scan_ckpt_elems": ([ctypes.c_int64] * 4, ctypes.c_int64),
    "ssm_scan_ckpt_interval": ([], ctypes.c_int),
    "ssm_poll_status": ([ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "ssm_clear_status": ([ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "ssm_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "ssm_last_launch_count": ([], ctypes.c_int),
    "ssm_conv1d_fwd": ([ctypes.POINTER(ConvArgs), ctypes.c_void_p], ctypes.c_int),
    "ssm_conv1d_bwd": ([ctypes.POINTER(ConvBwdArgs), ctypes.c_void_p], ctypes.c_int),
    "ssm_dtproj_fwd": ([ctypes.POINTER(DtProjArgs), ctypes.c_void_p], ctypes.c_int),
    "ssm_dtproj_bwd": ([ctypes.POINTER(DtProjBwdArgs), ctypes.c_void_p], ctypes.c_int),
    "ssm_dA_log_grad": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p],
                        ctypes.c_int),
    "ssm_debug_arm_wait_fault": ([ctypes.c_int64, ctypes.c_uint64], ctypes.c_int),
    "ssm_exp2_fma": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p], ctypes.c_int),
    "gdn2_chunk_fwd": ([ctypes.POINTER(Gdn2Args), ctypes.c_void_p], ctypes.c_int),
    "gdn2_debug_arm_wait_fault": ([ctypes.c_int64, ctypes.c_uint64], ctypes.c_int),
    "gdn2_step": ([ctypes.POINTER(Gdn2StepArgs), ctypes.c_void_p], ctypes.c_int),
    "mlstm_chunk_fwd": ([ctypes.POINTER(MlstmArgs), ctypes.c_void_p], ctypes.c_int),
    "mlstm_debug_arm_wait_fault": ([ctypes.c_int64, ctypes.c_uint64], ctypes.c_int),
    "mlstm_step": ([ctypes.POINTER(MlstmStepArgs), ctypes.c_void_p], ctypes.c_int),
}


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libssmscan.so for sm_103a (no-op when up to date)."""
    import importlib
    return importlib.import_module(__name__ + "._builder").build(force=force, verbose=verbose)


def lib():
    """The loaded CUDA library. Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: build it with selective_state_space_07_gb300.build()")
            h = ctypes.CDLL(LIB_PATH)
            for name, (argt, rest) in EXPORTS.items():
                f = getattr(h, name)
                f.argtypes = argt
                f.restype = rest
            _lib = h
    return _lib


def _p(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need(t, name, shape, dtype, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (the library reads raw row-major memory)")
    if t.numel() and t.data_ptr() % 16:
        raise ValueError(f"{name} must be 16-byte aligned")


def _opt(t, name, shape, dtype, device):
    if t is not None:
        _need(t, name, shape, dtype, device)
    return t


def _stream(device, stream):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def workspace_bytes(B: int, L: int, D: int, N: int = 16) -> int:
    return int(lib().ssm_scan_workspace_bytes(B, L, D, N))


def ckpt_elems(B: int, L: int, D: int, N: int = 16) -> int:
    return int(lib().ssm_scan_ckpt_elems(B, L, D, N))


def ckpt_states(ckpt: torch.Tensor, B: int, L: int, D: int, N: int = 16) -> torch.Tensor:
    """The checkpoint buffer as states [B, ceil(L/8), D, N] (a copy): entry [b, k] is the state [D, N]
    before token 8k of batch row b. The buffer itself is laid out [B, ceil(L/8), N/2, D, 2]."""
    nck = (L + CKPT_INTERVAL - 1) // CKPT_INTERVAL
    v = ckpt[: B * nck * N * D].view(B, nck, N // 2, D, 2)
    return v.permute(0, 1, 3, 2, 4).reshape(B, nck, D, N)


def arm_wait_fault(tile: int, wait_ns: int) -> None:
    """Testing hook: the next scan_fwd on this thread stages tile ``tile`` of every warp without issuing its
    copies and bounds its waits by ``wait_ns``; poll_status then reports the timeout."""
    _check(lib().ssm_debug_arm_wait_fault(int(tile), int(wait_ns)), "ssm_debug_arm_wait_fault")


def last_launch_count() -> int:
    """Kernels the library launched in the last fwd / bwd / step call of this thread."""
    return int(lib().ssm_last_launch_count())


class Workspace:
    """Caller-owned scratch for fwd / bwd: status word + carries along L."""

    def __init__(self, B: int, L: int, D: int, device, N: int = 16):
        self.nbytes = workspace_bytes(B, L, D, N)
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device)

    def fits(self, B, L, D, N=16) -> bool:
        return self.nbytes >= workspace_bytes(B, L, D, N)


def _ws(ws, B, L, D, device):
    if ws is None or not ws.fits(B, L, D):
        ws = Workspace(B, L, D, device)
    return ws


def _check(rc: int, where: str):
    if rc != 0:
        raise SsmError(rc, where)


def _fwd_struct(x, dt, A, Bm, Cm, z, Dskip, dt_bias, h0, delta_softplus, y, h_last, ckpt, ws, nsplit, groups):
    B, L, D = x.shape
    N = A.shape[1]
    return FwdArgs(B=B, L=L, D=D, N=N, io_dtype=_IO[x.dtype], delta_softplus=int(bool(delta_softplus)),
                   x=_p(x), z=_p(z), Bm=_p(Bm), Cm=_p(Cm), dt=_p(dt), dt_bias=_p(dt_bias), A=_p(A),
                   Dskip=_p(Dskip), h0=_p(h0), y=_p(y), h_last=_p(h_last), ckpt=_p(ckpt),
                   workspace=ws.buf.data_ptr(), workspace_bytes=ws.nbytes, nsplit=nsplit, groups=groups,
                   bc_stride=_bc_stride_pair(Bm, Cm, B, L, N))


def _token_rows(t, name, lead, N, dtype, device):
    """Check a [*lead, N] tensor whose rows (the last dim) are contiguous and evenly spaced, as in a column
    slice of the x_proj output; returns the row stride in elements."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(lead) + (N,):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(lead) + (N,)}")
    if t.numel() == 0:
        return N
    if N > 1 and t.stride(-1) != 1:
        raise ValueError(f"{name}: the {N} values of a row must be contiguous")
    # the row stride: rows of the flattened leading dims must be s elements apart
    s, span = None, 1
    for size, stride in zip(reversed(t.shape[:-1]), reversed(t.stride()[:-1])):
        if size > 1:
            if s is None:
                s = stride
            elif stride != s * span:
                raise ValueError(f"{name}: rows must be evenly spaced (a slice of a [rows, width] buffer)")
        span *= size
    s = N if s is None else s
    if s < N:
        raise ValueError(f"{name}: rows overlap (row stride {s} < {N})")
    if t.data_ptr() % 16 or (s * t.element_size()) % 16:
        raise ValueError(f"{name} must start on a 16-byte boundary with rows a multiple of 16 bytes apart")
    return s


def _bc_stride_pair(Bm, Cm, *lead_and_N):
    *lead, N = lead_and_N
    sb = _token_rows(Bm, "Bm", lead, N, Bm.dtype, Bm.device)
    sc = _token_rows(Cm, "Cm", lead, N, Bm.dtype, Bm.device)
    if sb != sc:
        raise ValueError(f"Bm and Cm must have the same row stride ({sb} != {sc})")
    return 0 if sb == N else sb


def _check_inputs(x, dt, A, Bm, Cm, z, Dskip, dt_bias, h0):
    if x.dim() != 3:
        raise ValueError("x must be [B, L, D]")
    B, L, D = x.shape
    dev, io = x.device, x.dtype
    if dev.type != "cuda":
        raise ValueError("the scan runs on a CUDA device; x is on " + str(dev))
    if io not in _IO:
        raise TypeError(f"x dtype must be float32 or bfloat16, got {io}")
    if A.dim() != 2 or A.shape[0] != D:
        raise ValueError("A must be [D, N]")
    N = A.shape[1]
    _need(x, "x", (B, L, D), io, dev)
    _need(dt, "dt", (B, L, D), torch.float32, dev)
    _need(A, "A", (D, N), torch.float32, dev)
    # Bm, Cm: dense [B, L, N], or column slices of the x_proj output (rows evenly spaced)
    _token_rows(Bm, "Bm", (B, L), N, io, dev)
    _token_rows(Cm, "Cm", (B, L), N, io, dev)
    _opt(z, "z", (B, L, D), io, dev)
    _opt(Dskip, "Dskip", (D,), torch.float32, dev)
    _opt(dt_bias, "dt_bias", (D,), torch.float32, dev)
    _opt(h0, "h0", (B, D, N), torch.float32, dev)
    return B, L, D, N, dev, io


def scan_fwd(x, dt, A, Bm, Cm, z=None, Dskip=None, dt_bias=None, h0=None, delta_softplus=True, *,
             return_last_state=False, save_ckpt=True, y=None, h_last=None, ckpt=None, workspace=None,
             nsplit=0, groups=0, stream=None):
    """Sequence forward. Returns (y, h_last or None, ckpt or None, workspace)."""
    B, L, D, N, dev, io = _check_inputs(x, dt, A, Bm, Cm, z, Dskip, dt_bias, h0)
    y = torch.empty_like(x) if y is None else y
    _need(y, "y", (B, L, D), io, dev)
    if return_last_state and h_last is None:
        h_last = torch.empty(B, D, N, dtype=torch.float32, device=dev)
    _opt(h_last, "h_last", (B, D, N), torch.float32, dev)
    if save_ckpt and ckpt is None:
        ckpt = torch.empty(max(1, ckpt_elems(B, L, D, N)), dtype=torch.float32, device=dev)
    if ckpt is not None and ckpt.numel() < ckpt_elems(B, L, D, N):
        raise ValueError("ckpt is smaller than ckpt_elems(B, L, D, N)")
    ws = _ws(workspace, B, L, D, dev)
    args = _fwd_struct(x, dt, A, Bm, Cm, z, Dskip, dt_bias, h0, delta_softplus, y, h_last, ckpt, ws, nsplit,
                       groups)
    _check(lib().ssm_scan_fwd(ctypes.byref(args), _stream(dev, stream)), "ssm_scan_fwd")
    return y, h_last, ckpt, ws


def scan_bwd(x, dt, A, Bm, Cm, dy, ckpt, z=None, Dskip=None, dt_bias=None, h0=None, dh_last=None,
             delta_softplus=True, *, return_dh0=False, inplace=False, out: Optional[Dict] = None,
             workspace=None, nsplit=0, groups=0, stream=None) -> Dict[str, torch.Tensor]:
    """Reverse pass for loss = <dy, y> + <dh_last, h_last>. Returns a dict with dx, dz (if z), d_dt,
    dA, dD, d_dt_bias, dB, dC and dh0 (if asked). ``inplace`` writes dx into dy, dz into z and d_dt
    into dt."""
    B, L, D, N, dev, io = _check_inputs(x, dt, A, Bm, Cm, z, Dskip, dt_bias, h0)
    _need(dy, "dy", (B, L, D), io, dev)
    _opt(dh_last, "dh_last", (B, D, N), torch.float32, dev)
    if ckpt is None or ckpt.numel() < ckpt_elems(B, L, D, N) or ckpt.dtype != torch.float32:
        raise ValueError("ckpt must be the fp32 checkpoint buffer scan_fwd filled")
    o = dict(out or {})
    if inplace:
        o.setdefault("dx", dy)
        o.setdefault("d_dt", dt)
        if z is not None:
            o.setdefault("dz", z)
    f32 = dict(dtype=torch.float32, device=dev)
    want = {"dx": lambda: torch.empty_like(x), "d_dt": lambda: torch.empty(B, L, D, **f32),
            "dA": lambda: torch.empty(D, N, **f32), "dD": lambda: torch.empty(D, **f32),
            "d_dt_bias": lambda: torch.empty(D, **f32), "dB": lambda: torch.empty(B, L, N, **f32),
            "dC": lambda: torch.empty(B, L, N, **f32)}
    if z is not None:
        want["dz"] = lambda: torch.empty_like(x)
    if return_dh0:
        want["dh0"] = lambda: torch.empty(B, D, N, **f32)
    for k, make in want.items():
        if k not in o:
            o[k] = make()
    for k, shp, dt_ in (("dx", (B, L, D), io), ("dz", (B, L, D), io), ("d_dt", (B, L, D), torch.float32),
                        ("dA", (D, N), torch.float32), ("dD", (D,), torch.float32),
                        ("d_dt_bias", (D,), torch.float32), ("dB", (B, L, N), torch.float32),
                        ("dC", (B, L, N), torch.float32), ("dh0", (B, D, N), torch.float32)):
        _opt(o.get(k), k, shp, dt_, dev)
    ws = _ws(workspace, B, L, D, dev)
    fa = _fwd_struct(x, dt, A, Bm, Cm, z, Dskip, dt_bias, h0, delta_softplus, None, None, ckpt, ws, nsplit,
                     groups)
    args = BwdArgs(f=fa, dy=_p(dy), dh_last=_p(dh_last), dx=_p(o["dx"]), dz=_p(o.get("dz")),
                   d_dt=_p(o["d_dt"]), dA=_p(o["dA"]), dD=_p(o["dD"]), d_dt_bias=_p(o["d_dt_bias"]),
                   dB=_p(o["dB"]), dC=_p(o["dC"]), dh0=_p(o.get("dh0")))
    _check(lib().ssm_scan_bwd(ctypes.byref(args), _stream(dev, stream)), "ssm_scan_bwd")
    o["workspace"] = ws
    return o


def step(state, x_t, dt_t, A, Bm_t, Cm_t, z_t=None, Dskip=None, dt_bias=None, delta_softplus=True, *,
         y_t=None, workspace=None, nsplit=0, stream=None):
    """One token for every channel; ``state`` [B, D, 16] fp32 is updated in place. Returns y_t [B, D]."""
    if x_t.dim() != 2:
        raise ValueError("x_t must be [B, D]")
    B, D = x_t.shape
    dev, io = x_t.device, x_t.dtype
    if dev.type != "cuda":
        raise ValueError("the step runs on a CUDA device; x_t is on " + str(dev))
    if io not in _IO:
        raise TypeError(f"x_t dtype must be float32 or bfloat16, got {io}")
    N = A.shape[1]
    _need(state, "state", (B, D, N), torch.float32, dev)
    _need(x_t, "x_t", (B, D), io, dev)
    _need(dt_t, "dt_t", (B, D), torch.float32, dev)
    _need(A, "A", (D, N), torch.float32, dev)
    _token_rows(Bm_t, "Bm_t", (B,), N, io, dev)
    _token_rows(Cm_t, "Cm_t", (B,), N, io, dev)
    _opt(z_t, "z_t", (B, D), io, dev)
    _opt(Dskip, "Dskip", (D,), torch.float32, dev)
    _opt(dt_bias, "dt_bias", (D,), torch.float32, dev)
    y_t = torch.empty_like(x_t) if y_t is None else y_t
    _need(y_t, "y_t", (B, D), io, dev)
    args = StepArgs(B=B, D=D, N=N, io_dtype=_IO[io], delta_softplus=int(bool(delta_softplus)), x_t=_p(x_t),
                    z_t=_p(z_t), Bm_t=_p(Bm_t), Cm_t=_p(Cm_t), dt_t=_p(dt_t), dt_bias=_p(dt_bias), A=_p(A),
                    Dskip=_p(Dskip), state=_p(state), y_t=_p(y_t),
                    workspace=None if workspace is None else workspace.buf.data_ptr(), nsplit=nsplit,
                    bc_stride=_bc_stride_pair(Bm_t, Cm_t, B, N))
    _check(lib().ssm_step(ctypes.byref(args), _stream(dev, stream)), "ssm_step")
    return y_t


def dA_log_grad(dA, A, out=None, stream=None):
    """Gradient of A_log for A = -exp(A_log): dA_log = dA * A (elementwise, on the GPU)."""
    _need(A, "A", tuple(A.shape), torch.float32, A.device)
    _need(dA, "dA", tuple(A.shape), torch.float32, A.device)
    out = torch.empty_like(A) if out is None else out
    _need(out, "out", tuple(A.shape), torch.float32, A.device)
    _check(lib().ssm_dA_log_grad(_p(dA), _p(A), _p(out), A.numel(), _stream(A.device, stream)),
           "ssm_dA_log_grad")
    return out


def _conv_struct(xin, w, bias, state_in, x, state_out, workspace):
    if xin.dim() != 3:
        raise ValueError("xin must be [B, L, D]")
    B, L, D = xin.shape
    dev, io = xin.device, xin.dtype
    if dev.type != "cuda":
        raise ValueError("the conv runs on a CUDA device; xin is on " + str(dev))
    if io not in _IO:
        raise TypeError(f"xin dtype must be float32 or bfloat16, got {io}")
    if w.dim() != 2 or w.shape[0] != D:
        raise ValueError("w must be [D, K]")
    K = w.shape[1]
    _need(xin, "xin", (B, L, D), io, dev)
    _need(w, "w", (D, K), torch.float32, dev)
    _opt(bias, "bias", (D,), torch.float32, dev)
    _opt(state_in, "state_in", (B, D, K - 1), torch.float32, dev)
    _opt(x, "x", (B, L, D), io, dev)
    _opt(state_out, "state_out", (B, D, K - 1), torch.float32, dev)
    return ConvArgs(B=B, L=L, D=D, K=K, io_dtype=_IO[io], xin=_p(xin), w=_p(w), bias=_p(bias),
                    state_in=_p(state_in), x=_p(x), state_out=_p(state_out),
                    workspace=None if workspace is None else workspace.buf.data_ptr())


def conv1d_fwd(xin, w, bias=None, state_in=None, *, x=None, state_out=None, want_state=False, workspace=None,
               stream=None):
    """Causal depthwise conv1d + SiLU in front of the scan:
    x[b,t,d] = silu(bias[d] + sum_k w[d,k] * xin[b, t-(K-1)+k, d]), with the K-1 inputs before t = 0 taken
    from ``state_in`` [B, D, K-1] (zeros when None). xin, x [B, L, D] fp32 or bf16; w [D, K] fp32, K <= 4;
    D a multiple of 8. Returns (x, state_out); state_out ([B, D, K-1], the last K-1 inputs) is None unless
    given or ``want_state``."""
    B, L, D = xin.shape
    K = w.shape[1] if w.dim() == 2 else 0
    x = torch.empty_like(xin) if x is None else x
    if state_out is None and want_state:
        state_out = torch.empty(B, D, max(K - 1, 0), dtype=torch.float32, device=xin.device)
    args = _conv_struct(xin, w, bias, state_in, x, state_out, workspace)
    _check(lib().ssm_conv1d_fwd(ctypes.byref(args), _stream(xin.device, stream)), "ssm_conv1d_fwd")
    return x, state_out


def conv1d_bwd(xin, w, dx, bias=None, state_in=None, *, dxin=None, want_dstate=False, workspace=None,
               stream=None):
    """Reverse pass of conv1d_fwd for loss = <dx, x>. Returns dict dxin [B, L, D] (xin's dtype), dw [D, K],
    dbias [D] (when ``bias`` is given) and dstate_in [B, D, K-1] (when ``want_dstate``), all fp32 but dxin."""
    B, L, D = xin.shape
    K = w.shape[1] if w.dim() == 2 else 0
    dev = xin.device
    f = _conv_struct(xin, w, bias, state_in, None, None, workspace)
    _need(dx, "dx", (B, L, D), xin.dtype, dev)
    dxin = torch.empty_like(xin) if dxin is None else dxin
    _need(dxin, "dxin", (B, L, D), xin.dtype, dev)
    dw = torch.empty(D, K, dtype=torch.float32, device=dev)
    dbias = torch.empty(D, dtype=torch.float32, device=dev) if bias is not None else None
    dstate = torch.empty(B, D, max(K - 1, 0), dtype=torch.float32, device=dev) if want_dstate else None
    args = ConvBwdArgs(f=f, dx=_p(dx), dxin=_p(dxin), dw=_p(dw), dbias=_p(dbias), dstate_in=_p(dstate))
    _check(lib().ssm_conv1d_bwd(ctypes.byref(args), _stream(dev, stream)), "ssm_conv1d_bwd")
    return {"dxin": dxin, "dw": dw, "dbias": dbias, "dstate_in": dstate}


def conv1d_step(ring, xin_t, w, bias=None, *, x_t=None, workspace=None, stream=None):
    """One decoding token through the conv: ``ring`` [B, D, K-1] fp32 (the last K-1 inputs, oldest first)
    is read and then advanced in place. xin_t [B, D]; returns x_t [B, D]."""
    if xin_t.dim() != 2:
        raise ValueError("xin_t must be [B, D]")
    B, D = xin_t.shape
    xin = xin_t.view(B, 1, D)
    x = torch.empty_like(xin) if x_t is None else x_t.view(B, 1, D)
    conv1d_fwd(xin, w, bias, ring, x=x, state_out=ring, workspace=workspace, stream=stream)
    return x.view(B, D)


def _dtproj_struct(a, w, bias, softplus, delta, workspace):
    if a.dim() < 2:
        raise ValueError("a must be [..., R] (e.g. [B, L, R] columns of the x_proj output)")
    dev = a.device
    if dev.type != "cuda":
        raise ValueError("the dt projection runs on a CUDA device; a is on " + str(dev))
    lead, R = tuple(a.shape[:-1]), a.shape[-1]
    M = 1
    for v in lead:
        M *= v
    if w.dim() != 2 or w.shape[1] != R:
        raise ValueError("w must be [D, R]")
    D = w.shape[0]
    stride = _token_rows(a, "a", lead, R, torch.bfloat16, dev)
    _need(w, "w", (D, R), torch.bfloat16, dev)
    _opt(bias, "bias", (D,), torch.float32, dev)
    _opt(delta, "delta", lead + (D,), torch.float32, dev)
    args = DtProjArgs(M=M, D=D, R=R, a_stride=0 if stride == R else stride, softplus=int(bool(softplus)),
                      a=_p(a), w=_p(w), bias=_p(bias), delta=_p(delta),
                      workspace=None if workspace is None else workspace.buf.data_ptr())
    return args, lead, D


def dtproj_fwd(a, w, bias=None, softplus=True, *, delta=None, workspace=None, stream=None):
    """The dt projection with its softplus on the tensor cores: delta = softplus(a @ w.T + bias), fp32
    [..., D]. a [..., R] bf16 may be the first R columns of the x_proj output (rows evenly spaced,
    16-byte aligned); w [D, R] bf16; bias [D] fp32. Feed delta to scan_fwd as dt with
    delta_softplus=False and no dt_bias."""
    lead, D = tuple(a.shape[:-1]), w.shape[0]
    delta = torch.empty(lead + (D,), dtype=torch.float32, device=a.device) if delta is None else delta
    args, _, _ = _dtproj_struct(a, w, bias, softplus, delta, workspace)
    _check(lib().ssm_dtproj_fwd(ctypes.byref(args), _stream(a.device, stream)), "ssm_dtproj_fwd")
    return delta


def dtproj_bwd(a, w, ddelta, bias=None, softplus=True, *, dpre=None, inplace=False, workspace=None, stream=None):
    """Reverse pass up to the pre-activation: dpre = ddelta * sigmoid(a @ w.T + bias) (recomputed on the
    tensor cores) and dbias = dpre summed over rows (None without a bias). The gradients of a and w are
    dpre @ w and dpre^T @ a. ``inplace`` writes dpre over ddelta."""
    args, lead, D = _dtproj_struct(a, w, bias, softplus, None, workspace)
    _need(ddelta, "ddelta", lead + (D,), torch.float32, a.device)
    dpre = ddelta if inplace else (torch.empty_like(ddelta) if dpre is None else dpre)
    _need(dpre, "dpre", lead + (D,), torch.float32, a.device)
    dbias = torch.empty(D, dtype=torch.float32, device=a.device) if bias is not None else None
    bargs = DtProjBwdArgs(f=args, ddelta=_p(ddelta), dpre=_p(dpre), dbias=_p(dbias))
    _check(lib().ssm_dtproj_bwd(ctypes.byref(bargs), _stream(a.device, stream)), "ssm_dtproj_bwd")
    return {"dpre": dpre, "dbias": dbias}


def gdn2_fwd(q, k, v, g, b, w, state=None, scale=None, *, out=None, state_out=None, want_state=True,
             workspace=None, stream=None):
    """Gated DeltaNet-2 chunkwise forward (C ABI in ``include/gdn2.h``; docs.rs, burn-gdn2 0.1.4,
    src/forward.rs, chunk_wy_forward) on the tensor cores, chunks of 64 tokens.
    q, k, b [B, H, T, 128] bf16; g [B, H, T, 128] fp32 log-gates; v, w [B, H, T, 128] bf16;
    state [B, H, 128, 128] fp32 or None (zeros); scale defaults to 1/sqrt(K).
    Returns (out [B, H, T, V] bf16, final state [B, H, K, V] fp32 or None)."""
    if q.dim() != 4:
        raise ValueError("q must be [B, H, T, K]")
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("the GDN2 forward runs on a CUDA device; q is on " + str(dev))
    Bn, H, T, K = q.shape
    V = v.shape[-1] if v.dim() == 4 else -1
    bf, f32 = torch.bfloat16, torch.float32
    for t, n in ((q, "q"), (k, "k"), (b, "b")):
        _need(t, n, (Bn, H, T, K), bf, dev)
    _need(g, "g", (Bn, H, T, K), f32, dev)
    for t, n in ((v, "v"), (w, "w")):
        _need(t, n, (Bn, H, T, V), bf, dev)
    _opt(state, "state", (Bn, H, K, V), f32, dev)
    out = torch.empty((Bn, H, T, V), dtype=bf, device=dev) if out is None else out
    _need(out, "out", (Bn, H, T, V), bf, dev)
    if want_state and state_out is None:
        state_out = torch.empty((Bn, H, K, V), dtype=f32, device=dev)
    _opt(state_out, "state_out", (Bn, H, K, V), f32, dev)
    args = Gdn2Args(B=Bn, H=H, T=T, K=K, V=V, chunk=GDN2_CHUNK,
                    scale=float(K ** -0.5 if scale is None else scale),
                    q=_p(q), k=_p(k), v=_p(v), g=_p(g), b=_p(b), w=_p(w), state_in=_p(state), out=_p(out),
                    state_out=_p(state_out), workspace=None if workspace is None else workspace.buf.data_ptr())
    _check(lib().gdn2_chunk_fwd(ctypes.byref(args), _stream(dev, stream)), "gdn2_chunk_fwd")
    return out, state_out


def gdn2_step(q, k, v, g, b, w, state, scale=None, *, out=None, workspace=None, stream=None):
    """One token of the Gated DeltaNet-2 mixer, the per-token form (C ABI in ``include/gdn2.h``): q, k, b [B, H, 128]
    bf16; g [B, H, 128] fp32 log-gates; v, w [B, H, 128] bf16; state [B, H, 128, 128] fp32, updated in place;
    scale defaults to 1/sqrt(K). Returns out [B, H, V] bf16."""
    if q.dim() != 3:
        raise ValueError("q must be [B, H, K]")
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("the GDN2 step runs on a CUDA device; q is on " + str(dev))
    Bn, H, K = q.shape
    V = v.shape[-1] if v.dim() == 3 else -1
    bf, f32 = torch.bfloat16, torch.float32
    for t, n in ((q, "q"), (k, "k"), (b, "b")):
        _need(t, n, (Bn, H, K), bf, dev)
    _need(g, "g", (Bn, H, K), f32, dev)
    for t, n in ((v, "v"), (w, "w")):
        _need(t, n, (Bn, H, V), bf, dev)
    _need(state, "state", (Bn, H, K, V), f32, dev)
    out = torch.empty((Bn, H, V), dtype=bf, device=dev) if out is None else out
    _need(out, "out", (Bn, H, V), bf, dev)
    args = Gdn2StepArgs(B=Bn, H=H, K=K, V=V, scale=float(K ** -0.5 if scale is None else scale), q=_p(q), k=_p(k),
                        v=_p(v), g=_p(g), b=_p(b), w=_p(w), state=_p(state), out=_p(out),
                        workspace=None if workspace is None else workspace.buf.data_ptr())
    _check(lib().gdn2_step(ctypes.byref(args), _stream(dev, stream)), "gdn2_step")
    return out


def gdn2_arm_wait_fault(chunk: int, wait_ns: int) -> None:
    """Test hook: the next gdn2_fwd of this thread does not issue chunk `chunk`'s q, k, b copies and bounds every
    wait by wait_ns, so the call ends with SSM_ERR_TIMEOUT in the status word. chunk < 0 disarms."""
    _check(lib().gdn2_debug_arm_wait_fault(int(chunk), int(wait_ns)), "gdn2_debug_arm_wait_fault")


def mlstm_fwd(q, k, v, igate, fgate, state=None, scale=None, *, norm_weight=None, norm_eps=1e-5, h=None,
              state_out=None, want_state=True, workspace=None, stream=None):
    """mLSTM stabilized chunkwise forward (C ABI in ``include/mlstm.h``; Evil-Inference-Code,
    README_FIX_RUST.md, "mLSTM Equivalence Fixes (Rust vs Python)") on the tensor cores, chunks of 64 tokens.
    q, k [B, H, T, 128] bf16; v [B, H, T, 128] bf16; igate, fgate [B, H, T] fp32 gate pre-activations;
    state = (C [B, H, 128, 128], n [B, H, 128], m [B, H]) fp32 stabilized, or None (zeros, m = 0);
    norm_weight [H, 128] fp32 applies the head-wise norm (no bias) to h; scale defaults to 1/sqrt(K).
    Returns (h [B, H, T, V] bf16, final state (C, n, m) or None)."""
    if q.dim() != 4:
        raise ValueError("q must be [B, H, T, K]")
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("the mLSTM forward runs on a CUDA device; q is on " + str(dev))
    Bn, H, T, K = q.shape
    V = v.shape[-1] if v.dim() == 4 else -1
    bf, f32 = torch.bfloat16, torch.float32
    _need(q, "q", (Bn, H, T, K), bf, dev)
    _need(k, "k", (Bn, H, T, K), bf, dev)
    _need(v, "v", (Bn, H, T, V), bf, dev)
    _need(igate, "igate", (Bn, H, T), f32, dev)
    _need(fgate, "fgate", (Bn, H, T), f32, dev)
    shapes = ((Bn, H, K, V), (Bn, H, K), (Bn, H))
    if state is not None:
        if len(state) != 3:
            raise ValueError("state must be (C, n, m)")
        for t, n, shp in zip(state, ("C", "n", "m"), shapes):
            _need(t, n, shp, f32, dev)
    if norm_weight is not None:
        _need(norm_weight, "norm_weight", (H, V), f32, dev)
    h = torch.empty((Bn, H, T, V), dtype=bf, device=dev) if h is None else h
    _need(h, "h", (Bn, H, T, V), bf, dev)
    if want_state and state_out is None:
        state_out = tuple(torch.empty(shp, dtype=f32, device=dev) for shp in shapes)
    if state_out is not None:
        for t, n, shp in zip(state_out, ("C_out", "n_out", "m_out"), shapes):
            _need(t, n, shp, f32, dev)
    si = state if state is not None else (None, None, None)
    so = state_out if state_out is not None else (None, None, None)
    args = MlstmArgs(B=Bn, H=H, T=T, K=K, V=V, chunk=MLSTM_CHUNK,
                     scale=float(K ** -0.5 if scale is None else scale), norm_eps=float(norm_eps),
                     q=_p(q), k=_p(k), v=_p(v), igate=_p(igate), fgate=_p(fgate),
                     C_in=_p(si[0]), n_in=_p(si[1]), m_in=_p(si[2]), norm_weight=_p(norm_weight), h=_p(h),
                     C_out=_p(so[0]), n_out=_p(so[1]), m_out=_p(so[2]),
                     workspace=None if workspace is None else workspace.buf.data_ptr())
    _check(lib().mlstm_chunk_fwd(ctypes.byref(args), _stream(dev, stream)), "mlstm_chunk_fwd")
    return h, state_out


def mlstm_step(q, k, v, igate, fgate, state, scale=None, *, norm_weight=None, norm_eps=1e-5, h=None, workspace=None,
               stream=None):
    """One token of the mLSTM cell, the recurrent step (C ABI in ``include/mlstm.h``): q, k [B, H, 128] and v
    [B, H, 128] bf16; igate, fgate [B, H] fp32 gate pre-activations; state = (C [B, H, 128, 128], n [B, H, 128],
    m [B, H]) fp32 stabilized, updated in place (zeros and m = 0 for a fresh sequence); norm_weight [H, 128] fp32
    applies the head-wise norm; scale defaults to 1/sqrt(K). Returns h [B, H, V] bf16."""
    if q.dim() != 3:
        raise ValueError("q must be [B, H, K]")
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("the mLSTM step runs on a CUDA device; q is on " + str(dev))
    Bn, H, K = q.shape
    V = v.shape[-1] if v.dim() == 3 else -1
    bf, f32 = torch.bfloat16, torch.float32
    _need(q, "q", (Bn, H, K), bf, dev)
    _need(k, "k", (Bn, H, K), bf, dev)
    _need(v, "v", (Bn, H, V), bf, dev)
    _need(igate, "igate", (Bn, H), f32, dev)
    _need(fgate, "fgate", (Bn, H), f32, dev)
    if state is None or len(state) != 3:
        raise ValueError("state must be (C, n, m)")
    for t, n, shp in zip(state, ("C", "n", "m"), ((Bn, H, K, V), (Bn, H, K), (Bn, H))):
        _need(t, n, shp, f32, dev)
    if norm_weight is not None:
        _need(norm_weight, "norm_weight", (H, V), f32, dev)
    h = torch.empty((Bn, H, V), dtype=bf, device=dev) if h is None else h
    _need(h, "h", (Bn, H, V), bf, dev)
    args = MlstmStepArgs(B=Bn, H=H, K=K, V=V, scale=float(K ** -0.5 if scale is None else scale),
                         norm_eps=float(norm_eps), q=_p(q), k=_p(k), v=_p(v), igate=_p(igate), fgate=_p(fgate),
                         C=_p(state[0]), n=_p(state[1]), m=_p(state[2]), norm_weight=_p(norm_weight), h=_p(h),
                         workspace=None if workspace is None else workspace.buf.data_ptr())
    _check(lib().mlstm_step(ctypes.byref(args), _stream(dev, stream)), "mlstm_step")
    return h


def mlstm_arm_wait_fault(chunk: int, wait_ns: int) -> None:
    """Test hook: the next mlstm_fwd of this thread does not issue chunk `chunk`'s q copy and bounds every
    wait by wait_ns, so the call ends with SSM_ERR_TIMEOUT in the status word. chunk < 0 disarms."""
    _check(lib().mlstm_debug_arm_wait_fault(int(chunk), int(wait_ns)), "mlstm_debug_arm_wait_fault")


def exp2_fma(x, *, out=None, stream=None):
    """The library's FMA-pipe 2^x (Cody-Waite split + degree-6 polynomial; C ABI ssm_exp2_fma) on an fp32
    device tensor: for tests and error-bound checks of the exponential a kernel can use instead of the MUFU."""
    if not isinstance(x, torch.Tensor) or x.dtype != torch.float32 or x.device.type != "cuda" or not x.is_contiguous():
        raise TypeError("x must be a contiguous fp32 CUDA tensor")
    out = torch.empty_like(x) if out is None else out
    _need(out, "out", tuple(x.shape), torch.float32, x.device)
    _check(lib().ssm_exp2_fma(_p(x), _p(out), x.numel(), _stream(x.device, stream)), "ssm_exp2_fma")
    return out


def poll_status(workspace, stream=None) -> int:
    """Synchronise, read and clear the status word. 0 = ok, -7 = non-finite output seen, -6 = a bounded
    wait inside a kernel ran out."""
    dev = workspace.buf.device
    return int(lib().ssm_poll_status(workspace.buf.data_ptr(), _stream(dev, stream)))


def clear_status(workspace, stream=None) -> None:
    dev = workspace.buf.device
    _check(lib().ssm_clear_status(workspace.buf.data_ptr(), _stream(dev, stream)), "ssm_clear_status")


class HostPipeline:
    """Back-to-back end-to-end calls for host callers, overlapped.

    Each ``step`` copies one batch of inputs from pinned host memory to the
    device, runs ssm_scan_fwd and ssm_scan_bwd, and copies y and every
    gradient back into the pinned ``results`` buffers; it returns without
    waiting. Copies in, compute and copies out run on three streams over two
    sets of device buffers, so step k's inputs travel while step k-1
    computes and step k-2's results travel back (the host link carries both
    directions at once). Within a step the forward starts once its own
    inputs are in (dy follows), and y leaves while the backward runs.
    ``synchronize`` waits for every enqueued step; results of a step are
    valid after it."""

    _FWD_INPUTS = ("x", "dt", "A", "Bm", "Cm", "z", "Dskip", "dt_bias")

    def __init__(self, host: Dict[str, torch.Tensor], device, delta_softplus=True, depth=2):
        self.dev = torch.device(device)
        self.sp = delta_softplus
        self.depth = depth
        self.s_in, self.s_comp, self.s_out = (torch.cuda.Stream(self.dev) for _ in range(3))
        self.sets = []
        for _ in range(depth):
            # one plain call per set allocates (and zero-fills) every device
            # buffer up front, so no allocation happens on the pipeline's streams
            res, d = scan_fwd_bwd_host(host, self.dev, delta_softplus=delta_softplus)
            ev = {n: torch.cuda.Event() for n in ("in_fwd", "in_bwd", "fwd", "bwd", "out")}
            self.sets.append({"dev": d, "ev": ev, "used": False})
        torch.cuda.synchronize(self.dev)
        self.k = 0

    def step(self, host: Dict[str, torch.Tensor], results: Optional[Dict] = None) -> Dict[str, torch.Tensor]:
        st = self.sets[self.k % self.depth]
        self.k += 1
        d, ev = st["dev"], st["ev"]
        if st["used"]:
            self.s_in.wait_event(ev["bwd"])     # the set's inputs are no longer read
        with torch.cuda.stream(self.s_in):
            for k in self._FWD_INPUTS:
                if host.get(k) is not None:
                    d[k].copy_(host[k], non_blocking=True)
            ev["in_fwd"].record(self.s_in)
            d["dy"].copy_(host["dy"], non_blocking=True)
            ev["in_bwd"].record(self.s_in)
        self.s_comp.wait_event(ev["in_fwd"])
        if st["used"]:
            self.s_comp.wait_event(ev["out"])   # the set's outputs have left
        y, _, ck, ws = scan_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d.get("z"), d.get("Dskip"),
                                d.get("dt_bias"), None, self.sp, y=d.get("y"), ckpt=d.get("ckpt"),
                                workspace=d.get("ws"), stream=self.s_comp)
        d["y"], d["ckpt"], d["ws"] = y, ck, ws
        ev["fwd"].record(self.s_comp)
        self.s_comp.wait_event(ev["in_bwd"])
        g = scan_bwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["dy"], ck, d.get("z"), d.get("Dskip"),
                     d.get("dt_bias"), None, None, self.sp, out=d.get("grads"), workspace=ws, stream=self.s_comp)
        g.pop("workspace", None)
        d["grads"] = g
        ev["bwd"].record(self.s_comp)
        if results is None:
            results = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in {"y": y, **g}.items()}
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(ev["fwd"])
            results["y"].copy_(y, non_blocking=True)
            self.s_out.wait_event(ev["bwd"])
            for k, v in g.items():
                results[k].copy_(v, non_blocking=True)
            ev["out"].record(self.s_out)
        st["used"] = True
        return results

    def synchronize(self):
        for s_ in (self.s_in, self.s_comp, self.s_out):
            s_.synchronize()


def scan_fwd_bwd_host(host: Dict[str, torch.Tensor], device, *, dev_buffers: Optional[Dict] = None,
                      results: Optional[Dict] = None, stream=None, delta_softplus=True):
    """End-to-end call for host callers: copies the inputs from (pinned) host memory to the device,
    runs ssm_scan_fwd then ssm_scan_bwd, and copies y and every gradient back to host memory.
    ``host`` holds x, dt, A, Bm, Cm, z, Dskip, dt_bias, dy as CPU tensors. Device buffers and
    pinned result buffers are reused when passed in. Returns (results, dev_buffers)."""
    s = stream if stream is not None else torch.cuda.current_stream(device)
    dv = dev_buffers if dev_buffers is not None else {
        k: torch.empty(v.shape, dtype=v.dtype, device=device) for k, v in host.items() if v is not None}
    with torch.cuda.stream(s):
        for k, v in host.items():
            if v is not None:
                dv[k].copy_(v, non_blocking=True)
        y, _, ckpt, ws = scan_fwd(dv["x"], dv["dt"], dv["A"], dv["Bm"], dv["Cm"], dv.get("z"), dv.get("Dskip"),
                                  dv.get("dt_bias"), None, delta_softplus, y=dv.get("y"), ckpt=dv.get("ckpt"),
                                  workspace=dv.get("ws"), stream=s)
        dv["y"], dv["ckpt"], dv["ws"] = y, ckpt, ws
        g = scan_bwd(dv["x"], dv["dt"], dv["A"], dv["Bm"], dv["Cm"], dv["dy"], ckpt, dv.get("z"),
                     dv.get("Dskip"), dv.get("dt_bias"), None, None, delta_softplus, out=dv.get("grads"),
                     workspace=ws, stream=s)
        g.pop("workspace", None)
        dv["grads"] = g
        outs = {"y": y, **g}
        if results is None:
            results = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in outs.items()}
        for k, v in outs.items():
            results[k].copy_(v, non_blocking=True)
    return results, dv
