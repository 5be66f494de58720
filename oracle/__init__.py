"""CPU oracle for the S6 selective scan -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (the
``selective_state_space_07_gb300`` package and its CUDA library) never does.

The arithmetic lives in ``ssm_oracle.cpp`` (plain sequential C++, built here
with g++ -O2 -ffp-contract=off). This module only builds that file, marshals
numpy arrays and calls it. Parity status: every function is pinned by the
``-m "not gpu"`` tests in ``tests/test_oracle_pins.py`` (closed forms,
brute-force quadratic form, special cases, finite differences, adjoint and
step identities) and, for the conv1d + SiLU in front of the scan
(``conv_oracle.cpp``), in ``tests/test_conv_oracle_pins.py`` (numpy's
convolution, special kernels, causality, state chaining, finite
differences), and, for the dt projection with its softplus
(``dtproj_oracle.cpp``), in ``tests/test_dtproj_oracle_pins.py`` (numpy's
matrix product, softplus identities, finite differences); none is "parity
unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.cpp")
_SRCS = [_SRC, os.path.join(_HERE, "conv_oracle.cpp"), os.path.join(_HERE, "dtproj_oracle.cpp")]
_LIB = os.path.join(_HERE, "libssm_oracle.so")
_lock = threading.Lock()
_lib = None

CXXFLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
            "-pthread"]


def build(force: bool = False) -> str:
    """Compile the oracle library if it is missing or older than its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(os.path.getmtime(f) for f in _SRCS):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", *CXXFLAGS, *_SRCS, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


class _Args(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("L", ctypes.c_int64), ("D", ctypes.c_int64),
                ("N", ctypes.c_int64), ("delta_softplus", ctypes.c_int32),
                ("threads", ctypes.c_int32)] + [
        (name, ctypes.c_void_p) for name in (
            "x", "dt", "z", "Bm", "Cm", "A", "Dskip", "dt_bias", "h0", "y", "h_last", "dy",
            "dh_last", "dx", "ddt", "dz", "dA", "dD", "ddt_bias", "dB", "dC", "dh0", "ddelta")]


class _StepArgs(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("D", ctypes.c_int64), ("N", ctypes.c_int64),
                ("delta_softplus", ctypes.c_int32), ("pad_", ctypes.c_int32)] + [
        (name, ctypes.c_void_p) for name in (
            "x_t", "dt_t", "z_t", "Bm_t", "Cm_t", "A", "Dskip", "dt_bias", "state", "y_t")]


class _ConvArgs(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("L", ctypes.c_int64), ("D", ctypes.c_int64), ("K", ctypes.c_int64)] + [
        (name, ctypes.c_void_p) for name in (
            "xin", "w", "bias", "state", "x", "state_out", "dx", "dxin", "dw", "dbias", "dstate")]


class _DtProjArgs(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("D", ctypes.c_int64), ("R", ctypes.c_int64),
                ("softplus", ctypes.c_int32), ("pad_", ctypes.c_int32)] + [
        (name, ctypes.c_void_p) for name in ("a", "w", "bias", "delta", "ddelta", "dpre", "dbias")]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            for name in ("fwd", "bwd"):
                for dt in ("f64", "f32"):
                    f = getattr(_lib, f"ssm_oracle_{name}_{dt}")
                    f.argtypes = [ctypes.POINTER(_Args)]
                    f.restype = ctypes.c_int
            for dt in ("f64", "f32"):
                f = getattr(_lib, f"ssm_oracle_step_{dt}")
                f.argtypes = [ctypes.POINTER(_StepArgs)]
                f.restype = ctypes.c_int
            _lib.ssm_oracle_hardware_threads.restype = ctypes.c_int
            for name in ("fwd", "bwd"):
                for dt in ("f64", "f32"):
                    f = getattr(_lib, f"conv_oracle_{name}_{dt}")
                    f.argtypes = [ctypes.POINTER(_ConvArgs)]
                    f.restype = ctypes.c_int
                    f = getattr(_lib, f"dtproj_oracle_{name}_{dt}")
                    f.argtypes = [ctypes.POINTER(_DtProjArgs)]
                    f.restype = ctypes.c_int
    return _lib


def hardware_threads() -> int:
    return int(lib().ssm_oracle_hardware_threads())


def _np(a, dtype):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def _ptr(a) -> Optional[int]:
    return None if a is None else a.ctypes.data


_NP = {"f64": np.float64, "f32": np.float32}


def _fill(args, keep, dtype, **arrays):
    for k, v in arrays.items():
        a = _np(v, dtype)
        keep.append(a)
        setattr(args, k, _ptr(a))


def fwd(inp, dtype: str = "f64", threads: int = 0, *, h0="inp") -> Dict[str, np.ndarray]:
    """Sequence forward. Returns y [B,L,D] and h_last [B,D,N]."""
    t = _NP[dtype]
    B, L, D, N = inp.B, inp.L, inp.D, inp.N
    args = _Args(B=B, L=L, D=D, N=N, delta_softplus=inp.delta_softplus, threads=threads)
    keep = []
    _fill(args, keep, t, x=inp.x, dt=inp.dt, z=inp.z, Bm=inp.Bm, Cm=inp.Cm, A=inp.A,
          Dskip=inp.Dskip, dt_bias=inp.dt_bias, h0=inp.h0 if h0 == "inp" else h0)
    y = np.zeros((B, L, D), t)
    h_last = np.zeros((B, D, N), t)
    args.y, args.h_last = _ptr(y), _ptr(h_last)
    rc = getattr(lib(), f"ssm_oracle_fwd_{dtype}")(ctypes.byref(args))
    if rc != 0:
        raise ValueError(f"oracle fwd rejected the arguments ({rc})")
    return {"y": y, "h_last": h_last}


def bwd(inp, dtype: str = "f64", threads: int = 0) -> Dict[str, np.ndarray]:
    """Reverse pass for loss = <dy, y> + <dh_last, h_last>. Returns dx, ddt, dz,
    dA, dD, ddt_bias, dB, dC, dh0 and ddelta (dLoss/dDelta before softplus'
    chain rule)."""
    t = _NP[dtype]
    B, L, D, N = inp.B, inp.L, inp.D, inp.N
    args = _Args(B=B, L=L, D=D, N=N, delta_softplus=inp.delta_softplus, threads=threads)
    keep = []
    _fill(args, keep, t, x=inp.x, dt=inp.dt, z=inp.z, Bm=inp.Bm, Cm=inp.Cm, A=inp.A,
          Dskip=inp.Dskip, dt_bias=inp.dt_bias, h0=inp.h0, dy=inp.dy, dh_last=inp.dh_last)
    out = {
        "dx": np.zeros((B, L, D), t), "ddt": np.zeros((B, L, D), t),
        "dz": np.zeros((B, L, D), t) if inp.z is not None else None,
        "dA": np.zeros((D, N), t), "dD": np.zeros((D,), t), "ddt_bias": np.zeros((D,), t),
        "dB": np.zeros((B, L, N), t), "dC": np.zeros((B, L, N), t),
        "dh0": np.zeros((B, D, N), t), "ddelta": np.zeros((B, L, D), t),
    }
    for k, v in out.items():
        setattr(args, k, _ptr(v))
    rc = getattr(lib(), f"ssm_oracle_bwd_{dtype}")(ctypes.byref(args))
    if rc != 0:
        raise ValueError(f"oracle bwd rejected the arguments ({rc})")
    return out


def step(state: np.ndarray, x_t, dt_t, z_t, Bm_t, Cm_t, A, Dskip, dt_bias,
         delta_softplus: int = 1, dtype: str = "f64") -> np.ndarray:
    """One token for every (b,d). ``state`` [B,D,N] (of the oracle's dtype,
    contiguous) is updated in place; returns y_t [B,D]."""
    t = _NP[dtype]
    assert state.dtype == t and state.flags.c_contiguous
    B, D, N = state.shape
    args = _StepArgs(B=B, D=D, N=N, delta_softplus=delta_softplus)
    keep = []
    _fill(args, keep, t, x_t=x_t, dt_t=dt_t, z_t=z_t, Bm_t=Bm_t, Cm_t=Cm_t, A=A, Dskip=Dskip,
          dt_bias=dt_bias)
    y = np.zeros((B, D), t)
    args.state, args.y_t = _ptr(state), _ptr(y)
    rc = getattr(lib(), f"ssm_oracle_step_{dtype}")(ctypes.byref(args))
    if rc != 0:
        raise ValueError(f"oracle step rejected the arguments ({rc})")
    return y


def conv_fwd(xin, w, bias=None, state=None, dtype: str = "f64") -> Dict[str, np.ndarray]:
    """Causal depthwise conv1d + SiLU ("in_proj -> causal depthwise conv1d ->
    SiLU"): xin [B,L,D], w [D,K], bias [D] (None = 0), state [B,D,K-1] (the
    K-1 inputs before t = 0; None = zeros). Returns x = silu(conv) [B,L,D]
    and state_out [B,D,K-1] (the last K-1 inputs)."""
    t = _NP[dtype]
    xin = _np(xin, t)
    B, L, D = xin.shape
    K = int(np.asarray(w).shape[1])
    args = _ConvArgs(B=B, L=L, D=D, K=K)
    keep = [xin]
    args.xin = _ptr(xin)
    _fill(args, keep, t, w=w, bias=bias, state=state)
    x = np.zeros((B, L, D), t)
    so = np.zeros((B, D, max(K - 1, 0)), t)
    args.x, args.state_out = _ptr(x), _ptr(so)
    rc = getattr(lib(), f"conv_oracle_fwd_{dtype}")(ctypes.byref(args))
    if rc != 0:
        raise ValueError(f"oracle conv fwd rejected the arguments ({rc})")
    return {"x": x, "state_out": so}


def conv_bwd(xin, w, dx, bias=None, state=None, dtype: str = "f64") -> Dict[str, np.ndarray]:
    """Reverse pass of conv_fwd for loss = <dx, x>. Returns dxin [B,L,D],
    dw [D,K] and dbias [D] (summed over batch and tokens) and dstate
    [B,D,K-1] (the gradient of the initial conv state)."""
    t = _NP[dtype]
    xin = _np(xin, t)
    B, L, D = xin.shape
    K = int(np.asarray(w).shape[1])
    args = _ConvArgs(B=B, L=L, D=D, K=K)
    keep = [xin]
    args.xin = _ptr(xin)
    _fill(args, keep, t, w=w, bias=bias, state=state, dx=dx)
    out = {"dxin": np.zeros((B, L, D), t), "dw": np.zeros((D, K), t), "dbias": np.zeros((D,), t),
           "dstate": np.zeros((B, D, max(K - 1, 0)), t)}
    for k, v in out.items():
        setattr(args, k, _ptr(v))
    rc = getattr(lib(), f"conv_oracle_bwd_{dtype}")(ctypes.byref(args))
    if rc != 0:
        raise ValueError(f"oracle conv bwd rejected the arguments ({rc})")
    return out


def dtproj_fwd(a, w, bias=None, softplus: bool = True, dtype: str = "f64") -> np.ndarray:
    """The dt projection ("delta=softplus(dt.dt_proj+dt_bias)"): a [M,R] (the
    dt_rank columns of the x_proj output), w [D,R], bias [D] (None = 0).
    Returns delta [M,D] = softplus(a @ w.T + bias) (without the softplus when
    ``softplus`` is False)."""
    t = _NP[dtype]
    a = _np(a, t)
    M, R = a.shape
    D = int(np.asarray(w).shape[0])
    args = _DtProjArgs(M=M, D=D, R=R, softplus=int(bool(softplus)))
    keep = [a]
    args.a = _ptr(a)
    _fill(args, keep, t, w=w, bias=bias)
    out = np.zeros((M, D), t)
    args.delta = _ptr(out)
    if getattr(lib(), f"dtproj_oracle_fwd_{dtype}")(ctypes.byref(args)) != 0:
        raise ValueError("oracle dt projection rejected the arguments")
    return out


def dtproj_bwd(a, w, ddelta, bias=None, softplus: bool = True, dtype: str = "f64") -> Dict[str, np.ndarray]:
    """Reverse pass of dtproj_fwd up to the pre-activation: dpre [M,D] =
    ddelta * sigmoid(pre) and dbias [D] = sum over m of dpre."""
    t = _NP[dtype]
    a = _np(a, t)
    M, R = a.shape
    D = int(np.asarray(w).shape[0])
    args = _DtProjArgs(M=M, D=D, R=R, softplus=int(bool(softplus)))
    keep = [a]
    args.a = _ptr(a)
    _fill(args, keep, t, w=w, bias=bias, ddelta=ddelta)
    out = {"dpre": np.zeros((M, D), t), "dbias": np.zeros((D,), t)}
    args.dpre, args.dbias = _ptr(out["dpre"]), _ptr(out["dbias"])
    if getattr(lib(), f"dtproj_oracle_bwd_{dtype}")(ctypes.byref(args)) != 0:
        raise ValueError("oracle dt projection backward rejected the arguments")
    return out
