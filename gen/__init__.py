"""Seeded synthetic inputs for the S6 selective scan.

This module only draws numbers. It holds no part of the scan's arithmetic
(no softplus, no exponentials of delta*A, no recurrence). The oracle tests,
the GPU parity tests and ``bench.py`` all take their inputs from here, so
both sides of every comparison see the same values.

Generator
---------
* SplitMix64 (Vigna's published mixer): ``state += 0x9E3779B97F4A7C15`` then
  ``z = (z ^ z>>30) * 0xBF58476D1CE4E5B9``,
  ``z = (z ^ z>>27) * 0x94D049BB133111EB``, ``z ^= z>>31``.
  Output i of the stream seeded with s is the mix of ``s + (i+1)*golden``,
  so any slice of a stream can be drawn on its own.
* Uniforms: the top 53 bits of an output times 2**-53, in [0, 1).
* Normals: Box-Muller on consecutive output pairs (u1, u2) with
  r = sqrt(-2 ln(1 - u1)), theta = 2*pi*u2, giving r*cos(theta) and
  r*sin(theta) in that order; computed in float64, scaled, then rounded
  to float32.
* Per-tensor seeds: the workload seed feeds one SplitMix64 stream whose
  successive outputs seed x, z, Bm, Cm, dt, dy, h0, dh_last in that order
  (the per-tensor SplitMix64-derived seeding the rustytorch commit log on
  ``MambaBlock::new_seeded`` describes).
* bf16 workloads round x, z, Bm, Cm and dy to bfloat16 (round to nearest
  even) here, once; both sides then read the same rounded values.

Workloads
---------
The five workload recipes follow the sizes and distributions of the
selective-scan configurations this library is measured on: A[d, n] =
-(n + 1) (the canonical A_log = ln(1..N) init), D = 1, gate on, h0 = 0,
dh_last = 0, and dt_bias chosen so that softplus(dt_bias) equals a target
delta (0.69 for the "active" tiny block, 0.01 for the canonical init).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, Optional

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

TENSOR_ORDER = ("x", "z", "Bm", "Cm", "dt", "dy", "h0", "dh_last")


def splitmix64(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Outputs start .. start+n-1 of the SplitMix64 stream seeded with ``seed``."""
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform53(seed: int, n: int, start: int = 0) -> np.ndarray:
    """float64 uniforms in [0, 1) from the top 53 bits of each output."""
    return (splitmix64(seed, n, start) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal_f32(seed: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """n float32 samples of N(mean, std^2) by Box-Muller, drawn in chunks."""
    out = np.empty(n, dtype=np.float32)
    pairs = (n + 1) // 2
    done = 0
    while done < pairs:
        m = min(_CHUNK, pairs - done)
        u = uniform53(seed, 2 * m, 2 * done)
        r = np.sqrt(-2.0 * np.log1p(-u[0::2]))
        th = (2.0 * math.pi) * u[1::2]
        zz = np.empty(2 * m, dtype=np.float64)
        zz[0::2] = r * np.cos(th)
        zz[1::2] = r * np.sin(th)
        lo = 2 * done
        hi = min(n, lo + 2 * m)
        out[lo:hi] = (mean + std * zz[: hi - lo]).astype(np.float32)
        done += m
    return out


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    bias = np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    r = ((u + bias) & np.uint64(0xFFFF0000)).astype(np.uint32)
    return r.view(np.float32)


def tensor_seeds(seed: int) -> Dict[str, int]:
    s = splitmix64(seed, len(TENSOR_ORDER))
    return {name: int(v) for name, v in zip(TENSOR_ORDER, s)}


def inverse_softplus(target: float) -> float:
    """The dt_bias whose softplus is ``target``: ln(e^target - 1)."""
    return math.log(math.expm1(target))


@dataclass
class Workload:
    name: str
    B: int
    L: int
    D: int
    N: int
    io: str            # "f32" or "bf16": dtype of x, z, Bm, Cm, y, dy, dx, dz
    seed: int
    dt_std: float
    delta_target: float  # softplus(dt_bias) = delta_target
    note: str = ""

    @property
    def tc(self) -> int:
        return self.B * self.L * self.D


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in (
        Workload("s6-tiny-active-f32", 1, 64, 16, 16, "f32", 0, 0.1, 0.69,
                 "active block: delta ~ 0.69"),
        Workload("s6-small-f32", 2, 512, 256, 16, "f32", 1, 1.0, 0.01,
                 "canonical dt_bias, dt ~ N(0,1): delta spread ~1e-3..1"),
        Workload("mamba130m-bf16", 8, 2048, 1536, 16, "bf16", 2, 1.0, 0.01,
                 "Mamba-130M-shaped: d_model 768, expand 2"),
        Workload("mamba1.4b-bf16", 4, 4096, 4096, 16, "bf16", 3, 1.0, 0.01,
                 "Mamba-1.4B-shaped: d_model 2048, expand 2"),
        Workload("long65k-bf16", 1, 65536, 2048, 16, "bf16", 4, 1.0, 0.01,
                 "long sequence, needs the multi-CTA carry along L"),
    )
}
WORKLOAD_ORDER = list(WORKLOADS)


@dataclass
class Inputs:
    """All inputs of one scan problem as float32 numpy arrays (bf16-rounded
    where the workload's I/O dtype is bf16). Layouts: x, z, dt, dy [B,L,D];
    Bm, Cm [B,L,N]; A [D,N]; Dskip, dt_bias [D]; h0, dh_last [B,D,N]."""
    B: int
    L: int
    D: int
    N: int
    io: str
    x: np.ndarray
    dt: np.ndarray
    z: Optional[np.ndarray]
    Bm: np.ndarray
    Cm: np.ndarray
    A: np.ndarray
    Dskip: Optional[np.ndarray]
    dt_bias: Optional[np.ndarray]
    h0: Optional[np.ndarray]
    dy: np.ndarray
    dh_last: Optional[np.ndarray]
    delta_softplus: int = 1
    meta: dict = field(default_factory=dict)


def make_inputs(B: int, L: int, D: int, N: int, *, io: str = "f32", seed: int = 0,
                dt_std: float = 1.0, delta_target: float = 0.01, gate: bool = True,
                skip: bool = True, bias: bool = True, with_h0: bool = False,
                with_dh_last: bool = False, delta_softplus: int = 1,
                x_std: float = 1.0) -> Inputs:
    """Draw one problem. ``with_h0`` / ``with_dh_last`` draw N(0, 1) initial
    state and final-state gradient instead of zeros."""
    s = tensor_seeds(seed)
    tc = B * L * D
    bl = B * L * N
    rnd = round_bf16 if io == "bf16" else (lambda a: a)
    x = rnd(normal_f32(s["x"], tc, 0.0, x_std)).reshape(B, L, D)
    z = rnd(normal_f32(s["z"], tc)).reshape(B, L, D) if gate else None
    Bm = rnd(normal_f32(s["Bm"], bl)).reshape(B, L, N)
    Cm = rnd(normal_f32(s["Cm"], bl)).reshape(B, L, N)
    dt = normal_f32(s["dt"], tc, 0.0, dt_std).reshape(B, L, D)
    dy = rnd(normal_f32(s["dy"], tc)).reshape(B, L, D)
    A = np.tile(-np.arange(1, N + 1, dtype=np.float32), (D, 1))
    Dskip = np.ones(D, dtype=np.float32) if skip else None
    dt_bias = np.full(D, inverse_softplus(delta_target), dtype=np.float32) if bias else None
    h0 = normal_f32(s["h0"], B * D * N).reshape(B, D, N) if with_h0 else None
    dh_last = normal_f32(s["dh_last"], B * D * N).reshape(B, D, N) if with_dh_last else None
    return Inputs(B, L, D, N, io, x, dt, z, Bm, Cm, A, Dskip, dt_bias, h0, dy, dh_last,
                  delta_softplus, {"seed": seed, "dt_std": dt_std, "delta_target": delta_target})


def workload_inputs(name: str, **kw) -> Inputs:
    w = WORKLOADS[name]
    return make_inputs(w.B, w.L, w.D, w.N, io=w.io, seed=w.seed, dt_std=w.dt_std,
                       delta_target=w.delta_target, **kw)


@dataclass
class ConvInputs:
    """One problem for the conv1d + SiLU in front of the scan: xin [B,L,D]
    (the in_proj output), w [D,K], bias [D] (None = 0), state [B,D,K-1]
    (None = zeros), dx [B,L,D] (the gradient arriving at the conv output)."""
    B: int
    L: int
    D: int
    K: int
    io: str
    xin: np.ndarray
    w: np.ndarray
    bias: Optional[np.ndarray]
    state: Optional[np.ndarray]
    dx: np.ndarray


def make_conv_inputs(B: int, L: int, D: int, K: int = 4, *, io: str = "f32", seed: int = 0,
                     bias: bool = True, with_state: bool = False) -> ConvInputs:
    """Draw a conv problem: xin, dx ~ N(0,1) (bf16-rounded for bf16 I/O);
    w ~ N(0, 1/K) (the scale of the usual 1/sqrt(fan_in) init); bias ~
    N(0, 0.1^2) when drawn (the canonical init sets it to zero); state ~
    N(0,1) when drawn. Per-tensor seeds come from the same SplitMix64
    streams as make_inputs (x, dt, z, dy, h0 slots), so the draws are fixed
    by (seed, shape)."""
    s = tensor_seeds(seed)
    tc = B * L * D
    rnd = round_bf16 if io == "bf16" else (lambda a: a)
    xin = rnd(normal_f32(s["x"], tc)).reshape(B, L, D)
    w = normal_f32(s["dt"], D * K, 0.0, float(1.0 / np.sqrt(K))).reshape(D, K)
    b = normal_f32(s["z"], D, 0.0, 0.1) if bias else None
    st = normal_f32(s["h0"], B * D * (K - 1)).reshape(B, D, K - 1) if with_state and K > 1 else None
    dx = rnd(normal_f32(s["dy"], tc)).reshape(B, L, D)
    return ConvInputs(B, L, D, K, io, xin, w, b, st, dx)


@dataclass
class DtProjInputs:
    """One problem for the dt projection in front of the scan: a [B,L,R] (the
    dt_rank columns of the x_proj output), w [D,R] (dt_proj weight), bias [D],
    ddelta [B,L,D] (the gradient arriving at Delta)."""
    B: int
    L: int
    D: int
    R: int
    a: np.ndarray
    w: np.ndarray
    bias: np.ndarray
    ddelta: np.ndarray


def make_dtproj_inputs(B: int, L: int, D: int, R: int, *, seed: int = 0) -> DtProjInputs:
    """Draw a dt-projection problem with bf16 operands (the tensor-core path):
    a ~ N(0,1) and w ~ N(0, 1/R), both bf16-rounded, so a.w ~ N(0,1); bias[d]
    = the inverse softplus of a log-uniform Delta in [1e-3, 1e-1] (Mamba's
    dt_proj bias init), so softplus(a.w + bias) has the scan inputs'
    distribution; ddelta ~ N(0,1) fp32. Per-tensor seeds from the same
    SplitMix64 streams as make_inputs (x, dt, z, dy slots)."""
    s = tensor_seeds(seed)
    a = round_bf16(normal_f32(s["x"], B * L * R)).reshape(B, L, R)
    w = round_bf16(normal_f32(s["dt"], D * R, 0.0, float(1.0 / np.sqrt(R)))).reshape(D, R)
    u = uniform53(s["z"], D)
    delta0 = np.exp(np.log(1e-3) + u * (np.log(1e-1) - np.log(1e-3)))
    bias = np.log(np.expm1(delta0)).astype(np.float32)
    ddelta = normal_f32(s["dy"], B * L * D).reshape(B, L, D)
    return DtProjInputs(B, L, D, R, a, w, bias, ddelta)


@dataclass
class Gdn2Inputs:
    """One problem for the Gated DeltaNet-2 chunkwise forward (layout
    [batch, heads, time, dim] as on its page): q, k, g, b [B,H,T,K]; v, w
    [B,H,T,V]; state [B,H,K,V]; scale."""
    B: int
    H: int
    T: int
    K: int
    V: int
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    g: np.ndarray
    b: np.ndarray
    w: np.ndarray
    state: np.ndarray
    scale: float


GDN2_WORKLOADS = {
    # name: (B, H, T, K, V, seed); chunks of 64 tokens
    "gdn2-small": (1, 2, 200, 128, 128, 11),
    "gdn2-1.3b-like": (8, 16, 2048, 128, 128, 12),
}


def make_gdn2_inputs(B: int, H: int, T: int, K: int, V: int, *, seed: int = 0, io: str = "bf16",
                     with_state: bool = True, key_uniform_gates: bool = False) -> Gdn2Inputs:
    """Draw a Gated DeltaNet-2 problem: q, k ~ N(0, 1/K) (so q.k ~ N(0,1));
    v ~ N(0,1); the log-gates g uniform in [-0.3, -0.001] per (token, key
    channel) (one value per token, shared by all key channels, with
    key_uniform_gates); the erase gates b and write gates w uniform in
    (0, 1); the initial state ~ N(0, 0.1^2) (zeros without with_state);
    scale = 1/sqrt(K). With io = "bf16", q, k, v, b, w are rounded to
    bfloat16 once; g and the state stay float32. Per-tensor seeds from the
    same SplitMix64 streams as make_inputs (x, z, Bm, Cm, dt, dy, h0, dh_last
    slots in order)."""
    s = tensor_seeds(seed)
    nk, nv = B * H * T * K, B * H * T * V
    rnd = round_bf16 if io == "bf16" else (lambda a: np.asarray(a, np.float32))
    q = rnd(normal_f32(s["x"], nk, 0.0, float(1.0 / np.sqrt(K)))).reshape(B, H, T, K)
    k = rnd(normal_f32(s["z"], nk, 0.0, float(1.0 / np.sqrt(K)))).reshape(B, H, T, K)
    v = rnd(normal_f32(s["Bm"], nv)).reshape(B, H, T, V)
    if key_uniform_gates:
        gt = (-0.001 - 0.299 * uniform53(s["Cm"], B * H * T)).astype(np.float32).reshape(B, H, T, 1)
        g = np.ascontiguousarray(np.broadcast_to(gt, (B, H, T, K)))
    else:
        g = (-0.001 - 0.299 * uniform53(s["Cm"], nk)).astype(np.float32).reshape(B, H, T, K)
    b = rnd(uniform53(s["dt"], nk).astype(np.float32)).reshape(B, H, T, K)
    w = rnd(uniform53(s["dy"], nv).astype(np.float32)).reshape(B, H, T, V)
    state = (normal_f32(s["h0"], B * H * K * V, 0.0, 0.1).reshape(B, H, K, V) if with_state
             else np.zeros((B, H, K, V), np.float32))
    return Gdn2Inputs(B, H, T, K, V, q, k, v, g, b, w, state, float(1.0 / np.sqrt(K)))


@dataclass
class MlstmInputs:
    """One problem for the mLSTM chunkwise forward (layout [batch, heads,
    time, dim]): q, k [B,H,T,K]; v [B,H,T,V]; igate, fgate [B,H,T] (gate
    pre-activations); the stabilized initial state C0 [B,H,K,V], n0 [B,H,K],
    m0 [B,H]; the head-wise norm's weight [H,V]; scale."""
    B: int
    H: int
    T: int
    K: int
    V: int
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    igate: np.ndarray
    fgate: np.ndarray
    C0: np.ndarray
    n0: np.ndarray
    m0: np.ndarray
    norm_weight: np.ndarray
    scale: float


MLSTM_WORKLOADS = {
    # name: (B, H, T, K, V, seed); chunks of 64 tokens
    "mlstm-small": (1, 2, 200, 128, 128, 13),
    "mlstm-8x16x2048": (8, 16, 2048, 128, 128, 14),
}


def make_mlstm_inputs(B: int, H: int, T: int, K: int, V: int, *, seed: int = 0, io: str = "bf16",
                      with_state: bool = True, igate_mean: float = 0.0) -> MlstmInputs:
    """Draw an mLSTM problem: q, k, v ~ N(0, 1); input-gate pre-activations
    ~ N(igate_mean, 1) (i = exp(.) around 1); forget-gate pre-activations
    uniform in [3, 6] (f = sigmoid(.) between 0.95 and 0.998: long memory);
    with with_state, C0 ~ N(0, 0.1^2), n0 ~ N(0, 0.1^2) and m0 uniform in
    [-2, 2] (else zeros); the norm weight ~ 1 + N(0, 0.1^2); scale =
    1/sqrt(K). With io = "bf16", q, k, v are rounded to bfloat16 once; the
    gates, the state and the weight stay float32. Per-tensor seeds from the
    same SplitMix64 streams as make_inputs (x, z, Bm, Cm, dt, dy, h0,
    dh_last slots in order)."""
    s = tensor_seeds(seed)
    nk, nv, nt = B * H * T * K, B * H * T * V, B * H * T
    rnd = round_bf16 if io == "bf16" else (lambda a: np.asarray(a, np.float32))
    q = rnd(normal_f32(s["x"], nk)).reshape(B, H, T, K)
    k = rnd(normal_f32(s["z"], nk)).reshape(B, H, T, K)
    v = rnd(normal_f32(s["Bm"], nv)).reshape(B, H, T, V)
    igate = normal_f32(s["Cm"], nt, igate_mean, 1.0).reshape(B, H, T)
    fgate = (3.0 + 3.0 * uniform53(s["dt"], nt)).astype(np.float32).reshape(B, H, T)
    if with_state:
        st = normal_f32(s["h0"], B * H * (K * V + K), 0.0, 0.1)
        C0 = st[:B * H * K * V].reshape(B, H, K, V)
        n0 = st[B * H * K * V:].reshape(B, H, K)
        m0 = (-2.0 + 4.0 * uniform53(s["dh_last"], B * H)).astype(np.float32).reshape(B, H)
    else:
        C0 = np.zeros((B, H, K, V), np.float32)
        n0 = np.zeros((B, H, K), np.float32)
        m0 = np.zeros((B, H), np.float32)
    wgt = (1.0 + normal_f32(s["dy"], H * V, 0.0, 0.1)).astype(np.float32).reshape(H, V)
    return MlstmInputs(B, H, T, K, V, q, k, v, igate, fgate, C0, n0, m0, wgt, float(1.0 / np.sqrt(K)))


def recipe_text() -> str:
    lines = []
    for w in WORKLOADS.values():
        lines.append(f"{w.name}: B={w.B} L={w.L} D={w.D} N={w.N} io={w.io} seed={w.seed} "
                     f"dt~N(0,{w.dt_std}^2) softplus(dt_bias)={w.delta_target} ({w.note})")
    return "\n".join(lines)
