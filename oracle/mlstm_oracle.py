"""CPU oracle for the mLSTM stabilized cell -- TEST INFRASTRUCTURE ONLY (the
same rule as the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it; the product path never does).

What it follows: Evil-Inference-Code, README_FIX_RUST.md, "mLSTM Equivalence
Fixes (Rust vs Python)". The page records how a second implementation of
the mLSTM cell was made to agree with the first: a recurrent ``step()``
that must match the parallel form (section 1, "Fixed: Recurrent gradient
now correctly matches the parallel gradient"), a cumulative sum of the
log forget gates built by iteration rather than as a product with a
lower-triangular matrix (section 2, "Cumulative Sum (cumsum_matrix)"), a
stabilized denominator taken as the larger of the normaliser's magnitude
and exp(-max_log_D) (section 2, "Stabilization Logic"), the stabilizer
state m starting at 0 (section 3, "m_state Initialization") and a head-wise
layer norm computed by hand from the mean and variance, with weights and no
bias (section 3, "LayerNorm (ln.rs)"). It states the fixes, not the cell's
equations; the cell they are fixes to is the published mLSTM (matrix
memory C, normaliser n, exponential input gate, sigmoid forget gate,
log-domain stabilizer m), and that is the reading taken here, per (batch,
head) and token t, with q scaled by ``scale`` (1/sqrt(K) by default):

    log f_t = log sigmoid(fgate_t),   log i_t = igate_t
    m_t     = max(log f_t + m_{t-1}, log i_t)
    C_t     = exp(log f_t + m_{t-1} - m_t) C_{t-1} + exp(log i_t - m_t) k_t v_t^T
    n_t     = exp(log f_t + m_{t-1} - m_t) n_{t-1} + exp(log i_t - m_t) k_t
    h_t     = (q_t^T C_t) / max(|q_t . n_t|, exp(-m_t))

(C is [K, V], n is [K]; the stabilized C, n are the plain ones times
exp(-m_t), so h equals the plain (q^T C) / max(|q . n|, 1) for any choice
of m: the stabilizer changes the rounding, never the value.)

Functions, each a separate evaluation:
- ``recurrent``: the per-token step above, m_0 = 0 unless given;
- ``parallel``: the page's parallel form for a zero initial state:
  cumulative log forget gates by iteration, log D[t, s] = F_t - F_s +
  log i_s (s <= t), max_log_D[t] its row maximum, D = exp(log D -
  max_log_D), Cm = (q k^T) * D, h = (Cm / max(|row sums of Cm|,
  exp(-max_log_D))) v;
- ``chunkwise``: the chunked evaluation the GPU kernel implements (the
  chunkwise form of the cell: the parallel form inside a chunk, the
  recurrent form across chunks) -- derived here, not printed on the page:
  per chunk with state (C, n, m_prev) and F the chunk's inclusive cumulative
  log forget gates, g_s = log i_s - F_s, M_t = max_{s<=t} g_s, mx_t =
  max(m_prev, M_t) and m_t = F_t + mx_t (the recurrent m unrolled), then
  alpha_t = exp(m_prev - mx_t), P[t, s] = (q_t . k_s) exp(g_s - mx_t)
  (s <= t), num_t = alpha_t q_t^T C + sum_s P[t, s] v_s, den_t = alpha_t
  q_t . n + sum_s P[t, s], h_t = num_t / max(|den_t|, exp(-m_t)); the state
  moves to the chunk's last token with gamma_s = exp(g_s - mx_last):
  C <- alpha_last C + sum_s gamma_s k_s v_s^T, n likewise, m <- m_last;
- ``plain``: the unstabilized definition (f = sigmoid, i = exp, no m),
  usable while exp(igate) stays in range;
- ``head_layer_norm``: mean and (biased) variance over the value channels
  of each (token, head), (h - mean) / sqrt(var + eps) * weight[head], no
  bias.

Everything is float64 numpy; products are numpy's (a library primitive
serving as one step). Pins: ``tests/test_mlstm_oracle_pins.py`` (the four
evaluations against each other, the single-token closed form, the
invariance to m_0 that section 3's fix relies on, large input gates, the
layer norm's moments and scale invariance).
"""
from __future__ import annotations

from typing import Optional, Tuple

import numpy as np


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def log_sigmoid(x):
    """log(1 / (1 + exp(-x))) without overflow for either sign of x."""
    x = _f64(x)
    return np.where(x >= 0, -np.log1p(np.exp(-np.abs(x))), x - np.log1p(np.exp(-np.abs(x))))


def _shapes(q, v):
    Bn, H, T, K = q.shape
    return Bn, H, T, K, v.shape[-1]


def recurrent(q, k, v, igate, fgate, C0=None, n0=None, m0=None, scale: Optional[float] = None
              ) -> Tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]:
    """The stabilized per-token step. q, k [B,H,T,K]; v [B,H,T,V]; igate,
    fgate [B,H,T]; C0 [B,H,K,V], n0 [B,H,K], m0 [B,H] (zeros when None).
    Returns (h [B,H,T,V], C, n, m), float64."""
    q, k, v, ig, fg = (_f64(a) for a in (q, k, v, igate, fgate))
    Bn, H, T, K, V = _shapes(q, v)
    sc = 1.0 / np.sqrt(K) if scale is None else float(scale)
    C = np.zeros((Bn, H, K, V)) if C0 is None else _f64(C0).copy()
    n = np.zeros((Bn, H, K)) if n0 is None else _f64(n0).copy()
    m = np.zeros((Bn, H)) if m0 is None else _f64(m0).copy()
    lf = log_sigmoid(fg)
    h = np.zeros((Bn, H, T, V))
    for t in range(T):
        m_new = np.maximum(lf[:, :, t] + m, ig[:, :, t])
        fs = np.exp(lf[:, :, t] + m - m_new)
        is_ = np.exp(ig[:, :, t] - m_new)
        kt, vt = k[:, :, t], v[:, :, t]
        C = fs[..., None, None] * C + is_[..., None, None] * kt[..., :, None] * vt[..., None, :]
        n = fs[..., None] * n + is_[..., None] * kt
        m = m_new
        qt = q[:, :, t] * sc
        num = np.einsum("bhk,bhkv->bhv", qt, C)
        den = np.einsum("bhk,bhk->bh", qt, n)
        h[:, :, t] = num / np.maximum(np.abs(den), np.exp(-m))[..., None]
    return h, C, n, m


def parallel(q, k, v, igate, fgate, scale: Optional[float] = None) -> np.ndarray:
    """The parallel stabilized form for a zero initial state. Returns h
    [B,H,T,V], float64."""
    q, k, v, ig, fg = (_f64(a) for a in (q, k, v, igate, fgate))
    Bn, H, T, K, V = _shapes(q, v)
    sc = 1.0 / np.sqrt(K) if scale is None else float(scale)
    lf = log_sigmoid(fg)
    F = np.zeros((Bn, H, T))
    acc = np.zeros((Bn, H))
    for t in range(T):  # the cumulative sum by iteration
        acc = acc + lf[:, :, t]
        F[:, :, t] = acc
    causal = np.tril(np.ones((T, T), dtype=bool))
    logD = F[..., :, None] - F[..., None, :] + ig[..., None, :]
    logD = np.where(causal, logD, -np.inf)
    max_log_D = logD.max(axis=-1) if T else np.zeros((Bn, H, 0))
    Dm = np.exp(logD - max_log_D[..., None])
    Cm = np.einsum("bhtk,bhsk->bhts", q * sc, k) * Dm
    normaliser = np.maximum(np.abs(Cm.sum(axis=-1)), np.exp(-max_log_D))
    return np.einsum("bhts,bhsv->bhtv", Cm / normaliser[..., None], v)


def chunkwise(q, k, v, igate, fgate, C0=None, n0=None, m0=None, scale: Optional[float] = None, chunk: int = 64
              ) -> Tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]:
    """The chunked evaluation (parallel inside a chunk of ``chunk`` tokens,
    recurrent across chunks; the last chunk ragged). Same arguments and
    results as ``recurrent``."""
    q, k, v, ig, fg = (_f64(a) for a in (q, k, v, igate, fgate))
    Bn, H, T, K, V = _shapes(q, v)
    sc = 1.0 / np.sqrt(K) if scale is None else float(scale)
    C = np.zeros((Bn, H, K, V)) if C0 is None else _f64(C0).copy()
    n = np.zeros((Bn, H, K)) if n0 is None else _f64(n0).copy()
    m = np.zeros((Bn, H)) if m0 is None else _f64(m0).copy()
    lf = log_sigmoid(fg)
    h = np.zeros((Bn, H, T, V))
    for t0 in range(0, T, chunk):
        c = min(chunk, T - t0)
        sl = slice(t0, t0 + c)
        # 1. the chunk's cumulative log forget gates, by iteration
        F = np.zeros((Bn, H, c))
        acc = np.zeros((Bn, H))
        for j in range(c):
            acc = acc + lf[:, :, t0 + j]
            F[:, :, j] = acc
        # 2. stabilizer: m_t = F_t + max(m_prev, max_{s<=t} (log i_s - F_s))
        g = ig[:, :, sl] - F
        M = np.maximum.accumulate(g, axis=-1)
        mx = np.maximum(m[..., None], M)
        mt = F + mx
        # 3. the decayed, stabilized intra-chunk scores and the inter-chunk weight
        alpha = np.exp(m[..., None] - mx)
        causal = np.tril(np.ones((c, c), dtype=bool))
        w = np.exp(np.where(causal, g[..., None, :] - mx[..., :, None], -np.inf))
        qs = q[:, :, sl] * sc
        P = np.einsum("bhtk,bhsk->bhts", qs, k[:, :, sl]) * w
        # 4. numerator and denominator: the state's term plus the chunk's own
        num = alpha[..., None] * np.einsum("bhtk,bhkv->bhtv", qs, C) + np.einsum("bhts,bhsv->bhtv", P, v[:, :, sl])
        den = alpha * np.einsum("bhtk,bhk->bht", qs, n) + P.sum(axis=-1)
        # 5. the stabilized division
        h[:, :, sl] = num / np.maximum(np.abs(den), np.exp(-mt))[..., None]
        # 6. the state at the chunk's last token
        gamma = np.exp(g - mx[..., -1:])
        beta = alpha[..., -1]
        C = beta[..., None, None] * C + np.einsum("bhs,bhsk,bhsv->bhkv", gamma, k[:, :, sl], v[:, :, sl])
        n = beta[..., None] * n + np.einsum("bhs,bhsk->bhk", gamma, k[:, :, sl])
        m = mt[..., -1]
    return h, C, n, m


def plain(q, k, v, igate, fgate, C0=None, n0=None, scale: Optional[float] = None
          ) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """The unstabilized cell: f = sigmoid(fgate), i = exp(igate), C_t = f C
    + i k v^T, n_t = f n + i k, h = (q^T C) / max(|q . n|, 1). C0, n0 are
    the plain (unscaled) state. Returns (h, C, n), float64."""
    q, k, v, ig, fg = (_f64(a) for a in (q, k, v, igate, fgate))
    Bn, H, T, K, V = _shapes(q, v)
    sc = 1.0 / np.sqrt(K) if scale is None else float(scale)
    C = np.zeros((Bn, H, K, V)) if C0 is None else _f64(C0).copy()
    n = np.zeros((Bn, H, K)) if n0 is None else _f64(n0).copy()
    f = 1.0 / (1.0 + np.exp(-fg))
    i = np.exp(ig)
    h = np.zeros((Bn, H, T, V))
    for t in range(T):
        C = f[:, :, t, None, None] * C + i[:, :, t, None, None] * k[:, :, t, :, None] * v[:, :, t, None, :]
        n = f[:, :, t, None] * n + i[:, :, t, None] * k[:, :, t]
        qt = q[:, :, t] * sc
        num = np.einsum("bhk,bhkv->bhv", qt, C)
        den = np.einsum("bhk,bhk->bh", qt, n)
        h[:, :, t] = num / np.maximum(np.abs(den), 1.0)[..., None]
    return h, C, n


def head_layer_norm(h, weight, eps: float = 1e-5) -> np.ndarray:
    """Per (batch, head, token): (h - mean) / sqrt(var + eps) * weight[head]
    over the value channels, var the mean squared deviation; no bias.
    h [B,H,T,V], weight [H,V]."""
    h = _f64(h)
    mu = h.mean(axis=-1, keepdims=True)
    var = ((h - mu) ** 2).mean(axis=-1, keepdims=True)
    return (h - mu) / np.sqrt(var + eps) * _f64(weight)[None, :, None, :]
