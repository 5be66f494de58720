"""CPU oracle for the Gated DeltaNet-2 chunkwise WY forward -- TEST
INFRASTRUCTURE ONLY (the same rule as the rest of ``oracle/``: only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it; the product path never does).

What it follows: docs.rs, burn-gdn2 0.1.4, ``src/forward.rs``,
``chunk_wy_forward`` ("Gated DeltaNet 2 -- linear recurrent token mixer with
channel-wise erase/write gates"). Per (batch, head), the sequence is cut
into chunks of ``chunk`` tokens (the last one ragged) and, per chunk, in the
page's order:

1. ``G`` = cumulative sum of the log-gates g over the chunk's tokens (the
   page multiplies by a lower-triangular matrix of ones; a cumulative sum is
   that product written out);
2. ``decay[i, j]`` = mean over the key channels of exp(G[i] - G[j]);
3. ``aqk`` = (q k^T) * decay * scale on and below the diagonal;
   ``akk`` = ((b * k) k^T) * decay strictly below it;
4. ``rhs_k`` = b * k * exp(G), ``rhs_v`` = w * v;
5. the WY rows by forward substitution, row i after rows 0..i-1:
   W[i] = rhs_k[i] - akk[i, :i] W[:i],  U[i] = rhs_v[i] - akk[i, :i] U[:i];
6. ``v_new`` = U - W S with S the state before the chunk;
7. output = aqk v_new + (q * exp(G)) S * scale;
8. S <- S * exp(G[last]) (per key row) + (k * exp(G[last] - G))^T v_new.

Everything is float64 numpy; matrix products are numpy's (a library
primitive serving as one step), with no reordering beyond the steps above.

``recurrent`` is the per-token form the chunked steps reduce to with chunks
of one token (derived here from steps 1-8 with c = 1, not printed on the
page):
   S' = diag(exp(g_t)) S;  v_new = w_t * v_t - (b_t * k_t)^T S';
   S  = S' + k_t v_new^T;   o_t = scale * q_t^T S.
With key-uniform gates (g[t, k] the same for every k) the chunked steps
equal it for every chunk size (the mean in step 2 is then exact); with
gates that differ across key channels, step 2 averages the per-channel
decays and the chunked result depends on the chunk size -- that is the
page's method, and the oracle follows it. Pins: ``tests/test_gdn2_oracle_pins.py``
(chunk size 1, key-uniform gates, a single key channel, the linear-attention
closed form, chunk-boundary state chaining, channel-permutation symmetry).
The intra-chunk key-mean of step 2 with channel-varying gates and chunks
longer than one token is "parity unpinned" beyond its symmetry: no other
evaluation of it exists.
"""
from __future__ import annotations

from typing import Tuple

import numpy as np


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def chunk_wy_forward(q, k, v, g, b, w, state, scale: float, chunk: int) -> Tuple[np.ndarray, np.ndarray]:
    """q, k, g, b: [B, H, T, K]; v, w: [B, H, T, V]; state: [B, H, K, V].
    Returns (output [B, H, T, V], final state [B, H, K, V]), float64."""
    q, k, v, g, b, w = (_f64(a) for a in (q, k, v, g, b, w))
    S = _f64(state).copy()
    Bn, H, T, K = q.shape
    V = v.shape[3]
    out = np.zeros((Bn, H, T, V))
    for c0 in range(0, T, chunk):
        c1 = min(c0 + chunk, T)
        c = c1 - c0
        qc, kc, vc, gc, bc, wc = (a[:, :, c0:c1] for a in (q, k, v, g, b, w))
        G = np.cumsum(gc, axis=2)                                         # step 1: [B,H,c,K]
        decay = np.exp(G[:, :, :, None, :] - G[:, :, None, :, :]).mean(axis=4)  # step 2: [B,H,c,c]
        causal = np.tril(np.ones((c, c)))
        strict = np.tril(np.ones((c, c)), -1)
        aqk = (qc @ np.swapaxes(kc, 2, 3)) * decay * scale * causal      # step 3
        akk = ((bc * kc) @ np.swapaxes(kc, 2, 3)) * decay * strict
        gexp = np.exp(G)
        rhs_k = bc * kc * gexp                                            # step 4
        rhs_v = wc * vc
        W = np.zeros((Bn, H, c, K))
        U = np.zeros((Bn, H, c, V))
        for i in range(c):                                                # step 5
            W[:, :, i] = rhs_k[:, :, i] - np.einsum("bhj,bhjk->bhk", akk[:, :, i, :i], W[:, :, :i])
            U[:, :, i] = rhs_v[:, :, i] - np.einsum("bhj,bhjv->bhv", akk[:, :, i, :i], U[:, :, :i])
        v_new = U - W @ S                                                 # step 6
        out[:, :, c0:c1] = aqk @ v_new + (qc * gexp) @ S * scale          # step 7
        g_last = gexp[:, :, c - 1]                                        # step 8
        to_last = np.exp(G[:, :, c - 1:c] - G)
        S = S * g_last[:, :, :, None] + np.swapaxes(kc * to_last, 2, 3) @ v_new
    return out, S


def recurrent(q, k, v, g, b, w, state, scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """The per-token form of the same mixer (the chunked steps with chunks of
    one token), float64."""
    q, k, v, g, b, w = (_f64(a) for a in (q, k, v, g, b, w))
    S = _f64(state).copy()
    Bn, H, T, K = q.shape
    out = np.zeros((Bn, H, T, v.shape[3]))
    for t in range(T):
        S = S * np.exp(g[:, :, t])[:, :, :, None]
        v_new = w[:, :, t] * v[:, :, t] - np.einsum("bhk,bhkv->bhv", b[:, :, t] * k[:, :, t], S)
        S = S + k[:, :, t][:, :, :, None] * v_new[:, :, None, :]
        out[:, :, t] = scale * np.einsum("bhk,bhkv->bhv", q[:, :, t], S)
    return out, S
