"""Float64 oracle of the generalised delta rule: a rank-one transition
I - a b^T between linear-attention steps ("Talk Linear Attention", section
7.1, generalised linear Transformer).

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module;
only tests/ and bench.py's CPU legs do. It shares no code with the CUDA path.

The page writes the value-major state S [dv, dk] as

    S_t = S_{t-1} (I - a_t b_t^T) + v_t k_t^T,   o_t = S_t q_t,

a structured (identity plus rank-one) transition that mixes key channels at
O(d^2) per token. In this library's key-major orientation (the transpose,
S [dk, dv], o_t = S_t^T q_t) the same recurrence reads

    S_t = (I - b_t a_t^T) S_{t-1} + k_t v_t^T:

retrieve u_t = S_{t-1}^T a_t with a_t, erase it along b_t, write k_t v_t^T.
The page names DeltaNet as the case a_t = b_t = sqrt(beta_t) k_t; the write
here is the page's unit write k v^T (pass beta_t k_t as the write key for
the beta-weighted DeltaNet write). Per (b, h), from S0 (zero when absent).

chunk_form restates it chunkwise (C tokens, WY-style): with the chunk's
incoming state S and rows a_r, b_r, k_r, v_r, q_r,

    U = (I + L_ab)^{-1} (A S + L_ak V),   L_ab[r, s] = a_r . b_s,
                                          L_ak[r, s] = a_r . k_s  (s < r)
    O = Q S + M(Q K^T) V - M(Q B^T) U     (M: inclusive causal mask)
    S <- S + K^T V - B^T U

where row r of U is u_r = S_{r-1}^T a_r.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular

__all__ = ["recurrence_gdelta", "chunk_form_gdelta"]


def recurrence_gdelta(q, k, v, a, b, S0=None):
    """q, k, a, b [B, H, T, dk]; v [B, H, T, dv]; S0 [B, H, dk, dv] or None.
    Returns (o [B, H, T, dv], S [B, H, dk, dv]) in float64."""
    q, k, v, a, b = (np.asarray(x, dtype=np.float64) for x in (q, k, v, a, b))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    S = np.zeros((B, H, dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((B, H, T, dv))
    for t in range(T):
        u = np.einsum("bhc,bhcv->bhv", a[:, :, t], S)                      # S^T a_t
        S = S - b[:, :, t][..., :, None] * u[..., None, :] + k[:, :, t][..., :, None] * v[:, :, t][..., None, :]
        o[:, :, t] = np.einsum("bhc,bhcv->bhv", q[:, :, t], S)
    return o, S


def chunk_form_gdelta(q, k, v, a, b, S0=None, C=64):
    """One head: q, k, a, b [T, dk], v [T, dv]. The chunkwise form above."""
    q, k, v, a, b = (np.asarray(x, dtype=np.float64) for x in (q, k, v, a, b))
    T, dk = q.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((T, dv))
    for t0 in range(0, T, C):
        t1 = min(T, t0 + C)
        n = t1 - t0
        Q, K, V, Am, Bm = q[t0:t1], k[t0:t1], v[t0:t1], a[t0:t1], b[t0:t1]
        strict = np.tril(np.ones((n, n)), -1)
        incl = np.tril(np.ones((n, n)))
        L_ab = (Am @ Bm.T) * strict
        L_ak = (Am @ K.T) * strict
        U = solve_triangular(np.eye(n) + L_ab, Am @ S + L_ak @ V, lower=True, unit_diagonal=True)
        o[t0:t1] = Q @ S + ((Q @ K.T) * incl) @ V - ((Q @ Bm.T) * incl) @ U
        S = S + K.T @ V - Bm.T @ U
    return o, S
