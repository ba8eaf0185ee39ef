"""Alternative float64 statements of the same computation, used to pin the oracle.

TEST INFRASTRUCTURE ONLY. Each function below restates one form the pages
give for linear attention or one of its special cases. The recurrence in
``oracle.recurrence`` must agree with every one of them; because they are
different formulas (quadratic masked products, explicit normalised sums, the
four-step DeltaNet memory update, a Kronecker-product brute force, the
chunkwise form), a dropped term, a wrong sign, a wrong index or a transposed
operand in the recurrence shows up as a mismatch.

All inputs are single-head float64 arrays: q, k [T, dk], v [T, dv].
Key-major state S [dk, dv] with o_t = S^T q_t unless stated otherwise.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular



def _phi(x):
    """elu(x) + 1 written as max(x, 0) + exp(min(x, 0)): equal to x + 1 for
    x > 0 and to exp(x) for x <= 0 (kept independent of the recurrence's
    own helper so that a mistake there cannot hide in both)."""
    x = np.asarray(x, dtype=np.float64)
    return np.maximum(x, 0.0) + np.exp(np.minimum(x, 0.0))

__all__ = ["parallel_linear", "parallel_gated", "normalised_sum",
           "deltanet_four_step", "kronecker_delta", "chunk_form"]


def parallel_linear(q, k, v):
    """Quadratic parallel form O = (Q K^T ⊙ M) V with an inclusive causal mask
    M and no softmax or 1/sqrt(d) scale ("Talk Linear Attention", section
    2.1). Also returns the closed-form final state S_T = K^T V (the sum of
    k_j v_j^T over all tokens, same section)."""
    T = q.shape[0]
    M = np.tril(np.ones((T, T)))
    return (q @ k.T * M) @ v, k.T @ v


def parallel_gated(q, k, v, log_alpha):
    """Decay-aware parallel form O = ((Q ⊙ B)(K / B)^T ⊙ M) V with cumulative
    decay b_t = prod_{j<=t} alpha_j ("Talk Linear Attention", section 5.2).

    log_alpha: [T] (one scalar gate per token, RetNet and Mamba-2 style) or
    [T, dk] (GLA, one gate per key channel). Zero initial state. Also returns
    the final state S_T = sum_s Diag(b_T / b_s) k_s v_s^T.
    Only for short T: B and 1/B are formed explicitly, as the page writes.
    """
    T, dk = q.shape
    la = np.asarray(log_alpha, dtype=np.float64)
    if la.ndim == 1:
        la = np.repeat(la[:, None], dk, axis=1)
    Bm = np.exp(np.cumsum(la, axis=0))            # [T, dk], b_t per channel
    M = np.tril(np.ones((T, T)))
    O = (((q * Bm) @ (k / Bm).T) * M) @ v
    S = ((k * (Bm[-1][None, :] / Bm)).T) @ v
    return O, S


def normalised_sum(q, k, v):
    """Causal normalised kernel attention written as explicit sums:
    o_i = sum_{j<=i} (phi(q_i).phi(k_j)) v_j / sum_{j<=i} phi(q_i).phi(k_j),
    phi = elu + 1 ("Linear Attention" glossary, kernel decomposition; kernel
    attention notes, section 13). Also returns the final (S, z) with
    S = sum_j phi(k_j) v_j^T and z = sum_j phi(k_j)."""
    qh, kh = _phi(q), _phi(k)
    T = q.shape[0]
    o = np.zeros((T, v.shape[1]))
    for i in range(T):
        w = kh[: i + 1] @ qh[i]                 # kernel values phi(q_i).phi(k_j)
        o[i] = (w[:, None] * v[: i + 1]).sum(0) / w.sum()
    return o, kh.T @ v, kh.sum(0)


def deltanet_four_step(q, k, v, beta, S0=None, log_alpha=None):
    """DeltaNet memory update in the page's four steps, value-major state
    S [dv, dk] ("Talk Linear Attention", section 6.1):
      v_old = S k_t ; v_new = beta v_t + (1 - beta) v_old ;
      S <- S - v_old k_t^T + v_new k_t^T ; o_t = S q_t.
    With log_alpha, the state is first decayed S <- alpha_t S (Gated
    DeltaNet, decay then delta rule). Returns o and the key-major final
    state (the transpose of the value-major one)."""
    T = q.shape[0]
    S = np.zeros((v.shape[1], k.shape[1])) if S0 is None else np.array(S0, dtype=np.float64).T
    o = np.zeros((T, v.shape[1]))
    for t in range(T):
        if log_alpha is not None:
            S = np.exp(log_alpha[t]) * S
        v_old = S @ k[t]
        v_new = beta[t] * v[t] + (1.0 - beta[t]) * v_old
        S = S - np.outer(v_old, k[t]) + np.outer(v_new, k[t])
        o[t] = S @ q[t]
    return o, S.T


def kronecker_delta(q, k, v, beta, S0=None, log_alpha=None):
    """Brute force on the vectorised state: with vec() stacking the columns
    of the key-major S [dk, dv],
      vec(S_t) = (I_dv ⊗ alpha_t (I - beta_t k_t k_t^T)) vec(S_{t-1})
                 + beta_t vec(k_t v_t^T),
    the Kronecker-product statement of the reparameterised delta rule
    S_t = (I - beta k k^T) alpha S_{t-1} + beta k v^T ("Talk Linear
    Attention", section 6.2, transposed to key-major). With a per-channel
    log_alpha [T, dk] the factor is (I - beta k k^T) Diag(alpha_t), the Kimi
    Delta Attention update as the "LLM attention optimisation" page writes it
    (its Kimi Delta Attention section). Tiny sizes only."""
    T, dk = k.shape
    dv = v.shape[1]
    s = np.zeros(dk * dv) if S0 is None else np.asarray(S0, dtype=np.float64).reshape(-1, order="F")
    o = np.zeros((T, dv))
    for t in range(T):
        if log_alpha is None:
            D = np.eye(dk)
        else:
            D = np.diag(np.broadcast_to(np.exp(np.asarray(log_alpha[t], dtype=np.float64)), (dk,)))
        Ht = (np.eye(dk) - beta[t] * np.outer(k[t], k[t])) @ D
        s = np.kron(np.eye(dv), Ht) @ s + beta[t] * np.outer(k[t], v[t]).reshape(-1, order="F")
        St = s.reshape(dk, dv, order="F")
        o[t] = St.T @ q[t]
    return o, s.reshape(dk, dv, order="F")


def chunk_form(q, k, v, mode, g=None, beta=None, S0=None, C=64):
    """Chunkwise-parallel form, float64, one head.

    The sequence is cut into chunks of C tokens ("Talk Linear Attention",
    section 3.2). Inside a chunk with inclusive log-gate prefix b_r
    (section 5.2, b_t = prod alpha_j taken in log space from the chunk start):
      P  = (Q K^T) ⊙ exp(b_r - b_s) ⊙ M     (decay-masked local attention)
      Qt = Q ⊙ exp(b), Kt = K ⊙ exp(b_last - b)
      U  = V                                  for the unit-write modes;
      U  = T (diag(beta) V - diag(beta e^b) K S),  T = (I + A)^{-1},
           A_rs = beta_r exp(b_r - b_s) k_r.k_s for s < r   (delta rule: the
           WY/UT form of section 6.2 that removes the serial dependency)
    kda takes the per-channel prefix of gla into the delta rule: the factors
    e^{b} act channel by channel, A_rs = beta_r sum_c k_rc k_sc e^{b_rc - b_sc},
    U = T (diag(beta) V - diag(beta) (K ⊙ e^b) S), S <- Diag(e^{b_last}) S + Kt^T U.
    outer adds the value-axis prefix bv (log beta): each value column v is a
    decay e^{bv_r - bv_s} of its own, so V is divided by e^{bv} before the
    products and O multiplied by it after, and the state decays by
    e^{b_last} on the key axis and e^{bv_last} on the value axis.
      O  = Qt S + P U                         (inter-chunk + local, section 3.2)
      S <- Diag(exp(b_last)) S + Kt^T U       (state passing, section 3.2)
    elu1 applies phi to q and k first and divides by Qt z + P 1, carrying
    z <- z + sum phi(k). C=1 reduces this to the recurrence and C=T to the
    parallel form (section 3.3).

    g: retnet scalar log gamma for this head; scalar/gdn [T]; gla/kda/outer [T, dk];
    outer takes the value-axis log-gates [T, dv] in beta.
    Returns (o [T, dv], S [dk, dv] or [dk, dv + 1] for elu1).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, dk = q.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv))
    z = np.zeros(dk)
    if S0 is not None:
        S0 = np.asarray(S0, dtype=np.float64)
        if mode == "elu1":
            S, z = S0[:, :dv].copy(), S0[:, dv].copy()
        else:
            S = S0.copy()
    o = np.zeros((T, dv))
    for t0 in range(0, T, C):
        t1 = min(T, t0 + C)
        n = t1 - t0
        Q, K, V = q[t0:t1], k[t0:t1], v[t0:t1]
        if mode == "elu1":
            Q, K = _phi(Q), _phi(K)
        if mode == "retnet":
            lg = np.full(n, float(g))
        elif mode in ("scalar",) or (mode == "gdn" and g is not None):
            lg = np.asarray(g[t0:t1], dtype=np.float64)
        elif mode in ("gla", "kda", "outer"):
            lg = np.asarray(g[t0:t1], dtype=np.float64)
        else:
            lg = np.zeros(n)
        b = np.cumsum(lg, axis=0)
        tril = np.tril(np.ones((n, n)))
        if mode in ("gla", "kda", "outer"):
            P = ((Q * np.exp(b)) @ (K * np.exp(-b)).T) * tril
            Qt = Q * np.exp(b)
            Kt = K * np.exp(b[-1][None, :] - b)
            decay = np.exp(b[-1])[:, None]
        else:
            P = (Q @ K.T) * np.exp(b[:, None] - b[None, :]) * tril
            Qt = Q * np.exp(b)[:, None]
            Kt = K * np.exp(b[-1] - b)[:, None]
            decay = np.exp(b[-1])
        if mode == "gdn":
            bet = np.ones(n) if beta is None else np.asarray(beta[t0:t1], dtype=np.float64)
            A = np.tril(bet[:, None] * np.exp(b[:, None] - b[None, :]) * (K @ K.T), -1)
            rhs = bet[:, None] * V - (bet * np.exp(b))[:, None] * (K @ S)
            U = solve_triangular(np.eye(n) + A, rhs, lower=True, unit_diagonal=True)
        elif mode == "kda":
            bet = np.ones(n) if beta is None else np.asarray(beta[t0:t1], dtype=np.float64)
            A = np.tril(bet[:, None] * ((K * np.exp(b)) @ (K * np.exp(-b)).T), -1)
            rhs = bet[:, None] * (V - (K * np.exp(b)) @ S)
            U = solve_triangular(np.eye(n) + A, rhs, lower=True, unit_diagonal=True)
        elif mode == "outer":
            bv = np.cumsum(np.asarray(beta[t0:t1], dtype=np.float64), axis=0)   # [n, dv]
            U = V * np.exp(-bv)
        else:
            U = V
        O = Qt @ S + P @ U
        if mode == "outer":
            O = O * np.exp(bv)
        if mode == "elu1":
            den = Qt @ z + P.sum(1)
            O = O / den[:, None]
            z = z + K.sum(0)
        o[t0:t1] = O
        if mode == "outer":  # decay of both axes to the chunk end
            S = decay * np.exp(bv[-1])[None, :] * S + Kt.T @ (U * np.exp(bv[-1])[None, :])
        else:
            S = decay * S + Kt.T @ U
    if mode == "elu1":
        S = np.concatenate([S, z[:, None]], axis=1)
    return o, S
