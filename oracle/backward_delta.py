"""Float64 oracle of the backward pass of the delta-rule forward (Gated
DeltaNet and Kimi Delta Attention): the gradients of the token recurrence,
taken by reverse-mode differentiation of its steps, one token at a time.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module;
only tests/ and bench.py's CPU legs do. It shares no code with the CUDA path.

Forward, per (b, h), key-major state S [dk, dv], for t = 0 .. T-1
("LLM attention optimisation" page, Gated DeltaNet and Kimi Delta Attention
sections; "Talk Linear Attention" section 6.2, the delta rule):

  R_t = alpha_t S_{t-1}             (gdn: scalar alpha_t = exp(g_t);
                                     kda: Diag(alpha_t) on the key axis, alpha_t = exp(g_t[c]))
  r_t = v_t - R_t^T k_t             (what the key k_t reads back, subtracted from v_t)
  S_t = R_t + beta_t k_t r_t^T      (= (I - beta k k^T) R_t + beta k v^T)
  o_t = S_t^T q_t ,  S_final = S_{T-1}

"Talk Linear Attention" section 4.1.2 says the backward pass recomputes the
states instead of storing them; the pages give no gradient formulas, so the
ones below are the chain rule applied to the four lines above, last line
first. With Gh = dL/dS_t (the gradient arriving from later tokens plus the
read of o_t):

  Gh   = G + q_t dO_t^T             (o_t = S_t^T q_t reads S_t)
  dq_t = S_t dO_t
  Gk   = Gh^T k_t                   (shared by the terms through r_t)
  dv_t = beta_t Gk                  (r_t enters S_t as beta k r^T)
  dbeta_t = Gk . r_t
  dk_t = beta_t (Gh r_t - R_t Gk)   (k_t writes, and reads through r_t)
  dR   = Gh - beta_t k_t Gk^T       (= (I - beta k k^T) Gh)
  dg_t = <dR, R_t>                  (gdn: a scalar; kda: one value per key
                                     channel c, the row sum of dR ⊙ R_t)
  G    = alpha_t dR                 (dL/dS_{t-1}; dS0 = G after token 0)

starting from G = dS (= dL/dS_final). alpha = 1 when g is absent (plain
DeltaNet, gdn only) and beta = 1 when beta is absent, as in the forward.

The reverse sweep needs S_{t-1} for every t. The forward states are kept
every `checkpoint` tokens and the steps between two checkpoints are re-run
forward, in the same float64 operations, when the sweep reaches them: the
values are bit-identical to storing every state, with memory for T/checkpoint
states instead of T.
"""
from __future__ import annotations

import numpy as np

__all__ = ["backward_delta"]


def _f64(x):
    return None if x is None else np.asarray(x, dtype=np.float64)


def _token_grads(G, q_t, k_t, dO_t, beta_t, alpha_t, R, r, S_t, per_channel):
    """The reverse of one token (the lines of the module docstring, in order):
    G = dL/dS_t from later tokens, R = R_t, r = r_t, S_t the state after the
    token. Returns dq_t, dk_t, dv_t, dbeta_t, dg_t, dL/dS_{t-1}."""
    Gh = G + np.outer(q_t, dO_t)
    dq = S_t @ dO_t
    Gk = Gh.T @ k_t
    dv = beta_t * Gk
    dbeta = Gk @ r
    dk = beta_t * (Gh @ r - R @ Gk)
    dR = Gh - beta_t * np.outer(k_t, Gk)
    dg = np.sum(dR * R, axis=1) if per_channel else np.sum(dR * R)
    return dq, dk, dv, dbeta, dg, alpha_t[:, None] * dR


def backward_delta(q, k, v, dO, mode="gdn", g=None, beta=None, S0=None, dS=None, checkpoint=256):
    """q, k [B,H,T,dk]; v, dO [B,H,T,dv]; g [B,H,T] (gdn) or [B,H,T,dk] (kda),
    or None (gdn only: alpha = 1); beta [B,H,T] or None (beta = 1); S0, dS
    [B,H,dk,dv] or None (zero).

    Returns dq [B,H,T,dk], dk [B,H,T,dk], dv [B,H,T,dv], dbeta [B,H,T],
    dg (like g, or None when g is None), dS0 [B,H,dk,dv] (float64)."""
    if mode not in ("gdn", "kda"):
        raise ValueError(f"backward_delta covers gdn and kda, not {mode!r}")
    if mode == "kda" and g is None:
        raise ValueError("kda needs per-channel log-gates g")
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    g, beta, S0, dS = _f64(g), _f64(beta), _f64(S0), _f64(dS)
    B, H, T, dkk = q.shape
    dvv = v.shape[-1]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dbeta = np.zeros((B, H, T))
    dg = None if g is None else np.zeros_like(g)
    dS0 = np.zeros((B, H, dkk, dvv))
    for b in range(B):
        for h in range(H):
            Q, K, V, dOh = q[b, h], k[b, h], v[b, h], dO[b, h]
            bet = np.ones(T) if beta is None else beta[b, h]
            if g is None:
                alpha = np.ones((T, 1))
            elif mode == "gdn":
                alpha = np.exp(g[b, h])[:, None]           # [T, 1]: one factor per token
            else:
                alpha = np.exp(g[b, h])                    # [T, dk]: one factor per key channel

            def step(S_prev, t):
                """One forward token: returns (R_t, r_t, S_t)."""
                R = alpha[t][:, None] * S_prev
                r = V[t] - R.T @ K[t]
                return R, r, R + bet[t] * np.outer(K[t], r)

            # forward: states at the checkpoints (S_{t-1} for t = 0, c, 2c, ...)
            S = np.zeros((dkk, dvv)) if S0 is None else S0[b, h].copy()
            ckpt = []
            for t in range(T):
                if t % checkpoint == 0:
                    ckpt.append(S.copy())
                S = step(S, t)[2]
            # reverse sweep, one checkpoint segment at a time (last segment first)
            G = np.zeros((dkk, dvv)) if dS is None else dS[b, h].copy()
            for seg in range(len(ckpt) - 1, -1, -1):
                t0, t1 = seg * checkpoint, min(T, (seg + 1) * checkpoint)
                prev = [ckpt[seg]]                          # S_{t-1} for t = t0 .. t1-1
                for t in range(t0, t1 - 1):
                    prev.append(step(prev[-1], t)[2])
                for t in range(t1 - 1, t0 - 1, -1):
                    R, r, S_t = step(prev[t - t0], t)
                    dq[b, h, t], dk[b, h, t], dv[b, h, t], dbeta[b, h, t], dgt, G = _token_grads(
                        G, Q[t], K[t], dOh[t], bet[t], alpha[t], R, r, S_t, mode == "kda")
                    if dg is not None:
                        dg[b, h, t] = dgt
            dS0[b, h] = G
    return dq, dk, dv, dbeta, dg, dS0
