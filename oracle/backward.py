"""Float64 oracle of the backward pass of the causal forward, for the modes
whose decay is not a learned input: plain linear attention and RetNet's fixed
per-head decay.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module;
only tests/ and bench.py's CPU legs do. It shares no code with the CUDA path.

Forward, per (b, h), with alpha = 1 (linear) or gamma_h = exp(g_h) (RetNet):

  S_t = alpha S_{t-1} + k_t v_t^T,  o_t = S_t^T q_t,  S_final = S_{T-1}
  so  o_t = alpha^(t+1) S0^T q_t + sum_{s<=t} alpha^(t-s) (q_t . k_s) v_s
      S_final = alpha^T S0 + sum_s alpha^(T-1-s) k_s v_s^T

("Talk Linear Attention" sections 2.1 and 5.2; section 4.1.2 of the same page
notes that the backward pass recomputes the chunk states rather than storing
them).
Given dO = dL/do and dS = dL/dS_final, the gradients are the plain sums

  dq_t = alpha^(t+1) S0 dO_t + sum_{s<=t} alpha^(t-s) (dO_t . v_s) k_s
  dk_s = sum_{t>=s} alpha^(t-s) (dO_t . v_s) q_t + alpha^(T-1-s) dS v_s
  dv_s = sum_{t>=s} alpha^(t-s) (q_t . k_s) dO_t + alpha^(T-1-s) dS^T k_s
  dS0  = sum_t alpha^(t+1) q_t dO_t^T + alpha^T dS

written out below with explicit decay matrices (no reordering beyond the sums).
"""
from __future__ import annotations

import numpy as np

__all__ = ["backward", "backward_scalar", "backward_gla"]


def backward(q, k, v, dO, mode, g=None, S0=None, dS=None):
    """q, k [B,H,T,dk]; v, dO [B,H,T,dv]; g [H] log-decay for retnet; S0, dS
    [B,H,dk,dv] or None. Returns dq, dk, dv, dS0 (float64)."""
    q, k, v, dO = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dO))
    B, H, T, dkk = q.shape
    dvv = v.shape[-1]
    if mode == "linear":
        logs = np.zeros(H)
    elif mode == "retnet":
        logs = np.asarray(g, dtype=np.float64).reshape(H)
    else:
        raise ValueError(f"backward is defined here for linear and retnet, not {mode}")
    S0 = np.zeros((B, H, dkk, dvv)) if S0 is None else np.asarray(S0, dtype=np.float64)
    dS = np.zeros((B, H, dkk, dvv)) if dS is None else np.asarray(dS, dtype=np.float64)
    t = np.arange(T)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dS0 = np.zeros_like(S0)
    for h in range(H):
        la = logs[h]
        # D[t, s] = alpha^(t-s) for s <= t, else 0
        diff = t[:, None] - t[None, :]
        D = np.where(diff >= 0, np.exp(la * np.maximum(diff, 0)), 0.0)
        a_t1 = np.exp(la * (t + 1))        # alpha^(t+1)
        a_last = np.exp(la * (T - 1 - t))  # alpha^(T-1-s)
        aT = np.exp(la * T)
        for b in range(B):
            Q, K, V, G = q[b, h], k[b, h], v[b, h], dO[b, h]
            Mo = (G @ V.T) * D                  # [t, s] = alpha^(t-s) (dO_t . v_s), s <= t
            Mk = (Q @ K.T) * D                  # [t, s] = alpha^(t-s) (q_t . k_s)
            dq[b, h] = a_t1[:, None] * (G @ S0[b, h].T) + Mo @ K
            dk[b, h] = Mo.T @ Q + a_last[:, None] * (V @ dS[b, h].T)
            dv[b, h] = Mk.T @ G + a_last[:, None] * (K @ dS[b, h])
            dS0[b, h] = (Q * a_t1[:, None]).T @ G + aT * dS[b, h]
    return dq, dk, dv, dS0


def backward_scalar(q, k, v, dO, g, S0=None, dS=None):
    """The same gradients for the data-dependent scalar decay (alpha_t =
    exp(g_t), g [B, H, T]), plus the gradient of the log-gates. With the
    inclusive prefix G_t = sum_{tau<=t} g_tau the decay between positions is
    alpha(t, s) = exp(G_t - G_s), so dq, dk, dv and dS0 are the sums above with
    those factors, and, since G_u enters with + where u reads (o_u, and
    S_final through G_{T-1}) and with - where u writes,

      dL/dG_u = q_u . dq_u - k_u . dk_u + [u = T-1] sum(dS ⊙ S_final),
      dg_tau  = sum_{u >= tau} dL/dG_u.

    Returns dq, dk, dv, dS0, dg (float64)."""
    q, k, v, dO, g = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dO, g))
    B, H, T, dkk = q.shape
    dvv = v.shape[-1]
    S0 = np.zeros((B, H, dkk, dvv)) if S0 is None else np.asarray(S0, dtype=np.float64)
    dS = np.zeros((B, H, dkk, dvv)) if dS is None else np.asarray(dS, dtype=np.float64)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dS0 = np.zeros_like(S0)
    dg = np.zeros((B, H, T))
    tri = np.tril(np.ones((T, T)))
    for b in range(B):
        for h in range(H):
            G = np.cumsum(g[b, h])
            D = np.exp(np.where(tri > 0, G[:, None] - G[None, :], -np.inf))   # alpha(t, s), s <= t
            a_t1 = np.exp(G)                  # alpha(t, -1)
            a_last = np.exp(G[-1] - G)        # alpha(T-1, s)
            aT = np.exp(G[-1])
            Q, K, V, Gd = q[b, h], k[b, h], v[b, h], dO[b, h]
            Mo = (Gd @ V.T) * D
            Mk = (Q @ K.T) * D
            dq[b, h] = a_t1[:, None] * (Gd @ S0[b, h].T) + Mo @ K
            dk[b, h] = Mo.T @ Q + a_last[:, None] * (V @ dS[b, h].T)
            dv[b, h] = Mk.T @ Gd + a_last[:, None] * (K @ dS[b, h])
            dS0[b, h] = (Q * a_t1[:, None]).T @ Gd + aT * dS[b, h]
            S_T = aT * S0[b, h] + (K * a_last[:, None]).T @ V
            dG = np.sum(Q * dq[b, h], axis=1) - np.sum(K * dk[b, h], axis=1)
            dG[-1] += np.sum(dS[b, h] * S_T)
            dg[b, h] = np.cumsum(dG[::-1])[::-1]
    return dq, dk, dv, dS0, dg


def backward_gla(q, k, v, dO, g, S0=None, dS=None):
    """The gradients for GLA's per-key-channel decay (alpha_t[c] = exp(g_t[c]),
    g [B, H, T, dk]). With the inclusive prefix G_t[c], the decay of channel c
    between positions is alpha_c(t, s) = exp(G_t[c] - G_s[c]), and

      dq_t[c] = sum_{s<=t} (dO_t . v_s) alpha_c(t, s) k_s[c] + alpha_c(t, -1) (S0 dO_t)[c]
      dk_s[c] = sum_{t>=s} (dO_t . v_s) alpha_c(t, s) q_t[c] + alpha_c(T-1, s) (dS v_s)[c]
      dv_s    = sum_{t>=s} (sum_c q_t[c] alpha_c(t, s) k_s[c]) dO_t + dS^T (alpha(T-1, s) ⊙ k_s)
      dS0[c]  = sum_t alpha_c(t, -1) q_t[c] dO_t + alpha_c(T-1, -1) dS[c]
      dg_tau[c] = sum_{u>=tau} (q_u[c] dq_u[c] - k_u[c] dk_u[c]) + sum_j dS[c, j] S_final[c, j]

    (G_u[c] enters with + where u reads and with - where u writes, as for the
    scalar decay, now channel by channel). Written as explicit sums over token
    pairs. Returns dq, dk, dv, dS0, dg (float64)."""
    q, k, v, dO, g = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dO, g))
    B, H, T, dkk = q.shape
    dvv = v.shape[-1]
    S0 = np.zeros((B, H, dkk, dvv)) if S0 is None else np.asarray(S0, dtype=np.float64)
    dS = np.zeros((B, H, dkk, dvv)) if dS is None else np.asarray(dS, dtype=np.float64)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dS0 = np.zeros_like(S0)
    dg = np.zeros_like(g)
    for b in range(B):
        for h in range(H):
            G = np.cumsum(g[b, h], axis=0)                       # [T, dk]
            Q, K, V, Gd = q[b, h], k[b, h], v[b, h], dO[b, h]
            S_T = np.exp(G[-1])[:, None] * S0[b, h]
            for t in range(T):
                a0 = np.exp(G[t])                                # alpha(t, -1)
                dq[b, h, t] += a0 * (S0[b, h] @ Gd[t])
                dS0[b, h] += np.outer(a0 * Q[t], Gd[t])
                for s in range(t + 1):
                    a = np.exp(G[t] - G[s])                      # alpha(t, s) per channel
                    w = Gd[t] @ V[s]
                    dq[b, h, t] += w * a * K[s]
                    dk[b, h, s] += w * a * Q[t]
                    dv[b, h, s] += (Q[t] @ (a * K[s])) * Gd[t]
            aT = np.exp(G[-1])
            dS0[b, h] += aT[:, None] * dS[b, h]
            for s in range(T):
                al = np.exp(G[-1] - G[s])                        # alpha(T-1, s)
                dk[b, h, s] += al * (dS[b, h] @ V[s])
                dv[b, h, s] += dS[b, h].T @ (al * K[s])
                S_T += np.outer(al * K[s], V[s])
            dGu = Q * dq[b, h] - K * dk[b, h]                    # [T, dk]
            dGu[-1] += np.sum(dS[b, h] * S_T, axis=1)
            dg[b, h] = np.cumsum(dGu[::-1], axis=0)[::-1]
    return dq, dk, dv, dS0, dg
