"""Float64 token-by-token recurrence: the definition the chunked GPU path must reproduce.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this
module; only tests/, the smoke check and bench.py's CPU-baseline leg do.

Orientation. The state S is key-major, shape [dk, dv], and the output is
o_t = S_t^T q_t. The pages write the same recurrence both ways: "Talk Linear
Attention" section 2.1 and the kernel-attention notes (section 13) use
S = sum k v^T read as q^T S; "Talk Linear Attention" section 6 and the
"LLM attention optimisation: linear attention" page write S = sum v k^T read
as S q. The two states are transposes of one another and give identical o.

Per (b, h), starting from S0 (zero when absent), for t = 0..T-1:

  linear  S <- S + k_t v_t^T                      o_t = S^T q_t
          ("Talk Linear Attention", section 2.1, the recurrent form)
  elu1    qh, kh = phi(q_t), phi(k_t), phi(x) = elu(x) + 1
          S <- S + kh v_t^T ; z <- z + kh          o_t = (S^T qh) / (z^T qh)
          (kernel-attention notes, sections 13-14, causal form with the
          normaliser z; "Linear Attention" glossary, kernel decomposition)
  retnet  S <- gamma_h S + k_t v_t^T               o_t = S^T q_t
          (fixed, data-independent decay; linear-attention page, decay section)
  scalar  S <- alpha_t S + k_t v_t^T               (data-dependent scalar decay)
  gla     S <- Diag(alpha_t) S + k_t v_t^T         ("Talk Linear Attention",
          section 5.1, gate G_t = alpha_t 1^T acting on the key axis)
  gdn     S <- alpha_t S ; u = beta_t (v_t - S^T k_t) ; S <- S + k_t u^T
          o_t = S^T q_t  (Gated DeltaNet: decay first, then the delta rule,
          "LLM attention optimisation" page, Gated DeltaNet section;
          "Talk Linear Attention" section 6.2 reparameterised form)
  kda     S <- Diag(alpha_t) S ; u = beta_t (v_t - S^T k_t) ; S <- S + k_t u^T
          (Kimi Delta Attention: Gated DeltaNet with a per-key-channel gate,
          S_t = (I - beta k k^T) Diag(alpha_t) S_{t-1} + beta k v^T in this
          key-major orientation; "LLM attention optimisation" page, Kimi Delta
          Attention section)
  outer   S <- (alpha_t beta_t^T) ⊙ S + k_t v_t^T  o_t = S^T q_t
          (gate G_t = alpha_t beta_t^T, an outer product of a key-axis and a
          value-axis gate: the form "Talk Linear Attention" section 5.4 gives
          for gated linear attention that stays a matrix product; alpha_t
          scales row c of S, beta_t column v)

Gates are natural logs: alpha = exp(g). retnet takes g of shape [H]; scalar
and gdn take [B, H, T]; gla and kda take [B, H, T, dk]. gdn and kda take beta
[B, H, T]; a missing g means alpha = 1 (plain DeltaNet, gdn only) and a
missing beta means 1. outer takes g = log alpha [B, H, T, dk] and, in the
beta argument, log beta [B, H, T, dv] (both required).

For elu1 the state carries z as an extra value column: S has shape
[dk, dv + 1] with z in column dv, both in S0 and in the returned state.

Parity of this module is pinned in tests/test_oracle_pins.py against the
pages' parallel forms, the DeltaNet four-step form, a Kronecker-product
brute force, the C=1 / C=T limits of the chunk form, the exact-retrieval
invariant and golden values built from the pages' recall examples.
"""
from __future__ import annotations

import numpy as np

__all__ = ["recurrence", "phi_elu1", "MODES"]

MODES = ("linear", "elu1", "retnet", "gla", "scalar", "gdn", "kda", "outer")


def phi_elu1(x):
    """elu(x) + 1: x + 1 for x > 0, exp(x) otherwise (always positive)."""
    x = np.asarray(x, dtype=np.float64)
    return np.where(x > 0.0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def _f64(x):
    return None if x is None else np.asarray(x, dtype=np.float64)


def recurrence(q, k, v, mode, g=None, beta=None, S0=None):
    """Run the per-token recurrence for every (b, h) in float64.

    q, k: [B, H, T, dk]; v: [B, H, T, dv]; any real dtype, upcast exactly.
    Returns (o [B, H, T, dv], S [B, H, dk, dv] or [B, H, dk, dv + 1] for elu1).
    """
    if mode not in MODES:
        raise ValueError(f"unknown mode {mode!r}")
    q, k, v = _f64(q), _f64(k), _f64(v)
    g, beta, S0 = _f64(g), _f64(beta), _f64(S0)
    B, H, T, dk = q.shape
    dv = v.shape[-1]

    S = np.zeros((B, H, dk, dv))
    z = np.zeros((B, H, dk))
    if S0 is not None:
        if mode == "elu1":
            S[:] = S0[..., :dv]
            z[:] = S0[..., dv]
        else:
            S[:] = S0
    o = np.zeros((B, H, T, dv))

    for t in range(T):
        qt, kt, vt = q[:, :, t], k[:, :, t], v[:, :, t]          # [B,H,d]
        if mode == "linear":
            S += kt[..., :, None] * vt[..., None, :]
            o[:, :, t] = np.einsum("bhc,bhcv->bhv", qt, S)
        elif mode == "elu1":
            qh, kh = phi_elu1(qt), phi_elu1(kt)
            S += kh[..., :, None] * vt[..., None, :]
            z += kh
            num = np.einsum("bhc,bhcv->bhv", qh, S)
            den = np.einsum("bhc,bhc->bh", qh, z)
            o[:, :, t] = num / den[..., None]
        elif mode in ("retnet", "scalar"):
            if mode == "retnet":
                alpha = np.exp(g)[None, :, None, None]            # [1,H,1,1]
            else:
                alpha = np.exp(g[:, :, t])[..., None, None]       # [B,H,1,1]
            S = alpha * S + kt[..., :, None] * vt[..., None, :]
            o[:, :, t] = np.einsum("bhc,bhcv->bhv", qt, S)
        elif mode == "gla":
            alpha = np.exp(g[:, :, t])[..., :, None]              # [B,H,dk,1]
            S = alpha * S + kt[..., :, None] * vt[..., None, :]
            o[:, :, t] = np.einsum("bhc,bhcv->bhv", qt, S)
        elif mode == "outer":
            G = np.exp(g[:, :, t])[..., :, None] * np.exp(beta[:, :, t])[..., None, :]  # [B,H,dk,dv]
            S = G * S + kt[..., :, None] * vt[..., None, :]
            o[:, :, t] = np.einsum("bhc,bhcv->bhv", qt, S)
        else:  # gdn, kda: decay first, then the delta rule
            if mode == "kda":
                S = np.exp(g[:, :, t])[..., :, None] * S          # Diag(alpha_t) on the key axis
            elif g is not None:
                S = np.exp(g[:, :, t])[..., None, None] * S
            b = 1.0 if beta is None else beta[:, :, t][..., None]   # [B,H,1]
            retrieved = np.einsum("bhc,bhcv->bhv", kt, S)         # S^T k_t
            u = b * (vt - retrieved)
            S = S + kt[..., :, None] * u[..., None, :]
            o[:, :, t] = np.einsum("bhc,bhcv->bhv", qt, S)

    if mode == "elu1":
        S = np.concatenate([S, z[..., None]], axis=-1)
    return o, S
