"""Float64 oracle of the non-causal form: every token reads the state of the
whole sequence.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module;
only tests/ and bench.py's CPU legs do. It shares no code with the CUDA path.

Per (b, h), from the exact (upcast) inputs:

  linear  S_T = S0 + sum_s k_s v_s^T            o_t = S_T^T q_t
  elu1    S_T = S0 + sum_s phi(k_s) v_s^T,  z_T = z0 + sum_s phi(k_s)
          o_t = (S_T^T phi(q_t)) / (z_T . phi(q_t)),  phi(x) = elu(x) + 1

that is, O = Q (K^T V) computed right to left (kernel-attention notes,
section 3: with no softmax the product associates, and K^T V is a dk x dv
matrix whatever the sequence length). S_final is S_T (elu1: z_T in column dv),
as in the causal form.
"""
from __future__ import annotations

import numpy as np

from .recurrence import phi_elu1

__all__ = ["noncausal"]


def noncausal(q, k, v, mode, S0=None):
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if mode == "linear":
        S = np.zeros((B, H, dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
        S = S + np.einsum("bhtc,bhtv->bhcv", k, v)
        return np.einsum("bhtc,bhcv->bhtv", q, S), S
    if mode == "elu1":
        qh, kh = phi_elu1(q), phi_elu1(k)
        S = np.zeros((B, H, dk, dv + 1)) if S0 is None else np.array(S0, dtype=np.float64)
        S[..., :dv] += np.einsum("bhtc,bhtv->bhcv", kh, v)
        S[..., dv] += kh.sum(axis=2)
        num = np.einsum("bhtc,bhcv->bhtv", qh, S[..., :dv])
        den = np.einsum("bhtc,bhc->bht", qh, S[..., dv])
        return num / den[..., None], S
    raise ValueError(f"the non-causal form is defined for linear and elu1, not {mode}")
