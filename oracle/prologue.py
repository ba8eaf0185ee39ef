"""Float64 oracle of the prologue: the per-token steps between the q/k/v/gate
projections and the chunk forward pass.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module;
only tests/, the smoke check and bench.py's CPU legs do. It shares no code
with the CUDA path.

Steps, per (b, h), all in float64 from the exact (upcast) inputs:

  short convolution   x~_t[c] = sum_{tau=0}^{K-1} w[h, c, tau] * x_{t-tau}[c]
      ("LLM attention optimisation: linear attention", DeltaNet section: a
      depthwise short convolution over the last K tokens after the q/k/v
      projections, K = 4 in DeltaNet). Tokens before the first one come from
      the history (the last K-1 raw rows of the previous call), else zero.
      Applied to q, k and v, each with its own weights (w = None: no
      convolution for that tensor).
  L2 normalisation    x <- x / max(||x||_2, 1e-6) per token, optional for q
      and k (the pages do not state it; the Gated DeltaNet workload uses
      L2-normalised q and k, with this guard for a zero vector).
  gate activation     g = logsigmoid(a) / tau  (log of alpha = sigmoid(.)^(1/tau),
      "Talk Linear Attention" section 5.1, the GLA gate), or
      g = -softplus(a) / tau  (a log-decay in (-inf, 0), so alpha in (0, 1),
      as the Gated DeltaNet section requires; the pages give no formula),
      scalar [B, H, T] or per key channel [B, H, T, dk].
  write strength      beta = sigmoid(a_beta), in (0, 1).

The history returned is the last K-1 raw rows (before the convolution) of
the concatenation history ++ x, so a call on x[:T1] followed by a call on
x[T1:] with that history equals one call on x.
"""
from __future__ import annotations

import numpy as np

GATE_KINDS = ("none", "logsigmoid", "neg_softplus")

__all__ = ["short_conv", "l2norm", "gate_activation", "beta_activation", "prologue", "GATE_KINDS"]


def short_conv(x, w, hist=None):
    """x [B, H, T, d], w [H, d, K] (w[..., 0] multiplies the current token),
    hist [B, H, K-1, d] raw rows before x (oldest first) or None for zeros.
    Returns (y [B, H, T, d], new_hist [B, H, K-1, d])."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    B, H, T, d = x.shape
    K = w.shape[-1]
    if hist is None:
        hist = np.zeros((B, H, K - 1, d))
    hist = np.asarray(hist, dtype=np.float64)
    full = np.concatenate([hist, x], axis=2)  # row K-1+t is token t
    y = np.zeros_like(x)
    for tau in range(K):
        # token t reads row K-1+t-tau of the padded sequence
        y += w[None, :, None, :, tau] * full[:, :, K - 1 - tau:K - 1 - tau + T, :]
    return y, full[:, :, full.shape[2] - (K - 1):, :].copy()


def l2norm(x, eps=1e-6):
    x = np.asarray(x, dtype=np.float64)
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / np.maximum(n, eps)


def _softplus(a):
    # log(1 + e^a), written to stay finite for large |a|
    return np.maximum(a, 0.0) + np.log1p(np.exp(-np.abs(a)))


def gate_activation(a, kind, tau=1.0):
    a = np.asarray(a, dtype=np.float64)
    if kind == "logsigmoid":
        return -_softplus(-a) / tau          # log(1 / (1 + e^-a))
    if kind == "neg_softplus":
        return -_softplus(a) / tau
    raise ValueError(kind)


def beta_activation(a):
    a = np.asarray(a, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-a))


def prologue(xq, xk, xv, wq=None, wk=None, wv=None, hist=None, l2q=False, l2k=False,
             a_gate=None, gate_kind="none", tau=1.0, a_beta=None, K=None):
    """Whole prologue. hist is a dict with keys q, k, v ([B, H, K-1, d]) or None.
    Returns a dict with q, k, v, g (or None), beta (or None) and hist (the new
    history dict, None when K == 1)."""
    if K is None:
        K = next((w.shape[-1] for w in (wq, wk, wv) if w is not None), 1)
    out, new_hist = {}, {}
    for name, x, w in (("q", xq, wq), ("k", xk, wk), ("v", xv, wv)):
        x = np.asarray(x, dtype=np.float64)
        h_in = None if hist is None else hist[name]
        if w is None:  # identity: the current token with weight 1
            B, H, T, d = x.shape
            w = np.zeros((H, d, K))
            w[..., 0] = 1.0
        y, h_out = short_conv(x, w, h_in)
        out[name], new_hist[name] = y, h_out
    if l2q:
        out["q"] = l2norm(out["q"])
    if l2k:
        out["k"] = l2norm(out["k"])
    out["g"] = None if gate_kind == "none" else gate_activation(a_gate, gate_kind, tau)
    out["beta"] = None if a_beta is None else beta_activation(a_beta)
    out["hist"] = new_hist if K > 1 else None
    return out
