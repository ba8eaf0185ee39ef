"""Helpers for the GPU parity tests: run the CUDA path, run the oracle, compare.

Tolerances (for both o and the final state):
  bf16 inputs: max-abs error <= 2e-2 and relative Frobenius error <= 5e-3
  fp32 inputs: relative Frobenius error <= 1e-4 and max-abs error
               <= 1e-4 * max(1, max |reference|)
"""
from __future__ import annotations

import numpy as np
import torch

import gated_delta_rule_linear_gb300 as la
import oracle
import workloads

BF16_MAX_ABS = 2e-2
BF16_REL_FRO = 5e-3
F32_REL = 1e-4


def f64(t):
    return None if t is None else t.detach().float().cpu().numpy().astype(np.float64)


def to_dev(inp, dev="cuda"):
    return {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inp.items()}


def run_cuda(inp, C=0, with_state=True, S0=None):
    d = to_dev(inp)
    wl = inp["wl"]
    torch.cuda.synchronize()
    o, S = la.chunk_fwd(d["q"], d["k"], d["v"], wl.mode, g=d["g"], beta=d["beta"],
                        S0=d["S0"] if S0 is None else S0, C=C, with_state=with_state)
    torch.cuda.synchronize()
    return o, S


def run_oracle(inp, heads=None, use_c=None):
    """Oracle on all heads, or on a list of (b, h) heads (returned stacked as
    [1, len(heads), ...])."""
    wl = inp["wl"]
    q, k, v, g, beta, S0 = (inp[n] for n in ("q", "k", "v", "g", "beta", "S0"))
    if heads is not None:
        sel = lambda x: None if x is None else torch.stack([x[b, h] for b, h in heads])[None]
        q, k, v, beta, S0 = sel(q), sel(k), sel(v), sel(beta), sel(S0)
        if g is not None:
            g = torch.stack([g[h] for _, h in heads]) if wl.mode == "retnet" else sel(g)
    args = [f64(q), f64(k), f64(v), wl.mode]
    kw = dict(g=f64(g), beta=f64(beta), S0=f64(S0))
    if use_c is None:
        use_c = q.shape[2] * q.shape[1] * q.shape[0] > 4096
    if use_c:
        return oracle.recurrence_c(*args, **kw)
    return oracle.recurrence(*args, **kw)


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in the CUDA result"
    diff = got - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-30))
    return max_abs, rel


def assert_close(got, ref, dtype, what=""):
    max_abs, rel = errors(got, ref)
    if dtype == "bf16":
        ok = max_abs <= BF16_MAX_ABS and rel <= BF16_REL_FRO
    else:
        scale = max(1.0, float(np.max(np.abs(ref))) if np.size(ref) else 1.0)
        ok = rel <= F32_REL and max_abs <= F32_REL * scale
    assert ok, f"{what}: max_abs={max_abs:.3e} rel_fro={rel:.3e} ({dtype})"
    return max_abs, rel


def make(name, **sizes):
    return workloads.make_inputs(name, **sizes)
