"""ctypes binding of libla.so: the C ABI of include/la.h under the same names.

Argument marshalling only. The raw entry points (``la_chunk_fwd``,
``la_recurrent_step``, ...) take integers for device pointers exactly like the
C functions; ``chunk_fwd`` / ``recurrent_step`` accept torch CUDA tensors,
allocate the outputs and raise ``LAError`` on a non-zero status. Every step of
the computation runs in the library's CUDA kernels; there is no fallback: if
the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libla.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "la.h")


def _read_constants(path):
    consts = {}
    with open(path) as f:
        for line in f:
            m = re.match(r"#define\s+(LA_[A-Z0-9_]+)\s+(0x[0-9a-fA-F]+|\d+)", line)
            if m:
                consts[m.group(1)] = int(m.group(2), 0)
    return consts


CONSTANTS = _read_constants(HEADER)
globals().update(CONSTANTS)

MODE_IDS = {
    "linear": CONSTANTS["LA_LINEAR"],
    "elu1": CONSTANTS["LA_ELU1_NORM"],
    "retnet": CONSTANTS["LA_RETNET"],
    "gla": CONSTANTS["LA_GLA"],
    "scalar": CONSTANTS["LA_SCALAR_GATE"],
    "gdn": CONSTANTS["LA_GDN"],
    "kda": CONSTANTS["LA_KDA"],
    "outer": CONSTANTS["LA_OUTER_GATE"],  # beta carries the value-axis log-gates
}

# Every function the header declares, with its ctypes signature.
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
SIGNATURES = {
    "la_chunk_fwd": ([_P] * 8 + [_I] * 7 + [_P], _I),
    "la_chunk_fwd_gdelta": ([_P] * 8 + [_I] * 7 + [_P], _I),
    "la_chunk_fwd_noalloc": ([_P] * 8 + [_I] * 7 + [_P], _I),
    "la_recurrent_step": ([_P] * 7 + [_I] * 5 + [_P], _I),
    "la_chunk_bwd": ([_P] * 12 + [_I] * 7 + [_P], _I),
    "la_chunk_bwd_delta": ([_P] * 14 + [_I] * 7 + [_P], _I),
    "la_prologue": ([_P] * 6 + [_I] + [_P] * 3 + [_I, _I, _F] + [_P] * 6 + [_I] * 6 + [_P], _I),
    "la_stream_status": ([_P], _I),
    "la_last_error": ([], ctypes.c_char_p),
    "la_version": ([], _I),
}


class LAError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"[{code}] {msg}")
        self.code = code


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libla.so (once) and bind every declared symbol. Raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libla.so is not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


# ---- raw C entry points (same names and argument order as la.h) -----------

def la_chunk_fwd(q, k, v, g, beta, o, S0, S_final, B, H, T, dk, dv, C, mode, stream):
    return load_library().la_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(o),
                                       _ptr(S0), _ptr(S_final), B, H, T, dk, dv, C, mode, stream)


def la_chunk_fwd_noalloc(q, k, v, g, beta, o, S0, S_final, B, H, T, dk, dv, C, mode, stream):
    return load_library().la_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                               _ptr(o), _ptr(S0), _ptr(S_final), B, H, T, dk, dv,
                                               C, mode, stream)


def la_chunk_fwd_gdelta(q, k, v, a, b, o, S0, S_final, B, H, T, dk, dv, C, mode, stream):
    return load_library().la_chunk_fwd_gdelta(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(o),
                                              _ptr(S0), _ptr(S_final), B, H, T, dk, dv, C, mode, stream)


def la_chunk_bwd(q, k, v, g, dO, dS_final, S0, dq_out, dk_out, dv_out, dS0, dg_out, B, H, T, dk, dv, C, mode,
                 stream):
    return load_library().la_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(dO), _ptr(dS_final), _ptr(S0),
                                       _ptr(dq_out), _ptr(dk_out), _ptr(dv_out), _ptr(dS0), _ptr(dg_out), B, H, T,
                                       dk, dv, C, mode, stream)


def la_chunk_bwd_delta(q, k, v, g, beta, dO, dS_final, S0, dq_out, dk_out, dv_out, dbeta_out, dg_out, dS0,
                       B, H, T, dk, dv, C, mode, stream):
    return load_library().la_chunk_bwd_delta(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(dO),
                                             _ptr(dS_final), _ptr(S0), _ptr(dq_out), _ptr(dk_out), _ptr(dv_out),
                                             _ptr(dbeta_out), _ptr(dg_out), _ptr(dS0), B, H, T, dk, dv, C, mode,
                                             stream)


def la_recurrent_step(q, k, v, g, beta, o, S, B, H, dk, dv, mode, stream):
    return load_library().la_recurrent_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                            _ptr(o), _ptr(S), B, H, dk, dv, mode, stream)


def la_prologue(xq, xk, xv, wq, wk, wv, K, hist_in, hist_out, a_gate, gate_kind, gate_width, tau,
                a_beta, q, k, v, g, beta, B, H, T, dk, dv, flags, stream):
    return load_library().la_prologue(_ptr(xq), _ptr(xk), _ptr(xv), _ptr(wq), _ptr(wk), _ptr(wv), K,
                                      _ptr(hist_in), _ptr(hist_out), _ptr(a_gate), gate_kind,
                                      gate_width, float(tau), _ptr(a_beta), _ptr(q), _ptr(k), _ptr(v),
                                      _ptr(g), _ptr(beta), B, H, T, dk, dv, flags, stream)


def la_stream_status(stream):
    return load_library().la_stream_status(stream)


def la_last_error() -> str:
    return load_library().la_last_error().decode()


def la_version() -> int:
    return load_library().la_version()


# ---- torch-tensor convenience wrappers --------------------------------------

def _mode_id(mode, dtype):
    import torch
    mid = MODE_IDS[mode] if isinstance(mode, str) else int(mode)
    if dtype == torch.float32:
        mid |= CONSTANTS["LA_F32"]
    elif dtype != torch.bfloat16:
        raise TypeError(f"q/k/v must be bfloat16 or float32, got {dtype}")
    return mid


def _check(t, name):
    if t is not None and (not t.is_cuda or not t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def _stream_handle(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def chunk_fwd(q, k, v, mode, g=None, beta=None, S0=None, C=0, with_state=True,
              o=None, S_final=None, stream=None):
    """Chunkwise causal forward. q, k [B,H,T,dk], v [B,H,T,dv] (bf16 or fp32,
    CUDA, contiguous). Returns (o, S_final or None)."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("S0", S0)):
        _check(t, name)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    mid = _mode_id(mode, q.dtype)
    if o is None:
        o = torch.empty((B, H, T, dv), dtype=q.dtype, device=q.device)
    if with_state and S_final is None:
        W = dv + 1 if (mid & 0xFF) == CONSTANTS["LA_ELU1_NORM"] else dv
        S_final = torch.empty((B, H, dk, W), dtype=torch.float32, device=q.device)
    rc = la_chunk_fwd(q, k, v, g, beta, o, S0, S_final if with_state else None,
                      B, H, T, dk, dv, C, mid, _stream_handle(stream))
    if rc != 0:
        raise LAError(rc, la_last_error())
    return o, (S_final if with_state else None)


GATE_KINDS = {"none": CONSTANTS["LA_GATE_NONE"], "logsigmoid": CONSTANTS["LA_GATE_LOGSIGMOID"],
              "neg_softplus": CONSTANTS["LA_GATE_NEG_SOFTPLUS"]}


def prologue(xq, xk, xv, wq=None, wk=None, wv=None, K=None, hist_in=None, with_hist=False,
             l2q=False, l2k=False, a_gate=None, gate_kind="none", tau=1.0, a_beta=None, stream=None):
    """Short convolution, L2 normalisation and gate/beta activations (la_prologue).
    xq, xk [B,H,T,dk], xv [B,H,T,dv] bf16 CUDA tensors; w* [H,d,K] fp32 or None.
    Returns a dict with q, k, v, g (or None), beta (or None), hist (or None)."""
    import torch
    for name, t in (("xq", xq), ("xk", xk), ("xv", xv), ("wq", wq), ("wk", wk), ("wv", wv),
                    ("hist_in", hist_in), ("a_gate", a_gate), ("a_beta", a_beta)):
        _check(t, name)
    B, H, T, dk = xq.shape
    dv = xv.shape[-1]
    if K is None:
        K = next((w.shape[-1] for w in (wq, wk, wv) if w is not None), 1)
    kind = GATE_KINDS[gate_kind]
    dev = xq.device
    q = torch.empty_like(xq)
    k = torch.empty_like(xk)
    v = torch.empty_like(xv)
    g = torch.empty_like(a_gate) if kind != 0 else None
    beta = torch.empty_like(a_beta) if a_beta is not None else None
    hist_out = (torch.empty((B, H, K - 1, 2 * dk + dv), dtype=torch.bfloat16, device=dev)
                if with_hist and K > 1 else None)
    width = 1 if a_gate is None or a_gate.dim() == 3 else a_gate.shape[-1]
    flags = (CONSTANTS["LA_PRO_L2NORM_Q"] if l2q else 0) | (CONSTANTS["LA_PRO_L2NORM_K"] if l2k else 0)
    rc = la_prologue(xq, xk, xv, wq, wk, wv, K, hist_in, hist_out, a_gate if kind else None, kind,
                     width, tau, a_beta, q, k, v, g, beta, B, H, T, dk, dv, flags, _stream_handle(stream))
    if rc != 0:
        raise LAError(rc, la_last_error())
    return {"q": q, "k": k, "v": v, "g": g, "beta": beta, "hist": hist_out}


def chunk_fwd_gdelta(q, k, v, a, b, S0=None, C=0, with_state=True, o=None, S_final=None, stream=None):
    """Generalised delta rule S <- (I - b a^T) S + k v^T (la_chunk_fwd_gdelta).
    q, k, a, b [B,H,T,dk], v [B,H,T,dv] (bf16 or fp32, CUDA, contiguous).
    Returns (o, S_final or None)."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b), ("S0", S0)):
        _check(t, name)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    mode = CONSTANTS["LA_F32"] if q.dtype == torch.float32 else 0
    if o is None:
        o = torch.empty((B, H, T, dv), dtype=q.dtype, device=q.device)
    if with_state and S_final is None:
        S_final = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    rc = la_chunk_fwd_gdelta(q, k, v, a, b, o, S0, S_final if with_state else None,
                             B, H, T, dk, dv, C, mode, _stream_handle(stream))
    if rc != 0:
        raise LAError(rc, la_last_error())
    return o, (S_final if with_state else None)


def chunk_bwd(q, k, v, dO, mode, g=None, S0=None, dS_final=None, with_dS0=True, with_dg=True, C=0, stream=None):
    """Backward pass of chunk_fwd for "linear", "retnet", "scalar" and "gla":
    returns dq, dk, dv (dtype of q), dS0 (float32, or None) and dg (float32,
    [B,H,T] for "scalar", [B,H,T,dk] for "gla", with with_dg; else None)."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("dO", dO), ("g", g), ("S0", S0), ("dS_final", dS_final)):
        _check(t, name)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    mid = _mode_id(mode, q.dtype)
    dq, dk_, dv_ = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dS0 = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device) if with_dS0 else None
    kind = mid & 0xFF
    dg = None
    if with_dg and kind == CONSTANTS["LA_SCALAR_GATE"]:
        dg = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    elif with_dg and kind == CONSTANTS["LA_GLA"]:
        dg = torch.empty((B, H, T, dk), dtype=torch.float32, device=q.device)
    rc = la_chunk_bwd(q, k, v, g, dO, dS_final, S0, dq, dk_, dv_, dS0, dg, B, H, T, dk, dv, C, mid,
                      _stream_handle(stream))
    if rc != 0:
        raise LAError(rc, la_last_error())
    return dq, dk_, dv_, dS0, dg


def chunk_bwd_delta(q, k, v, dO, g=None, beta=None, S0=None, dS_final=None, with_dS0=True, with_dg=True,
                    with_dbeta=True, C=0, stream=None, mode="gdn"):
    """Delta-rule backward (la_chunk_bwd_delta), mode "gdn" (Gated DeltaNet) or
    "kda" (Kimi Delta Attention). q, k [B,H,T,dk], v, dO [B,H,T,dv] bf16 CUDA
    tensors; beta [B,H,T] fp32 or None; g [B,H,T] (gdn, or None) or
    [B,H,T,dk] (kda, required) fp32; S0, dS_final [B,H,dk,dv] fp32 or None.
    Returns dq, dk, dv, dbeta, dg, dS0 (None where not requested; dg None
    without g; dg has g's shape)."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("dO", dO), ("g", g), ("beta", beta), ("S0", S0),
                    ("dS_final", dS_final)):
        _check(t, name)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    mid = _mode_id(mode, q.dtype)
    dq, dk_, dv_ = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    f32 = dict(dtype=torch.float32, device=q.device)
    dbeta = torch.empty((B, H, T), **f32) if with_dbeta else None
    dg = torch.empty(tuple(g.shape), **f32) if (with_dg and g is not None) else None
    dS0 = torch.empty((B, H, dk, dv), **f32) if with_dS0 else None
    rc = la_chunk_bwd_delta(q, k, v, g, beta, dO, dS_final, S0, dq, dk_, dv_, dbeta, dg, dS0, B, H, T, dk, dv,
                            C, mid, _stream_handle(stream))
    if rc != 0:
        raise LAError(rc, la_last_error())
    return dq, dk_, dv_, dbeta, dg, dS0


def recurrent_step(q, k, v, S, mode, g=None, beta=None, o=None, stream=None):
    """One decode step. q, k [B,H,dk], v [B,H,dv]; S [B,H,dk,W] fp32 updated in place."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("S", S)):
        _check(t, name)
    B, H, dk = q.shape
    dv = v.shape[-1]
    mid = _mode_id(mode, q.dtype)
    if o is None:
        o = torch.empty((B, H, dv), dtype=q.dtype, device=q.device)
    rc = la_recurrent_step(q, k, v, g, beta, o, S, B, H, dk, dv, mid, _stream_handle(stream))
    if rc != 0:
        raise LAError(rc, la_last_error())
    return o
