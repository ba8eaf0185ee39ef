"""Float64 CPU oracle for the chunkwise linear-attention forward pass.

TEST INFRASTRUCTURE ONLY. The product (the CUDA library and its Python
binding) never imports, links or runs anything in this package; only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg do. It shares no code with the CUDA path: the only common
dependency is the seeded input generator in ``workloads``.

Contents
  recurrence   numpy float64 token recurrence -- the definition (every mode)
  forms        the pages' other statements of the same computation, used as
               pins (parallel masked forms, normalised sums, the DeltaNet
               four-step update, a Kronecker brute force, the chunk form)
  recurrence_c the same recurrence in plain C (la_oracle.c), multi-threaded
               over heads, for full-length sequences and CPU timing
  prologue     short convolution, L2 normalisation, gate and beta activations
  noncausal    the non-causal form O = Q (K^T V) (linear, elu+1)
  gdelta       the generalised delta rule S <- (I - b a^T) S + k v^T
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .recurrence import MODES, phi_elu1, recurrence
from . import forms

__all__ = ["recurrence", "recurrence_c", "forms", "phi_elu1", "MODES", "build_c",
           "c_threads_default"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "la_oracle.c")
_LIB = os.path.join(_HERE, "liblaoracle.so")
_MODE_ID = {m: i for i, m in enumerate(MODES)}
_lib = None


def build_c(force: bool = False) -> str:
    """Compile la_oracle.c with the system C compiler (plain -O2, no
    machine-specific flags, so x86_64 and aarch64 builds agree)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_c())
        dp = ctypes.POINTER(ctypes.c_double)
        lib.la_oracle_fwd.argtypes = [dp] * 8 + [ctypes.c_int] * 7
        lib.la_oracle_fwd.restype = ctypes.c_int
        lib.la_oracle_threads_default.restype = ctypes.c_int
        _lib = lib
    return _lib


def c_threads_default() -> int:
    return int(_load().la_oracle_threads_default())


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def recurrence_c(q, k, v, mode, g=None, beta=None, S0=None, nthreads: int = 0):
    """Same contract as ``recurrence`` (shapes, modes, gate meaning), computed
    by the C implementation with ``nthreads`` threads (0 = all cores)."""
    lib = _load()
    as64 = lambda x: None if x is None else np.ascontiguousarray(x, dtype=np.float64)
    q, k, v, g, beta, S0 = map(as64, (q, k, v, g, beta, S0))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    W = dv + 1 if mode == "elu1" else dv
    o = np.zeros((B, H, T, dv))
    S = np.zeros((B, H, dk, W))
    rc = lib.la_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0),
                           _ptr(o), _ptr(S), B, H, T, dk, dv, _MODE_ID[mode], int(nthreads))
    if rc != 0:
        raise RuntimeError(f"la_oracle_fwd failed with {rc}")
    return o, S
