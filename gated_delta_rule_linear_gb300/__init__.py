"""Chunkwise linear-attention forward for NVIDIA GB300 (sm_103a).

The compute lives in libla.so (C ABI, include/la.h): hand-written CUDA
kernels for the chunkwise causal forward pass of the gated delta-rule family
(plain linear attention, elu+1 normalised attention, RetNet decay, GLA gates,
scalar decay, Gated DeltaNet, Kimi Delta Attention, the outer-product gate;
the generalised delta rule), its one-token decode
step, the backward pass (linear, RetNet, scalar decay, GLA, Gated DeltaNet),
and the prologue in front of it (short convolution, L2 normalisation,
gate activations). This package is
only the binding: ctypes marshalling plus a build helper.
"""
from ._binding import (CONSTANTS, GATE_KINDS, LIB_PATH, MODE_IDS, SIGNATURES, LAError, chunk_bwd,
                       chunk_bwd_delta, chunk_fwd, chunk_fwd_gdelta, la_chunk_bwd, la_chunk_bwd_delta, la_chunk_fwd, la_chunk_fwd_gdelta, la_chunk_fwd_noalloc,
                       la_last_error, la_prologue,
                       la_recurrent_step, la_stream_status, la_version, load_library, prologue, recurrent_step)
from ._binding import *  # noqa: F401,F403  (LA_* constants)

__all__ = ["chunk_fwd", "chunk_bwd", "chunk_bwd_delta", "chunk_fwd_gdelta", "recurrent_step", "prologue",
           "la_chunk_fwd", "la_chunk_bwd", "la_chunk_bwd_delta", "la_chunk_fwd_gdelta", "la_chunk_fwd_noalloc",
           "la_prologue", "la_recurrent_step", "GATE_KINDS",
           "la_stream_status", "la_last_error", "la_version", "load_library", "LAError",
           "CONSTANTS", "MODE_IDS", "SIGNATURES", "LIB_PATH"]
