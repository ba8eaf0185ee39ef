"""Seeded synthetic inputs for the chunkwise linear-attention forward pass.

This module is shared by the float64 oracle's tests and by the CUDA path's
tests and benchmark. It holds only input recipes -- shapes, dtypes, value
distributions and draw order -- and none of the method's arithmetic.

Five workloads stand in for the long-sequence training forward the pages on
linear attention describe ("Talk Linear Attention", sections 3-6; "Linear
Attention" glossary, applications list). No public dataset is involved:
every tensor is drawn from one CPU ``torch.Generator`` seeded per workload,
in the fixed order q, k, v, g, beta, S0, in float32, and then cast to the
workload's input dtype. Consumers must use the cast values (the oracle
upcasts them exactly to float64).

Gate convention: ``g`` holds natural-log gates, so the decay factor applied
to the state is ``alpha = exp(g)``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch
import torch.nn.functional as F

__all__ = ["Workload", "WORKLOADS", "make_inputs", "MODES", "PrologueWorkload", "PROLOGUE_WORKLOADS",
           "make_prologue_inputs"]

# Mode names used throughout the Python side. The C ABI has its own enum;
# the binding maps these names onto it.
MODES = ("linear", "elu1", "retnet", "gla", "scalar", "gdn", "kda", "outer", "gdelta")


@dataclass(frozen=True)
class Workload:
    name: str
    mode: str
    B: int
    H: int
    T: int
    dk: int
    dv: int
    dtype: str            # "bf16" or "f32": dtype of q, k, v and o
    C: int                # chunk length the workload is specified with
    seed: int
    qkv_scale: float = 1.0
    l2norm_qk: bool = False
    s0: bool = False      # random initial state
    extra: dict = field(default_factory=dict)

    def with_sizes(self, **kw) -> "Workload":
        return replace(self, **kw)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


WORKLOADS = {
    # Plain causal linear attention, fp32 inputs.
    "linear_fp32": Workload("linear_fp32", "linear", 1, 1, 256, 64, 64, "f32", 64,
                            seed=1, qkv_scale=1.0 / 8.0),
    # elu(x)+1 kernelised attention with the causal normaliser.
    "elu1": Workload("elu1", "elu1", 4, 8, 2048, 64, 64, "bf16", 64, seed=2),
    # RetNet fixed per-head decay gamma_h = 1 - 2^(-5-h).
    "retnet": Workload("retnet", "retnet", 8, 16, 4096, 128, 128, "bf16", 64, seed=3,
                       qkv_scale=1.0 / math.sqrt(128.0)),
    # GLA per-key-channel data-dependent gate, log alpha = logsigmoid(N(0,1))/16.
    "gla": Workload("gla", "gla", 8, 16, 8192, 128, 128, "bf16", 64, seed=4,
                    qkv_scale=1.0 / math.sqrt(128.0)),
    # Gated DeltaNet: L2-normalised q,k; beta = sigmoid(N); alpha = exp(-softplus(N)/8).
    "gdn": Workload("gdn", "gdn", 4, 16, 16384, 128, 128, "bf16", 64, seed=5,
                    l2norm_qk=True, s0=True),
    # Data-dependent scalar decay (the Mamba-2 style update, unit write).
    # Not one of the five headline workloads; used by parity tests only.
    "scalar": Workload("scalar", "scalar", 2, 4, 1024, 128, 128, "bf16", 64, seed=6,
                       qkv_scale=1.0 / math.sqrt(128.0), s0=True),
    # Kimi Delta Attention (Gated DeltaNet with a per-key-channel gate): the Gated
    # DeltaNet shape and q/k/beta recipe with the GLA gate distribution per channel.
    # The next row after the headline workloads; parity tests and its own bench line.
    "kda": Workload("kda", "kda", 4, 16, 16384, 128, 128, "bf16", 64, seed=7,
                    l2norm_qk=True, s0=True),
    # Non-causal linear attention O = Q (K^T V) (a next row): the RetNet shape
    # and q/k/v distribution, no gates.
    "noncausal": Workload("noncausal", "linear", 8, 16, 4096, 128, 128, "bf16", 64, seed=8,
                          qkv_scale=1.0 / math.sqrt(128.0), extra={"noncausal": True}),
    # Backward pass of the RetNet workload (a next row): q, k, v as retnet; the
    # output gradient dO ~ N(0,1)/sqrt(128) and dS_final ~ N(0, 0.01), drawn
    # after S0 by bench.py's backward leg from the same generator recipe.
    "backward": Workload("backward", "retnet", 8, 16, 4096, 128, 128, "bf16", 64, seed=9,
                         qkv_scale=1.0 / math.sqrt(128.0), extra={"backward": True}),
    # Backward of the data-dependent scalar decay, with the log-gate gradient dg:
    # the retnet shape and q/k/v recipe, g = -softplus(N(0,1))/8 per token, dO and
    # dS_final as for the backward workload.
    "backward_scalar": Workload("backward_scalar", "scalar", 8, 16, 4096, 128, 128, "bf16", 64, seed=13,
                                qkv_scale=1.0 / math.sqrt(128.0), extra={"backward": True}),
    # Backward of GLA with the per-channel log-gate gradient: the retnet shape, the
    # gla q/k/v and gate recipe, dO and dS_final as for the backward workload.
    "backward_gla": Workload("backward_gla", "gla", 8, 16, 4096, 128, 128, "bf16", 64, seed=14,
                             qkv_scale=1.0 / math.sqrt(128.0), extra={"backward": True}),
    # Backward of Gated DeltaNet (dq, dk, dv, dbeta, dg, dS0): the gdn shape and
    # q/k/v/gate/beta recipe, dO and dS_final as for the backward workload.
    "backward_gdn": Workload("backward_gdn", "gdn", 4, 16, 16384, 128, 128, "bf16", 64, seed=15,
                             l2norm_qk=True, s0=True, extra={"backward": True}),
    # Backward of Kimi Delta Attention (dq, dk, dv, dbeta, the per-channel dg, dS0):
    # the kda shape and q/k/gate/beta recipe, dO and dS_final as for the backward workload.
    "backward_kda": Workload("backward_kda", "kda", 4, 16, 16384, 128, 128, "bf16", 64, seed=16,
                             l2norm_qk=True, s0=True, extra={"backward": True}),
    # Outer-product gate alpha_t beta_t^T (a next row): the GLA shape and q/k/v
    # recipe with GLA-distributed log-gates on both the key and the value axis.
    "outer": Workload("outer", "outer", 8, 16, 8192, 128, 128, "bf16", 64, seed=11,
                      qkv_scale=1.0 / math.sqrt(128.0)),
    # Generalised delta rule S <- (I - b a^T) S + k v^T (a next row): q, k
    # L2-normalised, v ~ N(0, 1/4), a = sqrt(beta) k and b = sqrt(beta) times a
    # unit vector near k (so a != b and a.b = beta cos < 1), beta = sigmoid(N(0,1)).
    "gdelta": Workload("gdelta", "gdelta", 4, 8, 2048, 64, 64, "bf16", 64, seed=12,
                       qkv_scale=0.5, l2norm_qk=True, s0=True),
    # One Gated DeltaNet decode step (la_recurrent_step) for a batch of 128
    # sequences x 16 heads with resident states: the gdn recipe with T = 1
    # and a random state S ~ N(0, 0.01).
    "decode": Workload("decode", "gdn", 128, 16, 1, 128, 128, "bf16", 64, seed=10,
                       l2norm_qk=True, s0=True, extra={"decode": True}),
}


def _normal(gen, shape, scale=1.0):
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x


def make_inputs(wl: Workload | str, **sizes) -> dict:
    """Draw one workload's inputs on the CPU.

    Returns a dict with q, k, v (workload dtype, [B,H,T,d] contiguous),
    g (float32 or None), beta (float32 or None), S0 (float32 or None), plus
    the workload itself under "wl". ``sizes`` overrides B, H, T, dk, dv
    (and optionally seed) while keeping the value distributions.
    """
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    if sizes:
        wl = wl.with_sizes(**sizes)
    B, H, T, dk, dv = wl.B, wl.H, wl.T, wl.dk, wl.dv
    gen = torch.Generator(device="cpu")
    gen.manual_seed(wl.seed)

    q = _normal(gen, (B, H, T, dk), wl.qkv_scale)
    k = _normal(gen, (B, H, T, dk), wl.qkv_scale)
    v = _normal(gen, (B, H, T, dv), wl.qkv_scale)
    if wl.l2norm_qk:
        q = q / q.norm(dim=-1, keepdim=True).clamp_min(1e-6)
        k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-6)

    g = None
    beta = None
    if wl.mode == "retnet":
        # gamma_h = 1 - 2^(-5-h), h = 0..H-1; stored as float32 log gamma_h.
        g = torch.tensor([math.log1p(-(2.0 ** (-5 - h))) for h in range(H)],
                         dtype=torch.float64).to(torch.float32)
    elif wl.mode == "gla":
        g = F.logsigmoid(_normal(gen, (B, H, T, dk))) / 16.0
    elif wl.mode == "scalar":
        g = -F.softplus(_normal(gen, (B, H, T))) / 8.0
    elif wl.mode == "gdn":
        g = -F.softplus(_normal(gen, (B, H, T))) / 8.0
        beta = torch.sigmoid(_normal(gen, (B, H, T)))
        # draw order is q,k,v,g,beta,S0: g above is drawn before beta
    elif wl.mode == "kda":
        g = F.logsigmoid(_normal(gen, (B, H, T, dk))) / 16.0
        beta = torch.sigmoid(_normal(gen, (B, H, T)))
    elif wl.mode == "gdelta":
        pass  # its own inputs a and b are drawn below, after S0
    elif wl.mode == "outer":
        # key-axis and value-axis log-gates, both with the GLA gate's distribution;
        # the value-axis gates travel in the beta slot
        g = F.logsigmoid(_normal(gen, (B, H, T, dk))) / 16.0
        beta = F.logsigmoid(_normal(gen, (B, H, T, dv))) / 16.0
    S0 = None
    if wl.s0:
        width = dv + 1 if wl.mode == "elu1" else dv
        S0 = _normal(gen, (B, H, dk, width), 0.1)  # N(0, 0.01): variance 0.01

    dt = wl.torch_dtype
    a = b = None
    if wl.mode == "gdelta":  # drawn after S0: sqrt(beta) k and sqrt(beta) (a unit vector near k)
        wb = torch.sigmoid(_normal(gen, (B, H, T)))
        e = _normal(gen, (B, H, T, dk), 1.0 / math.sqrt(dk))
        root = wb.sqrt()[..., None]
        a = (root * k).to(dt).contiguous()
        b = (root * F.normalize(k + 0.5 * e, dim=-1)).to(dt).contiguous()
    return {
        "wl": wl,
        "q": q.to(dt).contiguous(),
        "k": k.to(dt).contiguous(),
        "v": v.to(dt).contiguous(),
        "g": None if g is None else g.contiguous(),
        "beta": None if beta is None else beta.contiguous(),
        "S0": None if S0 is None else S0.contiguous(),
        "a": a,
        "b": b,
    }



# ---------------------------------------------------------------- prologue

@dataclass(frozen=True)
class PrologueWorkload:
    """Inputs of the prologue in front of the chunk forward pass: the raw
    q/k/v projections, depthwise convolution weights, and the gate and beta
    pre-activations (drawn here; the activations themselves are the method's)."""
    name: str
    B: int
    H: int
    T: int
    dk: int
    dv: int
    K: int                 # convolution length
    gate_kind: str         # "none", "logsigmoid" or "neg_softplus"
    gate_width: int        # 1 (scalar) or dk (per key channel)
    tau: float
    l2q: bool
    l2k: bool
    beta: bool
    seed: int

    def with_sizes(self, **kw) -> "PrologueWorkload":
        return replace(self, **kw)


PROLOGUE_WORKLOADS = {
    # The Gated DeltaNet shape: K = 4 convolution on q, k and v, L2-normalised
    # q and k, alpha = exp(-softplus(a)/8), beta = sigmoid(a_beta).
    "prologue": PrologueWorkload("prologue", 4, 16, 16384, 128, 128, 4, "neg_softplus", 1, 8.0,
                                 True, True, True, seed=11),
    # The GLA/KDA gate form: per-channel logsigmoid(a)/16, no beta.
    "prologue_gla": PrologueWorkload("prologue_gla", 2, 8, 4096, 128, 128, 4, "logsigmoid", 128, 16.0,
                                     False, False, False, seed=12),
}


def make_prologue_inputs(wl: PrologueWorkload | str, hist: bool = False, **sizes) -> dict:
    """Draw one prologue workload's inputs on the CPU, in the order xq, xk, xv,
    wq, wk, wv, a_gate, a_beta, history: projections N(0, 1) cast to bf16,
    weights N(0, 1/K) float32 [H, d, K], pre-activations N(0, 1) float32, and
    (hist=True) a random bf16 history [B, H, K-1, 2 dk + dv]."""
    if isinstance(wl, str):
        wl = PROLOGUE_WORKLOADS[wl]
    if sizes:
        wl = wl.with_sizes(**sizes)
    B, H, T, dk, dv, K = wl.B, wl.H, wl.T, wl.dk, wl.dv, wl.K
    gen = torch.Generator(device="cpu")
    gen.manual_seed(wl.seed)
    xq = _normal(gen, (B, H, T, dk)).to(torch.bfloat16).contiguous()
    xk = _normal(gen, (B, H, T, dk)).to(torch.bfloat16).contiguous()
    xv = _normal(gen, (B, H, T, dv)).to(torch.bfloat16).contiguous()
    ws = 1.0 / math.sqrt(K)
    wq = _normal(gen, (H, dk, K), ws).contiguous()
    wk = _normal(gen, (H, dk, K), ws).contiguous()
    wv = _normal(gen, (H, dv, K), ws).contiguous()
    a_gate = None
    if wl.gate_kind != "none":
        shape = (B, H, T) if wl.gate_width == 1 else (B, H, T, wl.gate_width)
        a_gate = _normal(gen, shape).contiguous()
    a_beta = _normal(gen, (B, H, T)).contiguous() if wl.beta else None
    h = None
    if hist and K > 1:
        h = _normal(gen, (B, H, K - 1, 2 * dk + dv)).to(torch.bfloat16).contiguous()
    return {"wl": wl, "xq": xq, "xk": xk, "xv": xv, "wq": wq, "wk": wk, "wv": wv,
            "a_gate": a_gate, "a_beta": a_beta, "hist": h}
