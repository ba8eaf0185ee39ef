"""GPU parity of the non-causal form (LA_NONCAUSAL with LA_LINEAR and
LA_ELU1_NORM: split-T state reduction, finalize, parallel output pass) with
the float64 oracle, through the C ABI, at the library's bf16 tolerance on o
and on S_final."""
import numpy as np
import pytest
import torch

from oracle.noncausal import noncausal
from paritylib import assert_close, f64, make

pytestmark = pytest.mark.gpu

RECIPE = {"linear": "retnet", "elu1": "elu1"}  # q, k, v distributions (no gates are used)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import gated_delta_rule_linear_gb300 as la
    from gated_delta_rule_linear_gb300 import build
    build.build()
    la.load_library()
    assert torch.cuda.is_available()


def _inputs(mode, B, H, T, dk, dv, s0, seed=None):
    from workloads import WORKLOADS
    wl = WORKLOADS[RECIPE[mode]].with_sizes(B=B, H=H, T=T, dk=dk, dv=dv, dtype="bf16", s0=False)
    if seed is not None:
        wl = wl.with_sizes(seed=seed)
    inp = make(wl)
    if s0:
        g = torch.Generator().manual_seed(99)
        W = dv + 1 if mode == "elu1" else dv
        S0 = torch.randn(B, H, dk, W, generator=g) * 0.1
        if mode == "elu1":
            S0[..., dv] = S0[..., dv].abs() + 1.0
        inp["S0"] = S0
    else:
        inp["S0"] = None
    return inp


def _run(inp, mode):
    import gated_delta_rule_linear_gb300 as la
    dev = torch.device("cuda")
    mid = la.MODE_IDS[mode] | la.LA_NONCAUSAL
    S0 = None if inp["S0"] is None else inp["S0"].to(dev).contiguous()
    o, S = la.chunk_fwd(inp["q"].to(dev), inp["k"].to(dev), inp["v"].to(dev), mid, S0=S0)
    torch.cuda.synchronize()
    assert la.la_stream_status(torch.cuda.current_stream().cuda_stream) == 0
    return o, S


def _ref(inp, mode):
    return noncausal(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), mode,
                     S0=None if inp["S0"] is None else f64(inp["S0"]))


@pytest.mark.parametrize("mode", ["linear", "elu1"])
@pytest.mark.parametrize("dims", [(128, 128), (64, 64), (64, 128), (128, 64)])
@pytest.mark.parametrize("T", [1, 63, 64, 200, 777])
def test_noncausal_parity(mode, dims, T):
    dk, dv = dims
    inp = _inputs(mode, 2, 3, T, dk, dv, s0=(T % 2 == 1))
    o, S = _run(inp, mode)
    o_ref, S_ref = _ref(inp, mode)
    assert_close(f64(o), o_ref, "bf16", f"{mode} non-causal o")
    assert_close(f64(S), S_ref, "bf16", f"{mode} non-causal S_final")


@pytest.mark.parametrize("mode", ["linear", "elu1"])
def test_noncausal_long_sequence_many_splits(mode):
    """Few heads and a long sequence: the T-range is split over many CTAs."""
    inp = _inputs(mode, 1, 2, 16384 + 37, 128, 128, s0=True)
    o, S = _run(inp, mode)
    o_ref, S_ref = _ref(inp, mode)
    assert_close(f64(o), o_ref, "bf16", f"{mode} long o")
    assert_close(f64(S), S_ref, "bf16", f"{mode} long S_final")


def test_noncausal_bench_shape_sampled():
    """The bench configuration (B=8 H=16 T=4096): sampled heads against the oracle."""
    import gated_delta_rule_linear_gb300 as la
    from workloads import WORKLOADS
    wl = WORKLOADS["noncausal"]
    inp = make(wl)
    dev = torch.device("cuda")
    o, S = la.chunk_fwd(inp["q"].to(dev), inp["k"].to(dev), inp["v"].to(dev),
                        la.MODE_IDS[wl.mode] | la.LA_NONCAUSAL)
    rng = np.random.default_rng(3)
    for _ in range(3):
        b, h = int(rng.integers(wl.B)), int(rng.integers(wl.H))
        sl = lambda t: f64(t[b:b + 1, h:h + 1])
        o_ref, S_ref = noncausal(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), wl.mode)
        assert_close(f64(o[b:b + 1, h:h + 1]), o_ref, "bf16", f"head {b},{h} o")
        assert_close(f64(S[b:b + 1, h:h + 1]), S_ref, "bf16", f"head {b},{h} S")
