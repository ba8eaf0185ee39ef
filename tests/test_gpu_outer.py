"""GPU parity of the outer-product gate (LA_OUTER_GATE: S_t = (alpha_t
beta_t^T) ⊙ S_{t-1} + k_t v_t^T) against the float64 oracle, through the C
ABI. The chunk forward runs on the pipelined unit-write kernel with both
axes' gates folded around the chunk midpoint; the decode step on the step
kernel. Same tolerances as every other mode (tests/paritylib.py).
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_linear_gb300 as la
from paritylib import assert_close, f64, make, run_cuda, run_oracle, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_linear_gb300 import build
    build.build()
    la.load_library()
    assert torch.cuda.is_available()


def _inputs(dtype="bf16", B=2, H=2, T=200, dk=128, dv=128, s0=True, seed=None):
    from workloads import WORKLOADS
    wl = WORKLOADS["outer"].with_sizes(B=B, H=H, T=T, dk=dk, dv=dv, dtype=dtype, s0=s0)
    if seed is not None:
        wl = wl.with_sizes(seed=seed)
    return make(wl)


@pytest.mark.parametrize("dims", [(128, 128), (64, 64), (64, 128), (128, 64)])
def test_outer_small_parity(dims):
    dk, dv = dims
    inp = _inputs(dk=dk, dv=dv)
    o, S = run_cuda(inp)
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", "outer o")
    assert_close(f64(S), S_ref, "bf16", "outer S_final")


@pytest.mark.parametrize("T", [1, 17, 63, 64, 65, 129, 1000])
def test_outer_ragged_lengths(T):
    inp = _inputs(B=1, H=3, T=T)
    o, S = run_cuda(inp)
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", f"outer T={T} o")
    assert_close(f64(S), S_ref, "bf16", f"outer T={T} S")


def test_outer_without_initial_state_or_state_output():
    inp = _inputs(B=1, H=2, T=150, s0=False)
    o, S = run_cuda(inp, with_state=False)
    assert S is None
    o_ref, _ = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", "outer o (S0 = 0)")


def test_outer_strong_and_uneven_value_decay():
    """Value columns with very different decay rates (one ~e^-1 per token)."""
    inp = _inputs(B=1, H=2, T=300)
    inp["beta"][..., 5] = inp["beta"][..., 5] * 16.0
    inp["beta"][..., 77] = 0.0
    o, S = run_cuda(inp)
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", "outer o (uneven value decay)")
    assert_close(f64(S), S_ref, "bf16", "outer S (uneven value decay)")


def test_outer_with_unit_value_gate_matches_gla_kernel():
    """log beta = 0: the outer-product gate is GLA's key-axis gate; the two
    kernels' outputs agree to float32 rounding."""
    inp = _inputs(B=1, H=2, T=260)
    d = to_dev(inp)
    zero = torch.zeros_like(d["beta"])
    o1, S1 = la.chunk_fwd(d["q"], d["k"], d["v"], "outer", g=d["g"], beta=zero, S0=d["S0"])
    o2, S2 = la.chunk_fwd(d["q"], d["k"], d["v"], "gla", g=d["g"], S0=d["S0"])
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 2.0 ** -7 * o2.float().abs().max().item()
    assert torch.allclose(S1, S2, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("T1", [128, 100])
def test_outer_split_call_resumes_from_final_state(T1):
    T = 300
    inp = _inputs(B=1, H=2, T=T)
    d = to_dev(inp)
    sl = lambda x, a, b: x[:, :, a:b].contiguous()
    o1, S1 = la.chunk_fwd(sl(d["q"], 0, T1), sl(d["k"], 0, T1), sl(d["v"], 0, T1), "outer",
                          g=sl(d["g"], 0, T1), beta=sl(d["beta"], 0, T1), S0=d["S0"])
    o2, S2 = la.chunk_fwd(sl(d["q"], T1, T), sl(d["k"], T1, T), sl(d["v"], T1, T), "outer",
                          g=sl(d["g"], T1, T), beta=sl(d["beta"], T1, T), S0=S1)
    torch.cuda.synchronize()
    o_ref, S_ref = run_oracle(inp)
    assert_close(np.concatenate([f64(o1), f64(o2)], axis=2), o_ref, "bf16", "split o")
    assert_close(f64(S2), S_ref, "bf16", "split S")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_outer_decode_steps_match_oracle(dtype):
    T = 6
    inp = _inputs(dtype=dtype, B=2, H=3, T=T)
    d = to_dev(inp)
    S = inp["S0"].cuda().clone()
    outs = []
    for t in range(T):
        outs.append(la.recurrent_step(d["q"][:, :, t].contiguous(), d["k"][:, :, t].contiguous(),
                                      d["v"][:, :, t].contiguous(), S, "outer",
                                      g=d["g"][:, :, t].contiguous(), beta=d["beta"][:, :, t].contiguous()))
    torch.cuda.synchronize()
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(torch.stack(outs, dim=2)), o_ref, dtype, "outer decode o")
    assert_close(f64(S), S_ref, dtype, "outer decode S")


def test_outer_full_size_workload_sampled_heads():
    """The bench configuration (B=8 H=16 T=8192): sampled heads against the oracle."""
    inp = make("outer")
    wl = inp["wl"]
    o, S = run_cuda(inp, C=wl.C)
    B, H = wl.B, wl.H
    heads = [(0, 0), (B - 1, H - 1), (B // 2, H // 3)]
    o_ref, S_ref = run_oracle(inp, heads=heads, use_c=True)
    o_got = np.stack([f64(o[b, h]) for b, h in heads])[None]
    S_got = np.stack([f64(S[b, h]) for b, h in heads])[None]
    assert_close(o_got, o_ref, "bf16", "outer o (sampled heads)")
    assert_close(S_got, S_ref, "bf16", "outer S_final (sampled heads)")
    assert torch.isfinite(o.float()).all()


def test_outer_rejects_float32_missing_value_gates_and_other_variants(monkeypatch):
    with pytest.raises(la.LAError) as e:
        run_cuda(_inputs(dtype="f32", B=1, H=1, T=64))
    assert e.value.code == la.CONSTANTS["LA_ERR_UNSUPPORTED"]
    inp = _inputs(B=1, H=1, T=64)
    inp["beta"] = None
    with pytest.raises(la.LAError) as e:
        run_cuda(inp)
    assert e.value.code == la.CONSTANTS["LA_ERR_INVALID_ARG"]
    for variant in ("mat", "simt"):
        monkeypatch.setenv("LA_VARIANT", variant)
        with pytest.raises(la.LAError) as e:
            run_cuda(_inputs(B=1, H=1, T=64))
        assert e.value.code == la.CONSTANTS["LA_ERR_UNSUPPORTED"]
