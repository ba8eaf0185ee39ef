"""GPU parity of Kimi Delta Attention (LA_KDA: Gated DeltaNet with a
per-key-channel gate) against the float64 oracle, through the C ABI.

The chunk forward runs on the two-phase path by default (every chunk's key
side in parallel, then the state chain on bf16 warp MMAs) and on the fused
tensor-core kernel with LA_KDA=tc; the decode step on the step kernel. Same
tolerances as every other mode (tests/paritylib.py).
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
    wl = WORKLOADS["kda"].with_sizes(B=B, H=H, T=T, dk=dk, dv=dv, dtype=dtype, s0=s0)
    if seed is not None:
        wl = wl.with_sizes(seed=seed)
    return make(wl)


@pytest.mark.parametrize("dims", [(128, 128), (64, 64), (64, 128), (128, 64)])
def test_kda_small_parity(dims):
    dk, dv = dims
    inp = _inputs(dk=dk, dv=dv)
    o, S = run_cuda(inp)
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", "kda o")
    assert_close(f64(S), S_ref, "bf16", "kda S_final")


@pytest.mark.parametrize("T", [1, 17, 63, 64, 65, 129, 1000])
def test_kda_ragged_lengths(T):
    inp = _inputs(B=1, H=3, T=T)
    o, S = run_cuda(inp)
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", f"kda T={T} o")
    assert_close(f64(S), S_ref, "bf16", f"kda T={T} S")


def test_kda_without_beta_and_initial_state():
    inp = _inputs(B=1, H=2, T=150, s0=False)
    inp["beta"] = None
    o, S = run_cuda(inp, with_state=False)
    assert S is None
    o_ref, _ = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", "kda o (beta = 1, S0 = 0)")


@pytest.mark.parametrize("T1", [128, 100])
def test_kda_split_call_resumes_from_final_state(T1):
    T = 300
    inp = _inputs(B=1, H=2, T=T)
    d = to_dev(inp)
    sl = lambda x, a, b: x[:, :, a:b].contiguous()
    o1, S1 = la.chunk_fwd(sl(d["q"], 0, T1), sl(d["k"], 0, T1), sl(d["v"], 0, T1), "kda",
                          g=sl(d["g"], 0, T1), beta=sl(d["beta"], 0, T1), S0=d["S0"])
    o2, S2 = la.chunk_fwd(sl(d["q"], T1, T), sl(d["k"], T1, T), sl(d["v"], T1, T), "kda",
                          g=sl(d["g"], T1, T), beta=sl(d["beta"], T1, T), S0=S1)
    torch.cuda.synchronize()
    o_ref, S_ref = run_oracle(inp)
    assert_close(np.concatenate([f64(o1), f64(o2)], axis=2), o_ref, "bf16", "split o")
    assert_close(f64(S2), S_ref, "bf16", "split S")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_kda_decode_steps_match_oracle(dtype):
    T = 6
    inp = _inputs(dtype=dtype, B=2, H=3, T=T)
    d = to_dev(inp)
    S = inp["S0"].cuda().clone()
    outs = []
    for t in range(T):
        outs.append(la.recurrent_step(d["q"][:, :, t].contiguous(), d["k"][:, :, t].contiguous(),
                                      d["v"][:, :, t].contiguous(), S, "kda",
                                      g=d["g"][:, :, t].contiguous(), beta=d["beta"][:, :, t].contiguous()))
    torch.cuda.synchronize()
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(torch.stack(outs, dim=2)), o_ref, dtype, "kda decode o")
    assert_close(f64(S), S_ref, dtype, "kda decode S")


def test_kda_decode_loop_equals_chunk_forward():
    T = 70
    inp = _inputs(B=1, H=2, T=T)
    o_chunk, S_chunk = run_cuda(inp)
    d = to_dev(inp)
    S = inp["S0"].cuda().clone()
    outs = []
    for t in range(T):
        outs.append(la.recurrent_step(d["q"][:, :, t].contiguous(), d["k"][:, :, t].contiguous(),
                                      d["v"][:, :, t].contiguous(), S, "kda",
                                      g=d["g"][:, :, t].contiguous(), beta=d["beta"][:, :, t].contiguous()))
    torch.cuda.synchronize()
    assert_close(f64(torch.stack(outs, dim=2)), f64(o_chunk), "bf16", "decode vs chunk o")
    assert_close(f64(S), f64(S_chunk), "bf16", "decode vs chunk S")


def test_kda_full_size_workload_sampled_heads():
    inp = make("kda")
    wl = inp["wl"]
    o, S = run_cuda(inp, C=wl.C)
    B, H = wl.B, wl.H
    heads = [(0, 0), (B - 1, H - 1), (B // 2, H // 3)]
    o_ref, S_ref = run_oracle(inp, heads=heads, use_c=True)
    o_got = np.stack([f64(o[b, h]) for b, h in heads])[None]
    S_got = np.stack([f64(S[b, h]) for b, h in heads])[None]
    assert_close(o_got, o_ref, "bf16", "kda o (sampled heads)")
    assert_close(S_got, S_ref, "bf16", "kda S_final (sampled heads)")
    assert torch.isfinite(o.float()).all()


def test_kda_rejects_float32_and_the_materialised_variant(monkeypatch):
    inp = _inputs(dtype="f32", B=1, H=1, T=64)
    with pytest.raises(la.LAError) as e:
        run_cuda(inp)
    assert e.value.code == la.CONSTANTS["LA_ERR_UNSUPPORTED"]
    monkeypatch.setenv("LA_VARIANT", "mat")
    with pytest.raises(la.LAError) as e:
        run_cuda(_inputs(B=1, H=1, T=64))
    assert e.value.code == la.CONSTANTS["LA_ERR_UNSUPPORTED"]


@pytest.mark.parametrize("dims", [(128, 128), (64, 64)])
@pytest.mark.parametrize("T", [1, 65, 300])
def test_kda_fused_kernel_parity(dims, T, monkeypatch):
    # the default is the two-phase path; LA_KDA=tc keeps the fused sequential-phase kernel
    monkeypatch.setenv("LA_KDA", "tc")
    dk, dv = dims
    inp = _inputs(B=1, H=2, T=T, dk=dk, dv=dv, seed=41)
    o, S = run_cuda(inp)
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", f"kda fused T={T} o")
    assert_close(f64(S), S_ref, "bf16", f"kda fused T={T} S")


def test_kda_paths_agree(monkeypatch):
    inp = _inputs(B=2, H=3, T=777, dk=128, dv=64, seed=42)
    o_a, S_a = run_cuda(inp)
    monkeypatch.setenv("LA_KDA", "tc")
    o_b, S_b = run_cuda(inp)
    assert_close(f64(o_a), f64(o_b), "bf16", "two-phase vs fused o")
    assert_close(f64(S_a), f64(S_b), "bf16", "two-phase vs fused S_final")
