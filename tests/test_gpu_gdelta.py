"""GPU parity of the generalised delta rule (la_chunk_fwd_gdelta:
S_t = (I - b_t a_t^T) S_{t-1} + k_t v_t^T, key-major) against the float64
oracle (oracle/gdelta.py), through the C ABI, at the library's tolerance
(bf16: max-abs 2e-2 and relative Frobenius 5e-3; fp32: relative 1e-4)."""
import numpy as np
import pytest
import torch

import gated_delta_rule_linear_gb300 as la
from oracle.gdelta import recurrence_gdelta
from paritylib import assert_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_linear_gb300 import build
    build.build()
    la.load_library()
    assert torch.cuda.is_available()


def _inputs(dtype="bf16", B=2, H=2, T=200, dk=64, dv=64, s0=True, seed=None):
    from workloads import WORKLOADS, make_inputs
    wl = WORKLOADS["gdelta"].with_sizes(B=B, H=H, T=T, dk=dk, dv=dv, dtype=dtype, s0=s0)
    if seed is not None:
        wl = wl.with_sizes(seed=seed)
    return make_inputs(wl)


def _gpu(inp, with_state=True, S0="inp", S_final=None):
    cu = lambda t: None if t is None else t.cuda().contiguous()
    s0 = cu(inp["S0"]) if S0 == "inp" else S0
    o, S = la.chunk_fwd_gdelta(cu(inp["q"]), cu(inp["k"]), cu(inp["v"]), cu(inp["a"]), cu(inp["b"]),
                               S0=s0, with_state=with_state, S_final=S_final)
    torch.cuda.synchronize()
    return o, S


def _ref(inp, heads=None):
    sel = (lambda x: x) if heads is None else (lambda x: None if x is None else
                                               torch.stack([x[b, h] for b, h in heads])[None])
    return recurrence_gdelta(*(f64(sel(inp[n])) for n in ("q", "k", "v", "a", "b")),
                             S0=None if inp["S0"] is None else f64(sel(inp["S0"])))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dims", [(64, 64), (128, 128), (64, 128), (128, 64)])
def test_gdelta_small_parity(dtype, dims):
    dk, dv = dims
    inp = _inputs(dtype, dk=dk, dv=dv)
    o, S = _gpu(inp)
    o_ref, S_ref = _ref(inp)
    assert_close(f64(o), o_ref, dtype, "gdelta o")
    assert_close(f64(S), S_ref, dtype, "gdelta S_final")


@pytest.mark.parametrize("T", [1, 17, 63, 64, 65, 129, 700])
def test_gdelta_ragged_lengths(T):
    inp = _inputs(B=1, H=3, T=T)
    o, S = _gpu(inp)
    o_ref, S_ref = _ref(inp)
    assert_close(f64(o), o_ref, "bf16", f"gdelta T={T} o")
    assert_close(f64(S), S_ref, "bf16", f"gdelta T={T} S")


def test_gdelta_zero_state_and_no_state_output():
    inp = _inputs(B=1, H=2, T=150, s0=False)
    o, S = _gpu(inp, with_state=False)
    assert S is None
    o_ref, _ = _ref(inp)
    assert_close(f64(o), o_ref, "bf16", "gdelta o (S0 = 0)")


def test_gdelta_final_state_may_alias_initial_state():
    inp = _inputs(B=2, H=2, T=130)
    S = inp["S0"].cuda().clone()
    _gpu(inp, S0=S, S_final=S)
    _, S_ref = _ref(inp)
    assert_close(f64(S), S_ref, "bf16", "aliased S")


def test_gdelta_deltanet_case_matches_the_deltanet_oracle():
    """a = b = sqrt(beta) k with beta k as the write key is DeltaNet (the page's
    special case, pinned on the CPU against the gdn recurrence): the kernel on
    those inputs against the oracle."""
    inp = _inputs(B=1, H=2, T=300, dk=128, dv=128)
    k = inp["k"].float()
    beta = torch.sigmoid(torch.randn(k.shape[:3], generator=torch.Generator().manual_seed(5)))
    ab = (beta.sqrt()[..., None] * k).to(torch.bfloat16)
    kw = (beta[..., None] * k).to(torch.bfloat16)
    run = dict(inp, a=ab, b=ab, k=kw)
    o, S = _gpu(run)
    # the oracle sees the rounded inputs the kernel saw: a = b = sqrt(beta) k_bf16 rounded
    o_ref, S_ref = recurrence_gdelta(f64(inp["q"]), f64(kw), f64(inp["v"]), f64(ab), f64(ab), S0=f64(inp["S0"]))
    assert_close(f64(o), o_ref, "bf16", "DeltaNet case o")
    assert_close(f64(S), S_ref, "bf16", "DeltaNet case S")


def test_gdelta_split_call_resumes_from_final_state():
    T, T1 = 300, 100
    inp = _inputs(B=1, H=2, T=T)
    sl = lambda d, a, b: {n: (x[:, :, a:b].contiguous() if n in ("q", "k", "v", "a", "b") else x)
                          for n, x in d.items()}
    o1, S1 = _gpu(sl(inp, 0, T1))
    o2, S2 = _gpu(sl(inp, T1, T), S0=S1)
    o_ref, S_ref = _ref(inp)
    assert_close(np.concatenate([f64(o1), f64(o2)], axis=2), o_ref, "bf16", "split o")
    assert_close(f64(S2), S_ref, "bf16", "split S")


def test_gdelta_full_size_workload_sampled_heads():
    """The bench configuration (B=4 H=8 T=2048 d=64): sampled heads against the oracle."""
    from workloads import make_inputs
    inp = make_inputs("gdelta")
    wl = inp["wl"]
    o, S = _gpu(inp)
    heads = [(0, 0), (wl.B - 1, wl.H - 1), (wl.B // 2, wl.H // 3)]
    o_ref, S_ref = _ref(inp, heads)
    assert_close(np.stack([f64(o[b, h]) for b, h in heads])[None], o_ref, "bf16", "gdelta o (sampled)")
    assert_close(np.stack([f64(S[b, h]) for b, h in heads])[None], S_ref, "bf16", "gdelta S (sampled)")


@pytest.mark.parametrize("dims", [(64, 64), (128, 128)])
@pytest.mark.parametrize("T", [1, 65, 300])
def test_gdelta_bf16_cuda_core_path_parity(dims, T, monkeypatch):
    # bfloat16 runs the two-phase tensor-core path by default; LA_GDELTA=simt keeps the
    # one-pass CUDA-core kernel for it, which must meet the same tolerance
    monkeypatch.setenv("LA_GDELTA", "simt")
    dk, dv = dims
    inp = _inputs("bf16", B=1, H=2, T=T, dk=dk, dv=dv, seed=31)
    o, S = _gpu(inp)
    o_ref, S_ref = _ref(inp)
    assert_close(f64(o), o_ref, "bf16", "gdelta (CUDA cores) o")
    assert_close(f64(S), S_ref, "bf16", "gdelta (CUDA cores) S_final")


def test_gdelta_bf16_paths_agree(monkeypatch):
    inp = _inputs("bf16", B=2, H=3, T=777, dk=64, dv=128, seed=32)
    o_a, S_a = _gpu(inp)
    monkeypatch.setenv("LA_GDELTA", "simt")
    o_b, S_b = _gpu(inp)
    assert_close(f64(o_a), f64(o_b), "bf16", "two-phase vs CUDA-core o")
    assert_close(f64(S_a), f64(S_b), "bf16", "two-phase vs CUDA-core S_final")


@pytest.mark.parametrize("dims", [(64, 64), (128, 128)])
def test_gdelta_many_heads_single_buffered_chain(dims):
    # more chain CTAs (heads x 16-column blocks) than SMs selects the single-buffered
    # chain (two CTAs an SM); sampled heads against the oracle, ragged tail included
    dk, dv = dims
    B, H = 4, 160 * 16 // dv
    assert B * H * (dv // 16) > torch.cuda.get_device_properties(0).multi_processor_count
    inp = _inputs("bf16", B=B, H=H, T=321, dk=dk, dv=dv, seed=33)
    o, S = _gpu(inp)
    heads = [(0, 0), (B - 1, H - 1), (2, H // 2)]
    o_ref, S_ref = _ref(inp, heads)
    assert_close(np.stack([f64(o[b, h]) for b, h in heads])[None], o_ref, "bf16", "gdelta o (many heads)")
    assert_close(np.stack([f64(S[b, h]) for b, h in heads])[None], S_ref, "bf16", "gdelta S (many heads)")
