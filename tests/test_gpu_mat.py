"""GPU parity of the materialised (two-phase) variant against the float64 oracle.

The variant writes every chunk's incoming state to a workspace in a state
pass (serial per head; for linear and elu+1 attention every chunk's K^T V at
once and a prefix scan, unless LA_MAT_STATE=serial) and then computes all
chunks' outputs in parallel; it covers the unit-write modes (everything but
the delta rule). It is selected with
LA_VARIANT=mat and must agree with the oracle to the same tolerance as the
fused kernel, and with the fused kernel itself.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_linear_gb300 as la
from paritylib import assert_close, f64, make, run_cuda, run_oracle, to_dev
from test_gpu_parity import _inputs

pytestmark = pytest.mark.gpu

UNIT_WRITE = ["linear", "elu1", "retnet", "gla", "scalar"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_linear_gb300 import build
    build.build()
    la.load_library()
    assert torch.cuda.is_available()


@pytest.fixture
def mat(monkeypatch):
    monkeypatch.setenv("LA_VARIANT", "mat")


@pytest.mark.parametrize("mode", UNIT_WRITE)
@pytest.mark.parametrize("dims", [(128, 128), (64, 64), (64, 128), (128, 64)])
def test_mat_small_parity(mode, dims, mat):
    dk, dv = dims
    inp = _inputs(mode, "bf16", dk=dk, dv=dv)
    o, S = run_cuda(inp)
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", f"{mode} o")
    assert_close(f64(S), S_ref, "bf16", f"{mode} S_final")


@pytest.mark.parametrize("mode", UNIT_WRITE)
@pytest.mark.parametrize("T", [1, 17, 63, 64, 65, 129, 1000])
def test_mat_ragged_lengths(mode, T, mat):
    inp = _inputs(mode, "bf16", B=1, H=3, T=T)
    o, S = run_cuda(inp)
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", f"{mode} T={T} o")
    assert_close(f64(S), S_ref, "bf16", f"{mode} T={T} S")


@pytest.mark.parametrize("mode", UNIT_WRITE)
def test_mat_zero_initial_state_and_no_state_output(mode, mat):
    inp = _inputs(mode, "bf16", B=1, H=2, T=150, s0=False)
    o, S = run_cuda(inp, with_state=False)
    assert S is None
    o_ref, _ = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", f"{mode} o")


@pytest.mark.parametrize("mode", ["gla", "elu1", "retnet"])
def test_mat_split_call_resumes_from_final_state(mode, mat):
    T, T1 = 300, 100
    inp = _inputs(mode, "bf16", B=1, H=2, T=T)
    d = to_dev(inp)

    def sl(x, a, b):
        if x is None or (mode == "retnet" and x is d["g"]):
            return x
        return x[:, :, a:b].contiguous()

    o1, S1 = la.chunk_fwd(sl(d["q"], 0, T1), sl(d["k"], 0, T1), sl(d["v"], 0, T1), mode,
                          g=sl(d["g"], 0, T1), S0=d["S0"])
    o2, S2 = la.chunk_fwd(sl(d["q"], T1, T), sl(d["k"], T1, T), sl(d["v"], T1, T), mode,
                          g=sl(d["g"], T1, T), S0=S1)
    torch.cuda.synchronize()
    o_ref, S_ref = run_oracle(inp)
    assert_close(np.concatenate([f64(o1), f64(o2)], axis=2), o_ref, "bf16", "split o")
    assert_close(f64(S2), S_ref, "bf16", "split S")


@pytest.mark.parametrize("mode", ["retnet", "gla"])
def test_mat_agrees_with_fused_kernel(mode, monkeypatch):
    inp = _inputs(mode, "bf16", B=2, H=3, T=700)
    monkeypatch.setenv("LA_VARIANT", "tc")
    o_a, S_a = run_cuda(inp)
    monkeypatch.setenv("LA_VARIANT", "mat")
    o_b, S_b = run_cuda(inp)
    assert_close(f64(o_b), f64(o_a), "bf16", "mat vs fused o")
    assert_close(f64(S_b), f64(S_a), "bf16", "mat vs fused S")


def test_mat_delta_rule_runs_the_two_phase_path(mat):
    # LA_VARIANT=mat on the delta rule selects its two-phase path (dk = dv = 128 only)
    inp = _inputs("gdn", "bf16", B=1, H=2, T=200)
    o, S = run_cuda(inp)
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", "gdn two-phase o")
    assert_close(f64(S), S_ref, "bf16", "gdn two-phase S_final")
    inp = _inputs("gdn", "bf16", B=1, H=1, T=64, dk=64, dv=64)
    with pytest.raises(la.LAError) as e:
        run_cuda(inp)
    assert e.value.code == la.CONSTANTS["LA_ERR_UNSUPPORTED"]
    assert "two-phase" in str(e.value)


@pytest.mark.parametrize("name", ["elu1", "retnet", "gla"])
def test_mat_full_size_workload_sampled_heads(name, mat):
    inp = make(name)
    wl = inp["wl"]
    o, S = run_cuda(inp, C=wl.C)
    B, H = wl.B, wl.H
    heads = [(0, 0), (B - 1, H - 1), (B // 2, H // 3)]
    o_ref, S_ref = run_oracle(inp, heads=heads, use_c=True)
    o_got = np.stack([f64(o[b, h]) for b, h in heads])[None]
    S_got = np.stack([f64(S[b, h]) for b, h in heads])[None]
    assert_close(o_got, o_ref, wl.dtype, f"{name} o (sampled heads)")
    assert_close(S_got, S_ref, wl.dtype, f"{name} S_final (sampled heads)")
    assert torch.isfinite(o.float()).all()


# ------------------------------------------------------------ C = 128
# The 128-token chunk: the state pass writes one image per 128 tokens and the
# output pass computes 128-token chunks (modes without per-channel gates).
C128 = ["linear", "elu1", "retnet", "scalar"]


@pytest.mark.parametrize("mode", C128)
@pytest.mark.parametrize("dims", [(128, 128), (64, 64), (64, 128), (128, 64)])
def test_c128_small_parity(mode, dims):
    dk, dv = dims
    inp = _inputs(mode, "bf16", dk=dk, dv=dv)
    o, S = run_cuda(inp, C=128)
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", f"{mode} C=128 o")
    assert_close(f64(S), S_ref, "bf16", f"{mode} C=128 S_final")


@pytest.mark.parametrize("mode", C128)
@pytest.mark.parametrize("T", [1, 17, 127, 128, 129, 255, 256, 257, 1000])
def test_c128_ragged_lengths(mode, T):
    inp = _inputs(mode, "bf16", B=1, H=3, T=T)
    o, S = run_cuda(inp, C=128)
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", f"{mode} C=128 T={T} o")
    assert_close(f64(S), S_ref, "bf16", f"{mode} C=128 T={T} S")


@pytest.mark.parametrize("mode", C128)
def test_c128_zero_initial_state_and_no_state_output(mode):
    inp = _inputs(mode, "bf16", B=1, H=2, T=300, s0=False)
    o, S = run_cuda(inp, C=128, with_state=False)
    assert S is None
    o_ref, _ = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", f"{mode} C=128 o")


@pytest.mark.parametrize("mode", C128)
def test_c128_agrees_with_c64(mode, mat):
    inp = _inputs(mode, "bf16", B=2, H=3, T=700)
    o_a, S_a = run_cuda(inp, C=64)
    o_b, S_b = run_cuda(inp, C=128)
    assert_close(f64(o_b), f64(o_a), "bf16", "C=128 vs C=64 o")
    # the state pass is the same serial scan at either C: identical final states
    assert torch.equal(S_a, S_b)


def test_c128_split_call_resumes_from_final_state():
    T, T1 = 600, 200
    inp = _inputs("scalar", "bf16", B=1, H=2, T=T)
    d = to_dev(inp)
    sl = lambda x, a, b: x[:, :, a:b].contiguous()
    o1, S1 = la.chunk_fwd(sl(d["q"], 0, T1), sl(d["k"], 0, T1), sl(d["v"], 0, T1), "scalar",
                          g=sl(d["g"], 0, T1), S0=d["S0"], C=128)
    o2, S2 = la.chunk_fwd(sl(d["q"], T1, T), sl(d["k"], T1, T), sl(d["v"], T1, T), "scalar",
                          g=sl(d["g"], T1, T), S0=S1, C=128)
    torch.cuda.synchronize()
    o_ref, S_ref = run_oracle(inp)
    assert_close(np.concatenate([f64(o1), f64(o2)], axis=2), o_ref, "bf16", "split o")
    assert_close(f64(S2), S_ref, "bf16", "split S")


@pytest.mark.parametrize("forced", ["tc", "simt"])
def test_c128_rejects_a_forced_non_materialised_variant(forced, monkeypatch):
    monkeypatch.setenv("LA_VARIANT", forced)
    inp = _inputs("retnet", "bf16", B=1, H=1, T=256)
    with pytest.raises(la.LAError) as e:
        run_cuda(inp, C=128)
    assert e.value.code == la.CONSTANTS["LA_ERR_UNSUPPORTED"]


@pytest.mark.parametrize("name", ["elu1", "retnet"])
def test_c128_full_size_workload_sampled_heads(name):
    inp = make(name)
    wl = inp["wl"]
    o, S = run_cuda(inp, C=128)
    B, H = wl.B, wl.H
    heads = [(0, 0), (B - 1, H - 1), (B // 2, H // 3)]
    o_ref, S_ref = run_oracle(inp, heads=heads, use_c=True)
    o_got = np.stack([f64(o[b, h]) for b, h in heads])[None]
    S_got = np.stack([f64(S[b, h]) for b, h in heads])[None]
    assert_close(o_got, o_ref, wl.dtype, f"{name} C=128 o (sampled heads)")
    assert_close(S_got, S_ref, wl.dtype, f"{name} C=128 S_final (sampled heads)")
    assert torch.isfinite(o.float()).all()


@pytest.mark.parametrize("mode", ["linear", "elu1"])
@pytest.mark.parametrize("C", [64, 128])
@pytest.mark.parametrize("dims", [(128, 128), (64, 64)])
def test_parallel_state_pass_matches_oracle_and_serial_pass(mode, C, dims, mat, monkeypatch):
    # linear and elu+1: the parallel state pass (every chunk's partial, then a prefix
    # scan into the images) against the oracle and the serial walk; S0 given, a tail
    # chunk, several images per head
    dk, dv = dims
    inp = _inputs(mode, "bf16", B=2, H=3, T=777, dk=dk, dv=dv)
    o, S = run_cuda(inp, C=C)
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", f"{mode} C={C} parallel o")
    assert_close(f64(S), S_ref, "bf16", f"{mode} C={C} parallel S_final")
    monkeypatch.setenv("LA_MAT_STATE", "serial")
    o_s, S_s = run_cuda(inp, C=C)
    assert_close(f64(o), f64(o_s), "bf16", f"{mode} C={C} parallel vs serial o")
    assert_close(f64(S), f64(S_s), "bf16", f"{mode} C={C} parallel vs serial S_final")
