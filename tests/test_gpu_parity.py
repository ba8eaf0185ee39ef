"""GPU parity: the CUDA path against the float64 oracle, element by element.

Small shapes span several chunks and a ragged tail; the full-size workloads
run in the launch configuration the benchmark times and are compared on
sampled heads, which the oracle computes one at a time over the whole
sequence. All calls go through the C ABI (libla.so).
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_linear_gb300 as la
import oracle
from paritylib import assert_close, f64, make, run_cuda, run_oracle, to_dev

pytestmark = pytest.mark.gpu

MODES = ["linear", "elu1", "retnet", "gla", "scalar", "gdn"]
RECIPE = {"linear": "linear_fp32", "elu1": "elu1", "retnet": "retnet", "gla": "gla",
          "scalar": "scalar", "gdn": "gdn"}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_linear_gb300 import build
    build.build()
    la.load_library()
    assert torch.cuda.is_available()


def _inputs(mode, dtype, B=2, H=2, T=200, dk=128, dv=128, s0=True, seed=None):
    from workloads import WORKLOADS
    wl = WORKLOADS[RECIPE[mode]].with_sizes(B=B, H=H, T=T, dk=dk, dv=dv, dtype=dtype, s0=s0)
    if seed is not None:
        wl = wl.with_sizes(seed=seed)
    inp = make(wl)
    if mode == "elu1" and inp["S0"] is not None:
        inp["S0"][..., dv] = inp["S0"][..., dv].abs() + 1.0   # positive normaliser z0
    return inp


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("dtype,variant", [("bf16", "tc"), ("bf16", "simt"), ("f32", "simt")])
@pytest.mark.parametrize("dims", [(128, 128), (64, 64), (64, 128), (128, 64)])
def test_small_parity(mode, dtype, variant, dims, monkeypatch):
    monkeypatch.setenv("LA_VARIANT", variant)
    dk, dv = dims
    inp = _inputs(mode, dtype, dk=dk, dv=dv)
    o, S = run_cuda(inp)
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(o), o_ref, dtype, f"{mode} o")
    assert_close(f64(S), S_ref, dtype, f"{mode} S_final")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("T", [1, 17, 63, 64, 65, 128, 129])
def test_ragged_lengths(mode, T):
    inp = _inputs(mode, "bf16", B=1, H=3, T=T)
    o, S = run_cuda(inp)
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", f"{mode} T={T} o")
    assert_close(f64(S), S_ref, "bf16", f"{mode} T={T} S")


@pytest.mark.parametrize("mode", MODES)
def test_zero_initial_state_and_no_state_output(mode):
    inp = _inputs(mode, "bf16", B=1, H=2, T=150, s0=False)
    o, S = run_cuda(inp, with_state=False)
    assert S is None
    o_ref, _ = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", f"{mode} o")


@pytest.mark.parametrize("mode", ["gdn", "gla", "elu1", "retnet"])
@pytest.mark.parametrize("T1", [128, 100])
def test_split_call_resumes_from_final_state(mode, T1):
    T = 300
    inp = _inputs(mode, "bf16", B=1, H=2, T=T)
    d = to_dev(inp)
    o_full, S_full = la.chunk_fwd(d["q"], d["k"], d["v"], mode, g=d["g"], beta=d["beta"], S0=d["S0"])

    def sl(x, a, b):
        if x is None or (mode == "retnet" and x is d["g"]):
            return x
        return x[:, :, a:b].contiguous()

    o1, S1 = la.chunk_fwd(sl(d["q"], 0, T1), sl(d["k"], 0, T1), sl(d["v"], 0, T1), mode,
                          g=sl(d["g"], 0, T1), beta=sl(d["beta"], 0, T1), S0=d["S0"])
    o2, S2 = la.chunk_fwd(sl(d["q"], T1, T), sl(d["k"], T1, T), sl(d["v"], T1, T), mode,
                          g=sl(d["g"], T1, T), beta=sl(d["beta"], T1, T), S0=S1)
    torch.cuda.synchronize()
    o_ref, S_ref = run_oracle(inp)
    assert_close(np.concatenate([f64(o1), f64(o2)], axis=2), o_ref, "bf16", "split o")
    assert_close(f64(S2), S_ref, "bf16", "split S")
    assert_close(f64(o_full), o_ref, "bf16", "full o")


@pytest.mark.parametrize("mode", ["gdn", "linear"])
def test_final_state_may_alias_initial_state(mode):
    inp = _inputs(mode, "bf16", B=2, H=2, T=130)
    d = to_dev(inp)
    S = d["S0"].clone()
    la.chunk_fwd(d["q"], d["k"], d["v"], mode, g=d["g"], beta=d["beta"], S0=S, S_final=S)
    torch.cuda.synchronize()
    _, S_ref = run_oracle(inp)
    assert_close(f64(S), S_ref, "bf16", "aliased S")


def test_outputs_write_nothing_outside_their_extent():
    inp = _inputs("gdn", "bf16", B=1, H=2, T=77)
    d = to_dev(inp)
    B, H, T, dv = 1, 2, 77, 128
    pad = 1024
    n = B * H * T * dv
    buf = torch.full((n + 2 * pad,), float("nan"), dtype=torch.bfloat16, device="cuda")
    o = buf[pad:pad + n].view(B, H, T, dv)
    sbuf = torch.full((B * H * 128 * dv + 2 * pad,), float("nan"), device="cuda")
    S = sbuf[pad:pad + B * H * 128 * dv].view(B, H, 128, dv)
    la.chunk_fwd(d["q"], d["k"], d["v"], "gdn", g=d["g"], beta=d["beta"], S0=d["S0"], o=o,
                 S_final=S)
    torch.cuda.synchronize()
    assert torch.isnan(buf[:pad].float()).all() and torch.isnan(buf[pad + n:].float()).all()
    assert torch.isnan(sbuf[:pad]).all() and torch.isnan(sbuf[-pad:]).all()
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", "o")


def test_gdn_retrieval_on_gpu():
    # beta = 1, alpha = 1, S0 = 0, orthonormal keys: the state returns every value
    # exactly up to the kernel's bf16 rounding.
    dk = dv = 128
    rng = np.random.default_rng(7)
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = torch.tensor(Qm.T, dtype=torch.float32)
    vals = torch.randn(dk, dv, generator=torch.Generator().manual_seed(3))
    k = keys.to(torch.bfloat16)[None, None].cuda().contiguous()
    v = vals.to(torch.bfloat16)[None, None].cuda().contiguous()
    q = k.clone()
    o, S = la.chunk_fwd(q, k, v, "gdn")
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.recurrence(f64(q), f64(k), f64(v), "gdn")
    assert_close(f64(S), S_ref, "bf16", "S")
    assert_close(f64(o), o_ref, "bf16", "o")


# --- decode step ---------------------------------------------------------------

def _step_slices(inp, t):
    d = to_dev(inp)
    mode = inp["wl"].mode
    g = d["g"]
    if g is not None and mode != "retnet":
        g = g[:, :, t].contiguous()
    beta = None if d["beta"] is None else d["beta"][:, :, t].contiguous()
    return (d["q"][:, :, t].contiguous(), d["k"][:, :, t].contiguous(),
            d["v"][:, :, t].contiguous(), g, beta)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_steps_match_oracle(mode, dtype):
    T = 6
    inp = _inputs(mode, dtype, B=2, H=3, T=T)
    S = inp["S0"].cuda().clone()
    outs = []
    for t in range(T):
        q, k, v, g, beta = _step_slices(inp, t)
        outs.append(la.recurrent_step(q, k, v, S, mode, g=g, beta=beta))
    torch.cuda.synchronize()
    o = torch.stack(outs, dim=2)
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(o), o_ref, dtype, f"{mode} decode o")
    assert_close(f64(S), S_ref, dtype, f"{mode} decode S")


@pytest.mark.parametrize("mode", ["gdn", "gla", "elu1"])
def test_decode_loop_equals_chunk_forward(mode):
    T = 70
    inp = _inputs(mode, "bf16", B=1, H=2, T=T)
    o_chunk, S_chunk = run_cuda(inp)
    S = inp["S0"].cuda().clone()
    outs = []
    for t in range(T):
        q, k, v, g, beta = _step_slices(inp, t)
        outs.append(la.recurrent_step(q, k, v, S, mode, g=g, beta=beta))
    torch.cuda.synchronize()
    assert_close(f64(torch.stack(outs, dim=2)), f64(o_chunk), "bf16", "decode vs chunk o")
    assert_close(f64(S), f64(S_chunk), "bf16", "decode vs chunk S")


# --- full-size workloads, sampled heads ------------------------------------------

FULL = ["linear_fp32", "elu1", "retnet", "gla", "gdn"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload_sampled_heads(name):
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
    # every head: finite output
    assert torch.isfinite(o.float()).all()


# --- delta rule: one CTA per head, a CTA pair per head, or the two-phase path
# (the solve for every chunk first, then the state chain on a CTA pair) -------

@pytest.mark.parametrize("path", ["single", "pair", "wy"])
@pytest.mark.parametrize("T", [1, 64, 65, 200, 1000])
@pytest.mark.parametrize("gated", [True, False])
def test_delta_kernel_paths(path, T, gated, monkeypatch):
    monkeypatch.setenv("LA_DELTA", path)
    inp = _inputs("gdn", "bf16", B=2, H=3, T=T)
    if not gated:
        inp["g"] = None
    o, S = run_cuda(inp)
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", f"{path} T={T} o")
    assert_close(f64(S), S_ref, "bf16", f"{path} T={T} S")


@pytest.mark.parametrize("path", ["single", "pair", "wy"])
def test_delta_kernel_paths_aliased_state_and_split(path, monkeypatch):
    monkeypatch.setenv("LA_DELTA", path)
    inp = _inputs("gdn", "bf16", B=1, H=2, T=300)
    d = to_dev(inp)
    S = d["S0"].clone()
    o, _ = la.chunk_fwd(d["q"], d["k"], d["v"], "gdn", g=d["g"], beta=d["beta"], S0=S, S_final=S)
    torch.cuda.synchronize()
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", "aliased o")
    assert_close(f64(S), S_ref, "bf16", "aliased S")


def test_delta_pair_and_single_agree():
    inp = _inputs("gdn", "bf16", B=2, H=4, T=777)
    import os
    outs = []
    for path in ("single", "pair", "wy"):
        os.environ["LA_DELTA"] = path
        try:
            outs.append(run_cuda(inp))
        finally:
            del os.environ["LA_DELTA"]
    assert_close(f64(outs[1][0]), f64(outs[0][0]), "bf16", "pair vs single o")
    assert_close(f64(outs[1][1]), f64(outs[0][1]), "bf16", "pair vs single S")
    assert_close(f64(outs[2][0]), f64(outs[0][0]), "bf16", "two-phase vs single o")
    assert_close(f64(outs[2][1]), f64(outs[0][1]), "bf16", "two-phase vs single S")
