"""GPU parity of la_chunk_bwd (linear, RetNet, scalar decay; three chunk-forward passes,
two of them the kernels' reversed runs over the stored tensors) with the
float64 backward oracle, through the C ABI, at the library's tolerance (bf16:
max-abs 2e-2 and relative Frobenius 5e-3; fp32: relative 1e-4) on dq, dk, dv
and dS0. Lengths that 64 does not divide put the last reversed window above
row 0 (zero-filled rows, row-by-row output); 700 tokens wrap the kernels'
three-stage ring several times."""
import numpy as np
import pytest
import torch

from oracle.backward import backward, backward_gla, backward_scalar
from paritylib import assert_close, f64, make

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import gated_delta_rule_linear_gb300 as la
    from gated_delta_rule_linear_gb300 import build
    build.build()
    la.load_library()
    assert torch.cuda.is_available()


def _case(mode, dtype, B, H, T, dk, dv, s0, ds, seed=0):
    from workloads import WORKLOADS
    wl = WORKLOADS["retnet"].with_sizes(B=B, H=H, T=T, dk=dk, dv=dv, dtype=dtype, s0=False, seed=20 + seed)
    inp = make(wl)
    gen = torch.Generator().manual_seed(40 + seed)
    dO = (torch.randn(B, H, T, dv, generator=gen) / np.sqrt(dv)).to(wl.torch_dtype)
    S0 = torch.randn(B, H, dk, dv, generator=gen) * 0.1 if s0 else None
    dS = torch.randn(B, H, dk, dv, generator=gen) * 0.1 if ds else None
    g = inp["g"] if mode == "retnet" else None
    return inp["q"], inp["k"], inp["v"], g, dO, S0, dS


def _run(mode, q, k, v, g, dO, S0, dS):
    import gated_delta_rule_linear_gb300 as la
    dev = torch.device("cuda")
    cu = lambda t: None if t is None else t.to(dev).contiguous()
    out = la.chunk_bwd(cu(q), cu(k), cu(v), cu(dO), mode, g=cu(g), S0=cu(S0), dS_final=cu(dS))
    torch.cuda.synchronize()
    assert out[4] is None or mode in ("scalar", "gla")
    return out[:4] if mode not in ("scalar", "gla") else out


@pytest.mark.parametrize("mode", ["linear", "retnet"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dims", [(128, 128), (64, 128), (128, 64), (64, 64)])
@pytest.mark.parametrize("T", [1, 64, 129, 200, 700])
def test_backward_parity(mode, dtype, dims, T):
    dk, dv = dims
    q, k, v, g, dO, S0, dS = _case(mode, dtype, 2, 3, T, dk, dv, s0=True, ds=True)
    dq, dk_, dv_, dS0 = _run(mode, q, k, v, g, dO, S0, dS)
    ref = backward(f64(q), f64(k), f64(v), f64(dO), mode, g=None if g is None else f64(g),
                   S0=f64(S0), dS=f64(dS))
    for name, got, r in (("dq", dq, ref[0]), ("dk", dk_, ref[1]), ("dv", dv_, ref[2]), ("dS0", dS0, ref[3])):
        assert_close(f64(got), r, dtype, f"{mode} {dtype} {name}")


@pytest.mark.parametrize("mode", ["linear", "retnet"])
def test_backward_without_states(mode):
    q, k, v, g, dO, S0, dS = _case(mode, "bf16", 1, 2, 333, 128, 128, s0=False, ds=False, seed=1)
    dq, dk_, dv_, dS0 = _run(mode, q, k, v, g, dO, None, None)
    ref = backward(f64(q), f64(k), f64(v), f64(dO), mode, g=None if g is None else f64(g))
    for name, got, r in (("dq", dq, ref[0]), ("dk", dk_, ref[1]), ("dv", dv_, ref[2]), ("dS0", dS0, ref[3])):
        assert_close(f64(got), r, "bf16", f"{mode} {name}")


def test_backward_bench_shape_sampled():
    """The bench configuration (RetNet, B=8 H=16 T=4096): sampled heads against the oracle."""
    q, k, v, g, dO, S0, dS = _case("retnet", "bf16", 8, 16, 4096, 128, 128, s0=False, ds=True, seed=2)
    dq, dk_, dv_, dS0 = _run("retnet", q, k, v, g, dO, None, dS)
    rng = np.random.default_rng(9)
    for _ in range(2):
        b, h = int(rng.integers(8)), int(rng.integers(16))
        sl = lambda t: f64(t[b:b + 1, h:h + 1])
        ref = backward(sl(q), sl(k), sl(v), sl(dO), "retnet", g=f64(g)[h:h + 1], dS=sl(dS))
        for name, got, r in (("dq", dq, ref[0]), ("dk", dk_, ref[1]), ("dv", dv_, ref[2]), ("dS0", dS0, ref[3])):
            assert_close(f64(got[b:b + 1, h:h + 1]), r, "bf16", f"head {b},{h} {name}")


# --- the data-dependent scalar decay, with dg ------------------------------------------
# dg is a suffix sum over up to T tokens of w_u = q_u.dq_u - k_u.dk_u, formed
# from the dq and dk the passes write. Expanding dq and dk fully, each element
# is a sum of elementary products (for the scalar decay, e.g. dq_t[c] =
# sum_j a(t) S0[c,j] dO_t[j] + sum_{s<=t} sum_j a(t,s) dO_t[j] v_s[j] k_s[c]).
# Every rounding on a product's way through the chunk passes perturbs it by at
# most one unit roundoff u relative to its own size: in bf16 the decayed
# operand copy, the intermediate score or state tile and the bf16 MMA operand
# (2^-9 each) and the output rounding (2^-9), at most four, so 4u = 2^-7;
# in float32 (LA_F32) up to eight float32 roundings, 8 * 2^-24 = 2^-21. So
# with M_dq, M_dk the same sums taken over the products' absolute values (the
# oracle's backward evaluated on |q|, |k|, |v|, |dO|, |S0|, |dS| with the
# same, positive, decay factors):
#   |dg_tau - ref_tau| <= eps * sum_{u>=tau} sum_c (|q_u,c| M_dq(u,c) + |k_u,c| M_dk(u,c)) + 1e-6,
# eps = 2^-7 for bf16 and 2^-21 for float32. Cancellation inside w or inside
# dq and dk cannot break it, since M bounds every intermediate's size; a
# relative bound on dg itself would not follow from the arithmetic.

def _dg_bound(q, k, v, dO, g, S0, dS, eps, backward_fn):
    """Suffix sums of eps * (|q| M_dq + |k| M_dk) along the token axis (axis 2),
    per token for the scalar decay and per channel for GLA."""
    a = np.abs
    M = backward_fn(a(q), a(k), a(v), a(dO), g, S0=None if S0 is None else a(S0),
                    dS=None if dS is None else a(dS))
    mag = a(q) * M[0] + a(k) * M[1]
    if M[4].ndim == 3:                         # scalar decay: one gate per token
        mag = mag.sum(-1)
    return eps * np.flip(np.cumsum(np.flip(mag, 2), 2), 2) + 1e-6


def _scalar_case(dtype, B, H, T, dk, dv, seed=0):
    from workloads import WORKLOADS
    wl = WORKLOADS["scalar"].with_sizes(B=B, H=H, T=T, dk=dk, dv=dv, dtype=dtype, s0=True, seed=60 + seed)
    inp = make(wl)
    gen = torch.Generator().manual_seed(70 + seed)
    dO = (torch.randn(B, H, T, dv, generator=gen) / np.sqrt(dv)).to(wl.torch_dtype)
    dS = torch.randn(B, H, dk, dv, generator=gen) * 0.1
    return inp["q"], inp["k"], inp["v"], inp["g"], dO, inp["S0"], dS


def _check_dg(got, ref, dtype, what, q, k, v, dO, g, S0, dS):
    """ref = backward_scalar's outputs; the rest the float64 inputs."""
    assert np.all(np.isfinite(got)), what
    if dtype == "f32":
        assert_close(got, ref[4], dtype, what)
    bound = _dg_bound(q, k, v, dO, g, S0, dS, 2.0 ** -7 if dtype == "bf16" else 2.0 ** -21, backward_scalar)
    bad = np.abs(got - ref[4]) > bound
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside the rounding bound"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dims", [(128, 128), (64, 128), (64, 64)])
@pytest.mark.parametrize("T", [1, 64, 129, 700])
def test_scalar_backward_parity(dtype, dims, T):
    dk, dv = dims
    q, k, v, g, dO, S0, dS = _scalar_case(dtype, 2, 3, T, dk, dv)
    dq, dk_, dv_, dS0, dg = _run("scalar", q, k, v, g, dO, S0, dS)
    ref = backward_scalar(f64(q), f64(k), f64(v), f64(dO), f64(g), S0=f64(S0), dS=f64(dS))
    for name, got, r in (("dq", dq, ref[0]), ("dk", dk_, ref[1]), ("dv", dv_, ref[2]), ("dS0", dS0, ref[3])):
        assert_close(f64(got), r, dtype, f"scalar {dtype} T={T} {name}")
    _check_dg(f64(dg), ref, dtype, f"scalar {dtype} T={T} dg", f64(q), f64(k), f64(v), f64(dO), f64(g),
              f64(S0), f64(dS))


def test_scalar_backward_without_states_or_dS():
    q, k, v, g, dO, S0, dS = _scalar_case("bf16", 1, 2, 333, 128, 128, seed=1)
    dq, dk_, dv_, dS0, dg = _run("scalar", q, k, v, g, dO, None, None)
    ref = backward_scalar(f64(q), f64(k), f64(v), f64(dO), f64(g))
    for name, got, r in (("dq", dq, ref[0]), ("dk", dk_, ref[1]), ("dv", dv_, ref[2]), ("dS0", dS0, ref[3])):
        assert_close(f64(got), r, "bf16", f"scalar {name}")
    _check_dg(f64(dg), ref, "bf16", "scalar dg", f64(q), f64(k), f64(v), f64(dO), f64(g), None, None)


# --- GLA's per-channel decay, with the per-channel dg ------------------------------------
# dq and dk come from outer-product-gate passes (the decay on their value axis),
# dv from a reversed GLA run; dg[c] is held to the same bound as the scalar
# decay's, channel by channel.

def _gla_case(B, H, T, dk, dv, seed=0):
    from workloads import WORKLOADS
    wl = WORKLOADS["gla"].with_sizes(B=B, H=H, T=T, dk=dk, dv=dv, s0=True, seed=80 + seed)
    inp = make(wl)
    gen = torch.Generator().manual_seed(90 + seed)
    dO = (torch.randn(B, H, T, dv, generator=gen) / np.sqrt(dv)).to(torch.bfloat16)
    dS = torch.randn(B, H, dk, dv, generator=gen) * 0.1
    S0 = torch.randn(B, H, dk, dv, generator=gen) * 0.1
    return inp["q"], inp["k"], inp["v"], inp["g"], dO, S0, dS


def _check_dgc(got, ref, what, q, k, v, dO, g, S0, dS):
    """The bound of the scalar decay, channel by channel (eps = 2^-7), plus the
    final-state term sum_j dS[c, j] S_final[c, j], whose S_final comes from the
    bf16 forward kernel: held to eps * sum_j |dS| S_abs, S_abs the final state
    of the same recurrence on the absolute values (a bound on every product
    that forms S_final)."""
    from oracle import recurrence
    assert np.all(np.isfinite(got)), what
    eps = 2.0 ** -7
    bound = _dg_bound(q, k, v, dO, g, S0, dS, eps, backward_gla)
    if dS is not None:
        a = np.abs
        _, S_abs = recurrence(a(q), a(k), a(v), "gla", g=g, S0=None if S0 is None else a(S0))
        bound = bound + eps * np.sum(a(dS) * S_abs, axis=-1)[:, :, None, :]
    bad = np.abs(got - ref[4]) > bound
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside the rounding bound"


@pytest.mark.parametrize("dims", [(128, 128), (64, 64), (64, 128)])
@pytest.mark.parametrize("T", [1, 64, 129, 300])
def test_gla_backward_parity(dims, T):
    dk, dv = dims
    q, k, v, g, dO, S0, dS = _gla_case(1, 2, T, dk, dv)
    dq, dk_, dv_, dS0, dg = _run("gla", q, k, v, g, dO, S0, dS)
    ref = backward_gla(f64(q), f64(k), f64(v), f64(dO), f64(g), S0=f64(S0), dS=f64(dS))
    for name, got, r in (("dq", dq, ref[0]), ("dk", dk_, ref[1]), ("dv", dv_, ref[2]), ("dS0", dS0, ref[3])):
        assert_close(f64(got), r, "bf16", f"gla T={T} {name}")
    _check_dgc(f64(dg), ref, f"gla T={T} dg", f64(q), f64(k), f64(v), f64(dO), f64(g), f64(S0), f64(dS))


def test_gla_backward_without_states_or_dS():
    q, k, v, g, dO, S0, dS = _gla_case(1, 2, 200, 128, 128, seed=1)
    dq, dk_, dv_, dS0, dg = _run("gla", q, k, v, g, dO, None, None)
    ref = backward_gla(f64(q), f64(k), f64(v), f64(dO), f64(g))
    for name, got, r in (("dq", dq, ref[0]), ("dk", dk_, ref[1]), ("dv", dv_, ref[2]), ("dS0", dS0, ref[3])):
        assert_close(f64(got), r, "bf16", f"gla {name}")
    _check_dgc(f64(dg), ref, "gla dg", f64(q), f64(k), f64(v), f64(dO), f64(g), None, None)
