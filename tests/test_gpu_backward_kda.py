"""GPU parity of la_chunk_bwd_delta for Kimi Delta Attention (LA_KDA: the
delta rule with a per-key-channel gate; dq, dk, dv, dbeta, the per-channel
dg and dS0) with the float64 delta-rule backward oracle in its "kda" mode,
through the C ABI, at the library's bf16 tolerance on every output (relative
Frobenius 5e-3; max-abs 2e-2 taken at the output's own scale, as for Gated
DeltaNet's backward). Inputs follow the Kimi Delta Attention workload recipe
(L2-normalised q and k, beta = sigmoid(N(0,1)), per-channel log-gates),
with dO ~ N(0,1)/sqrt(dv) and dS_final ~ N(0, 0.01). Lengths that 64 does
not divide exercise the padded tail chunk."""
import numpy as np
import pytest
import torch

from oracle.backward_delta import backward_delta
from paritylib import BF16_MAX_ABS, BF16_REL_FRO, errors, f64, make

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import gated_delta_rule_linear_gb300 as la
    from gated_delta_rule_linear_gb300 import build
    build.build()
    la.load_library()
    assert torch.cuda.is_available()


def _case(B, H, T, dk, dv, s0=True, ds=True, betas=True, seed=0):
    from workloads import WORKLOADS
    wl = WORKLOADS["kda"].with_sizes(B=B, H=H, T=T, dk=dk, dv=dv, s0=s0, seed=120 + seed)
    inp = make(wl)
    gen = torch.Generator().manual_seed(130 + seed)
    dO = (torch.randn(B, H, T, dv, generator=gen) / np.sqrt(dv)).to(torch.bfloat16)
    dS = torch.randn(B, H, dk, dv, generator=gen) * 0.1 if ds else None
    return dict(q=inp["q"], k=inp["k"], v=inp["v"], g=inp["g"], beta=inp["beta"] if betas else None,
                S0=inp["S0"], dO=dO, dS=dS)


def _run(c, **kw):
    import gated_delta_rule_linear_gb300 as la
    cu = lambda t: None if t is None else t.cuda().contiguous()
    out = la.chunk_bwd_delta(cu(c["q"]), cu(c["k"]), cu(c["v"]), cu(c["dO"]), g=cu(c["g"]), beta=cu(c["beta"]),
                             S0=cu(c["S0"]), dS_final=cu(c["dS"]), mode="kda", **kw)
    torch.cuda.synchronize()
    return out


def _oracle(c, sel=lambda t: t):
    s = lambda t: None if t is None else sel(f64(t))
    return backward_delta(s(c["q"]), s(c["k"]), s(c["v"]), s(c["dO"]), "kda", g=s(c["g"]), beta=s(c["beta"]),
                          S0=s(c["S0"]), dS=s(c["dS"]))


NAMES = ("dq", "dk", "dv", "dbeta", "dg", "dS0")


def _check(got, ref, what, sel=lambda t: t):
    for name, a, r in zip(NAMES, got, ref):
        if r is None:
            assert a is None, f"{what} {name}"
            continue
        max_abs, rel = errors(sel(f64(a)), r)
        scale = max(1.0, float(np.max(np.abs(r))) if np.size(r) else 1.0)
        assert max_abs <= BF16_MAX_ABS * scale and rel <= BF16_REL_FRO, \
            f"{what} {name}: max_abs={max_abs:.3e} (scale {scale:.2f}) rel_fro={rel:.3e}"


@pytest.mark.parametrize("dims", [(128, 128), (64, 64), (64, 128), (128, 64)])
@pytest.mark.parametrize("T", [1, 17, 64, 65, 200])
def test_kda_backward_parity(dims, T):
    dk, dv = dims
    c = _case(1, 2, T, dk, dv)
    _check(_run(c), _oracle(c), f"T={T} dk={dk} dv={dv}")


def test_kda_backward_without_beta_or_states():
    c = _case(1, 2, 150, 128, 128, betas=False, seed=1)
    _check(_run(c), _oracle(c), "beta = 1")
    c = _case(2, 2, 333, 128, 128, s0=False, ds=False, seed=2)
    _check(_run(c), _oracle(c), "no S0 / dS")


def test_kda_backward_optional_outputs_are_skipped():
    c = _case(1, 2, 100, 128, 128, seed=3)
    full = _run(c)
    part = _run(c, with_dS0=False, with_dg=False, with_dbeta=False)
    assert part[3] is None and part[4] is None and part[5] is None
    for a, b in zip(full[:3], part[:3]):
        assert torch.equal(a, b)


def test_kda_backward_multichunk_long():
    c = _case(1, 3, 1280, 128, 128, seed=4)
    _check(_run(c), _oracle(c), "T=1280")


def test_kda_backward_with_equal_channel_gates_is_gated_deltanet():
    # the same gate on every key channel is Gated DeltaNet: the two entry points agree
    # (dg summed over the channels)
    import gated_delta_rule_linear_gb300 as la
    c = _case(1, 2, 200, 128, 128, seed=5)
    g1 = c["g"][..., 0].contiguous()
    c["g"] = g1[..., None].expand(c["g"].shape).contiguous()
    kda = _run(c)
    cu = lambda t: None if t is None else t.cuda().contiguous()
    gdn = la.chunk_bwd_delta(cu(c["q"]), cu(c["k"]), cu(c["v"]), cu(c["dO"]), g=cu(g1), beta=cu(c["beta"]),
                             S0=cu(c["S0"]), dS_final=cu(c["dS"]), mode="gdn")
    torch.cuda.synchronize()
    for name, a, b in zip(NAMES, kda, gdn):
        if name == "dg":
            a = a.sum(-1)
        max_abs, rel = errors(f64(a), f64(b))
        assert rel <= 2 * BF16_REL_FRO, f"{name}: rel {rel:.2e}"


def test_kda_backward_bench_shape_sampled():
    """The Kimi Delta Attention workload shape (B=4, H=16, T=16384): sampled heads against the oracle."""
    c = _case(4, 16, 16384, 128, 128, seed=6)
    got = _run(c)
    for b, h in [(0, 0), (3, 15)]:
        sel = lambda t: t[b:b + 1, h:h + 1]
        _check(got, _oracle(c, sel), f"head {b},{h}", sel)
