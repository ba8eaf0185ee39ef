"""GPU edge cases against the float64 oracle, through the C ABI: the
degenerate cases of the method (no write, full overwrite, zero keys, a state
that forgets within a chunk), decay strong enough to take the kernels' exact
path, and tensors with more than 2^31 elements (index arithmetic past 32
bits), compared on sampled heads at the library's tolerance."""
import pytest
import torch

import gated_delta_rule_linear_gb300 as la
from paritylib import assert_close, f64, make, run_cuda, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_linear_gb300 import build
    build.build()
    la.load_library()
    assert torch.cuda.is_available()


def _small(name, **sizes):
    from workloads import WORKLOADS
    kw = dict(B=1, H=2, T=200)
    kw.update(sizes)
    return make(WORKLOADS[name].with_sizes(**kw))


def _check(inp, what):
    o, S = run_cuda(inp)
    o_ref, S_ref = run_oracle(inp)
    assert_close(f64(o), o_ref, "bf16", f"{what} o")
    assert_close(f64(S), S_ref, "bf16", f"{what} S")


@pytest.mark.parametrize("path", ["single", "pair", "wy"])
@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_delta_rule_with_no_write_and_full_overwrite(path, beta, monkeypatch):
    """beta = 0: the state only decays (o = alpha-decayed S0^T q); beta = 1: each
    token's value replaces what its key retrieves."""
    monkeypatch.setenv("LA_DELTA", path)
    inp = _small("gdn")
    inp["beta"] = torch.full_like(inp["beta"], beta)
    _check(inp, f"gdn beta={beta} ({path})")


@pytest.mark.parametrize("mode", ["gdn", "linear", "gla", "kda", "outer"])
def test_zero_keys_leave_the_state_alone(mode):
    """k = 0: nothing is written or erased; the output reads the (decayed) S0."""
    name = {"linear": "retnet", "gdn": "gdn", "gla": "gla", "kda": "kda", "outer": "outer"}[mode]
    inp = _small(name, s0=True)
    if mode == "linear":
        inp["g"] = None
        inp["wl"] = inp["wl"].with_sizes(mode="linear")
    inp["k"] = torch.zeros_like(inp["k"])
    _check(inp, f"{mode} k=0")


@pytest.mark.parametrize("mode", ["retnet", "scalar", "gdn"])
def test_decay_strong_enough_for_the_exact_path(mode):
    """Chunks whose total log2-decay exceeds the fast path's limit (and chunks
    that do not, in one sequence): every chunk forgets most of its past."""
    inp = _small({"retnet": "retnet", "scalar": "scalar", "gdn": "gdn"}[mode], T=300, s0=True)
    if mode == "retnet":
        inp["g"] = torch.tensor([-3.0, -0.01], dtype=torch.float32)
    else:
        g = inp["g"].clone()
        g[:, :, :128] = -3.0      # two chunks past the limit
        g[:, :, 128:] *= 0.5      # the rest mild
        inp["g"] = g
    _check(inp, f"{mode} strong decay")


@pytest.mark.parametrize("mode", ["gla", "kda", "outer"])
def test_per_channel_decay_near_the_fold_range(mode):
    """Per-channel log-gates of -2 per token (-64 over half a chunk, e^64 inside
    the midpoint fold, within the float range) on half the key channels; for the
    outer-product gate, whose two axes' half-chunk decays add up inside the fold,
    -1.2 per token on half the key channels and half the value columns (-77 for
    the pairs where both apply)."""
    inp = _small(mode, T=200)
    g = inp["g"].clone()
    g[..., ::2] = -1.2 if mode == "outer" else -2.0
    inp["g"] = g
    if mode == "outer":
        b = inp["beta"].clone()
        b[..., 1::2] = -1.2
        inp["beta"] = b
    _check(inp, f"{mode} strong channel decay")


# --- more than 2^31 elements per tensor -------------------------------------------

BIG_BH, BIG_T, BIG_D = 20480, 1024, 128   # 2.68e9 elements per q/k/v/o tensor


@pytest.mark.parametrize("mode", ["gla", "retnet", "gdn"])
def test_tensors_past_two_to_the_31_elements(mode):
    assert BIG_BH * BIG_T * BIG_D > 2 ** 31
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(99)
    B, H = BIG_BH // 16, 16
    shape = (B, H, BIG_T, BIG_D)
    rn = lambda *s: torch.randn(*s, generator=gen, device=dev)
    q = (rn(*shape) / BIG_D ** 0.5).to(torch.bfloat16)
    k = (rn(*shape) / BIG_D ** 0.5).to(torch.bfloat16)
    v = (rn(*shape) / BIG_D ** 0.5).to(torch.bfloat16)
    g = beta = None
    if mode == "gla":
        g = torch.nn.functional.logsigmoid(rn(*shape)) / 16.0
    elif mode == "retnet":
        g = torch.log1p(-(2.0 ** (-5.0 - torch.arange(H, device=dev, dtype=torch.float64)))).float()
    else:
        q = torch.nn.functional.normalize(q.float(), dim=-1).to(torch.bfloat16)
        k = torch.nn.functional.normalize(k.float(), dim=-1).to(torch.bfloat16)
        g = -torch.nn.functional.softplus(rn(B, H, BIG_T)) / 8.0
        beta = torch.sigmoid(rn(B, H, BIG_T))
    o, S = la.chunk_fwd(q, k, v, mode, g=g, beta=beta)
    torch.cuda.synchronize()
    assert la.la_stream_status(torch.cuda.current_stream().cuda_stream) == 0
    import oracle
    # the first head, the first head past 2^31 elements, the last head
    for bh in (0, 2 ** 31 // (BIG_T * BIG_D), BIG_BH - 1):
        b, h = divmod(bh, H)
        cpu = lambda t: None if t is None else t[b:b + 1, h:h + 1].cpu()
        gh = None
        if g is not None:
            gh = g[h:h + 1].cpu() if mode == "retnet" else cpu(g)
        o_ref, S_ref = oracle.recurrence_c(f64(cpu(q)), f64(cpu(k)), f64(cpu(v)), mode, g=f64(gh),
                                           beta=f64(cpu(beta)))
        assert_close(f64(cpu(o)), o_ref, "bf16", f"{mode} head {bh} o")
        assert_close(f64(cpu(S)), S_ref, "bf16", f"{mode} head {bh} S")
    del q, k, v, g, beta, o, S
    torch.cuda.empty_cache()
