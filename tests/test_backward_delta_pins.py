"""Pins of the delta-rule backward oracle (Gated DeltaNet, Kimi Delta
Attention) to gradients obtained another way:

  * central finite differences of the float64 forward recurrence
    (oracle.recurrence, a separate module) on tiny inputs, for every input
    (q, k, v, g, beta, S0);
  * reverse-mode automatic differentiation (torch.autograd, float64) of a
    step-by-step forward written afresh in the pages' product form
    S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T;
  * special cases with a known answer: beta = 0 leaves only the decay, whose
    gradients the scalar-decay oracle gives (and dk = dv = 0); KDA with the
    same gate on every channel is Gated DeltaNet (its dg summed over channels);
    exact retrieval with orthonormal keys, beta = 1 and no decay;
  * checkpointing does not change a single bit;
  * mistakes planted in the oracle's per-token step are caught by the pins.
CPU only."""
import numpy as np
import pytest
import torch

import oracle.backward_delta as bd
from oracle import recurrence
from oracle.backward import backward_scalar
from oracle.backward_delta import backward_delta

RNG = np.random.default_rng(17)


def _case(mode="gdn", B=1, H=2, T=7, dk=3, dv=4, gates=True, betas=True):
    q = RNG.standard_normal((B, H, T, dk)) * 0.5
    k = RNG.standard_normal((B, H, T, dk)) * 0.5
    v = RNG.standard_normal((B, H, T, dv))
    gshape = (B, H, T, dk) if mode == "kda" else (B, H, T)
    g = -np.abs(RNG.standard_normal(gshape)) * 0.3 if gates else None
    beta = RNG.uniform(0.1, 0.9, (B, H, T)) if betas else None
    S0 = RNG.standard_normal((B, H, dk, dv)) * 0.3
    dO = RNG.standard_normal((B, H, T, dv))
    dS = RNG.standard_normal((B, H, dk, dv))
    return dict(q=q, k=k, v=v, g=g, beta=beta, S0=S0, dO=dO, dS=dS)


def _loss(c, mode):
    o, S = recurrence(c["q"], c["k"], c["v"], mode, g=c["g"], beta=c["beta"], S0=c["S0"])
    return float(np.sum(o * c["dO"]) + np.sum(S * c["dS"]))


def _grads(c, mode, **kw):
    dq, dk, dv, dbeta, dg, dS0 = backward_delta(c["q"], c["k"], c["v"], c["dO"], mode, g=c["g"],
                                                beta=c["beta"], S0=c["S0"], dS=c["dS"], **kw)
    return {"q": dq, "k": dk, "v": dv, "beta": dbeta, "g": dg, "S0": dS0}


def _finite_differences(c, mode, name, eps=1e-6):
    x = c[name]
    num = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        old = x[idx]
        x[idx] = old + eps
        lp = _loss(c, mode)
        x[idx] = old - eps
        lm = _loss(c, mode)
        x[idx] = old
        num[idx] = (lp - lm) / (2 * eps)
    return num


@pytest.mark.parametrize("mode", ["gdn", "kda"])
def test_delta_backward_matches_finite_differences(mode):
    c = _case(mode)
    got = _grads(c, mode, checkpoint=3)
    for name in ("q", "k", "v", "g", "beta", "S0"):
        assert np.allclose(got[name], _finite_differences(c, mode, name), rtol=1e-6, atol=1e-7), name


@pytest.mark.parametrize("gates,betas", [(False, True), (True, False), (False, False)])
def test_delta_backward_without_gates_or_betas_matches_finite_differences(gates, betas):
    # absent g means alpha = 1 (plain DeltaNet), absent beta means beta = 1
    c = _case("gdn", T=6, gates=gates, betas=betas)
    got = _grads(c, "gdn")
    names = ["q", "k", "v", "S0"] + (["g"] if gates else [])
    for name in names:
        assert np.allclose(got[name], _finite_differences(c, "gdn", name), rtol=1e-6, atol=1e-7), name
    assert (got["g"] is None) == (not gates)
    if not betas:  # dbeta is still the gradient at beta = 1: check it against a perturbed beta
        c["beta"] = np.ones(c["q"].shape[:3])
        assert np.allclose(got["beta"], _finite_differences(c, "gdn", "beta"), rtol=1e-6, atol=1e-7)


def _torch_forward(q, k, v, g, beta, S0, mode):
    """Written for autograd in the product form (I - b k k^T) Diag(alpha) S + b k v^T."""
    B, H, T, dk = q.shape
    eye = torch.eye(dk, dtype=torch.float64)
    S = S0
    outs = []
    for t in range(T):
        kt = k[:, :, t]
        if mode == "gdn":
            a = torch.exp(g[:, :, t])[..., None, None] * torch.ones(dk, 1, dtype=torch.float64)
        else:
            a = torch.exp(g[:, :, t])[..., :, None]
        proj = eye - beta[:, :, t, None, None] * kt[..., :, None] * kt[..., None, :]
        S = proj @ (a * S) + beta[:, :, t, None, None] * kt[..., :, None] * v[:, :, t, None, :]
        outs.append(torch.einsum("bhc,bhcv->bhv", q[:, :, t], S))
    return torch.stack(outs, dim=2), S


@pytest.mark.parametrize("mode", ["gdn", "kda"])
def test_delta_backward_matches_autograd(mode):
    c = _case(mode, B=2, H=2, T=33, dk=5, dv=6)
    names = ("q", "k", "v", "g", "beta", "S0")
    tens = {n: torch.tensor(c[n], requires_grad=True) for n in names}
    o, S = _torch_forward(*(tens[n] for n in names), mode)
    (o * torch.tensor(c["dO"])).sum().add((S * torch.tensor(c["dS"])).sum()).backward()
    got = _grads(c, mode, checkpoint=8)
    for n in names:
        assert np.allclose(got[n], tens[n].grad.numpy(), rtol=1e-10, atol=1e-11), n


def test_checkpoint_length_changes_no_bit():
    c = _case("gdn", T=23)
    ref = _grads(c, "gdn", checkpoint=1)
    for ck in (2, 5, 23, 256):
        got = _grads(c, "gdn", checkpoint=ck)
        for n in ref:
            assert np.array_equal(got[n], ref[n]), (ck, n)


def test_beta_zero_leaves_the_decay_alone():
    # beta = 0: S_t = alpha_t S_{t-1} and nothing is written, which is the scalar decay
    # with v = 0; dk and dv vanish
    c = _case("gdn", T=11)
    c["beta"] = np.zeros_like(c["beta"])
    got = _grads(c, "gdn")
    dq, dk, dv, dS0, dg = backward_scalar(c["q"], c["k"], np.zeros_like(c["v"]), c["dO"], c["g"],
                                          S0=c["S0"], dS=c["dS"])
    assert np.allclose(got["q"], dq, atol=1e-12)
    assert np.allclose(got["S0"], dS0, atol=1e-12)
    assert np.allclose(got["g"], dg, atol=1e-12)
    assert np.all(got["k"] == 0) and np.all(got["v"] == 0)


def test_kda_with_equal_channel_gates_is_gated_deltanet():
    c = _case("gdn", T=13)
    dkk = c["q"].shape[-1]
    ck = dict(c, g=np.repeat(c["g"][..., None], dkk, axis=-1))
    a, b = _grads(c, "gdn"), _grads(ck, "kda")
    for n in ("q", "k", "v", "beta", "S0"):
        assert np.allclose(a[n], b[n], atol=1e-12), n
    assert np.allclose(a["g"], b["g"].sum(axis=-1), atol=1e-12)


def test_exact_retrieval_gradient():
    # orthonormal keys, beta = 1, alpha = 1: token t writes v_t at key e_t and
    # o_{t'} = v_t for a later query q_{t'} = e_t, so dv_t = sum of dO over those queries
    dk_, dv_, T = 6, 3, 6
    keys = np.linalg.qr(RNG.standard_normal((dk_, dk_)))[0].T          # rows orthonormal
    k = keys[None, None]
    v = RNG.standard_normal((1, 1, T, dv_))
    perm = np.array([0, 0, 1, 2, 2, 4])                                 # query t reads key perm[t] <= t
    q = keys[perm][None, None]
    dO = RNG.standard_normal((1, 1, T, dv_))
    dq, dk, dv, dbeta, dg, dS0 = backward_delta(q, k, v, dO, "gdn")
    want = np.zeros((T, dv_))
    for t in range(T):
        want[perm[t]] += dO[0, 0, t]
    assert np.allclose(dv[0, 0], want, atol=1e-12)
    assert dg is None


# --- mistakes planted in the oracle's per-token step -----------------------------

def _plant(monkeypatch, which):
    orig = bd._token_grads

    def mutant(G, q_t, k_t, dO_t, beta_t, alpha_t, R, r, S_t, per_channel):
        dq, dk, dv, dbeta, dg, Gp = orig(G, q_t, k_t, dO_t, beta_t, alpha_t, R, r, S_t, per_channel)
        Gh = G + np.outer(q_t, dO_t)
        Gk = Gh.T @ k_t
        if which == "dk_read_term_dropped":
            dk = beta_t * (Gh @ r)
        elif which == "dg_sign":
            dg = -dg
        elif which == "dv_without_beta":
            dv = Gk
        elif which == "q_read_after_the_step":       # o_t read as S_{t-1}^T q_t
            dq = (S_t - beta_t * np.outer(k_t, r)) @ dO_t / 1.0
        elif which == "state_grad_not_projected":     # G = alpha Gh, the (I - b k k^T) dropped
            Gp = alpha_t[:, None] * Gh
        elif which == "dbeta_uses_v":                 # r_t replaced by v_t
            dbeta = Gk @ (r + R.T @ k_t)
        return dq, dk, dv, dbeta, dg, Gp

    monkeypatch.setattr(bd, "_token_grads", mutant)


@pytest.mark.parametrize("which,name", [
    ("dk_read_term_dropped", "k"), ("dg_sign", "g"), ("dv_without_beta", "v"),
    ("q_read_after_the_step", "q"), ("state_grad_not_projected", "S0"), ("dbeta_uses_v", "beta"),
])
def test_planted_mistakes_are_caught(monkeypatch, which, name):
    c = _case("gdn", T=5)
    num = _finite_differences(c, "gdn", name)
    assert np.allclose(_grads(c, "gdn")[name], num, rtol=1e-6, atol=1e-7)
    _plant(monkeypatch, which)
    assert not np.allclose(_grads(c, "gdn")[name], num, rtol=1e-3, atol=1e-4), which
