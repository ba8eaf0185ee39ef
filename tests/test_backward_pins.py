"""Pins of the backward oracle (linear, RetNet) to gradients computed another
way: central finite differences of the float64 token recurrence on tiny
inputs, and reverse-mode automatic differentiation (torch.autograd, float64)
of a separately written step-by-step recurrence. The last test plants
mistakes and checks that the pins catch them. CPU only."""
import numpy as np
import pytest
import torch

from oracle import recurrence
from oracle.backward import backward, backward_gla, backward_scalar

RNG = np.random.default_rng(5)


def _case(mode, B=1, H=2, T=9, dk=3, dv=4):
    q = RNG.standard_normal((B, H, T, dk)) * 0.5
    k = RNG.standard_normal((B, H, T, dk)) * 0.5
    v = RNG.standard_normal((B, H, T, dv))
    g = np.log(np.array([0.9, 0.6])[:H]) if mode == "retnet" else None
    S0 = RNG.standard_normal((B, H, dk, dv)) * 0.3
    dO = RNG.standard_normal((B, H, T, dv))
    dS = RNG.standard_normal((B, H, dk, dv))
    return q, k, v, g, S0, dO, dS


def _loss(q, k, v, g, S0, dO, dS, mode):
    o, S = recurrence(q, k, v, mode, g=g, S0=S0)
    return float(np.sum(o * dO) + np.sum(S * dS))


@pytest.mark.parametrize("mode", ["linear", "retnet"])
def test_backward_matches_finite_differences(mode):
    q, k, v, g, S0, dO, dS = _case(mode)
    dq, dk, dv, dS0 = backward(q, k, v, dO, mode, g=g, S0=S0, dS=dS)
    eps = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv), ("S0", S0, dS0)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + eps
            lp = _loss(q, k, v, g, S0, dO, dS, mode)
            x[idx] = old - eps
            lm = _loss(q, k, v, g, S0, dO, dS, mode)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        assert np.allclose(grad, num, rtol=1e-6, atol=1e-7), name


def _torch_recurrence(q, k, v, g, S0, mode):
    """A step-by-step recurrence in torch (float64), written for autograd."""
    B, H, T, dk = q.shape
    S = S0.clone()
    outs = []
    alpha = torch.ones(H, dtype=torch.float64) if mode == "linear" else torch.exp(g)
    for t in range(T):
        S = alpha[None, :, None, None] * S + k[:, :, t, :, None] * v[:, :, t, None, :]
        outs.append(torch.einsum("bhc,bhcv->bhv", q[:, :, t], S))
    return torch.stack(outs, dim=2), S


@pytest.mark.parametrize("mode", ["linear", "retnet"])
def test_backward_matches_autograd(mode):
    q, k, v, g, S0, dO, dS = _case(mode, B=2, H=2, T=40, dk=5, dv=6)
    tq, tk, tv, tS0 = (torch.tensor(x, requires_grad=True) for x in (q, k, v, S0))
    tg = None if g is None else torch.tensor(g)
    o, S = _torch_recurrence(tq, tk, tv, tg, tS0, mode)
    (o * torch.tensor(dO)).sum().add((S * torch.tensor(dS)).sum()).backward()
    dq, dk, dv, dS0 = backward(q, k, v, dO, mode, g=g, S0=S0, dS=dS)
    for name, a, b in (("q", dq, tq.grad), ("k", dk, tk.grad), ("v", dv, tv.grad), ("S0", dS0, tS0.grad)):
        assert np.allclose(a, b.numpy(), rtol=1e-11, atol=1e-11), name


def test_planted_mistakes_are_caught():
    q, k, v, g, S0, dO, dS = _case("retnet", T=12)
    tq, tk, tv, tS0 = (torch.tensor(x, requires_grad=True) for x in (q, k, v, S0))
    o, S = _torch_recurrence(tq, tk, tv, torch.tensor(g), tS0, "retnet")
    (o * torch.tensor(dO)).sum().add((S * torch.tensor(dS)).sum()).backward()
    dq, dk, dv, dS0 = backward(q, k, v, dO, "retnet", g=g, S0=S0, dS=dS)
    assert np.allclose(dk, tk.grad.numpy(), atol=1e-10)
    # a decay applied the wrong way round (alpha^(s-t)), and the final-state term dropped
    bad_dk, _, _, _ = backward(q, k, v, dO, "retnet", g=-np.asarray(g), S0=S0, dS=dS)
    _, bad2, _, _ = backward(q, k, v, dO, "retnet", g=g, S0=S0, dS=None)
    assert not np.allclose(bad_dk, tk.grad.numpy(), atol=1e-6)
    assert not np.allclose(bad2, tk.grad.numpy(), atol=1e-6)


# --- the data-dependent scalar decay, with the gradient of the log-gates ---------

def _scalar_case(B=1, H=2, T=9, dk=3, dv=4):
    q, k, v, _, S0, dO, dS = _case("linear", B=B, H=H, T=T, dk=dk, dv=dv)
    g = -np.abs(RNG.standard_normal((B, H, T))) * 0.3
    return q, k, v, g, S0, dO, dS


def test_scalar_backward_matches_finite_differences():
    q, k, v, g, S0, dO, dS = _scalar_case()
    grads = dict(zip(("q", "k", "v", "S0", "g"), (backward_scalar(q, k, v, dO, g, S0=S0, dS=dS)[i]
                                                   for i in (0, 1, 2, 3, 4))))
    eps = 1e-6
    for name, x in (("q", q), ("k", k), ("v", v), ("S0", S0), ("g", g)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + eps
            lp = _loss(q, k, v, g, S0, dO, dS, "scalar")
            x[idx] = old - eps
            lm = _loss(q, k, v, g, S0, dO, dS, "scalar")
            x[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        assert np.allclose(grads[name], num, rtol=1e-6, atol=1e-7), name


def test_scalar_backward_matches_autograd():
    q, k, v, g, S0, dO, dS = _scalar_case(B=2, H=2, T=40, dk=5, dv=6)
    tq, tk, tv, tg, tS0 = (torch.tensor(x, requires_grad=True) for x in (q, k, v, g, S0))
    S = tS0
    outs = []
    for t in range(40):  # written afresh for autograd: per-token scalar decay, then the write
        S = torch.exp(tg[:, :, t])[..., None, None] * S + tk[:, :, t, :, None] * tv[:, :, t, None, :]
        outs.append(torch.einsum("bhc,bhcv->bhv", tq[:, :, t], S))
    o = torch.stack(outs, dim=2)
    (o * torch.tensor(dO)).sum().add((S * torch.tensor(dS)).sum()).backward()
    got = backward_scalar(q, k, v, dO, g, S0=S0, dS=dS)
    for name, a, b in zip(("q", "k", "v", "S0", "g"), got, (tq.grad, tk.grad, tv.grad, tS0.grad, tg.grad)):
        assert np.allclose(a, b.numpy(), rtol=1e-10, atol=1e-11), name


def test_scalar_backward_with_zero_gates_is_linear():
    q, k, v, g, S0, dO, dS = _scalar_case(T=20)
    lin = backward(q, k, v, dO, "linear", S0=S0, dS=dS)
    sc = backward_scalar(q, k, v, dO, np.zeros_like(g), S0=S0, dS=dS)
    for a, b in zip(lin, sc[:4]):
        assert np.allclose(a, b, rtol=0, atol=1e-12)


def test_scalar_dg_pins_catch_an_exclusive_suffix_sum():
    q, k, v, g, S0, dO, dS = _scalar_case()
    dg = backward_scalar(q, k, v, dO, g, S0=S0, dS=dS)[4]
    eps = 1e-6
    num = np.zeros_like(g)
    for idx in np.ndindex(g.shape):
        old = g[idx]
        g[idx] = old + eps
        lp = _loss(q, k, v, g, S0, dO, dS, "scalar")
        g[idx] = old - eps
        lm = _loss(q, k, v, g, S0, dO, dS, "scalar")
        g[idx] = old
        num[idx] = (lp - lm) / (2 * eps)
    assert np.allclose(dg, num, rtol=1e-6, atol=1e-7)
    # the suffix sum taken exclusively (the token's own term dropped) is rejected
    shifted = np.concatenate([dg[..., 1:], np.zeros_like(dg[..., :1])], axis=-1)
    assert not np.allclose(shifted, num, rtol=1e-3, atol=1e-4)


# --- GLA's per-channel decay, with the per-channel log-gate gradient ------------------

def _gla_case(B=1, H=2, T=7, dk=3, dv=4):
    q, k, v, _, S0, dO, dS = _case("linear", B=B, H=H, T=T, dk=dk, dv=dv)
    g = -np.abs(RNG.standard_normal((B, H, T, dk))) * 0.3
    return q, k, v, g, S0, dO, dS


def test_gla_backward_matches_finite_differences():
    q, k, v, g, S0, dO, dS = _gla_case()
    got = backward_gla(q, k, v, dO, g, S0=S0, dS=dS)
    eps = 1e-6
    for name, x, grad in (("q", q, got[0]), ("k", k, got[1]), ("v", v, got[2]), ("S0", S0, got[3]), ("g", g, got[4])):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + eps
            lp = _loss(q, k, v, g, S0, dO, dS, "gla")
            x[idx] = old - eps
            lm = _loss(q, k, v, g, S0, dO, dS, "gla")
            x[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        assert np.allclose(grad, num, rtol=1e-6, atol=1e-7), name


def test_gla_backward_matches_autograd():
    q, k, v, g, S0, dO, dS = _gla_case(B=1, H=2, T=24, dk=5, dv=6)
    tq, tk, tv, tg, tS0 = (torch.tensor(x, requires_grad=True) for x in (q, k, v, g, S0))
    S = tS0
    outs = []
    for t in range(24):  # written afresh for autograd: per-key-channel decay, then the write
        S = torch.exp(tg[:, :, t])[..., :, None] * S + tk[:, :, t, :, None] * tv[:, :, t, None, :]
        outs.append(torch.einsum("bhc,bhcv->bhv", tq[:, :, t], S))
    o = torch.stack(outs, dim=2)
    (o * torch.tensor(dO)).sum().add((S * torch.tensor(dS)).sum()).backward()
    got = backward_gla(q, k, v, dO, g, S0=S0, dS=dS)
    for name, a, b in zip(("q", "k", "v", "S0", "g"), got, (tq.grad, tk.grad, tv.grad, tS0.grad, tg.grad)):
        assert np.allclose(a, b.numpy(), rtol=1e-10, atol=1e-11), name


def test_gla_backward_with_equal_channel_gates_is_the_scalar_decay():
    q, k, v, g, S0, dO, dS = _gla_case(T=15)
    gs = g[..., 0]
    gla = backward_gla(q, k, v, dO, np.repeat(gs[..., None], q.shape[-1], axis=-1), S0=S0, dS=dS)
    sc = backward_scalar(q, k, v, dO, gs, S0=S0, dS=dS)
    for a, b in zip(gla[:4], sc[:4]):
        assert np.allclose(a, b, rtol=0, atol=1e-12)
    assert np.allclose(gla[4].sum(-1), sc[4], rtol=0, atol=1e-12)  # dg summed over the shared channels
