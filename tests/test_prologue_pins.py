"""Pins of the prologue oracle (short convolution, L2 normalisation, gate and
write-strength activations) to results fixed independently of its code:
special weights that reduce the convolution to the identity or a shift,
numpy's own 1-D convolution, the unit-norm invariant, scipy's logistic
functions, closed-form values, and split-call invariance of the history.
The last test plants mistakes in copies of the oracle's steps and checks that
the pins catch them. CPU only.
"""
import numpy as np
import pytest

from oracle import prologue as P

RNG = np.random.default_rng(77)


def _x(B=2, H=3, T=19, d=8):
    return RNG.standard_normal((B, H, T, d))


def test_conv_with_unit_current_weight_is_identity():
    x = _x()
    w = np.zeros((3, 8, 4))
    w[..., 0] = 1.0
    y, _ = P.short_conv(x, w)
    assert np.array_equal(y, x)


def test_conv_with_unit_lag_weight_is_a_shift():
    x = _x()
    for lag in (1, 2, 3):
        w = np.zeros((3, 8, 4))
        w[..., lag] = 1.0
        y, _ = P.short_conv(x, w)
        assert np.array_equal(y[:, :, lag:], x[:, :, :-lag])
        assert np.array_equal(y[:, :, :lag], np.zeros_like(y[:, :, :lag]))


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_conv_equals_numpy_convolve_per_channel(K):
    x = _x(T=23)
    w = RNG.standard_normal((3, 8, K))
    y, _ = P.short_conv(x, w)
    for b in range(2):
        for h in range(3):
            for c in range(8):
                # full causal convolution, truncated to the sequence length
                ref = np.convolve(x[b, h, :, c], w[h, c, :])[: x.shape[2]]
                assert np.allclose(y[b, h, :, c], ref, rtol=0, atol=1e-12)


def test_conv_history_gives_split_call_invariance():
    x = _x(T=30)
    w = RNG.standard_normal((3, 8, 4))
    y_all, h_all = P.short_conv(x, w)
    for t1 in (1, 2, 3, 7, 29):
        y1, h1 = P.short_conv(x[:, :, :t1], w)
        y2, h2 = P.short_conv(x[:, :, t1:], w, h1)
        assert np.allclose(np.concatenate([y1, y2], axis=2), y_all, rtol=0, atol=1e-12)
        assert np.array_equal(h2, h_all)
    # the history is the last K-1 raw rows
    assert np.array_equal(h_all, x[:, :, -3:])


def test_history_shorter_call_than_window():
    x = _x(T=2)
    w = RNG.standard_normal((3, 8, 4))
    hist = RNG.standard_normal((2, 3, 3, 8))
    y, h = P.short_conv(x, w, hist)
    full = np.concatenate([hist, x], axis=2)
    assert np.array_equal(h, full[:, :, -3:])
    ref = sum(w[None, :, None, :, tau] * full[:, :, 3 - tau:5 - tau] for tau in range(4))
    assert np.allclose(y, ref, rtol=0, atol=1e-12)


def test_l2norm_unit_norm_and_direction():
    x = _x(d=64)
    y = P.l2norm(x)
    assert np.allclose(np.linalg.norm(y, axis=-1), 1.0, rtol=0, atol=1e-13)
    # same direction: y is a positive multiple of x
    ratio = y / x
    assert np.allclose(ratio, ratio[..., :1], rtol=1e-12, atol=0)
    assert np.all(ratio > 0)
    assert np.array_equal(P.l2norm(np.zeros((2, 4))), np.zeros((2, 4)))


def test_gate_activations_against_scipy():
    sp = pytest.importorskip("scipy.special")
    a = np.concatenate([RNG.standard_normal(1000) * 4, [-80.0, -30.0, 0.0, 30.0, 80.0]])
    for tau in (1.0, 8.0, 16.0):
        assert np.allclose(P.gate_activation(a, "logsigmoid", tau), sp.log_expit(a) / tau,
                           rtol=1e-13, atol=1e-15)
        assert np.allclose(P.gate_activation(a, "neg_softplus", tau), -np.logaddexp(0.0, a) / tau,
                           rtol=1e-13, atol=1e-15)
    assert np.allclose(P.beta_activation(a), sp.expit(a), rtol=1e-13, atol=1e-300)


def test_activation_closed_forms():
    assert P.gate_activation(0.0, "logsigmoid", 2.0) == pytest.approx(-np.log(2.0) / 2.0, abs=1e-15)
    assert P.gate_activation(0.0, "neg_softplus", 8.0) == pytest.approx(-np.log(2.0) / 8.0, abs=1e-15)
    assert P.beta_activation(0.0) == 0.5
    # alpha = exp(g) is in (0, 1) for both kinds
    a = RNG.standard_normal(500) * 10
    for kind in ("logsigmoid", "neg_softplus"):
        g = P.gate_activation(a, kind, 4.0)
        assert np.all(g < 0) and np.all(np.isfinite(g))


def test_prologue_composes_the_steps():
    xq, xk, xv = _x(d=8), _x(d=8), _x(d=6)
    wq, wk = RNG.standard_normal((3, 8, 3)), RNG.standard_normal((3, 8, 3))
    a_g, a_b = RNG.standard_normal((2, 3, 19, 8)), RNG.standard_normal((2, 3, 19))
    out = P.prologue(xq, xk, xv, wq, wk, None, l2q=True, l2k=True, a_gate=a_g,
                     gate_kind="logsigmoid", tau=16.0, a_beta=a_b)
    assert np.allclose(out["q"], P.l2norm(P.short_conv(xq, wq)[0]), rtol=0, atol=1e-14)
    assert np.allclose(out["k"], P.l2norm(P.short_conv(xk, wk)[0]), rtol=0, atol=1e-14)
    assert np.array_equal(out["v"], xv)  # no weights: identity
    assert np.array_equal(out["hist"]["v"], xv[:, :, -2:])


def test_planted_mistakes_are_caught():
    """Each plausible slip in the convolution fails one of the pins above."""
    x = _x(T=12)
    w = RNG.standard_normal((3, 8, 4))

    def conv_wrong_orientation(x, w):  # w[tau] applied to x_{t+tau-(K-1)} (flipped kernel)
        return P.short_conv(x, w[..., ::-1])[0]

    def conv_off_by_one(x, w):  # the window skips the current token
        y = np.zeros_like(x)
        for tau in range(4):
            y[:, :, tau + 1:] += w[None, :, None, :, tau] * x[:, :, : x.shape[2] - tau - 1]
        return y

    ref = np.stack([[[np.convolve(x[b, h, :, c], w[h, c])[:12] for c in range(8)]
                     for h in range(3)] for b in range(2)]).transpose(0, 1, 3, 2)
    assert np.allclose(P.short_conv(x, w)[0], ref, atol=1e-12)
    for bad in (conv_wrong_orientation, conv_off_by_one):
        assert not np.allclose(bad(x, w), ref, atol=1e-6)
    # gate slips: the sigmoid's argument negated, the softplus's sign dropped
    a = RNG.standard_normal(200) * 3
    sp = pytest.importorskip("scipy.special")
    assert not np.allclose(-P._softplus(a) / 4.0, sp.log_expit(a) / 4.0, atol=1e-6)
    assert not np.all(P._softplus(a) / 4.0 < 0)
