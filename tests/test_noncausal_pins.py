"""Pins of the non-causal oracle (O = Q (K^T V), and its elu+1 normalised
form) to statements computed another way: the left-to-right product with the
full n x n score matrix (kernel-attention notes, section 3: the two orders
agree when there is no softmax), explicit normalised sums over all tokens,
the causal recurrence (its final state, and its output at the last token,
which already sees every token), and constant-v invariance. The last test
plants mistakes and checks that the pins catch them. CPU only.
"""
import numpy as np
import pytest

from oracle import recurrence
from oracle.noncausal import noncausal
from oracle.recurrence import phi_elu1

RNG = np.random.default_rng(31)


def _qkv(B=2, H=2, T=23, dk=6, dv=5, scale=0.5):
    return (RNG.standard_normal((B, H, T, dk)) * scale, RNG.standard_normal((B, H, T, dk)) * scale,
            RNG.standard_normal((B, H, T, dv)))


def test_linear_equals_left_to_right_product():
    q, k, v = _qkv()
    S0 = RNG.standard_normal((2, 2, 6, 5)) * 0.3
    o, S = noncausal(q, k, v, "linear", S0=S0)
    for b in range(2):
        for h in range(2):
            scores = q[b, h] @ k[b, h].T          # n x n, no mask
            ref = scores @ v[b, h] + q[b, h] @ S0[b, h]
            assert np.allclose(o[b, h], ref, rtol=0, atol=1e-12)


def test_elu1_equals_explicit_normalised_sums():
    q, k, v = _qkv(T=17)
    o, S = noncausal(q, k, v, "elu1")
    qh, kh = phi_elu1(q), phi_elu1(k)
    for b in range(2):
        for h in range(2):
            for i in range(17):
                w = np.array([qh[b, h, i] @ kh[b, h, j] for j in range(17)])
                ref = (w[:, None] * v[b, h]).sum(0) / w.sum()
                assert np.allclose(o[b, h, i], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mode", ["linear", "elu1"])
def test_final_state_and_last_token_match_the_causal_recurrence(mode):
    q, k, v = _qkv(T=31)
    W = 5 + (1 if mode == "elu1" else 0)
    S0 = RNG.standard_normal((2, 2, 6, W)) * 0.2
    if mode == "elu1":
        S0[..., 5] = np.abs(S0[..., 5]) + 1.0
    o_nc, S_nc = noncausal(q, k, v, mode, S0=S0)
    o_c, S_c = recurrence(q, k, v, mode, S0=S0)
    assert np.allclose(S_nc, S_c, rtol=0, atol=1e-12)
    assert np.allclose(o_nc[:, :, -1], o_c[:, :, -1], rtol=1e-12, atol=1e-12)


def test_elu1_constant_values_give_that_constant():
    q, k, _ = _qkv(T=40)
    v = np.full((2, 2, 40, 5), 2.5)
    o, _ = noncausal(q, k, v, "elu1")
    assert np.allclose(o, 2.5, rtol=0, atol=1e-12)


def test_planted_mistakes_are_caught():
    q, k, v = _qkv(T=12)
    o, _ = noncausal(q, k, v, "linear")
    ref = np.einsum("bhij,bhjv->bhiv", np.einsum("bhic,bhjc->bhij", q, k), v)
    assert np.allclose(o, ref, atol=1e-12)
    causal, _ = recurrence(q, k, v, "linear")          # a mask left in
    swapped = np.einsum("bhij,bhjv->bhiv", np.einsum("bhic,bhjc->bhij", k, q), v)  # q and k swapped
    for bad in (causal, swapped):
        assert not np.allclose(bad, ref, atol=1e-6)
