"""Pins of the oracle's outer-product-gate mode ("outer": S_t = (alpha_t
beta_t^T) ⊙ S_{t-1} + k_t v_t^T, the gate form "Talk Linear Attention"
section 5.4 gives for gated linear attention that stays a matrix product) to
results fixed independently of its code: the key-axis-only case is the GLA
recurrence bit for bit, the value-axis-only case splits into one
scalar-decay linear attention per value column, and a brute-force sum over
tokens with explicit gate products gives every output. The last test plants
mistakes (axes exchanged, decay after the write, one axis dropped) and checks
that the pins catch them. CPU only.
"""
import numpy as np
import pytest

from oracle import forms, recurrence

RNG = np.random.default_rng(2024)


def _inputs(B=2, H=2, T=23, dk=5, dv=4, gate=0.2):
    q = RNG.standard_normal((B, H, T, dk)) * 0.5
    k = RNG.standard_normal((B, H, T, dk)) * 0.5
    v = RNG.standard_normal((B, H, T, dv))
    la = -np.abs(RNG.standard_normal((B, H, T, dk))) * gate   # log alpha, key axis
    lb = -np.abs(RNG.standard_normal((B, H, T, dv))) * gate   # log beta, value axis
    S0 = RNG.standard_normal((B, H, dk, dv)) * 0.3
    return q, k, v, la, lb, S0


def _brute(q, k, v, la, lb, S0):
    """o_t[j] = sum_c q_t[c] ( prod_{tau<=t} a_tau[c] b_tau[j] S0[c, j]
                + sum_{s<=t} prod_{s<tau<=t} a_tau[c] b_tau[j] k_s[c] v_s[j] ),
    written as explicit products of the gates over the covered tokens."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, H, T, dv))
    S = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            a = np.exp(la[b, h])  # [T, dk]
            be = np.exp(lb[b, h])  # [T, dv]
            for t in range(T + 1):
                st = np.zeros((dk, dv))
                for c in range(dk):
                    for j in range(dv):
                        w0 = 1.0
                        for tau in range(t):
                            w0 *= a[tau, c] * be[tau, j]
                        acc = w0 * S0[b, h, c, j]
                        for s in range(t):
                            w = 1.0
                            for tau in range(s + 1, t):
                                w *= a[tau, c] * be[tau, j]
                            acc += w * k[b, h, s, c] * v[b, h, s, j]
                        st[c, j] = acc
                if t > 0:
                    o[b, h, t - 1] = st.T @ q[b, h, t - 1]
                if t == T:
                    S[b, h] = st
    return o, S


def test_outer_with_unit_value_gate_is_gla_exactly():
    q, k, v, la, lb, S0 = _inputs()
    o1, S1 = recurrence(q, k, v, "outer", g=la, beta=np.zeros_like(lb), S0=S0)
    o2, S2 = recurrence(q, k, v, "gla", g=la, S0=S0)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)


def test_outer_with_unit_key_gate_is_a_scalar_decay_per_value_column():
    q, k, v, la, lb, S0 = _inputs()
    o, S = recurrence(q, k, v, "outer", g=np.zeros_like(la), beta=lb, S0=S0)
    for j in range(v.shape[-1]):
        oj, Sj = recurrence(q, k, v[..., j:j + 1], "scalar", g=lb[..., j], S0=S0[..., j:j + 1])
        assert np.allclose(o[..., j:j + 1], oj, rtol=0, atol=1e-13)
        assert np.allclose(S[..., j:j + 1], Sj, rtol=0, atol=1e-13)


def test_outer_equals_brute_force_sum():
    q, k, v, la, lb, S0 = _inputs(B=1, H=2, T=9, dk=3, dv=4, gate=0.4)
    o, S = recurrence(q, k, v, "outer", g=la, beta=lb, S0=S0)
    ob, Sb = _brute(q, k, v, la, lb, S0)
    assert np.allclose(o, ob, rtol=0, atol=1e-12)
    assert np.allclose(S, Sb, rtol=0, atol=1e-12)


@pytest.mark.parametrize("C", [1, 7, 16, 64])
def test_outer_chunk_form_with_extreme_value_gates(C):
    """The chunk form (value columns divided by their prefix decay, output
    multiplied back) holds for strong and uneven value-axis decay."""
    q, k, v, la, lb, S0 = _inputs(B=1, H=1, T=150, dk=6, dv=5, gate=0.3)
    lb[..., 2] *= 8.0  # one value column decays ~e^-2 per token
    o, S = recurrence(q, k, v, "outer", g=la, beta=lb, S0=S0)
    oc, Sc = forms.chunk_form(q[0, 0], k[0, 0], v[0, 0], "outer", g=la[0, 0], beta=lb[0, 0], S0=S0[0, 0], C=C)
    assert np.allclose(oc, o[0, 0], rtol=0, atol=1e-10)
    assert np.allclose(Sc, S[0, 0], rtol=0, atol=1e-10)


def test_outer_pins_detect_planted_mistakes():
    q, k, v, la, lb, S0 = _inputs(B=1, H=1, T=9, dk=4, dv=4, gate=0.4)
    ob, Sb = _brute(q, k, v, la, lb, S0)

    def passes(o, S):
        return np.allclose(o, ob, rtol=0, atol=1e-9) and np.allclose(S, Sb, rtol=0, atol=1e-9)

    assert passes(*recurrence(q, k, v, "outer", g=la, beta=lb, S0=S0))
    # the two axes exchanged (alpha on the value axis, beta on the key axis)
    assert not passes(*recurrence(q, k, v, "outer", g=lb, beta=la, S0=S0))
    # one axis dropped
    assert not passes(*recurrence(q, k, v, "gla", g=la, S0=S0))
    assert not passes(*recurrence(q, k, v, "outer", g=np.zeros_like(la), beta=lb, S0=S0))
    # the gate of the next token (off by one in time)
    assert not passes(*recurrence(q, k, v, "outer", g=np.roll(la, -1, axis=2), beta=lb, S0=S0))

    # the decay applied after the write: S <- G ⊙ (S + k v^T)
    def decay_after_write():
        S = S0[0, 0].copy()
        o = np.zeros((9, 4))
        for t in range(9):
            G = np.exp(la[0, 0, t])[:, None] * np.exp(lb[0, 0, t])[None, :]
            S = G * (S + np.outer(k[0, 0, t], v[0, 0, t]))
            o[t] = S.T @ q[0, 0, t]
        return o[None, None], S[None, None]

    assert not passes(*decay_after_write())
