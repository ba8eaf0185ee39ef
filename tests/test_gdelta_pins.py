"""Pins of the generalised-delta-rule oracle (S_t = (I - b_t a_t^T) S_{t-1} +
k_t v_t^T in key-major form, "Talk Linear Attention" section 7.1) to results
fixed independently of its code: the page's own DeltaNet special case
(a = b = sqrt(beta) k, with beta k as the write key, is the separately pinned
DeltaNet recurrence), zero a or b (plain linear attention), a Kronecker-product
brute force on the vectorised value-major state exactly as the page writes it,
the chunkwise (WY-style) form at several chunk lengths, and split calls. The
last test plants mistakes (a and b exchanged, the erase before the retrieval
of the same step, the write dropped from the retrieval) and checks that the
pins catch them. CPU only.
"""
import numpy as np
import pytest

from oracle import recurrence
from oracle.gdelta import chunk_form_gdelta, recurrence_gdelta

RNG = np.random.default_rng(31)


def _inputs(B=2, H=2, T=37, dk=6, dv=5, scale=0.4):
    q = RNG.standard_normal((B, H, T, dk)) * scale
    k = RNG.standard_normal((B, H, T, dk)) * scale
    v = RNG.standard_normal((B, H, T, dv))
    a = RNG.standard_normal((B, H, T, dk)) * scale
    b = RNG.standard_normal((B, H, T, dk)) * scale
    S0 = RNG.standard_normal((B, H, dk, dv)) * 0.3
    return q, k, v, a, b, S0


def _kron_value_major(q, k, v, a, b, S0):
    """The page's form on the value-major state Sv [dv, dk]: Sv <- Sv (I - a b^T)
    + v k^T, o = Sv q, vectorised: vec(Sv M) = (M^T ⊗ I_dv) vec(Sv)."""
    T, dk = q.shape
    dv = v.shape[1]
    s = np.asarray(S0).T.reshape(-1, order="F")  # vec of Sv = S0^T
    o = np.zeros((T, dv))
    for t in range(T):
        M = np.eye(dk) - np.outer(a[t], b[t])
        s = np.kron(M.T, np.eye(dv)) @ s + np.outer(v[t], k[t]).reshape(-1, order="F")
        Sv = s.reshape(dv, dk, order="F")
        o[t] = Sv @ q[t]
    return o, s.reshape(dv, dk, order="F").T  # back to key-major


def test_gdelta_with_a_equal_b_is_deltanet():
    q, k, v, _, _, S0 = _inputs()
    kn = k / np.linalg.norm(k, axis=-1, keepdims=True)
    beta = 1.0 / (1.0 + np.exp(-RNG.standard_normal(kn.shape[:3])))
    ab = np.sqrt(beta)[..., None] * kn
    o, S = recurrence_gdelta(q, beta[..., None] * kn, v, ab, ab, S0)
    o_ref, S_ref = recurrence(q, kn, v, "gdn", beta=beta, S0=S0)
    assert np.allclose(o, o_ref, rtol=0, atol=1e-12)
    assert np.allclose(S, S_ref, rtol=0, atol=1e-12)


def test_gdelta_without_erase_is_linear_attention():
    q, k, v, a, b, S0 = _inputs()
    o_ref, S_ref = recurrence(q, k, v, "linear", S0=S0)
    for a_, b_ in ((np.zeros_like(a), b), (a, np.zeros_like(b))):
        o, S = recurrence_gdelta(q, k, v, a_, b_, S0)
        assert np.allclose(o, o_ref, rtol=0, atol=1e-13)
        assert np.allclose(S, S_ref, rtol=0, atol=1e-13)


def test_gdelta_equals_value_major_kronecker_brute_force():
    q, k, v, a, b, S0 = _inputs(B=1, H=2, T=11, dk=4, dv=3, scale=0.6)
    o, S = recurrence_gdelta(q, k, v, a, b, S0)
    for h in range(2):
        ob, Sb = _kron_value_major(q[0, h], k[0, h], v[0, h], a[0, h], b[0, h], S0[0, h])
        assert np.allclose(o[0, h], ob, rtol=0, atol=1e-12)
        assert np.allclose(S[0, h], Sb, rtol=0, atol=1e-12)


@pytest.mark.parametrize("C", [1, 5, 16, 64, "T"])
def test_gdelta_chunk_form_matches_recurrence(C):
    q, k, v, a, b, S0 = _inputs(B=1, H=1, T=150, dk=8, dv=6, scale=0.3)
    o, S = recurrence_gdelta(q, k, v, a, b, S0)
    oc, Sc = chunk_form_gdelta(q[0, 0], k[0, 0], v[0, 0], a[0, 0], b[0, 0], S0[0, 0],
                               C=150 if C == "T" else C)
    scale = max(1.0, np.abs(o).max())
    assert np.max(np.abs(oc - o[0, 0])) / scale <= 1e-10
    assert np.max(np.abs(Sc - S[0, 0])) / max(1.0, np.abs(S).max()) <= 1e-10


@pytest.mark.parametrize("T1", [64, 37])
def test_gdelta_split_call_invariance(T1):
    q, k, v, a, b, S0 = _inputs(T=100)
    o, S = recurrence_gdelta(q, k, v, a, b, S0)
    sl = lambda x, i, j: x[:, :, i:j]
    o1, S1 = recurrence_gdelta(sl(q, 0, T1), sl(k, 0, T1), sl(v, 0, T1), sl(a, 0, T1), sl(b, 0, T1), S0)
    o2, S2 = recurrence_gdelta(sl(q, T1, 100), sl(k, T1, 100), sl(v, T1, 100), sl(a, T1, 100), sl(b, T1, 100), S1)
    assert np.allclose(np.concatenate([o1, o2], axis=2), o, rtol=0, atol=1e-12)
    assert np.allclose(S2, S, rtol=0, atol=1e-12)


def test_gdelta_pins_detect_planted_mistakes():
    q, k, v, a, b, S0 = _inputs(B=1, H=1, T=11, dk=4, dv=3, scale=0.6)
    ob, Sb = _kron_value_major(q[0, 0], k[0, 0], v[0, 0], a[0, 0], b[0, 0], S0[0, 0])

    def passes(o, S):
        return np.allclose(o[0, 0], ob, rtol=0, atol=1e-9) and np.allclose(S[0, 0], Sb, rtol=0, atol=1e-9)

    assert passes(*recurrence_gdelta(q, k, v, a, b, S0))
    assert not passes(*recurrence_gdelta(q, k, v, b, a, S0))          # a and b exchanged

    def variant(order):
        S = S0[0, 0].copy()
        o = np.zeros((11, 3))
        for t in range(11):
            at, bt, kt, vt = a[0, 0, t], b[0, 0, t], k[0, 0, t], v[0, 0, t]
            if order == "write_first":     # the write joins the retrieved value
                S = S + np.outer(kt, vt)
                S = S - np.outer(bt, at @ S)
            else:                          # the erase scaled by the wrong side
                S = S - np.outer(at, bt @ S) + np.outer(kt, vt)
            o[t] = S.T @ q[0, 0, t]
        return o[None, None], S[None, None]

    assert not passes(*variant("write_first"))
    assert not passes(*variant("transposed_erase"))
