"""The chunked form of the Kimi Delta Attention backward that the GPU path
computes (per chunk: the WY form with the per-channel gate folded around the
chunk's midpoint row; the gradients read off line by line, with the log-gate
gradient taken through the exponentials), restated in float64 numpy and
checked against the float64 delta-rule backward oracle, which differentiates
the token recurrence one step at a time. CPU only; a mistake planted in the
chunk form is caught."""
import numpy as np
import pytest

from oracle.backward_delta import backward_delta


def _chunk_form(q, k, v, dO, g, beta, S0, dS, C, plant=None):
    T, dk = q.shape
    mid = C // 2 - 1
    nch = (T + C - 1) // C
    dq, dkk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dbeta, dg = np.zeros(T), np.zeros_like(g)

    def chunk(i):
        t0, n = i * C, min(C, T - i * C)
        pad = lambda x: np.concatenate([x[t0:t0 + n], np.zeros((C - n,) + x.shape[1:])])
        qc, kc, vc, oc, gc, bc = (pad(x) for x in (q, k, v, dO, g, beta))
        B = np.cumsum(gc, axis=0)
        return t0, n, qc, kc, vc, oc, bc, B, B[-1], B[mid]

    def wy(kc, bc, B, bm, S, vc):
        Kp, Km = kc * np.exp(B - bm), kc * np.exp(bm - B)
        L = np.tril(Kp @ Km.T, -1)
        Tm = np.linalg.inv(np.eye(C) + bc[:, None] * L)
        Z = vc - (kc * np.exp(B)) @ S
        return Kp, Km, L, Tm, Z, Tm @ (bc[:, None] * Z)

    states, S = [], S0.copy()
    for i in range(nch):  # the states entering every chunk
        _, _, _, kc, vc, _, bc, B, BL, bm = chunk(i)
        states.append(S)
        U = wy(kc, bc, B, bm, S, vc)[-1]
        S = np.exp(BL)[:, None] * S + (kc * np.exp(BL - B)).T @ U
    E = dS.copy()
    for i in reversed(range(nch)):
        t0, n, qc, kc, vc, oc, bc, B, BL, bm = chunk(i)
        S = states[i]
        Kp, Km, L, Tm, Z, U = wy(kc, bc, B, bm, S, vc)
        Qp, EP = qc * np.exp(B - bm), np.exp(B - bm)
        P = np.tril(Qp @ Km.T)
        Kt = kc * np.exp(BL - B)
        Y = Tm.T @ (Kt @ E + P.T @ oc)
        dZ = bc[:, None] * Y
        dA = -np.tril(Y @ U.T, -1)
        dL, dP = bc[:, None] * dA, np.tril(oc @ U.T)
        X1 = np.exp(bm) * (-dZ @ S.T) + dL @ Km
        UE = np.exp(BL - bm) * (U @ E.T)
        X2 = UE + dL.T @ Kp + dP.T @ Qp
        dqc = EP * (np.exp(bm) * (oc @ S.T) + dP @ Km)
        dB = qc * dqc + kc * (EP * X1 - X2 / EP)
        dB[-1] += np.sum(kc * UE / EP, 0) + np.exp(BL) * np.sum(S * E, 1)
        if plant == "last_row_decay_term_dropped":
            dB[-1] -= np.exp(BL) * np.sum(S * E, 1)
        sl = slice(t0, t0 + n)
        dq[sl], dkk[sl], dv[sl] = dqc[:n], (EP * X1 + X2 / EP)[:n], dZ[:n]
        dbeta[sl] = (np.sum(Y * Z, 1) + np.sum(dA * L, 1))[:n]
        dg[sl] = np.cumsum(dB[::-1], axis=0)[::-1][:n]
        E = np.exp(BL)[:, None] * E + (qc * np.exp(B)).T @ oc - (kc * np.exp(B)).T @ dZ
    return dq, dkk, dv, dbeta, dg, E


def _case(T, dk, dv, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((T, dk)) * 0.5, rng.standard_normal((T, dk)) * 0.5, rng.standard_normal((T, dv)),
            rng.standard_normal((T, dv)), -np.abs(rng.standard_normal((T, dk))) * 0.3, rng.uniform(0.1, 0.9, T),
            rng.standard_normal((dk, dv)) * 0.3, rng.standard_normal((dk, dv)))


@pytest.mark.parametrize("T,dk,dv,C", [(7, 3, 4, 4), (21, 5, 6, 8), (100, 8, 8, 16), (130, 16, 8, 64)])
def test_chunk_form_matches_the_token_recurrence(T, dk, dv, C):
    q, k, v, dO, g, beta, S0, dS = _case(T, dk, dv, T)
    ref = backward_delta(*(x[None, None] for x in (q, k, v, dO)), "kda", g=g[None, None], beta=beta[None, None],
                         S0=S0[None, None], dS=dS[None, None])
    got = _chunk_form(q, k, v, dO, g, beta, S0, dS, C)
    for a, r in zip(got, ref):
        assert np.allclose(a, r[0, 0], rtol=1e-10, atol=1e-12)


def test_a_planted_mistake_in_the_chunk_form_is_caught():
    q, k, v, dO, g, beta, S0, dS = _case(40, 6, 5, 1)
    ref = backward_delta(*(x[None, None] for x in (q, k, v, dO)), "kda", g=g[None, None], beta=beta[None, None],
                         S0=S0[None, None], dS=dS[None, None])
    got = _chunk_form(q, k, v, dO, g, beta, S0, dS, 16, plant="last_row_decay_term_dropped")
    assert not np.allclose(got[4], ref[4][0, 0], rtol=1e-6, atol=1e-8)
