"""Pins of the float64 oracle to what the pages and the mathematics fix.

Each test compares the oracle's recurrence with a *different* statement of
the same computation (a quadratic masked product, an explicit normalised
sum, the four-step DeltaNet memory update, a Kronecker-product brute force,
the chunkwise form at its C=1 / C=T limits), with a closed form, with an
exact invariant, or with golden values built from the pages' recall
examples. The last test plants mistakes in the oracle's use and checks that
the pins catch them. CPU only.
"""
import os

import numpy as np
import pytest

import oracle
from oracle import forms, recurrence, recurrence_c

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def _rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


def _heads(B, H, T, dk, dv, scale=0.5):
    return _rand(B, H, T, dk, scale=scale), _rand(B, H, T, dk, scale=scale), _rand(B, H, T, dv)


def _close(a, b, tol):
    a, b = np.asarray(a), np.asarray(b)
    assert a.shape == b.shape, (a.shape, b.shape)
    err = np.max(np.abs(a - b)) / max(1.0, np.max(np.abs(b)))
    assert err <= tol, f"max scaled error {err:.3e} > {tol:.1e}"


# --- plain linear attention -------------------------------------------------

def test_linear_equals_quadratic_parallel_form():
    q, k, v = _heads(2, 2, 48, 8, 5)
    o, S = recurrence(q, k, v, "linear")
    for b in range(2):
        for h in range(2):
            O_par, S_closed = forms.parallel_linear(q[b, h], k[b, h], v[b, h])
            _close(o[b, h], O_par, 1e-12)
            _close(S[b, h], S_closed, 1e-12)


# --- decayed / gated forms ---------------------------------------------------

@pytest.mark.parametrize("mode", ["retnet", "scalar", "gla"])
def test_gated_equals_decay_masked_parallel_form(mode):
    B, H, T, dk, dv = 2, 3, 32, 6, 4
    q, k, v = _heads(B, H, T, dk, dv)
    if mode == "retnet":
        g = np.log1p(-(2.0 ** (-5.0 - np.arange(H)))) * 4.0
    elif mode == "scalar":
        g = -np.abs(_rand(B, H, T, scale=0.3))
    else:
        g = -np.abs(_rand(B, H, T, dk, scale=0.3))
    o, S = recurrence(q, k, v, mode, g=g)
    for b in range(B):
        for h in range(H):
            if mode == "retnet":
                la = np.full(T, g[h])
            else:
                la = g[b, h]
            O_par, S_par = forms.parallel_gated(q[b, h], k[b, h], v[b, h], la)
            _close(o[b, h], O_par, 1e-11)
            _close(S[b, h], S_par, 1e-11)


def test_retnet_with_gamma_one_is_linear():
    q, k, v = _heads(1, 2, 20, 4, 3)
    o1, S1 = recurrence(q, k, v, "retnet", g=np.zeros(2))
    o2, S2 = recurrence(q, k, v, "linear")
    _close(o1, o2, 1e-14)
    _close(S1, S2, 1e-14)


# --- elu+1 normalised attention ---------------------------------------------

def test_elu1_equals_explicit_normalised_sum():
    q, k, v = _heads(1, 2, 40, 6, 5, scale=1.0)
    o, S = recurrence(q, k, v, "elu1")
    for h in range(2):
        o_ref, S_ref, z_ref = forms.normalised_sum(q[0, h], k[0, h], v[0, h])
        _close(o[0, h], o_ref, 1e-12)
        _close(S[0, h, :, :5], S_ref, 1e-12)
        _close(S[0, h, :, 5], z_ref, 1e-12)


def test_elu1_feature_map_values():
    # elu(x)+1 at hand-checked points: x+1 for x>0, exp(x) for x<=0.
    x = np.array([-2.0, -0.5, 0.0, 0.25, 3.0])
    want = np.array([np.exp(-2.0), np.exp(-0.5), 1.0, 1.25, 4.0])
    np.testing.assert_allclose(oracle.phi_elu1(x), want, rtol=0, atol=1e-15)


def test_elu1_constant_values_give_constant_output():
    # A normalised convex combination of identical values returns that value.
    q, k, _ = _heads(1, 1, 30, 5, 3, scale=1.0)
    v = np.ones((1, 1, 30, 3)) * 2.5
    o, _ = recurrence(q, k, v, "elu1")
    np.testing.assert_allclose(o, 2.5, rtol=1e-13)


# --- gated delta rule --------------------------------------------------------

@pytest.mark.parametrize("gated", [False, True])
def test_gdn_equals_deltanet_four_step(gated):
    B, H, T, dk, dv = 1, 2, 40, 6, 5
    q, k, v = _heads(B, H, T, dk, dv)
    k = k / np.linalg.norm(k, axis=-1, keepdims=True)
    beta = 1.0 / (1.0 + np.exp(-_rand(B, H, T)))
    g = -np.abs(_rand(B, H, T, scale=0.2)) if gated else None
    S0 = _rand(B, H, dk, dv, scale=0.3)
    o, S = recurrence(q, k, v, "gdn", g=g, beta=beta, S0=S0)
    for h in range(H):
        o_ref, S_ref = forms.deltanet_four_step(q[0, h], k[0, h], v[0, h], beta[0, h], S0[0, h],
                                                None if g is None else g[0, h])
        _close(o[0, h], o_ref, 1e-12)
        _close(S[0, h], S_ref, 1e-12)


def test_gdn_equals_kronecker_brute_force():
    B, H, T, dk, dv = 1, 1, 6, 4, 3
    q, k, v = _heads(B, H, T, dk, dv)
    beta = 1.0 / (1.0 + np.exp(-_rand(B, H, T)))
    g = -np.abs(_rand(B, H, T, scale=0.3))
    S0 = _rand(B, H, dk, dv, scale=0.5)
    o, S = recurrence(q, k, v, "gdn", g=g, beta=beta, S0=S0)
    o_ref, S_ref = forms.kronecker_delta(q[0, 0], k[0, 0], v[0, 0], beta[0, 0], S0[0, 0], g[0, 0])
    _close(o[0, 0], o_ref, 1e-12)
    _close(S[0, 0], S_ref, 1e-12)


def test_gdn_without_gate_is_deltanet_and_zero_gate_matches():
    q, k, v = _heads(1, 1, 25, 4, 4)
    beta = np.full((1, 1, 25), 0.7)
    o1, S1 = recurrence(q, k, v, "gdn", g=None, beta=beta)
    o2, S2 = recurrence(q, k, v, "gdn", g=np.zeros((1, 1, 25)), beta=beta)
    _close(o1, o2, 1e-15)
    _close(S1, S2, 1e-15)
    o3, S3 = recurrence(q, k, v, "gdn", g=None, beta=None)
    o4, S4 = recurrence(q, k, v, "gdn", g=None, beta=np.ones((1, 1, 25)))
    _close(o3, o4, 1e-15)


def test_gdn_exact_retrieval_with_orthonormal_keys():
    # beta = 1, alpha = 1, S0 = 0, keys = rows of a random orthogonal matrix:
    # every stored value is read back exactly by its key.
    dk = dv = 8
    Qm, _ = np.linalg.qr(_rand(dk, dk))
    keys = Qm.T                                      # orthonormal rows
    vals = _rand(dk, dv)
    k = keys[None, None]
    v = vals[None, None]
    q = np.zeros_like(k)
    _, S = recurrence(q, k, v, "gdn", beta=np.ones((1, 1, dk)))
    _close(keys @ S[0, 0], vals, 1e-12)


def test_gdn_beta_one_overwrites_repeated_key():
    dk = dv = 4
    e = np.eye(dk)
    k = np.stack([e[0], e[1], e[0]])[None, None]
    v = np.stack([np.full(dv, 1.0), np.full(dv, 2.0), np.full(dv, 3.0)])[None, None]
    _, S = recurrence(np.zeros_like(k), k, v, "gdn", beta=np.ones((1, 1, 3)))
    np.testing.assert_allclose(S[0, 0].T @ e[0], 3.0, atol=1e-15)
    _, S_lin = recurrence(np.zeros_like(k), k, v, "linear")
    np.testing.assert_allclose(S_lin[0, 0].T @ e[0], 4.0, atol=1e-15)


# --- Kimi Delta Attention (per-key-channel gate) --------------------------------

def _kda_case(T=7, dk=4, dv=3):
    q, k, v = _heads(1, 1, T, dk, dv)
    beta = 1.0 / (1.0 + np.exp(-_rand(1, 1, T)))
    g = -np.abs(_rand(1, 1, T, dk, scale=0.4))
    S0 = _rand(1, 1, dk, dv, scale=0.5)
    return q, k, v, g, beta, S0


def test_kda_equals_kronecker_brute_force():
    # the page's product S_t = (I - beta k k^T) Diag(alpha_t) S_{t-1} + beta k v^T
    q, k, v, g, beta, S0 = _kda_case()
    o, S = recurrence(q, k, v, "kda", g=g, beta=beta, S0=S0)
    o_ref, S_ref = forms.kronecker_delta(q[0, 0], k[0, 0], v[0, 0], beta[0, 0], S0[0, 0], g[0, 0])
    _close(o[0, 0], o_ref, 1e-12)
    _close(S[0, 0], S_ref, 1e-12)


def test_kda_with_equal_channel_gates_is_gdn():
    q, k, v, g, beta, S0 = _kda_case(T=20, dk=5, dv=4)
    gs = g[..., 0]                                    # one gate per token
    gk = np.repeat(gs[..., None], 5, axis=-1)         # ... given to every channel
    o1, S1 = recurrence(q, k, v, "kda", g=gk, beta=beta, S0=S0)
    o2, S2 = recurrence(q, k, v, "gdn", g=gs, beta=beta, S0=S0)
    _close(o1, o2, 1e-13)
    _close(S1, S2, 1e-13)


def test_kda_beta_zero_is_pure_channel_decay():
    # beta = 0 writes nothing: S_t = Diag(exp(sum_{s<=t} g_s)) S0 row by row
    q, k, v, g, _, S0 = _kda_case(T=9, dk=4, dv=3)
    o, S = recurrence(q, k, v, "kda", g=g, beta=np.zeros((1, 1, 9)), S0=S0)
    cum = np.cumsum(g[0, 0], axis=0)                  # [T, dk]
    for t in range(9):
        St = np.exp(cum[t])[:, None] * S0[0, 0]
        _close(o[0, 0, t], St.T @ q[0, 0, t], 1e-13)
    _close(S[0, 0], np.exp(cum[-1])[:, None] * S0[0, 0], 1e-13)


def test_kda_pins_detect_planted_mistakes():
    q, k, v, g, beta, S0 = _kda_case()
    o_ref, S_ref = forms.kronecker_delta(q[0, 0], k[0, 0], v[0, 0], beta[0, 0], S0[0, 0], g[0, 0])

    def passes(o, S):
        return np.max(np.abs(o[0, 0] - o_ref)) < 1e-10 and np.max(np.abs(S[0, 0] - S_ref)) < 1e-10

    assert passes(*recurrence(q, k, v, "kda", g=g, beta=beta, S0=S0))
    # channels of the gate permuted (a wrong index on the key axis)
    assert not passes(*recurrence(q, k, v, "kda", g=g[..., ::-1], beta=beta, S0=S0))
    # the gate of the next token (off by one in time)
    assert not passes(*recurrence(q, k, v, "kda", g=np.roll(g, -1, axis=2), beta=beta, S0=S0))
    # wrong sign of the delta correction
    assert not passes(*recurrence(q, k, v, "kda", g=g, beta=-beta, S0=S0))
    # unit write instead of the delta rule
    assert not passes(*recurrence(q, k, v, "gla", g=g, S0=S0))
    # one scalar gate per token (the channel structure dropped)
    assert not passes(*recurrence(q, k, v, "gdn", g=g.mean(-1), beta=beta, S0=S0))


# --- chunk form limits and chunk sizes ---------------------------------------

def _mode_inputs(mode, T, dk=8, dv=6, s0=True):
    q, k, v = _heads(1, 1, T, dk, dv)
    g = beta = None
    if mode == "retnet":
        g = np.array([np.log1p(-2.0 ** -3)])
    elif mode in ("scalar", "gdn"):
        g = -np.abs(_rand(1, 1, T, scale=0.15))
    elif mode in ("gla", "kda", "outer"):
        g = -np.abs(_rand(1, 1, T, dk, scale=0.05))
    if mode == "outer":  # value-axis log-gates ride in beta
        beta = -np.abs(_rand(1, 1, T, dv, scale=0.05))
    if mode in ("gdn", "kda"):
        k = k / np.linalg.norm(k, axis=-1, keepdims=True)
        beta = 1.0 / (1.0 + np.exp(-_rand(1, 1, T)))
    S0 = None
    if s0:
        S0 = _rand(1, 1, dk, dv + (mode == "elu1"), scale=0.3)
        if mode == "elu1":
            S0[..., dv] = np.abs(S0[..., dv]) + 1.0       # a valid positive normaliser
    return q, k, v, g, beta, S0


@pytest.mark.parametrize("mode", oracle.MODES)
@pytest.mark.parametrize("C", [1, 16, 64, "T"])
def test_chunk_form_matches_recurrence(mode, C):
    T = 150
    q, k, v, g, beta, S0 = _mode_inputs(mode, T)
    o, S = recurrence(q, k, v, mode, g=g, beta=beta, S0=S0)
    gh = None
    if g is not None:
        gh = g[0] if mode == "retnet" else g[0, 0]
    o_c, S_c = forms.chunk_form(q[0, 0], k[0, 0], v[0, 0], mode, g=gh,
                                beta=None if beta is None else beta[0, 0],
                                S0=None if S0 is None else S0[0, 0],
                                C=T if C == "T" else C)
    _close(o_c, o[0, 0], 1e-10)
    _close(S_c, S[0, 0], 1e-10)


# --- checkpoint / resume: the final state is the next call's initial state ---

@pytest.mark.parametrize("mode", oracle.MODES)
@pytest.mark.parametrize("T1", [64, 37])
def test_split_call_invariance(mode, T1):
    T = 100
    q, k, v, g, beta, S0 = _mode_inputs(mode, T)
    full_o, full_S = recurrence(q, k, v, mode, g=g, beta=beta, S0=S0)

    def part(a, b):
        sl = lambda x: None if x is None or mode == "retnet" and x is g else x[:, :, a:b]
        return recurrence(q[:, :, a:b], k[:, :, a:b], v[:, :, a:b], mode,
                          g=g if mode == "retnet" else sl(g), beta=sl(beta), S0=S_mid if a else S0)

    S_mid = None
    o1, S_mid = part(0, T1)
    o2, S2 = part(T1, T)
    _close(np.concatenate([o1, o2], axis=2), full_o, 1e-12)
    _close(S2, full_S, 1e-12)


# --- the C implementation computes the same recurrence ------------------------

@pytest.mark.parametrize("mode", oracle.MODES)
def test_c_oracle_matches_numpy(mode):
    B, H, T, dk, dv = 2, 3, 70, 8, 6
    q, k, v = _heads(B, H, T, dk, dv)
    g = beta = S0 = None
    if mode == "retnet":
        g = np.log1p(-(2.0 ** (-5.0 - np.arange(H))))
    elif mode in ("scalar", "gdn"):
        g = -np.abs(_rand(B, H, T, scale=0.1))
    elif mode in ("gla", "kda", "outer"):
        g = -np.abs(_rand(B, H, T, dk, scale=0.1))
    if mode in ("gdn", "kda"):
        beta = 1.0 / (1.0 + np.exp(-_rand(B, H, T)))
    if mode == "outer":
        beta = -np.abs(_rand(B, H, T, dv, scale=0.1))
    S0 = _rand(B, H, dk, dv + (mode == "elu1"), scale=0.2)
    if mode == "elu1":
        S0[..., dv] = np.abs(S0[..., dv]) + 1.0
    o1, S1 = recurrence(q, k, v, mode, g=g, beta=beta, S0=S0)
    o2, S2 = recurrence_c(q, k, v, mode, g=g, beta=beta, S0=S0, nthreads=3)
    _close(o2, o1, 1e-12)
    _close(S2, S1, 1e-12)


# --- golden values from the pages' recall examples ---------------------------

def _load_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _recall_tokens(rows):
    names = sorted({r[1] for r in rows})
    dk = len(names)
    T = len(rows)
    q = np.zeros((1, 1, T, dk))
    k = np.zeros((1, 1, T, dk))
    v = np.zeros((1, 1, T, 1))
    for t, r in enumerate(rows):
        key = np.eye(dk)[names.index(r[1])]
        if r[0] == "write":
            k[0, 0, t] = key
            v[0, 0, t, 0] = float(r[2])
        else:
            q[0, 0, t] = key
    return q, k, v


@pytest.mark.parametrize("name", ["recall_ids.txt", "recall_A4B3C6.txt"])
@pytest.mark.parametrize("impl", ["numpy", "c"])
def test_golden_recall(name, impl):
    rows = _load_golden(name)
    q, k, v = _recall_tokens(rows)
    run = recurrence if impl == "numpy" else recurrence_c
    for mode, kw in (("linear", {}), ("gdn", {"beta": np.ones(q.shape[:3])})):
        o, _ = run(q, k, v, mode, **kw)
        for t, r in enumerate(rows):
            if r[0] == "query":
                assert o[0, 0, t, 0] == float(r[2]), (mode, r, o[0, 0, t, 0])


@pytest.mark.parametrize("impl", ["numpy", "c"])
def test_golden_overwrite(impl):
    rows = _load_golden("recall_overwrite.txt")
    toks = [[r[0], r[1], r[2] if r[0] == "write" else "0"] for r in rows]
    q, k, v = _recall_tokens(toks)
    run = recurrence if impl == "numpy" else recurrence_c
    o_d, _ = run(q, k, v, "gdn", beta=np.ones(q.shape[:3]))
    o_l, _ = run(q, k, v, "linear")
    for t, r in enumerate(rows):
        if r[0] == "query":
            assert o_d[0, 0, t, 0] == float(r[3])
            assert o_l[0, 0, t, 0] == float(r[4])


# --- the pins catch plausible mistakes ---------------------------------------

def _pin_linear(run):
    q, k, v = _heads(1, 1, 24, 5, 4)
    o, S = run(q, k, v)
    O_par, S_closed = forms.parallel_linear(q[0, 0], k[0, 0], v[0, 0])
    return np.max(np.abs(o[0, 0] - O_par)) < 1e-10 and np.max(np.abs(S[0, 0] - S_closed)) < 1e-10


def _pin_delta(run):
    q, k, v = _heads(1, 1, 24, 5, 4)
    beta = np.full((1, 1, 24), 0.6)
    g = np.full((1, 1, 24), -0.1)
    o, S = run(q, k, v, g, beta)
    o_ref, S_ref = forms.deltanet_four_step(q[0, 0], k[0, 0], v[0, 0], beta[0, 0], None, g[0, 0])
    return np.max(np.abs(o[0, 0] - o_ref)) < 1e-10 and np.max(np.abs(S[0, 0] - S_ref)) < 1e-10


def test_pins_detect_planted_mistakes():
    # Correct use passes.
    assert _pin_linear(lambda q, k, v: recurrence(q, k, v, "linear"))
    assert _pin_delta(lambda q, k, v, g, b: recurrence(q, k, v, "gdn", g=g, beta=b))
    # Exclusive instead of inclusive causality (o_t reads S_{t-1}).
    def shifted(q, k, v):
        o, S = recurrence(q, k, v, "linear")
        o2 = np.zeros_like(o)
        o2[:, :, 1:] = o[:, :, :-1]
        return o2, S
    assert not _pin_linear(shifted)
    # Swapped roles of q and k.
    assert not _pin_linear(lambda q, k, v: recurrence(k, q, v, "linear"))
    # Wrong sign of the delta correction (beta negated).
    assert not _pin_delta(lambda q, k, v, g, b: recurrence(q, k, v, "gdn", g=g, beta=-b))
    # Decay dropped.
    assert not _pin_delta(lambda q, k, v, g, b: recurrence(q, k, v, "gdn", g=None, beta=b))
    # Decay applied twice as strong (a wrong gate index / log scale).
    assert not _pin_delta(lambda q, k, v, g, b: recurrence(q, k, v, "gdn", g=2 * g, beta=b))
    # Unit write instead of the delta rule.
    assert not _pin_delta(lambda q, k, v, g, b: recurrence(q, k, v, "scalar", g=g))
