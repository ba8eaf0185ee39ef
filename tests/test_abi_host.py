"""Host-side checks of the C ABI (no GPU needed).

The library must build, load, export every function include/la.h declares,
and reject bad arguments on the host before touching a device.
"""
import ctypes
import os
import re
import subprocess

import pytest

import gated_delta_rule_linear_gb300 as la
from gated_delta_rule_linear_gb300 import build as labuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "la.h")


@pytest.fixture(scope="module")
def lib():
    labuild.build()
    return la.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(la_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    assert names == sorted(["la_chunk_fwd", "la_chunk_fwd_noalloc", "la_chunk_fwd_gdelta", "la_chunk_bwd",
                            "la_chunk_bwd_delta", "la_recurrent_step", "la_prologue", "la_stream_status", "la_last_error",
                            "la_version"])
    assert set(names) == set(la.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", la.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (la_[a-z_]+)\b", out))
    for name in _declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_version(lib):
    assert la.la_version() == 10000


# Fake but aligned device addresses: validation must reject the call on the
# host before any of them is dereferenced or any CUDA call is made.
A = 0x10000


def _call(**kw):
    args = dict(q=A, k=A, v=A, g=None, beta=None, o=A, S0=None, S_final=None,
                B=1, H=1, T=64, dk=64, dv=64, C=0, mode=la.LA_LINEAR, stream=None)
    args.update(kw)
    rc = la.la_chunk_fwd(**args)
    return rc, la.la_last_error()


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), "LA_ERR_INVALID_ARG"),
    (dict(o=None), "LA_ERR_INVALID_ARG"),
    (dict(T=0), "LA_ERR_INVALID_ARG"),
    (dict(B=0), "LA_ERR_INVALID_ARG"),
    (dict(H=-1), "LA_ERR_INVALID_ARG"),
    (dict(dk=96), "LA_ERR_UNSUPPORTED"),
    (dict(dv=32), "LA_ERR_UNSUPPORTED"),
    (dict(C=32), "LA_ERR_INVALID_ARG"),
    (dict(C=128, mode=3, g=A), "LA_ERR_UNSUPPORTED"),  # C = 128: not for the per-channel gates
    (dict(C=128, mode=5), "LA_ERR_UNSUPPORTED"),       # ... nor the delta rule
    (dict(C=128, mode=6, g=A), "LA_ERR_UNSUPPORTED"),
    (dict(C=128, mode=7, g=A, beta=A), "LA_ERR_UNSUPPORTED"),
    (dict(C=128, mode=0x100), "LA_ERR_UNSUPPORTED"),   # ... nor float32
    (dict(mode=9), "LA_ERR_INVALID_ARG"),
    (dict(mode=0x400), "LA_ERR_INVALID_ARG"),          # unknown flag
    (dict(q=A + 8), "LA_ERR_INVALID_ARG"),            # 16-byte alignment
    (dict(o=A + 2), "LA_ERR_INVALID_ARG"),
    (dict(g=A), "LA_ERR_INVALID_ARG"),                # linear takes no gates
    (dict(mode=2), "LA_ERR_INVALID_ARG"),             # retnet needs g
    (dict(mode=3), "LA_ERR_INVALID_ARG"),             # gla needs g
    (dict(mode=3, g=A + 4), "LA_ERR_INVALID_ARG"),    # gla g must be 16-byte aligned
    (dict(mode=2 | 0x200, g=A), "LA_ERR_INVALID_ARG"),  # non-causal: linear and elu1 only
    (dict(mode=0x200 | 0x100), "LA_ERR_UNSUPPORTED"),   # non-causal: bf16 only
    (dict(mode=0x200, C=128), "LA_ERR_UNSUPPORTED"),    # non-causal: C = 64
    (dict(mode=4), "LA_ERR_INVALID_ARG"),             # scalar needs g
    (dict(mode=2, g=A, beta=A), "LA_ERR_INVALID_ARG"),  # beta only for gdn
    (dict(mode=1, g=A), "LA_ERR_INVALID_ARG"),        # elu1 takes no gates
    (dict(mode=6), "LA_ERR_INVALID_ARG"),             # kda needs per-channel g
    (dict(mode=6, g=A + 4), "LA_ERR_INVALID_ARG"),    # kda g must be 16-byte aligned
    (dict(mode=8), "LA_ERR_INVALID_ARG"),             # no mode 8
    (dict(mode=7), "LA_ERR_INVALID_ARG"),             # outer gate needs g
    (dict(mode=7, g=A), "LA_ERR_INVALID_ARG"),        # ... and the value-axis gates in beta
    (dict(mode=7, g=A, beta=A + 4), "LA_ERR_INVALID_ARG"),  # beta 16-byte aligned
    (dict(mode=7, g=A + 4, beta=A), "LA_ERR_INVALID_ARG"),  # g 16-byte aligned
    (dict(mode=7 | 0x200, g=A, beta=A), "LA_ERR_INVALID_ARG"),  # non-causal: linear and elu1 only
    (dict(S0=A + 1), "LA_ERR_INVALID_ARG"),
])
def test_chunk_fwd_rejects_bad_arguments(lib, kw, code):
    rc, msg = _call(**kw)
    assert rc == la.CONSTANTS[code], (rc, msg)
    assert msg.startswith("la_chunk_fwd:"), msg


@pytest.mark.parametrize("kw,code", [
    (dict(S=None), "LA_ERR_INVALID_ARG"),
    (dict(B=0), "LA_ERR_INVALID_ARG"),
    (dict(dk=100), "LA_ERR_UNSUPPORTED"),
    (dict(mode=5, beta=A, g=A + 1), "LA_ERR_INVALID_ARG"),
    (dict(mode=0, beta=A), "LA_ERR_INVALID_ARG"),
    (dict(mode=7, g=A), "LA_ERR_INVALID_ARG"),        # outer gate: value-axis gates in beta
])
def test_recurrent_step_rejects_bad_arguments(lib, kw, code):
    args = dict(q=A, k=A, v=A, g=None, beta=None, o=A, S=A, B=1, H=1, dk=64, dv=64,
                mode=la.LA_LINEAR, stream=None)
    args.update(kw)
    rc = la.la_recurrent_step(**args)
    assert rc == la.CONSTANTS[code], (rc, la.la_last_error())
    assert la.la_last_error().startswith("la_recurrent_step:")


def test_error_message_is_thread_local(lib):
    import threading
    rc, _ = _call(T=0)
    assert rc != 0
    seen = []
    t = threading.Thread(target=lambda: seen.append(la.la_last_error()))
    t.start()
    t.join()
    assert seen == [""]
    assert "T must be" in la.la_last_error()


def test_binding_constants_match_header():
    text = open(HEADER).read()
    for name, val in la.CONSTANTS.items():
        assert re.search(rf"#define\s+{name}\s+{hex(val) if val >= 0x100 else val}\b", text), name


def test_product_does_not_reference_the_oracle():
    root = os.path.dirname(la.__file__)
    for dirpath, _, files in os.walk(root):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cuh", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "la_oracle" not in text, f


# ---- la_prologue argument checks (host only) --------------------------------

def _pro(**kw):
    args = dict(xq=A, xk=A, xv=A, wq=A, wk=A, wv=None, K=4, hist_in=None, hist_out=None,
                a_gate=A, gate_kind=la.LA_GATE_NEG_SOFTPLUS, gate_width=1, tau=8.0, a_beta=A,
                q=A, k=A, v=A, g=A, beta=A, B=1, H=1, T=64, dk=128, dv=128, flags=3, stream=None)
    args.update(kw)
    rc = la.la_prologue(**args)
    return rc, la.la_last_error()


@pytest.mark.parametrize("kw,code", [
    (dict(xq=None), "LA_ERR_INVALID_ARG"),
    (dict(v=None), "LA_ERR_INVALID_ARG"),
    (dict(T=0), "LA_ERR_INVALID_ARG"),
    (dict(B=70000), "LA_ERR_INVALID_ARG"),             # grid y limit on B*H
    (dict(dk=96), "LA_ERR_UNSUPPORTED"),
    (dict(K=0), "LA_ERR_INVALID_ARG"),
    (dict(K=5), "LA_ERR_INVALID_ARG"),
    (dict(flags=4), "LA_ERR_INVALID_ARG"),
    (dict(gate_kind=3), "LA_ERR_INVALID_ARG"),
    (dict(a_gate=None), "LA_ERR_INVALID_ARG"),         # a gate kind without its input
    (dict(gate_width=64), "LA_ERR_INVALID_ARG"),       # neither 1 nor dk
    (dict(tau=0.0), "LA_ERR_INVALID_ARG"),
    (dict(tau=float("nan")), "LA_ERR_INVALID_ARG"),
    (dict(beta=None), "LA_ERR_INVALID_ARG"),           # a_beta without beta
    (dict(hist_in=A, hist_out=A), "LA_ERR_INVALID_ARG"),  # aliasing histories
    (dict(xk=A + 8), "LA_ERR_INVALID_ARG"),            # 16-byte alignment
    (dict(hist_out=A + 4), "LA_ERR_INVALID_ARG"),
])
def test_prologue_rejects_bad_arguments(lib, kw, code):
    rc, msg = _pro(**kw)
    assert rc == la.CONSTANTS[code], (rc, msg)
    assert msg.startswith("la_prologue")


# ---- la_chunk_bwd argument checks (host only) -------------------------------

def _bwd(**kw):
    args = dict(q=A, k=A, v=A, g=None, dO=A, dS_final=None, S0=None, dq_out=A, dk_out=A, dv_out=A, dS0=None,
                dg_out=None, B=1, H=1, T=64, dk=128, dv=128, C=0, mode=la.LA_LINEAR, stream=None)
    args.update(kw)
    rc = la.la_chunk_bwd(**args)
    return rc, la.la_last_error()


@pytest.mark.parametrize("kw,code", [
    (dict(dO=None), "LA_ERR_INVALID_ARG"),
    (dict(dv_out=None), "LA_ERR_INVALID_ARG"),
    (dict(T=0), "LA_ERR_INVALID_ARG"),
    (dict(dk=96), "LA_ERR_UNSUPPORTED"),
    (dict(mode=5), "LA_ERR_UNSUPPORTED"),             # gdn: la_chunk_bwd_delta, not this entry point
    (dict(mode=9), "LA_ERR_INVALID_ARG"),
    (dict(mode=2), "LA_ERR_INVALID_ARG"),             # retnet needs g
    (dict(g=A), "LA_ERR_INVALID_ARG"),                # linear takes none
    (dict(C=128), "LA_ERR_UNSUPPORTED"),
    (dict(dq_out=A + 8), "LA_ERR_INVALID_ARG"),
    (dict(dS0=A + 4), "LA_ERR_INVALID_ARG"),
    (dict(mode=4), "LA_ERR_INVALID_ARG"),             # scalar decay needs g
    (dict(dg_out=A), "LA_ERR_INVALID_ARG"),           # dg only for the scalar decay
    (dict(mode=2, g=A, dg_out=A), "LA_ERR_INVALID_ARG"),
    (dict(mode=4, g=A, dg_out=A + 4), "LA_ERR_INVALID_ARG"),  # dg 16-byte aligned
    (dict(mode=6, g=A), "LA_ERR_UNSUPPORTED"),        # kda: no backward in this build
    (dict(mode=3 | 0x100, g=A), "LA_ERR_UNSUPPORTED"),  # gla backward: bf16 only
    (dict(mode=3), "LA_ERR_INVALID_ARG"),             # gla needs g
    (dict(mode=3, g=A, dg_out=A + 4), "LA_ERR_INVALID_ARG"),  # dg 16-byte aligned
    (dict(mode=7, g=A), "LA_ERR_UNSUPPORTED"),        # outer-product gate: no backward
    (dict(mode=4, g=A, dg_out=A, T=65535 * 256 + 1), "LA_ERR_UNSUPPORTED"),  # dg's tile grid
    (dict(mode=3, g=A, dg_out=A, T=65535 * 256 + 1), "LA_ERR_UNSUPPORTED"),
])
def test_chunk_bwd_rejects_bad_arguments(lib, kw, code):
    rc, msg = _bwd(**kw)
    assert rc == la.CONSTANTS[code], (rc, msg)
    assert msg.startswith("la_chunk_bwd")


@pytest.mark.parametrize("kw,code", [
    (dict(a=None), "LA_ERR_INVALID_ARG"),
    (dict(b=None), "LA_ERR_INVALID_ARG"),
    (dict(q=None), "LA_ERR_INVALID_ARG"),
    (dict(T=0), "LA_ERR_INVALID_ARG"),
    (dict(dk=96), "LA_ERR_UNSUPPORTED"),
    (dict(C=128), "LA_ERR_UNSUPPORTED"),
    (dict(mode=2), "LA_ERR_INVALID_ARG"),              # flags only: 0 or LA_F32
    (dict(a=A + 4), "LA_ERR_INVALID_ARG"),             # 16-byte alignment
    (dict(S0=A + 4), "LA_ERR_INVALID_ARG"),
])
def test_gdelta_rejects_bad_arguments(lib, kw, code):
    args = dict(q=A, k=A, v=A, a=A, b=A, o=A, S0=None, S_final=None, B=1, H=1, T=64, dk=64, dv=64,
                C=0, mode=0, stream=None)
    args.update(kw)
    rc = la.la_chunk_fwd_gdelta(**args)
    assert rc == la.CONSTANTS[code], (rc, la.la_last_error())
    assert la.la_last_error().startswith("la_chunk_fwd_gdelta:")


def _bwd_delta(**kw):
    args = dict(q=A, k=A, v=A, g=A, beta=A, dO=A, dS_final=None, S0=None, dq_out=A, dk_out=A, dv_out=A,
                dbeta_out=A, dg_out=A, dS0=None, B=1, H=1, T=64, dk=128, dv=128, C=0, mode=la.LA_GDN, stream=None)
    args.update(kw)
    rc = la.la_chunk_bwd_delta(**args)
    return rc, la.la_last_error()


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), "LA_ERR_INVALID_ARG"),
    (dict(dO=None), "LA_ERR_INVALID_ARG"),
    (dict(dv_out=None), "LA_ERR_INVALID_ARG"),
    (dict(T=0), "LA_ERR_INVALID_ARG"),
    (dict(B=65536), "LA_ERR_INVALID_ARG"),
    (dict(dk=96), "LA_ERR_UNSUPPORTED"),
    (dict(mode=la.LA_KDA, g=None, dg_out=None), "LA_ERR_INVALID_ARG"),  # KDA needs its per-channel gates
    (dict(mode=la.LA_KDA | la.LA_F32), "LA_ERR_UNSUPPORTED"),
    (dict(mode=la.LA_KDA, C=128), "LA_ERR_UNSUPPORTED"),
    (dict(mode=la.LA_RETNET), "LA_ERR_UNSUPPORTED"),      # la_chunk_bwd covers the unit-write modes
    (dict(mode=la.LA_GDN | la.LA_F32), "LA_ERR_UNSUPPORTED"),
    (dict(mode=9), "LA_ERR_INVALID_ARG"),
    (dict(mode=la.LA_GDN | 0x400), "LA_ERR_INVALID_ARG"),
    (dict(C=128), "LA_ERR_UNSUPPORTED"),
    (dict(C=32), "LA_ERR_UNSUPPORTED"),
    (dict(g=None), "LA_ERR_INVALID_ARG"),                  # dg requested without gates
    (dict(q=A + 8), "LA_ERR_INVALID_ARG"),
    (dict(dq_out=A + 2), "LA_ERR_INVALID_ARG"),
    (dict(beta=A + 4), "LA_ERR_INVALID_ARG"),
    (dict(dbeta_out=A + 4), "LA_ERR_INVALID_ARG"),
    (dict(S0=A + 4), "LA_ERR_INVALID_ARG"),
])
def test_chunk_bwd_delta_rejects_bad_arguments(lib, kw, code):
    rc, msg = _bwd_delta(**kw)
    assert rc == la.CONSTANTS[code], (rc, msg)
    assert msg.startswith("la_chunk_bwd_delta")
