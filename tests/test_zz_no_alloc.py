"""la_chunk_fwd_noalloc: the materialised variant with its workspace in the
library's static device array.

The GPU test calls the entry point through the C ABI twice in a row and
checks each result against la_chunk_fwd's materialised variant (same
kernels, workspace from the pool) on the same inputs; the host tests check
that oversized and unsupported requests are rejected before any CUDA call.
This file is collected last on purpose: it must pass after the other tests
have used the library, and alone in a fresh process.
"""
import pytest
import torch

import gated_delta_rule_linear_gb300 as la
from gated_delta_rule_linear_gb300 import build as labuild
import workloads

A = 0x10000  # fake aligned device address: rejected calls never dereference it


@pytest.fixture(scope="module")
def lib():
    labuild.build()
    return la.load_library()


def _host_call(**kw):
    args = dict(q=A, k=A, v=A, g=None, beta=None, o=A, S0=None, S_final=None,
                B=1, H=8, T=8192, dk=128, dv=128, C=0, mode=la.LA_LINEAR, stream=None)
    args.update(kw)
    return la.la_chunk_fwd_noalloc(**args)


def test_scratch_limit_is_exact(lib):
    limit = la.CONSTANTS["LA_NOALLOC_SCRATCH_BYTES"]
    assert 8 * (8192 // 64) * 128 * 256 == limit   # B*H*ceil(T/64)*dk*256 at the limit
    rc = _host_call(T=8193)                          # one chunk more than fits
    assert rc == la.LA_ERR_INVALID_ARG
    msg = la.la_last_error()
    assert "scratch" in msg and str(limit) in msg


@pytest.mark.parametrize("kw,code", [
    # every rejection the header lists
    (dict(mode=la.LA_GDN), "LA_ERR_UNSUPPORTED"),
    (dict(mode=la.LA_KDA, g=A), "LA_ERR_UNSUPPORTED"),
    (dict(mode=la.LA_OUTER_GATE, g=A, beta=A), "LA_ERR_UNSUPPORTED"),
    (dict(mode=la.LA_LINEAR | la.LA_F32), "LA_ERR_UNSUPPORTED"),
    (dict(mode=la.LA_GLA, g=A, C=128), "LA_ERR_UNSUPPORTED"),   # C = 128 without per-channel gates only
    (dict(C=32), "LA_ERR_INVALID_ARG"),
    (dict(mode=la.LA_LINEAR | la.LA_NONCAUSAL), "LA_ERR_INVALID_ARG"),
    (dict(mode=9), "LA_ERR_INVALID_ARG"),
    (dict(mode=la.LA_LINEAR, g=A), "LA_ERR_INVALID_ARG"),      # superfluous g
    (dict(mode=la.LA_GLA, g=A, beta=A), "LA_ERR_INVALID_ARG"),  # any beta
    (dict(mode=la.LA_RETNET), "LA_ERR_INVALID_ARG"),         # missing g
    (dict(q=None), "LA_ERR_INVALID_ARG"),
    (dict(o=A + 2), "LA_ERR_INVALID_ARG"),
    (dict(T=0), "LA_ERR_INVALID_ARG"),
])
def test_rejects_unsupported_requests_on_the_host(lib, kw, code):
    assert _host_call(**{"T": 64, **kw}) == la.CONSTANTS[code]
    assert la.la_last_error().startswith("la_chunk_fwd_noalloc")


def _inputs(mode, B, H, T, seed):
    wl = workloads.WORKLOADS[mode].with_sizes(B=B, H=H, T=T, seed=seed)
    inp = workloads.make_inputs(wl)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    if mode == "elu1" and d["S0"] is not None:
        d["S0"][..., wl.dv] = d["S0"][..., wl.dv].abs() + 1.0
    return wl, d


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["retnet", "gla", "elu1", "scalar"])
def test_noalloc_matches_materialised_entry_point_on_two_calls(lib, mode, monkeypatch):
    assert torch.cuda.is_available()
    stream = torch.cuda.current_stream()
    # two different problems in a row; the second also runs at the scratch limit (dk = 128)
    shapes = [(1, 2, 300, 11), (1, 8, 8192, 12) if mode != "elu1" else (2, 4, 4000, 12)]
    # references (la_chunk_fwd's materialised variant, workspace from the library's
    # pool) and output buffers first, so that nothing but the two no-alloc calls
    # runs between the device-memory readings below
    cases = []
    for B, H, T, seed in shapes:
        wl, d = _inputs(mode, B, H, T, seed)
        # the no-alloc entry point walks the chunk states serially; elu+1 and linear
        # attention otherwise take the parallel state pass, which sums in another order
        monkeypatch.setenv("LA_VARIANT", "mat")
        monkeypatch.setenv("LA_MAT_STATE", "serial")
        o_ref, S_ref = la.chunk_fwd(d["q"], d["k"], d["v"], wl.mode, g=d["g"], S0=d["S0"])
        monkeypatch.delenv("LA_VARIANT")
        monkeypatch.delenv("LA_MAT_STATE")
        o = torch.full_like(o_ref, float("nan"))
        S = torch.full_like(S_ref, float("nan"))
        cases.append((B, H, T, wl, d, o_ref, S_ref, o, S))
    torch.cuda.synchronize()
    free = []
    for B, H, T, wl, d, o_ref, S_ref, o, S in cases:
        rc = la.la_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["g"], None, o, d["S0"], S,
                                     B, H, T, wl.dk, wl.dv, 0, la.MODE_IDS[wl.mode], stream.cuda_stream)
        assert rc == 0, la.la_last_error()
        assert la.la_stream_status(stream.cuda_stream) == 0, la.la_last_error()
        free.append(torch.cuda.mem_get_info()[0])
    for B, H, T, wl, d, o_ref, S_ref, o, S in cases:
        assert torch.equal(o, o_ref), f"{mode} T={T}: o differs from la_chunk_fwd (materialised)"
        assert torch.equal(S, S_ref), f"{mode} T={T}: S_final differs from la_chunk_fwd (materialised)"
    # the first call may load the module that holds the static array; the second,
    # larger call must not take any device memory
    assert free[1] == free[0], f"device memory changed by {free[0] - free[1]} bytes across a no-alloc call"


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["retnet", "elu1"])
def test_noalloc_c128_matches_entry_point(lib, mode, monkeypatch):
    stream = torch.cuda.current_stream()
    wl, d = _inputs(mode, 1, 4, 1000, 13)
    monkeypatch.setenv("LA_MAT_STATE", "serial")  # the no-alloc entry point's state pass
    o_ref, S_ref = la.chunk_fwd(d["q"], d["k"], d["v"], wl.mode, g=d["g"], S0=d["S0"], C=128)
    monkeypatch.delenv("LA_MAT_STATE")
    o = torch.full_like(o_ref, float("nan"))
    S = torch.full_like(S_ref, float("nan"))
    rc = la.la_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["g"], None, o, d["S0"], S,
                                 1, 4, 1000, wl.dk, wl.dv, 128, la.MODE_IDS[wl.mode], stream.cuda_stream)
    assert rc == 0, la.la_last_error()
    assert la.la_stream_status(stream.cuda_stream) == 0, la.la_last_error()
    assert torch.equal(o, o_ref) and torch.equal(S, S_ref)
