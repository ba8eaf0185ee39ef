"""Failure detection on the GPU without a fault: a bounded device-side wait
that runs out is reported to the host as LA_ERR_TIMEOUT, the call returns
promptly, the CUDA context stays usable, and the next normal call is correct.

The failure is made by the library's test hook, off unless the environment
variable LA_TEST_FAULT is set: with LA_TEST_FAULT=prologue_wait, la_prologue
arms the mbarrier of k's bulk copy in every CTA without starting that copy
(so nothing is in flight), and the thread that waits on it gives up after a
short bounded wait, sets the device status word and skips the CTA's
arithmetic. la_stream_status reads and clears the word.
"""
import time

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import gated_delta_rule_linear_gb300 as la
    from gated_delta_rule_linear_gb300 import build
    build.build()
    la.load_library()
    assert torch.cuda.is_available()


def test_bounded_wait_reports_timeout_and_the_next_call_is_green(monkeypatch):
    import gated_delta_rule_linear_gb300 as la
    from test_gpu_prologue import _check, _run_gpu, _run_oracle

    wl = workloads.PROLOGUE_WORKLOADS["prologue"].with_sizes(B=1, H=2, T=300)
    inp = workloads.make_prologue_inputs(wl)
    stream = torch.cuda.current_stream().cuda_stream
    assert la.la_stream_status(stream) == la.LA_OK          # nothing pending from earlier tests

    monkeypatch.setenv("LA_TEST_FAULT", "prologue_wait")
    t0 = time.monotonic()
    _run_gpu(inp, wl)                                          # the launch itself succeeds
    rc = la.la_stream_status(stream)
    elapsed = time.monotonic() - t0
    assert rc == la.LA_ERR_TIMEOUT, (rc, la.la_last_error())
    assert "bounded device-side wait" in la.la_last_error()
    assert elapsed < 10.0, f"the timed-out call took {elapsed:.1f} s"
    assert la.la_stream_status(stream) == la.LA_OK            # the word was cleared

    monkeypatch.delenv("LA_TEST_FAULT")
    got = _run_gpu(inp, wl)
    assert la.la_stream_status(stream) == la.LA_OK, la.la_last_error()
    _check(got, _run_oracle(inp, wl), wl)
