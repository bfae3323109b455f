"""Device-side failure reporting without faulting the GPU: a bounded wait that
runs out reports SI_ERR_TIMEOUT and leaves the context usable; a workspace
whose counters were never zeroed is reported by the router's handshake."""
import time

import pytest
import torch

import gen
import moe_decode_ffn_gb300 as m

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    m.build()
    m.library()


def test_bounded_wait_reports_timeout_and_context_survives():
    ws = m.workspace(256)
    t0 = time.perf_counter()
    st = m.library().si_test_wait_timeout(5_000_000, ws.data_ptr(),
                                          torch.cuda.current_stream().cuda_stream)
    assert st == m.SI_OK
    assert m.si_workspace_status(ws) == m.SI_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 1.0
    assert m.si_workspace_status(ws) == m.SI_OK          # reading clears it
    # the context still runs kernels
    x = gen.make_tokens(1, 1).cuda()
    q = m.si_quantize_q8_1(x[0])
    torch.cuda.synchronize()
    assert q.numel() == 64 * 36


def test_stack_poll_reports_timeout_and_context_survives():
    """The persistent kernel's wait on a tagged slot of another block gives up
    after its budget when the slot never arrives (a block that died), records
    SI_ERR_TIMEOUT and leaves the context usable."""
    ws = m.workspace(512)
    t0 = time.perf_counter()
    assert m.library().si_test_poll_timeout(5_000_000, ws.data_ptr(),
                                            torch.cuda.current_stream().cuda_stream) == m.SI_OK
    assert m.si_workspace_status(ws) == m.SI_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 1.0
    assert m.si_workspace_status(ws) == m.SI_OK
    x = gen.make_tokens(2, 1).cuda()
    q = m.si_quantize_q8_1(x[0])
    torch.cuda.synchronize()
    assert q.numel() == 64 * 36


def test_timeout_budget_is_validated():
    ws = m.workspace(256)
    assert m.library().si_test_wait_timeout(3_000_000_000, ws.data_ptr(), None) == m.SI_ERR_INVALID_ARG
    assert m.library().si_test_poll_timeout(3_000_000_000, ws.data_ptr(), None) == m.SI_ERR_INVALID_ARG
