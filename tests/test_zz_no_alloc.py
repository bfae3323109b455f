"""The router entry point that allocates nothing.

Some callers cannot allocate device memory while they serve tokens (a
decode loop that bans cudaMalloc/cudaFree after start-up because they can
synchronise the device, or a plug-in whose host owns every byte of device
memory). si_moe_router_topk_noalloc serves them with scratch compiled into
the library. This checks, through the C ABI, that calls in a row give the
same selection, weights and logits (bit for bit: the same kernel on the same
inputs) as the workspace entry point - including a call whose geometry is
smaller than the previous one's, and the largest token count the scratch
takes (2048 tokens of 8 experts) - that the status query reports a clean run,
and that a call larger than the built-in scratch is refused.

Kept in its own file, collected last, so that a failure here is reported
after every other test has run.
"""
import ctypes

import numpy as np
import pytest
import torch

import gen
import moe_decode_ffn_gb300 as m

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    m.build()
    return m.library()


def _router_inputs(seed, n_experts, n_tokens):
    W = gen.to_bf16(gen.normal([gen.stream_key(seed, n_experts, 41)], n_experts * 2048, 0.0,
                               0.02)[0]).reshape(n_experts, 2048).cuda()
    X = gen.make_tokens(seed, n_tokens).cuda()
    return W, X


def _noalloc(lib, X, W, E, T, stream):
    ids = torch.full((T, 8), -7, dtype=torch.int32, device="cuda")
    wts = torch.zeros(T, 8, dtype=torch.float32, device="cuda")
    logits = torch.zeros(T, E, dtype=torch.float32, device="cuda")
    st = lib.si_moe_router_topk_noalloc(X.data_ptr(), m.SI_BF16, W.data_ptr(), m.SI_BF16,
                                        2048, E, 8, T, ids.data_ptr(), wts.data_ptr(),
                                        logits.data_ptr(), stream.cuda_stream)
    return st, ids, wts, logits


def test_noalloc_router_matches_workspace_router_on_calls_in_a_row(lib):
    stream = torch.cuda.current_stream()
    # 256 x 64 fills the scratch; 8 x 1 follows with a smaller geometry (its
    # counters and epochs sit where the larger call left tagged logits);
    # 8 x 2048 is the largest token count the scratch takes
    for call, (seed, E, T) in enumerate(((71, 256, 5), (72, 256, 64), (74, 8, 1), (75, 8, 2048),
                                         (76, 128, 64))):
        W, X = _router_inputs(seed, E, T)
        ids_ref, w_ref, l_ref = m.si_moe_router_topk(X, W, 8, want_logits=True)
        st, ids, wts, logits = _noalloc(lib, X, W, E, T, stream)
        assert st == m.SI_OK, (call, m.status_string(st))
        torch.cuda.synchronize()
        assert torch.equal(ids, ids_ref), call
        assert torch.equal(wts, w_ref), call
        assert torch.equal(logits, l_ref), call
        assert m.si_moe_router_noalloc_status() == m.SI_OK, call


def test_noalloc_router_refuses_more_than_its_scratch(lib):
    W, X = _router_inputs(73, 256, 65)          # 65 x 256 entries > 64 x 256
    ids = torch.empty(65, 8, dtype=torch.int32, device="cuda")
    wts = torch.empty(65, 8, dtype=torch.float32, device="cuda")
    st = lib.si_moe_router_topk_noalloc(X.data_ptr(), m.SI_BF16, W.data_ptr(), m.SI_BF16, 2048,
                                        256, 8, 65, ids.data_ptr(), wts.data_ptr(), None,
                                        torch.cuda.current_stream().cuda_stream)
    assert st == m.SI_ERR_UNSUPPORTED
