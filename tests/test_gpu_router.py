"""Fused router GEMV + top-k + softmax on the GPU against the oracle."""
import numpy as np
import pytest
import torch

import gen
import moe_decode_ffn_gb300 as m
from oracle import moe as M
from oracle import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    m.build()
    m.library()


@pytest.mark.parametrize("n_experts", [256, 128])
def test_router_tie_stress_4000_cases(n_experts):
    """4000 cases of small-integer x and W_r in [-3, 3] (fp32): logits are
    exact, so selection must equal the brute-force sort exactly."""
    cases = 0
    for group in range(40):
        W, X, fam = gen.tie_stress_group(2026, group, n_experts, 100)
        ids, w, logits = m.si_moe_router_topk(X.cuda(), W.cuda(), 8, want_logits=True)
        ref_logits = X.double().numpy() @ W.double().numpy().T
        assert np.array_equal(logits.cpu().double().numpy(), ref_logits), fam
        ids, w = ids.cpu().numpy(), w.cpu().double().numpy()
        for t in range(X.shape[0]):
            ref = M.topk_sort(ref_logits[t])
            assert ids[t].tolist() == ref, (fam, group, t)
            assert np.allclose(w[t], M.softmax_selected(ref_logits[t], ref), rtol=2e-6, atol=1e-7)
            cases += 1
    assert cases == 4000


@pytest.mark.parametrize("n_tokens", [1, 3, 8, 9, 64])
@pytest.mark.parametrize("n_experts", [256, 128, 8])
def test_router_bf16_random(n_tokens, n_experts):
    W = gen.to_bf16(gen.normal([gen.stream_key(1, n_experts, 3)], n_experts * 2048, 0.0, 0.02)[0]
                    ).reshape(n_experts, 2048)
    X = gen.make_tokens(31, n_tokens)
    ids, w, logits = m.si_moe_router_topk(X.cuda(), W.cuda(), 8, want_logits=True)
    ids, w, logits = ids.cpu().numpy(), w.cpu().double().numpy(), logits.cpu().double().numpy()
    Wf, Xf = M.as_f64(W), M.as_f64(X)
    mag = np.abs(Xf) @ np.abs(Wf).T
    for t in range(n_tokens):
        ref_l = Wf @ Xf[t]
        assert np.all(np.abs(logits[t] - ref_l) <= 1e-6 * mag[t] + 1e-30)
        ref_ids = M.topk_sort(ref_l)
        assert P.ids_valid(ids[t], ref_ids, ref_l)
        sel = ids[t].tolist()
        assert np.allclose(w[t], M.softmax_selected(ref_l, sel), rtol=1e-5, atol=1e-7)
        assert abs(w[t].sum() - 1) < 1e-5


@pytest.mark.parametrize("top_k", [1, 2, 5])
def test_router_smaller_top_k(top_k):
    W = gen.to_bf16(gen.normal([gen.stream_key(2, 7)], 256 * 2048, 0.0, 0.02)[0]).reshape(256, 2048)
    X = gen.make_tokens(32, 4)
    ids, w, _ = m.si_moe_router_topk(X.cuda(), W.cuda(), top_k)
    for t in range(4):
        ref_l = M.as_f64(W) @ M.as_f64(X[t])
        assert P.ids_valid(ids[t].cpu().numpy(), M.topk_sort(ref_l, top_k), ref_l)
        assert abs(w[t].sum().item() - 1) < 1e-5


def test_router_zero_input_selects_first_experts():
    W = gen.to_bf16(gen.normal([gen.stream_key(3)], 256 * 2048, 0.0, 0.02)[0]).reshape(256, 2048)
    X = torch.zeros(2, 2048, dtype=torch.bfloat16)
    ids, w, _ = m.si_moe_router_topk(X.cuda(), W.cuda(), 8)
    assert ids.cpu().tolist() == [list(range(8))] * 2
    assert torch.allclose(w.cpu(), torch.full((2, 8), 0.125))


def test_router_workspace_replay_and_determinism():
    """The completion counter returns to zero: the same workspace gives the
    same bits run after run (as a replayed graph would)."""
    W = gen.to_bf16(gen.normal([gen.stream_key(4)], 256 * 2048, 0.0, 0.02)[0]).reshape(256, 2048).cuda()
    X = gen.make_tokens(33, 5).cuda()
    ws = m.workspace(m.router_workspace_bytes(256, 2048, 5))
    first = m.si_moe_router_topk(X, W, 8, want_logits=True, ws=ws)
    for _ in range(5):
        again = m.si_moe_router_topk(X, W, 8, want_logits=True, ws=ws)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
    assert m.si_workspace_status(ws) == m.SI_OK


def test_router_detects_unzeroed_workspace():
    W = gen.to_bf16(gen.normal([gen.stream_key(5)], 256 * 2048, 0.0, 0.02)[0]).reshape(256, 2048).cuda()
    X = gen.make_tokens(34, 2).cuda()
    nb = m.router_workspace_bytes(256, 2048, 2)
    ws = torch.full((nb,), 0xFF, dtype=torch.uint8, device="cuda")
    ws[:256] = 0                                           # status word clear
    ids, w, _ = m.si_moe_router_topk(X, W, 8, ws=ws)
    assert m.si_workspace_status(ws) == m.SI_ERR_HANDSHAKE
    assert torch.all(ids == -1)
    ws.zero_()
    ids, w, _ = m.si_moe_router_topk(X, W, 8, ws=ws)
    assert m.si_workspace_status(ws) == m.SI_OK
    assert torch.all(ids >= 0)


@pytest.mark.parametrize("n_tokens", [16, 24, 32, 64, 100])
@pytest.mark.parametrize("n_experts,w_fp32,hidden", [(128, False, 2048), (100, False, 2048), (256, True, 2048),
                                                     (128, False, 4096)])
def test_router_chunks_equal_single_token_calls(n_tokens, n_experts, w_fp32, hidden):
    """Several chunks of tokens (several router rows per block) give the bits
    of one-token calls (one row per block): the same logits, ids and weights."""
    W = gen.to_bf16(gen.normal([gen.stream_key(6, n_experts, hidden)], n_experts * hidden, 0.0, 0.02)[0]
                    ).reshape(n_experts, hidden)
    if w_fp32:
        W = W.float()
    X = gen.make_tokens(35, n_tokens, hidden=hidden).cuda()
    W = W.cuda()
    ids, w, logits = m.si_moe_router_topk(X, W, 8, want_logits=True)
    for t in range(n_tokens):
        i1, w1, l1 = m.si_moe_router_topk(X[t:t + 1], W, 8, want_logits=True)
        assert torch.equal(logits[t:t + 1], l1), t
        assert torch.equal(ids[t:t + 1], i1), t
        assert torch.equal(w[t:t + 1], w1), t


@pytest.mark.parametrize("top_k", [1, 5])
def test_router_chunks_smaller_top_k_equal_single_token_calls(top_k):
    W = gen.to_bf16(gen.normal([gen.stream_key(7, top_k)], 128 * 2048, 0.0, 0.02)[0]).reshape(128, 2048).cuda()
    X = gen.make_tokens(36, 40).cuda()
    ids, w, _ = m.si_moe_router_topk(X, W, top_k)
    for t in range(40):
        i1, w1, _ = m.si_moe_router_topk(X[t:t + 1], W, top_k)
        assert torch.equal(ids[t:t + 1], i1), t
        assert torch.equal(w[t:t + 1], w1), t
