"""Load-time requant to Q4_K on the GPU against the oracle ("Q4_K
shared-expert FFN kernels + Q8_0/Q5_K->Q4_K requant of the MoE FFN stage",
PR #359, Summary bullets 1 and 2): the output bytes must equal the oracle's
bit for bit; a requantised layer stack runs on the persistent kernel and
matches the per-layer calls."""
import numpy as np
import pytest
import torch

import gen
import moe_decode_ffn_gb300 as m
from oracle import moe as M

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    m.build()
    m.library()


def _source(fmt, seed, rows, cols):
    w = gen.float_weights(seed, 0, gen.ROLE_SH_GATE, 0, rows, cols)
    return gen.encode(w, fmt)


@pytest.mark.parametrize("fmt", ["q8_0", "q5_k"])
@pytest.mark.parametrize("rows,cols", [(1, 256), (3, 512), (64, 2048), (37, 768), (2048, 512)])
def test_requant_bytes_equal_the_oracle(fmt, rows, cols):
    src = _source(fmt, rows * 7 + cols, rows, cols)
    got = m.si_requant_q4_k(src.cuda(), fmt, rows, cols)
    torch.cuda.synchronize()
    ref = M.requant_q4_k(fmt, src.numpy())
    assert np.array_equal(got.cpu().numpy(), ref)


def test_requant_full_shared_expert_and_routed_down_of_four_experts():
    """The full-size shared expert (Q8_0 gate/up 512 x 2048, down 2048 x 512)
    and the routed down rows of four experts (Q5_K, 4 x 2048 x 512)."""
    L = gen.make_layer(gen.NATIVE_LAYER_Q5K_DOWN, 61, 0, device="cpu", experts=[3, 77, 130, 255])
    for name, fmt, cols in (("sh_gate", "q8_0", 2048), ("sh_up", "q8_0", 2048),
                            ("sh_down", "q8_0", 512)):
        src = L[name]
        got = m.si_requant_q4_k(src.cuda(), fmt, src.shape[0], cols)
        assert np.array_equal(got.cpu().numpy(), M.requant_q4_k(fmt, src.numpy())), name
    down = L["down"].reshape(-1, L["down"].shape[-1])            # [4 * 2048, 352]
    got = m.si_requant_q4_k(down.cuda(), "q5_k", down.shape[0], 512)
    assert np.array_equal(got.cpu().numpy(), M.requant_q4_k("q5_k", down.numpy()))


def test_requant_edge_blocks():
    """All-zero blocks, a block with one non-zero weight, negative-only and
    positive-only blocks, and zero rows (nothing to do)."""
    w = torch.zeros(6, 512)
    w[1, 7] = 0.25
    w[2, 256:] = -torch.linspace(0.01, 0.2, 256)
    w[3, :256] = torch.linspace(0.0, 0.3, 256)
    w[4] = 1e-30                                    # subnormal-scale weights: d underflows
    w[5, ::2] = -1e-3
    for fmt in ("q8_0", "q5_k"):
        src = gen.encode(w, fmt)
        got = m.si_requant_q4_k(src.cuda(), fmt, 6, 512)
        assert np.array_equal(got.cpu().numpy(), M.requant_q4_k(fmt, src.numpy())), fmt
    out = torch.zeros(1, 144, dtype=torch.uint8, device="cuda")
    assert m.library().si_requant_q4_k(out.data_ptr(), m.SI_Q8_0, 0, 256, out.data_ptr(), None) == m.SI_OK
    assert m.library().si_requant_q4_k(out.data_ptr(), m.SI_Q8_0, 1, 100, out.data_ptr(), None) == \
        m.SI_ERR_INVALID_ARG
    assert m.library().si_requant_q4_k(out.data_ptr(), m.SI_Q4_K, 1, 256, out.data_ptr(), None) == \
        m.SI_ERR_UNSUPPORTED


def _requantised_layer(seed, layer):
    """A native layer (routed down Q5_K, shared Q8_0) requantised on the GPU
    into the Q4_K layer that the persistent kernel serves."""
    spec = gen.NATIVE_LAYER_Q5K_DOWN
    L = gen.make_layer(spec, seed, layer, device="cuda")
    E, H, I = spec.n_experts, spec.hidden, spec.inter
    t = {k: v for k, v in L.items() if isinstance(v, torch.Tensor)}
    t["down"] = m.si_requant_q4_k(t["down"].reshape(E * H, -1), "q5_k", E * H, I).reshape(E, H, -1)
    t["sh_gate"] = m.si_requant_q4_k(t["sh_gate"], "q8_0", spec.shared_inter, H)
    t["sh_up"] = m.si_requant_q4_k(t["sh_up"], "q8_0", spec.shared_inter, H)
    t["sh_down"] = m.si_requant_q4_k(t["sh_down"], "q8_0", H, spec.shared_inter)
    return m.Layer(gen.Q4K_LAYER_SHARED_Q4_K, t)


def test_requantised_stack_runs_on_the_persistent_kernel_and_equals_the_layer_calls():
    layers = [_requantised_layer(71, l) for l in range(3)]
    x = gen.make_tokens(72, 2).cuda()
    g = m.StackGraph(layers, x)
    assert g.persistent
    g.launch()
    torch.cuda.synchronize()
    assert m.si_workspace_status(g.ws) == m.SI_OK
    for t in range(2):
        xin, res = x[t], x[t]
        for l, L in enumerate(layers):
            out = m.si_moe_layer_decode(L, xin, res)
            assert torch.equal(out["ids"], g.ids[t, l])
            xin, res = out["y"], out["sum"]
        assert torch.equal(xin, g.y[t]) and torch.equal(res, g.sum[t])
    g.close()
