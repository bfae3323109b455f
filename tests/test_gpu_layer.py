"""Whole layer (router + experts + residual norm) and the graph-captured layer
stack on the GPU against the oracle."""
import numpy as np
import pytest
import torch

import gen
import moe_decode_ffn_gb300 as m
from oracle import moe as M
from oracle import parity as P
from tests.gpu_common import bf16_np, device_layer, host_layer_for, oracle_ids

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    m.build()
    m.library()


SPECS = {
    "q4k_shared_q8_0": gen.Q4K_LAYER_SHARED_Q8_0,
    "q4k_shared_q4k": gen.Q4K_LAYER_SHARED_Q4_K,
    "bf16": gen.BF16_LAYER,
    "q4k_128e_i768": gen.Q4K_LAYER_128E,
    "native_q5k_down_q8_0_shared": gen.NATIVE_LAYER_Q5K_DOWN,
}


def oracle_layer(spec, seed, layer, x, residual, gpu_ids):
    ref_ids, logits = oracle_ids(spec, seed, layer, x)
    assert P.ids_valid(gpu_ids, ref_ids, logits), (gpu_ids, ref_ids)
    use = ref_ids if list(gpu_ids) == ref_ids else list(gpu_ids)
    host = host_layer_for(spec, seed, layer, use)
    return M.layer_forward(host, x, residual, ids=use)


@pytest.mark.parametrize("name", list(SPECS))
def test_layer_decode_against_oracle(name):
    spec = SPECS[name]
    dev = device_layer(spec, 100, 0)
    for t in range(3):
        x = gen.make_tokens(700, 3)[t]
        out = m.si_moe_layer_decode(dev, x.cuda())
        torch.cuda.synchronize()
        ids = out["ids"].cpu().tolist()
        ref = oracle_layer(spec, 100, 0, x, None, ids)
        assert np.allclose(out["w"].cpu().double().numpy(), ref["w"], rtol=1e-5, atol=1e-7)
        for key in ("routed", "shared"):
            if key == "shared" and not spec.shared_inter:
                continue
            ok, rep = P.float_parity(bf16_np(out[key]), ref[key + "_bf16"])
            assert ok, f"{key}: {rep}"
        for key in ("sum", "y"):
            ok, rep = P.float_parity(bf16_np(out[key]), ref[key])
            assert ok, f"{key}: {rep}"


def _stack_layers(spec, n_layers, seed=200):
    return [device_layer(spec, seed, l) for l in range(n_layers)]


def test_stack_graph_against_oracle_per_layer():
    """3 layers x 2 tokens of the Q4_K layer captured as one graph (the
    persistent kernel). Every layer is checked against the oracle on the
    device's own input of that layer, at the standard tolerance: the
    single-layer calls reproduce the graph's outputs bit for bit and expose
    each layer's input (the previous layer's norm output and residual sum)."""
    spec = gen.Q4K_LAYER_SHARED_Q4_K
    layers = _stack_layers(spec, 3)
    x = gen.make_tokens(800, 2).cuda()
    g = m.StackGraph(layers, x)
    assert g.persistent
    g.launch()
    torch.cuda.synchronize()
    assert m.si_workspace_status(g.ws) == m.SI_OK
    for t in range(2):
        xin, res = x[t], x[t]
        for l, L in enumerate(layers):
            out = m.si_moe_layer_decode(L, xin, res)
            ids = out["ids"].cpu().tolist()
            assert ids == g.ids[t, l].cpu().tolist(), (t, l)
            ref = oracle_layer(spec, 200, l, xin.cpu(), res.cpu(), ids)
            for key in ("routed", "shared"):
                ok, rep = P.float_parity(bf16_np(out[key]), ref[key + "_bf16"])
                assert ok, f"token {t} layer {l} {key}: {rep}"
            for key in ("sum", "y"):
                ok, rep = P.float_parity(bf16_np(out[key]), ref[key])
                assert ok, f"token {t} layer {l} {key}: {rep}"
            xin, res = out["y"], out["sum"]
        assert torch.equal(xin, g.y[t]) and torch.equal(res, g.sum[t])
    g.close()


@pytest.mark.parametrize("name", ["q4k_shared_q8_0", "q4k_shared_q4k", "bf16"])
def test_stack_graph_equals_eager_layers_and_replays_bit_exact(name):
    """The Q4_K-shared, the Q8_0-shared and the bf16 stack each run as one
    persistent kernel: each must reproduce the per-layer calls bit for bit,
    and every replay of the graph must give the same bits."""
    spec = SPECS[name]
    layers = _stack_layers(spec, 4, seed=300)
    x = gen.make_tokens(900, 3).cuda()
    g = m.StackGraph(layers, x)
    assert g.persistent
    g.launch()
    torch.cuda.synchronize()
    y1, s1, i1 = g.y.clone(), g.sum.clone(), g.ids.clone()
    for _ in range(3):
        g.launch()
    torch.cuda.synchronize()
    assert torch.equal(g.y, y1) and torch.equal(g.sum, s1) and torch.equal(g.ids, i1)
    for t in range(3):
        xin, res = x[t], x[t]
        for l, L in enumerate(layers):
            out = m.si_moe_layer_decode(L, xin, res)
            assert torch.equal(out["ids"], i1[t, l])
            xin, res = out["y"], out["sum"]
        assert torch.equal(xin, y1[t]) and torch.equal(res, s1[t])
    g.close()


@pytest.mark.parametrize("name", ["q4k_shared_q4k", "q4k_shared_q8_0", "bf16"])
def test_stack_paths_agree_bit_exact_and_report_their_kind(name):
    """The same stack through the persistent kernel and through four kernels
    per layer: identical bits; a stack the persistent kernel does not serve
    (H = 4096 on 152 SMs: 28 output rows per block) is refused when that
    path is forced."""
    spec = SPECS[name]
    layers = _stack_layers(spec, 3, seed=310)
    x = gen.make_tokens(910, 2).cuda()
    gp = m.StackGraph(layers, x, mode=m.SI_STACK_PERSISTENT)
    gl = m.StackGraph(layers, x, mode=m.SI_STACK_PER_LAYER)
    ga = m.StackGraph(layers, x)
    assert gp.persistent and not gl.persistent and ga.persistent
    for g in (gp, gl):
        g.launch()
    torch.cuda.synchronize()
    assert torch.equal(gp.y, gl.y) and torch.equal(gp.sum, gl.sum) and torch.equal(gp.ids, gl.ids)
    for g in (gp, gl, ga):
        assert m.si_workspace_status(g.ws) == m.SI_OK
        g.close()
    wide = _stack_layers(gen.LayerSpec(hidden=4096, n_experts=64, top_k=2, inter=256, shared_inter=256,
                                       shared_type="q4_k"), 2, seed=311)
    xw = gen.make_tokens(912, 2).cuda()
    xw = torch.cat([xw, xw], dim=1).contiguous()   # bf16 [2, 4096]
    with pytest.raises(m.SiError) as e:
        m.StackGraph(wide, xw, mode=m.SI_STACK_PERSISTENT)
    assert e.value.status == m.SI_ERR_UNSUPPORTED
    assert not m.StackGraph(wide, xw).persistent


PERSISTENT_SHAPES = {
    "e128_shared_q4k": gen.LayerSpec(n_experts=128, shared_type="q4_k"),
    "e256_no_shared": gen.LayerSpec(shared_inter=0, shared_type="q4_k"),
    "e64_top4_shared_q4k": gen.LayerSpec(n_experts=64, top_k=4, shared_type="q4_k"),
    "i256_shared_q4k": gen.LayerSpec(inter=256, shared_type="q4_k"),
    "e128_shared_q8_0": gen.LayerSpec(n_experts=128, shared_type="q8_0"),
    "i256_shared_q8_0_is1024": gen.LayerSpec(inter=256, shared_inter=1024, shared_type="q8_0"),
    "bf16_no_shared": gen.LayerSpec(expert_type="bf16", shared_inter=0, shared_type="bf16"),
    # 192 gate/up units on 152 SMs (40 blocks take two), 6 down pieces per row
    "e128_i768_no_shared": gen.Q4K_LAYER_128E,
    # the shipped formats: Q5_K routed down rows (Q8_0 or Q4_K shared expert)
    "native_q5k_down_q8_0_shared": gen.NATIVE_LAYER_Q5K_DOWN,
    "q5k_down_q4k_shared": gen.LayerSpec(down_type="q5_k", shared_type="q4_k"),
    "e128_i768_q5k_down": gen.LayerSpec(n_experts=128, inter=768, shared_inter=0, shared_type="q4_k",
                                        down_type="q5_k"),
    "bf16_e128_top4_i768": gen.LayerSpec(expert_type="bf16", n_experts=128, top_k=4, inter=768,
                                         shared_type="bf16"),
    "bf16_e64_top2_i256": gen.LayerSpec(expert_type="bf16", n_experts=64, top_k=2, inter=256,
                                        shared_inter=256, shared_type="bf16"),
}


@pytest.mark.parametrize("name", list(PERSISTENT_SHAPES))
def test_persistent_kernel_shapes_equal_the_per_layer_path(name):
    """Other shapes the persistent kernel takes (router rows split over 8
    warps when E <= SMs, no shared expert, top-4, narrower experts): the same
    bits as four kernels per layer, and a clean status."""
    spec = PERSISTENT_SHAPES[name]
    layers = [device_layer(spec, 400 + len(name), l) for l in range(2)]
    x = gen.make_tokens(920, 3).cuda()
    gp = m.StackGraph(layers, x, mode=m.SI_STACK_PERSISTENT)
    gl = m.StackGraph(layers, x, mode=m.SI_STACK_PER_LAYER)
    for _ in range(2):                      # a replay continues the exchange epochs
        gp.launch()
    gl.launch()
    torch.cuda.synchronize()
    assert m.si_workspace_status(gp.ws) == m.SI_OK and m.si_workspace_status(gl.ws) == m.SI_OK
    assert torch.equal(gp.ids, gl.ids)
    assert torch.equal(gp.y, gl.y) and torch.equal(gp.sum, gl.sum)
    gp.close()
    gl.close()


def test_persistent_stack_at_its_layer_limit():
    """128 layers (the most one persistent launch takes; its layer table sits
    in shared memory) of a small layer shape x 2 tokens: the persistent
    kernel equals four kernels per layer bit for bit; 129 layers are refused
    by the persistent path and run per layer."""
    spec = gen.LayerSpec(n_experts=64, top_k=4, inter=256, shared_inter=256, shared_type="q4_k")
    layers = [device_layer(spec, 950, l) for l in range(128)]
    x = gen.make_tokens(951, 2).cuda()
    gp = m.StackGraph(layers, x, mode=m.SI_STACK_PERSISTENT)
    gl = m.StackGraph(layers, x, mode=m.SI_STACK_PER_LAYER)
    gp.launch()
    gl.launch()
    torch.cuda.synchronize()
    assert gp.persistent and not gl.persistent
    assert m.si_workspace_status(gp.ws) == m.SI_OK and m.si_workspace_status(gl.ws) == m.SI_OK
    assert torch.equal(gp.ids, gl.ids)
    assert torch.equal(gp.y, gl.y) and torch.equal(gp.sum, gl.sum)
    gp.close()
    gl.close()
    more = layers + [device_layer(spec, 950, 128)]
    with pytest.raises(m.SiError) as e:
        m.StackGraph(more, x, mode=m.SI_STACK_PERSISTENT)
    assert e.value.status == m.SI_ERR_UNSUPPORTED
    g = m.StackGraph(more, x)
    assert not g.persistent
    g.close()
