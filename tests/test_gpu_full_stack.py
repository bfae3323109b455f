"""The benchmark's own workload at full size, in the launch configuration it
times: 40 Qwen3.6-35B-A3B-shaped Q4_K layers (256 experts, top-8, I=512, Q4_K
shared expert, bf16 router) x 128 tokens captured as one graph on the
persistent kernel.

Checked three ways: every output of all 128 tokens (final y and residual, the
ids of every layer) equals, bit for bit, the same stack through four kernels
per layer; every token's layer-0 selection is valid against the oracle's fp64
logits; and three sampled tokens are replayed layer by layer through the
single-layer call, every layer's selection checked against the oracle's
logits on the device's own inputs, sampled layers also on their norm output
and residual against the full oracle layer, each chain ending on the
persistent kernel's exact output. (A full oracle layer costs about two
seconds of CPU, so the float check is sampled.)"""
import pytest
import torch

import bench
import gen
import moe_decode_ffn_gb300 as m
from oracle import moe as M
from oracle import parity as P
from tests.gpu_common import bf16_np, host_layer_for, oracle_ids

pytestmark = pytest.mark.gpu

SPEC = gen.Q4K_LAYER_SHARED_Q4_K
# token -> layers checked against the full oracle layer
SAMPLED = {0: (0, 39), 77: (13, 26), 127: (5, 20, 33, 39)}


@pytest.fixture(scope="module")
def stack():
    m.build()
    m.library()
    layers = [m.device_layer(SPEC, bench.SEED, l) for l in range(bench.N_LAYERS)]
    x = gen.make_tokens(bench.SEED, bench.N_TOKENS).cuda()   # rank 0's tokens
    g = m.StackGraph(layers, x)
    assert g.persistent
    g.launch()
    torch.cuda.synchronize()
    assert m.si_workspace_status(g.ws) == m.SI_OK
    yield layers, x, g
    g.close()
    del layers
    torch.cuda.empty_cache()


def test_full_stack_equals_four_kernel_path(stack):
    layers, x, g = stack
    gl = m.StackGraph(layers, x, mode=m.SI_STACK_PER_LAYER)
    assert not gl.persistent
    gl.launch()
    torch.cuda.synchronize()
    assert m.si_workspace_status(gl.ws) == m.SI_OK
    assert torch.equal(g.ids, gl.ids)
    assert torch.equal(g.y, gl.y) and torch.equal(g.sum, gl.sum)
    gl.close()


def test_full_stack_layer0_selection_against_oracle(stack):
    _, x, g = stack
    ids = g.ids.cpu()
    for t in range(bench.N_TOKENS):
        ref_ids, logits = oracle_ids(SPEC, bench.SEED, 0, x[t].cpu())
        assert P.ids_valid(ids[t, 0].tolist(), ref_ids, logits), (t, ids[t, 0].tolist(), ref_ids)


@pytest.mark.parametrize("t", sorted(SAMPLED))
def test_full_stack_sampled_token_layers_against_oracle(stack, t):
    layers, x, g = stack
    xin, res = x[t], x[t]
    for l, L in enumerate(layers):
        out = m.si_moe_layer_decode(L, xin, res)
        ids = out["ids"].cpu().tolist()
        assert ids == g.ids[t, l].cpu().tolist()
        ref_ids, logits = oracle_ids(SPEC, bench.SEED, l, xin.cpu())
        assert P.ids_valid(ids, ref_ids, logits), (l, ids, ref_ids)
        if l in SAMPLED[t]:
            use = ref_ids if ids == ref_ids else ids
            host = host_layer_for(SPEC, bench.SEED, l, use)
            ref = M.layer_forward(host, xin.cpu(), res.cpu(), ids=use)
            for key in ("y", "sum"):
                ok, rep = P.float_parity(bf16_np(out[key]), ref[key])
                assert ok, f"token {t} layer {l} {key}: {rep}"
        xin, res = out["y"], out["sum"]
    assert torch.equal(xin, g.y[t]) and torch.equal(res, g.sum[t])
