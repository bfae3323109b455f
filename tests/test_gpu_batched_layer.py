"""The batched layer (T tokens, each routed on its own: router + top-k,
grouped routed experts, residual norm of every row) and the batched layer
stack captured as one graph, on the Qwen3-30B-A3B-shaped layer (128 experts,
top-8, I=768, no shared expert, Q4_K).

Checked three ways: every token's results equal the single-token layer call
on that token alone, bit for bit; sampled tokens against the oracle layer on
the device's own inputs at the standard tolerance; the graph (3 layers, and
the 48-layer stack at T = 64) equals the same layers called one at a time."""
import numpy as np
import pytest
import torch

import gen
import moe_decode_ffn_gb300 as m
from oracle import moe as M
from oracle import parity as P
from tests.gpu_common import bf16_np, device_layer, host_layer_for, oracle_ids

pytestmark = pytest.mark.gpu

SPEC = gen.Q4K_LAYER_128E


@pytest.fixture(scope="module", autouse=True)
def _lib():
    m.build()
    m.library()


def _oracle_check(spec, seed, layer, x, res, out, t, where):
    ids = out["ids"][t].cpu().tolist()
    ref_ids, logits = oracle_ids(spec, seed, layer, x.cpu())
    assert P.ids_valid(ids, ref_ids, logits), (where, ids, ref_ids)
    use = ref_ids if ids == ref_ids else ids
    host = host_layer_for(spec, seed, layer, use)
    ref = M.layer_forward(host, x.cpu(), res.cpu(), ids=use)
    ok, rep = P.float_parity(bf16_np(out["routed"][t]), ref["routed_bf16"])
    assert ok, f"{where} routed: {rep}"
    for key in ("sum", "y"):
        ok, rep = P.float_parity(bf16_np(out[key][t]), ref[key])
        assert ok, f"{where} {key}: {rep}"


# 128 tokens x top-8 = 1024 (token, expert) pairs: the most the grouping takes
@pytest.mark.parametrize("T", [1, 4, 16, 64, 128])
def test_batched_layer_equals_single_token_layers_and_the_oracle(T):
    dev = device_layer(SPEC, 500, 0)
    x = gen.make_tokens(501 + T, T).cuda()
    res = gen.make_tokens(601 + T, T).cuda()       # a residual distinct from x
    out = m.si_moe_layer_decode_batched(dev, x, res, mode=m.SI_FFN_INT8)
    ws = m.workspace(m.layer_workspace_bytes(dev))
    torch.cuda.synchronize()
    for t in range(T):
        one = m.si_moe_layer_decode(dev, x[t], res[t], ws=ws)
        for key in ("ids", "w", "sum", "y", "routed"):
            assert torch.equal(out[key][t], one[key]), (t, key)
    assert m.si_workspace_status(ws) == m.SI_OK
    for t in sorted({0, T // 2, T - 1}):
        _oracle_check(SPEC, 500, 0, x[t], res[t], out, t, f"token {t}")


# 256 experts (the most the grouping takes), I=512: the longest-first active
# list over all 8 words of expert bits, several rows per router block
SPEC_256 = gen.LayerSpec(n_experts=256, inter=512, shared_inter=0, shared_type="q4_k")


@pytest.mark.parametrize("T", [16, 64])
def test_batched_layer_256_experts_equals_single_token_layers(T):
    dev = device_layer(SPEC_256, 520, 0)
    x = gen.make_tokens(521 + T, T).cuda()
    res = gen.make_tokens(621 + T, T).cuda()
    out = m.si_moe_layer_decode_batched(dev, x, res, mode=m.SI_FFN_AUTO)
    ws = m.workspace(m.layer_workspace_bytes(dev))
    torch.cuda.synchronize()
    for t in range(T):
        one = m.si_moe_layer_decode(dev, x[t], res[t], ws=ws)
        for key in ("ids", "w", "sum", "y", "routed"):
            assert torch.equal(out[key][t], one[key]), (t, key)
    assert m.si_workspace_status(ws) == m.SI_OK
    _oracle_check(SPEC_256, 520, 0, x[T - 1], res[T - 1], out, T - 1, f"token {T - 1}")


def test_batched_layer_auto_mode_is_the_integer_mode():
    dev = device_layer(SPEC, 500, 0)
    x = gen.make_tokens(505, 16).cuda()
    a = m.si_moe_layer_decode_batched(dev, x, mode=m.SI_FFN_AUTO)
    b = m.si_moe_layer_decode_batched(dev, x, mode=m.SI_FFN_INT8)
    torch.cuda.synchronize()
    for key in ("ids", "w", "sum", "y", "routed"):
        assert torch.equal(a[key], b[key]), key


def _replay(layers, x, mode=m.SI_FFN_AUTO):
    """The stack as one batched layer call after another; per layer the
    inputs and outputs."""
    steps = []
    xin, res = x, x
    for L in layers:
        out = m.si_moe_layer_decode_batched(L, xin, res, mode=mode)
        steps.append((xin, res, out))
        xin, res = out["y"], out["sum"]
    return steps


def test_batched_stack_graph_equals_layer_calls_and_the_oracle():
    layers = [device_layer(SPEC, 510, l) for l in range(3)]
    x = gen.make_tokens(511, 16).cuda()
    g = m.BatchedStackGraph(layers, x)
    for _ in range(2):                        # replays give the same bits
        g.launch()
    torch.cuda.synchronize()
    assert m.si_workspace_status(g.ws) == m.SI_OK
    steps = _replay(layers, x)
    torch.cuda.synchronize()
    for l, (_, _, out) in enumerate(steps):
        assert torch.equal(g.ids[l], out["ids"]), l
    assert torch.equal(g.y, steps[-1][2]["y"]) and torch.equal(g.sum, steps[-1][2]["sum"])
    for l, t in ((0, 3), (1, 9), (2, 15)):
        xin, res, out = steps[l]
        _oracle_check(SPEC, 510, l, xin[t], res[t], out, t, f"layer {l} token {t}")
    g.close()


def test_batched_48_layer_stack_at_64_tokens():
    """The 48-layer stack of the 128-expert layer at 64 tokens, the largest
    batch of the workload: the graph equals the layer calls, every token's
    first-layer selection is valid against the oracle's logits, and sampled
    (layer, token) pairs match the oracle layer on the device's inputs."""
    layers = [m.device_layer(SPEC, 520, l) for l in range(48)]
    x = gen.make_tokens(521, 64).cuda()
    g = m.BatchedStackGraph(layers, x)
    g.launch()
    torch.cuda.synchronize()
    assert m.si_workspace_status(g.ws) == m.SI_OK
    steps = _replay(layers, x)
    torch.cuda.synchronize()
    assert torch.equal(g.y, steps[-1][2]["y"]) and torch.equal(g.sum, steps[-1][2]["sum"])
    assert all(torch.equal(g.ids[l], steps[l][2]["ids"]) for l in range(48))
    ids0 = g.ids[0].cpu()
    for t in range(64):
        ref_ids, logits = oracle_ids(SPEC, 520, 0, x[t].cpu())
        assert P.ids_valid(ids0[t].tolist(), ref_ids, logits), t
    for l, t in ((0, 0), (17, 40), (47, 63)):
        xin, res, out = steps[l]
        _oracle_check(SPEC, 520, l, xin[t], res[t], out, t, f"layer {l} token {t}")
    g.close()
    del layers, steps
    torch.cuda.empty_cache()


def test_batched_stack_of_one_token_runs_on_the_persistent_kernel():
    """One token, automatic mode: the graph holds the persistent stack kernel
    (the layer has 192 gate/up units on 152 SMs) and gives the bits of the
    batched integer path, layer ids included."""
    layers = [device_layer(SPEC, 560, l) for l in range(6)]
    x = gen.make_tokens(561, 1).cuda()
    ga = m.BatchedStackGraph(layers, x)
    gi = m.BatchedStackGraph(layers, x, mode=m.SI_FFN_INT8)
    assert ga.persistent and not gi.persistent
    for _ in range(2):
        ga.launch()
    gi.launch()
    torch.cuda.synchronize()
    assert m.si_workspace_status(ga.ws) == m.SI_OK and m.si_workspace_status(gi.ws) == m.SI_OK
    assert torch.equal(ga.ids, gi.ids)
    assert torch.equal(ga.y, gi.y) and torch.equal(ga.sum, gi.sum)
    ga.close()
    gi.close()


def test_batched_layer_refuses_more_pairs_than_the_grouping_takes():
    """129 tokens x top-8 = 1032 pairs, above the 1024 the grouping holds:
    refused on the host, nothing enqueued."""
    dev = device_layer(SPEC, 500, 0)
    x = gen.make_tokens(540, 129).cuda()
    with pytest.raises(m.SiError) as e:
        m.si_moe_layer_decode_batched(dev, x, ws=m.workspace(1 << 20))
    assert e.value.status == m.SI_ERR_UNSUPPORTED


def test_batched_layer_rejects_a_shared_expert():
    spec = gen.Q4K_LAYER_SHARED_Q4_K
    dev = device_layer(spec, 530, 0)
    assert m.layer_batched_workspace_bytes(dev, 4) == 0
    x = gen.make_tokens(531, 4).cuda()
    with pytest.raises(m.SiError) as e:
        m.si_moe_layer_decode_batched(dev, x, ws=m.workspace(1 << 20))
    assert e.value.status == m.SI_ERR_UNSUPPORTED
