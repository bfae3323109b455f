"""Expert-parallel partitions on one GPU: the partitions' slot outputs
(si_moe_ffn_decode_ep over expert ranges that cover the experts), summed on
their bit patterns and combined (si_moe_combine_slots), equal the whole
routed FFN (si_moe_ffn_decode) bit for bit; every partition writes zero bits
for the slots it does not own and the full shared expert; a layer run as one
partition plus the other partition's slots equals the layer call."""
import pytest
import torch

import gen
import moe_decode_ffn_gb300 as m
from moe_decode_ffn_gb300 import ep
from tests.gpu_common import device_layer

pytestmark = pytest.mark.gpu

SPECS = {
    "q4k_shared_q4k": gen.Q4K_LAYER_SHARED_Q4_K,
    "q4k_shared_q8_0": gen.Q4K_LAYER_SHARED_Q8_0,
    "q4k_128e_i768": gen.Q4K_LAYER_128E,
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    m.build()
    m.library()


def _route(dev, x):
    ids, w, _ = m.si_moe_router_topk(x.view(1, -1), dev.t["w_router"], dev.spec.top_k)
    return ids.view(-1), w.view(-1)


@pytest.mark.parametrize("parts", [2, 4])
@pytest.mark.parametrize("name", list(SPECS))
def test_partitions_reproduce_the_whole_ffn(name, parts):
    spec = SPECS[name]
    dev = device_layer(spec, 700, 0)
    xs = gen.make_tokens(701, 3).cuda()
    for t in range(3):
        x = xs[t]
        ids, w = _route(dev, x)
        routed_ref, shared_ref = m.si_moe_ffn_decode(dev, x, ids, w)
        slots = []
        for e0, e1 in ep.expert_ranges(spec.n_experts, parts):
            y, sh = m.si_moe_ffn_decode_ep(dev, e0, e1, x, ids)
            own = (ids >= e0) & (ids < e1)
            assert not y[~own].view(torch.int32).any(), (t, e0, e1)
            if spec.shared_inter:
                assert torch.equal(sh, shared_ref)
            slots.append(y)
        full, _ = m.si_moe_ffn_decode_ep(dev, 0, spec.n_experts, x, ids)
        summed = ep.sum_slot_outputs(slots)
        assert torch.equal(summed.view(torch.int32), full.view(torch.int32)), t
        assert torch.equal(m.si_moe_combine_slots(summed, w), routed_ref), t


def test_ep_layer_equals_the_layer_call():
    spec = gen.Q4K_LAYER_SHARED_Q4_K
    dev = device_layer(spec, 710, 0)
    (a0, a1), (b0, b1) = ep.expert_ranges(spec.n_experts, 2)
    xs = gen.make_tokens(711, 2).cuda()
    res = gen.make_tokens(712, 2).cuda()
    for t in range(2):
        ids, _ = _route(dev, xs[t])
        other, _ = m.si_moe_ffn_decode_ep(dev, b0, b1, xs[t], ids)     # the other partition's slots
        got = ep.ep_layer_decode(dev, xs[t], res[t], a0, a1,
                                 reduce=lambda y: ep.sum_slot_outputs([y, other]))
        ref = m.si_moe_layer_decode(dev, xs[t], res[t])
        for key in ("ids", "w", "routed", "shared", "sum", "y"):
            assert torch.equal(got[key], ref[key]), (t, key)


def test_ep_rejects_bf16_experts_and_bad_ranges():
    dev = device_layer(gen.BF16_LAYER, 720, 0)
    x = gen.make_tokens(721, 1)[0].cuda()
    ids = torch.arange(8, dtype=torch.int32, device="cuda")
    with pytest.raises(m.SiError) as e:
        m.si_moe_ffn_decode_ep(dev, 0, 128, x, ids)
    assert e.value.status == m.SI_ERR_UNSUPPORTED
    q = device_layer(gen.Q4K_LAYER_SHARED_Q4_K, 700, 0)
    for e0, e1 in ((-1, 10), (10, 5), (0, 257)):
        with pytest.raises(m.SiError) as e:
            m.si_moe_ffn_decode_ep(q, e0, e1, x, ids)
        assert e.value.status == m.SI_ERR_INVALID_ARG
