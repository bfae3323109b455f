"""Expert-parallel partitions on CPU (gloo): the partition of the experts,
and the exact exchange of the partitions' slot outputs across two ranks.

Each rank computes the oracle's slot outputs y_r for the slots whose expert
it owns (zeros elsewhere, as si_moe_ffn_decode_ep writes them); after the
integer all-reduce every rank holds the single-rank slot outputs bit for bit,
so the rank-order combine that follows gives the single-rank routed output."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import gen
from moe_decode_ffn_gb300 import ep
from oracle import formats as F
from oracle import moe as M

SPEC = gen.LayerSpec(hidden=256, n_experts=16, top_k=4, inter=256, expert_type="q4_k",
                     shared_inter=0, shared_type="q4_k")
SEED = 62   # routes to experts 12, 14, 9 and 5: both halves of the experts


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _slot_outputs(e0, e1):
    """The oracle's slot outputs of one token (fp32 [k, H]), zero for the
    slots whose expert lies outside [e0, e1); and the routing."""
    L = gen.make_layer(SPEC, SEED, 0)
    x = M.as_f64(gen.make_tokens(SEED + 1, 1, hidden=SPEC.hidden)[0])
    ids, w = M.route(M.router_logits(x, L["w_router"]), SPEC.top_k)
    a = F.q8_1_quantize(F.fp32(x))
    out = np.zeros((SPEC.top_k, SPEC.hidden), np.float32)
    for r, e in enumerate(ids):
        if e0 <= e < e1:
            s = L["expert_ids"].index(e)
            out[r] = M.expert_ffn("q4_k", L["gate"][s], L["up"][s], L["down"][s], x, a)["y"]
    return torch.from_numpy(out), ids, w


def _combine(y, w):
    """routed = sum_r w_r y_r in rank order (the same host function on both
    sides of the comparison)."""
    acc = np.zeros(y.shape[1])
    for r in range(y.shape[0]):
        acc = acc + w[r] * y[r].numpy().astype(np.float64)
    return F.bf16(acc)


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        e0, e1 = ep.expert_ranges(SPEC.n_experts, world)[rank]
        y, ids, w = _slot_outputs(e0, e1)
        owned = sum(1 for e in ids if e0 <= e < e1)
        ep.all_reduce_slot_outputs(y)
        out.put((rank, owned, y.numpy().copy()))
    finally:
        dist.destroy_process_group()


def test_expert_ranges_partition_the_experts():
    for E, n in ((256, 2), (256, 8), (128, 3), (16, 16)):
        r = ep.expert_ranges(E, n)
        assert r[0][0] == 0 and r[-1][1] == E
        assert all(a[1] == b[0] for a, b in zip(r, r[1:]))
        assert max(e1 - e0 for e0, e1 in r) - min(e1 - e0 for e0, e1 in r) <= 1


def test_slot_sum_keeps_every_bit_pattern():
    """A float sum would turn -0 into +0; the integer sum does not."""
    a = torch.tensor([[-0.0, 1.5, 0.0], [0.0, 0.0, 0.0]])
    b = torch.tensor([[0.0, 0.0, 0.0], [-3.25e-39, 0.0, -2.0]])   # a subnormal too
    s = ep.sum_slot_outputs([a, b])
    want = torch.tensor([[-0.0, 1.5, 0.0], [-3.25e-39, 0.0, -2.0]])
    assert torch.equal(s.view(torch.int32), want.view(torch.int32))


def test_two_gloo_ranks_reproduce_the_single_rank_slots_and_routed_output():
    full, ids, w = _slot_outputs(0, SPEC.n_experts)
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted((out.get(timeout=300) for _ in procs), key=lambda g: g[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(owned > 0 for _, owned, _ in got), "the routing must use both partitions"
    assert sum(owned for _, owned, _ in got) == SPEC.top_k
    for rank, _, y in got:
        assert np.array_equal(y.view(np.int32), full.numpy().view(np.int32)), rank
        assert np.array_equal(_combine(torch.from_numpy(y), w), _combine(full, w)), rank
