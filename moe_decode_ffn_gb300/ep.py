"""Expert-parallel partitions of the routed experts (host side).

The routed expert weights that every token reads are what partitions across
GPUs ("Q4_K shared-expert FFN kernels + Q8_0/Q5_K->Q4_K requant of the MoE FFN
stage", Summary: the per-token expert weight read). Partition p owns experts
[e_p, e_{p+1}); for one token it computes the outputs y_r of the slots whose
expert it owns (si_moe_ffn_decode_ep: zero bits for the other slots), and
the router, the shared expert and the residual norm run replicated.

The exchange is a sum of the partitions' slot outputs taken on their 32-bit
patterns: every slot is non-zero in exactly one partition, so the integer sum
is that partition's value, bit for bit (a float sum would turn -0 into +0),
and the rank-order combine that follows (si_moe_combine_slots) gives exactly
the single-GPU routed output. The payload is k x H fp32 per token (64 KB at
k = 8, H = 2048).

Only argument marshalling and the collective live here; every step of the
computation runs in the library's kernels.
"""
from __future__ import annotations

import torch

from . import (Layer, si_add_rmsnorm3, si_moe_combine_slots, si_moe_ffn_decode_ep,
               si_moe_router_topk)


def expert_ranges(n_experts: int, n_parts: int) -> list:
    """Contiguous, near-equal expert ranges [(e0, e1), ...] of n_parts partitions."""
    if n_parts < 1 or n_parts > n_experts:
        raise ValueError(f"{n_parts} partitions of {n_experts} experts")
    b = [(i * n_experts) // n_parts for i in range(n_parts + 1)]
    return [(b[i], b[i + 1]) for i in range(n_parts)]


def sum_slot_outputs(parts) -> torch.Tensor:
    """Exact sum of the partitions' slot outputs (fp32 tensors of one shape)
    on their 32-bit patterns."""
    acc = parts[0].contiguous().view(torch.int32).clone()
    for p in parts[1:]:
        acc += p.contiguous().view(torch.int32)
    return acc.view(torch.float32)


def all_reduce_slot_outputs(slot_y: torch.Tensor, group=None) -> torch.Tensor:
    """The same sum across the ranks of a torch.distributed group, in place
    (an integer all-reduce: exact in any order)."""
    import torch.distributed as dist
    bits = slot_y.view(torch.int32)
    dist.all_reduce(bits, op=dist.ReduceOp.SUM, group=group)
    return bits.view(torch.float32)


def ep_layer_decode(layer: Layer, x: torch.Tensor, residual: torch.Tensor, e0: int, e1: int,
                    reduce=all_reduce_slot_outputs, stream=None) -> dict:
    """One layer for one token on the partition that owns experts [e0, e1):
    router and shared expert replicated, this partition's slots, the exact
    exchange `reduce(slot_y)` (by default an all-reduce over the default
    process group), the rank-order combine and the residual norm."""
    ids, w, _ = si_moe_router_topk(x.view(1, -1), layer.t["w_router"], layer.spec.top_k, stream=stream)
    slot_y, shared = si_moe_ffn_decode_ep(layer, e0, e1, x, ids.view(-1), stream=stream)
    slot_y = reduce(slot_y)
    routed = si_moe_combine_slots(slot_y, w.view(-1), stream=stream)
    eps = layer.spec.eps
    if shared is not None:
        s, y, _ = si_add_rmsnorm3(routed, shared, residual, layer.t["w_norm"], eps, stream=stream)
    else:
        s, y, _ = si_add_rmsnorm3(routed, residual, None, layer.t["w_norm"], eps, stream=stream)
    return {"ids": ids.view(-1), "w": w.view(-1), "slot_y": slot_y, "routed": routed,
            "shared": shared, "sum": s, "y": y}
