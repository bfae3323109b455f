"""Shared fixtures for the GPU parity tests (device layers are cached per
session: a full 256-expert Q4_K layer is ~0.45 GB, bf16 ~1.5 GB)."""
import functools

import numpy as np
import torch

import gen
import moe_decode_ffn_gb300 as m
from oracle import moe as M


@functools.lru_cache(maxsize=None)
def device_layer(spec, seed: int, layer: int = 0):
    L = gen.make_layer(spec, seed, layer, device="cuda")
    return m.Layer(spec, {k: v for k, v in L.items() if isinstance(v, torch.Tensor)})


@functools.lru_cache(maxsize=64)
def host_layer(spec, seed: int, layer: int, experts: tuple):
    return gen.make_layer(spec, seed, layer, device="cpu", experts=list(experts))


def host_layer_for(spec, seed, layer, ids):
    ids = tuple(sorted(set(int(i) for i in ids)))
    return host_layer(spec, seed, layer, ids)


def bf16_np(t: torch.Tensor) -> np.ndarray:
    return M.as_f64(t.detach().cpu())


def oracle_ids(spec, seed, layer, x):
    """Oracle routing of token x for a layer (router weights only)."""
    L = host_layer(spec, seed, layer, (0,))
    logits = M.router_logits(M.as_f64(x), L["w_router"])
    return M.topk_sort(logits, spec.top_k), logits
