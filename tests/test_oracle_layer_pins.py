"""Pins of the oracle's whole layer (router, top-k, softmax, routed and shared
experts, residual fold) against a layer worked out by hand.

The layer and the closed form of every expected value are written out in
tests/golden/layer_worked_example.py, which imports neither the oracle nor
the library; the values it wrote are in layer_worked_example.txt. The layer
exercises the tie rule at the top-k boundary ("perf(qwen3.6): fused router
GEMV+top-k + folded residual-norm (decode)", Summary item 1), the softmax over
the selected logits, silu-gated experts ("perf(qwen3.6): fuse decode kernel
launches", Summary item 1), the sigmoid gate of the shared expert, and the
3-input residual fold with its bf16 roundings (Summary item 2 of the first
page), and the 2-input fold of a layer without a shared expert.
"""
import os

import numpy as np
import torch

import gen
from oracle import moe as M

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "layer_worked_example.txt")
H = I = 256
E, K = 8, 2
C = (0.5, 1.0, -1.0, 2.0, 0.25, 1.0, -2.0, 0.0)


def golden():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, *v = line.split()
                out[k] = np.array([float(t) for t in v])
    return out


def _rows(t: torch.Tensor) -> torch.Tensor:
    """bf16 matrix -> the uint8 row bytes the oracle's bf16 GEMV reads."""
    return t.to(torch.bfloat16).contiguous().view(torch.uint8)


def hand_layer(with_shared: bool = True):
    """The layer of tests/golden/layer_worked_example.py."""
    spec = gen.LayerSpec(hidden=H, n_experts=E, top_k=K, inter=I, expert_type="bf16",
                         shared_inter=I if with_shared else 0, shared_type="bf16", eps=1e-6)
    wr = torch.zeros(E, H)
    wr[:, 0] = torch.tensor(C)
    gate, up, down = [], [], []
    for e in range(E):
        g = torch.zeros(I, H)
        g[0, 0] = 1.0
        u = torch.zeros(I, H)
        u[0, 1] = (e + 1) / 8
        d = torch.zeros(H, I)
        d[e, 0] = 1.0
        d[e + 8, 0] = -0.5
        gate.append(_rows(g))
        up.append(_rows(u))
        down.append(_rows(d))
    L = {"spec": spec, "expert_ids": list(range(E)), "w_router": wr.to(torch.bfloat16),
         "gate": torch.stack(gate), "up": torch.stack(up), "down": torch.stack(down),
         "w_norm": torch.tensor([1.0 + 0.5 * (h % 2) for h in range(H)]).to(torch.bfloat16)}
    if with_shared:
        g = torch.zeros(I, H)
        g[0, 0] = 1.0
        u = torch.zeros(I, H)
        u[0, 1] = 0.25
        d = torch.zeros(H, I)
        d[3, 0] = 11.0 / 32.0
        d[20, 0] = 1.0
        d[21, 0] = -1.0
        wsg = torch.zeros(H)
        wsg[1] = -0.5
        L.update(sh_gate=_rows(g), sh_up=_rows(u), sh_down=_rows(d), w_sg=wsg.to(torch.bfloat16))
    return L


def hand_inputs():
    x = torch.zeros(H)
    x[0], x[1] = 1.0, 2.0
    r = torch.tensor([(-0.75, -0.25, 0.25, 0.75)[h % 4] for h in range(H)])
    r[3] = 138.0 / 4096.0
    return x.to(torch.bfloat16), r.to(torch.bfloat16)


def _check(out, g, suffix):
    assert out["ids"] == [int(v) for v in g["ids" + suffix]], out["ids"]
    assert np.allclose(out["w"], g["w" + suffix], rtol=1e-15, atol=0)
    assert np.allclose(out["routed"], g["routed" + suffix], rtol=1e-14, atol=1e-17)
    for key in ("routed_bf16", "sum", "y"):
        assert np.array_equal(out[key], g[key + suffix]), key


def test_layer_worked_example():
    g = golden()
    x, r = hand_inputs()
    out = M.layer_forward(hand_layer(), x, r)
    _check(out, g, "")
    assert np.allclose(out["shared"], g["shared"], rtol=1e-14, atol=1e-17)
    assert np.array_equal(out["shared_bf16"], g["shared_bf16"])


def test_layer_worked_example_without_shared_expert():
    g = golden()
    x, r = hand_inputs()
    out = M.layer_forward(hand_layer(with_shared=False), x, r)
    _check(out, g, "_2in")
    assert not np.any(out["shared"])


def test_layer_residual_defaults_to_the_ffn_input():
    """A single layer takes x as both FFN input and residual."""
    x, _ = hand_inputs()
    L = hand_layer()
    a = M.layer_forward(L, x)
    b = M.layer_forward(L, x, x)
    for key in ("sum", "y", "routed_bf16", "shared_bf16"):
        assert np.array_equal(a[key], b[key]), key
