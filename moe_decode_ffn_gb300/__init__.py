"""Python binding of libsi_moe: the decode-time MoE FFN stage on GB300.

Argument marshalling only. Every step of the computation runs in the CUDA
kernels of ``libsi_moe.so`` (built in-tree from ``csrc/``); PyTorch supplies
device memory and streams. There is no CPU fallback: if the library is not
built, or a tensor is not on a CUDA device, the calls raise.

Names follow the C ABI in ``include/si_moe.h``.
"""
from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB, build  # noqa: F401

SI_OK, SI_ERR_INVALID_ARG, SI_ERR_UNSUPPORTED, SI_ERR_WORKSPACE = 0, 1, 2, 3
SI_ERR_CUDA, SI_ERR_HANDSHAKE, SI_ERR_TIMEOUT = 4, 5, 6
SI_F32, SI_F16, SI_Q8_0, SI_Q8_1, SI_Q4_K, SI_Q5_K, SI_BF16 = 0, 1, 8, 9, 12, 13, 30
DTYPES = {"f32": SI_F32, "f16": SI_F16, "q8_0": SI_Q8_0, "q8_1": SI_Q8_1, "q4_k": SI_Q4_K,
          "q5_k": SI_Q5_K, "bf16": SI_BF16}

_vp = ctypes.c_void_p
_i32, _i64, _sz, _f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float


class SiError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


class SiMoeLayer(ctypes.Structure):
    """Mirror of ``si_moe_layer``."""
    _fields_ = [
        ("hidden", _i32), ("n_experts", _i32), ("top_k", _i32), ("inter", _i32),
        ("expert_type", _i32), ("w_gate", _vp), ("w_up", _vp), ("w_down", _vp),
        ("shared_inter", _i32), ("shared_type", _i32),
        ("ws_gate", _vp), ("ws_up", _vp), ("ws_down", _vp), ("w_shared_sigmoid", _vp),
        ("w_router", _vp), ("router_type", _i32), ("w_norm", _vp), ("eps", _f32),
        ("down_type", _i32),
    ]


# name -> (restype, argtypes), exactly the exports of include/si_moe.h
SIGNATURES = {
    "si_status_string": (ctypes.c_char_p, [_i32]),
    "si_version": (_i32, []),
    "si_row_bytes": (_sz, [_i32, _i64]),
    "si_quantize_q8_1": (_i32, [_vp, _i32, _i64, _vp, _vp]),
    "si_moe_router_workspace_bytes": (_sz, [_i32, _i32, _i32]),
    "si_moe_router_topk": (_i32, [_vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp,
                                  _vp, _sz, _vp]),
    "si_moe_router_topk_noalloc": (_i32, [_vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp,
                                          _vp, _vp]),
    "si_moe_router_noalloc_status": (_i32, [_vp, ctypes.POINTER(_i32)]),
    "si_moe_ffn_workspace_bytes": (_sz, [ctypes.POINTER(SiMoeLayer), _i32]),
    "si_moe_ffn_decode": (_i32, [ctypes.POINTER(SiMoeLayer), _i32, _vp, _vp, _vp, _vp, _vp, _vp,
                                 _vp, _sz, _vp]),
    "si_moe_ffn_decode_ep": (_i32, [ctypes.POINTER(SiMoeLayer), _i32, _i32, _vp, _vp, _vp, _vp, _vp,
                                    _vp, _sz, _vp]),
    "si_moe_combine_slots": (_i32, [_vp, _vp, _i32, _i32, _vp, _vp]),
    "si_moe_ffn_batched_workspace_bytes": (_sz, [ctypes.POINTER(SiMoeLayer), _i32]),
    "si_moe_ffn_batched": (_i32, [ctypes.POINTER(SiMoeLayer), _i32, _i32, _vp, _vp, _vp, _vp, _vp,
                                  _sz, _vp]),
    "si_add_rmsnorm3": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _f32, _vp, _vp, _vp, _vp]),
    "si_moe_layer_workspace_bytes": (_sz, [ctypes.POINTER(SiMoeLayer)]),
    "si_moe_layer_decode": (_i32, [ctypes.POINTER(SiMoeLayer), _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                   _vp, _vp, _sz, _vp]),
    "si_moe_stack_workspace_bytes": (_sz, [ctypes.POINTER(SiMoeLayer), _i32]),
    "si_moe_stack_graph_create": (_i32, [ctypes.POINTER(SiMoeLayer), _i32, _i32, _vp, _vp, _vp,
                                         _vp, _vp, _sz, _vp, ctypes.POINTER(_vp)]),
    "si_moe_stack_graph_create_mode": (_i32, [ctypes.POINTER(SiMoeLayer), _i32, _i32, _vp, _vp,
                                              _vp, _vp, _vp, _sz, _i32, _vp,
                                              ctypes.POINTER(_vp)]),
    "si_graph_is_persistent": (_i32, [_vp]),
    "si_moe_layer_batched_workspace_bytes": (_sz, [ctypes.POINTER(SiMoeLayer), _i32]),
    "si_moe_layer_decode_batched": (_i32, [ctypes.POINTER(SiMoeLayer), _i32, _i32, _vp, _vp, _vp, _vp,
                                           _vp, _vp, _vp, _vp, _sz, _vp]),
    "si_moe_stack_batched_workspace_bytes": (_sz, [ctypes.POINTER(SiMoeLayer), _i32, _i32]),
    "si_moe_stack_graph_create_batched": (_i32, [ctypes.POINTER(SiMoeLayer), _i32, _i32, _i32, _vp,
                                                 _vp, _vp, _vp, _vp, _sz, _vp, ctypes.POINTER(_vp)]),
    "si_requant_q4_k": (_i32, [_vp, _i32, _i64, _i64, _vp, _vp]),
    "si_graph_launch": (_i32, [_vp, _vp]),
    "si_graph_destroy": (None, [_vp]),
    "si_workspace_status": (_i32, [_vp, _vp, ctypes.POINTER(_i32)]),
    "si_moe_ffn_gateup": (_i32, [ctypes.POINTER(SiMoeLayer), _i32, _vp, _vp, _vp, _vp, _sz, _vp]),
    "si_test_q4k_block_dots": (_i32, [_vp, _i32, _i32, _vp, _vp, _vp]),
    "si_test_block_dots": (_i32, [_i32, _vp, _i32, _i32, _vp, _i32, _vp, _vp]),
    "si_test_wait_timeout": (_i32, [ctypes.c_uint64, _vp, _vp]),
    "si_test_poll_timeout": (_i32, [ctypes.c_uint64, _vp, _vp]),
    "si_test_umma_f16": (_i32, [_vp, _vp, _i32, _i32, _vp, _vp, _vp]),
    "si_test_unfused_add_rmsnorm": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _f32, _vp, _vp, _vp,
                                           _vp]),
}

_lib = None


def library() -> ctypes.CDLL:
    """The loaded libsi_moe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is not built; run moe_decode_ffn_gb300.build() first")
        lib = ctypes.CDLL(LIB)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return library().si_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != SI_OK:
        raise SiError(status, where)


def _cuda(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _opt(t, name):
    return None if t is None else _cuda(t, name)


def _shaped(t, name: str, numel: int, dtypes) -> int:
    """Device pointer of ``t`` after checking that it holds exactly ``numel``
    elements of one of ``dtypes``: the C ABI takes raw pointers and cannot
    tell a short buffer from a long one."""
    p = _cuda(t, name)
    if t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {' or '.join(map(str, dtypes))}")
    return p


_BF16 = (torch.bfloat16,)
_FLOATS = (torch.bfloat16, torch.float32)
_I32 = (torch.int32,)
_F32 = (torch.float32,)
_U8 = (torch.uint8,)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _xtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SI_BF16
    if t.dtype == torch.float32:
        return SI_F32
    raise ValueError(f"unsupported dtype {t.dtype}")


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zeroed, 256-byte aligned device workspace of ``nbytes`` bytes."""
    if nbytes <= 0:
        raise ValueError("workspace size query returned 0 (invalid shapes)")
    return torch.zeros(int(nbytes), dtype=torch.uint8, device=device or "cuda")


# ----------------------------------------------------------------------------
# calls
# ----------------------------------------------------------------------------

def si_quantize_q8_1(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    n = x.numel()
    if out is None:
        out = torch.empty(n // 32 * 36, dtype=torch.uint8, device=x.device)
    _check(library().si_quantize_q8_1(_cuda(x, "x"), _xtype(x), n,
                                      _shaped(out, "out", n // 32 * 36, _U8), _stream(stream)),
           "si_quantize_q8_1")
    return out


def router_workspace_bytes(n_experts: int, hidden: int, n_tokens: int) -> int:
    return int(library().si_moe_router_workspace_bytes(n_experts, hidden, n_tokens))


def si_moe_router_topk(x: torch.Tensor, w_router: torch.Tensor, top_k: int = 8,
                       want_logits: bool = False, ws: torch.Tensor | None = None, stream=None):
    """x [T, H], w_router [E, H] (bf16 or fp32) -> (ids int32 [T, k], w fp32 [T, k], logits|None)."""
    T, H = x.shape
    E = w_router.shape[0]
    if tuple(w_router.shape) != (E, H):
        raise ValueError(f"w_router has shape {tuple(w_router.shape)}, expected ({E}, {H})")
    dev = x.device
    ids = torch.empty(T, top_k, dtype=torch.int32, device=dev)
    wts = torch.empty(T, top_k, dtype=torch.float32, device=dev)
    logits = torch.empty(T, E, dtype=torch.float32, device=dev) if want_logits else None
    if ws is None:
        ws = workspace(router_workspace_bytes(E, H, T), dev)
    _check(library().si_moe_router_topk(
        _cuda(x, "x"), _xtype(x), _cuda(w_router, "w_router"), _xtype(w_router), H, E, top_k, T,
        _cuda(ids, "ids"), _cuda(wts, "w"), _opt(logits, "logits"), _cuda(ws, "ws"), ws.numel(),
        _stream(stream)), "si_moe_router_topk")
    return ids, wts, logits


def si_moe_router_topk_noalloc(x: torch.Tensor, w_router: torch.Tensor, top_k: int = 8,
                               want_logits: bool = False, stream=None):
    """Router + top-k through the entry point that allocates nothing on the
    device side (its scratch is built into the library). The output tensors
    here are the caller's; the call itself needs no workspace."""
    T, H = x.shape
    E = w_router.shape[0]
    if tuple(w_router.shape) != (E, H):
        raise ValueError(f"w_router has shape {tuple(w_router.shape)}, expected ({E}, {H})")
    dev = x.device
    ids = torch.empty(T, top_k, dtype=torch.int32, device=dev)
    wts = torch.empty(T, top_k, dtype=torch.float32, device=dev)
    logits = torch.empty(T, E, dtype=torch.float32, device=dev) if want_logits else None
    _check(library().si_moe_router_topk_noalloc(
        _cuda(x, "x"), _xtype(x), _cuda(w_router, "w_router"), _xtype(w_router), H, E, top_k, T,
        _cuda(ids, "ids"), _cuda(wts, "w"), _opt(logits, "logits"), _stream(stream)),
        "si_moe_router_topk_noalloc")
    return ids, wts, logits


def si_moe_router_noalloc_status(stream=None) -> int:
    """Reads and clears the device status of the no-alloc router's scratch."""
    v = _i32(0)
    _check(library().si_moe_router_noalloc_status(_stream(stream), ctypes.byref(v)),
           "si_moe_router_noalloc_status")
    return v.value


class Layer:
    """Device weights of one layer plus the ``si_moe_layer`` descriptor.

    ``t`` maps the generator's names (gate, up, down, sh_gate, sh_up, sh_down,
    w_sg, w_router, w_norm) to CUDA tensors; formats come from ``spec``.
    """

    def __init__(self, spec, t: dict):
        self.spec, self.t = spec, t
        s = SiMoeLayer()
        s.hidden, s.n_experts, s.top_k, s.inter = spec.hidden, spec.n_experts, spec.top_k, spec.inter
        s.expert_type = DTYPES[spec.expert_type]
        s.w_gate, s.w_up, s.w_down = (_cuda(t[k], k) for k in ("gate", "up", "down"))
        s.shared_inter = spec.shared_inter
        s.shared_type = DTYPES[spec.shared_type]
        if spec.shared_inter > 0:
            s.ws_gate, s.ws_up, s.ws_down, s.w_shared_sigmoid = (
                _cuda(t[k], k) for k in ("sh_gate", "sh_up", "sh_down", "w_sg"))
        if "w_router" in t:
            s.w_router = _cuda(t["w_router"], "w_router")
            s.router_type = _xtype(t["w_router"])
        if "w_norm" in t:
            s.w_norm = _cuda(t["w_norm"], "w_norm")
        s.eps = spec.eps
        s.down_type = DTYPES[spec.down_type] if getattr(spec, "down_type", "") else SI_F32
        self.c = s

    @property
    def ref(self):
        return ctypes.byref(self.c)


def ffn_workspace_bytes(layer: Layer, n_tokens: int = 1) -> int:
    return int(library().si_moe_ffn_workspace_bytes(layer.ref, n_tokens))


def si_moe_ffn_decode(layer: Layer, x: torch.Tensor, ids: torch.Tensor, w: torch.Tensor,
                      x_q8_1: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                      stream=None):
    """One token: x bf16 [H] -> (routed bf16 [H], shared bf16 [H] or None)."""
    H = layer.spec.hidden
    routed = torch.empty(H, dtype=torch.bfloat16, device=x.device)
    shared = torch.empty(H, dtype=torch.bfloat16, device=x.device) if layer.spec.shared_inter else None
    if ws is None:
        ws = workspace(ffn_workspace_bytes(layer), x.device)
    k = layer.spec.top_k
    _check(library().si_moe_ffn_decode(
        layer.ref, 1, _shaped(x, "x", H, _BF16),
        None if x_q8_1 is None else _shaped(x_q8_1, "x_q8_1", H // 32 * 36, _U8),
        _shaped(ids, "ids", k, _I32), _shaped(w, "w", k, _F32),
        _cuda(routed, "routed"), _opt(shared, "shared"), _cuda(ws, "ws"), ws.numel(),
        _stream(stream)), "si_moe_ffn_decode")
    return routed, shared


def si_moe_ffn_decode_ep(layer: Layer, e0: int, e1: int, x: torch.Tensor, ids: torch.Tensor,
                         ws: torch.Tensor | None = None, stream=None):
    """The slots of experts in [e0, e1) for one token: -> (slot_y fp32 [k, H]
    with zeros for the other slots, shared bf16 [H] or None)."""
    H, k = layer.spec.hidden, layer.spec.top_k
    slot_y = torch.empty(k, H, dtype=torch.float32, device=x.device)
    shared = torch.empty(H, dtype=torch.bfloat16, device=x.device) if layer.spec.shared_inter else None
    if ws is None:
        ws = workspace(ffn_workspace_bytes(layer), x.device)
    _check(library().si_moe_ffn_decode_ep(
        layer.ref, e0, e1, _shaped(x, "x", H, _BF16), None, _shaped(ids, "ids", k, _I32),
        _cuda(slot_y, "slot_y"), _opt(shared, "shared"), _cuda(ws, "ws"), ws.numel(), _stream(stream)),
        "si_moe_ffn_decode_ep")
    return slot_y, shared


def si_moe_combine_slots(slot_y: torch.Tensor, w: torch.Tensor, stream=None) -> torch.Tensor:
    """routed = bf16(sum_r w[r] * slot_y[r]) in rank order: slot_y fp32 [k, H], w fp32 [k]."""
    k, H = slot_y.shape
    routed = torch.empty(H, dtype=torch.bfloat16, device=slot_y.device)
    _check(library().si_moe_combine_slots(_shaped(slot_y, "slot_y", k * H, _F32), _shaped(w, "w", k, _F32),
                                          k, H, _cuda(routed, "routed"), _stream(stream)),
           "si_moe_combine_slots")
    return routed


SI_FFN_AUTO, SI_FFN_INT8, SI_FFN_TENSOR = 0, 1, 2


def ffn_batched_workspace_bytes(layer: Layer, n_tokens: int) -> int:
    return int(library().si_moe_ffn_batched_workspace_bytes(layer.ref, n_tokens))


def si_moe_ffn_batched(layer: Layer, x: torch.Tensor, ids: torch.Tensor, w: torch.Tensor,
                       mode: int = SI_FFN_AUTO, ws: torch.Tensor | None = None, stream=None):
    """T tokens with per-token routing: x bf16 [T, H], ids int32 [T, k], w fp32 [T, k]
    -> routed bf16 [T, H]."""
    T = x.shape[0]
    H, k = layer.spec.hidden, layer.spec.top_k
    routed = torch.empty(T, H, dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = workspace(ffn_batched_workspace_bytes(layer, T), x.device)
    _check(library().si_moe_ffn_batched(
        layer.ref, T, mode, _shaped(x, "x", T * H, _BF16), _shaped(ids, "ids", T * k, _I32),
        _shaped(w, "w", T * k, _F32),
        _cuda(routed, "routed"), _cuda(ws, "ws"), ws.numel(), _stream(stream)),
        "si_moe_ffn_batched")
    return routed


def si_add_rmsnorm3(a, b, c, w_norm, eps: float = 1e-6, want_q8: bool = False, stream=None):
    """Rows [R, n] (or [n]) of bf16 -> (sum, norm, norm Q8_1 bytes | None)."""
    n = a.shape[-1]
    rows = a.numel() // n
    s = torch.empty_like(a)
    y = torch.empty_like(a)
    q8 = torch.empty(rows * (n // 32) * 36, dtype=torch.uint8, device=a.device) if want_q8 else None
    _check(library().si_add_rmsnorm3(_shaped(a, "a", rows * n, _BF16), _shaped(b, "b", rows * n, _BF16),
                                     None if c is None else _shaped(c, "c", rows * n, _BF16),
                                     _shaped(w_norm, "w_norm", n, _BF16), n, rows, eps, _cuda(s, "sum"),
                                     _cuda(y, "norm"), _opt(q8, "q8"), _stream(stream)),
           "si_add_rmsnorm3")
    return s, y, q8


def layer_workspace_bytes(layer: Layer) -> int:
    return int(library().si_moe_layer_workspace_bytes(layer.ref))


def si_moe_layer_decode(layer: Layer, x, residual=None, ws=None, stream=None) -> dict:
    H, k = layer.spec.hidden, layer.spec.top_k
    dev = x.device
    out = {n: torch.empty(H, dtype=torch.bfloat16, device=dev)
           for n in ("sum", "y", "routed", "shared")}
    out["ids"] = torch.empty(k, dtype=torch.int32, device=dev)
    out["w"] = torch.empty(k, dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(layer_workspace_bytes(layer), dev)
    res = x if residual is None else residual
    _check(library().si_moe_layer_decode(
        layer.ref, _shaped(x, "x", H, _BF16), _shaped(res, "residual", H, _BF16),
        _cuda(out["sum"], "sum"),
        _cuda(out["y"], "y"), _cuda(out["ids"], "ids"), _cuda(out["w"], "w"),
        _cuda(out["routed"], "routed"), _cuda(out["shared"], "shared"), _cuda(ws, "ws"),
        ws.numel(), _stream(stream)), "si_moe_layer_decode")
    return out


SI_STACK_AUTO, SI_STACK_PER_LAYER, SI_STACK_PERSISTENT = 0, 1, 2


class StackGraph:
    """n_layers x n_tokens decode captured as one CUDA graph (buffers owned here).

    mode: SI_STACK_AUTO (the persistent kernel when it supports the layers),
    SI_STACK_PER_LAYER or SI_STACK_PERSISTENT."""

    def __init__(self, layers, x_in: torch.Tensor, want_ids: bool = True, stream=None,
                 mode: int = SI_STACK_AUTO):
        self.layers = list(layers)
        arr = (SiMoeLayer * len(self.layers))(*[l.c for l in self.layers])
        self._arr = arr
        T, H = x_in.shape
        if H != self.layers[0].spec.hidden or x_in.dtype != torch.bfloat16:
            raise ValueError(f"x_in must be bf16 [T, {self.layers[0].spec.hidden}], got "
                             f"{x_in.dtype} {tuple(x_in.shape)}")
        k = self.layers[0].spec.top_k
        dev = x_in.device
        self.x_in = x_in
        self.y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        self.sum = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        self.ids = (torch.empty(T, len(self.layers), k, dtype=torch.int32, device=dev)
                    if want_ids else None)
        nb = int(library().si_moe_stack_workspace_bytes(arr, len(self.layers)))
        self.ws = workspace(nb, dev)
        h = _vp()
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(torch.cuda.current_stream())
        _check(library().si_moe_stack_graph_create_mode(
            arr, len(self.layers), T, _cuda(x_in, "x_in"), _cuda(self.y, "y"),
            _cuda(self.sum, "sum"), _opt(self.ids, "ids"), _cuda(self.ws, "ws"), self.ws.numel(),
            mode, _stream(cap), ctypes.byref(h)), "si_moe_stack_graph_create_mode")
        self.handle = h
        self.stream = stream
        self.persistent = bool(library().si_graph_is_persistent(h))

    def launch(self, stream=None):
        _check(library().si_graph_launch(self.handle, _stream(stream)), "si_graph_launch")

    def close(self):
        if self.handle:
            library().si_graph_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def layer_batched_workspace_bytes(layer: Layer, n_tokens: int) -> int:
    return int(library().si_moe_layer_batched_workspace_bytes(layer.ref, n_tokens))


def si_moe_layer_decode_batched(layer: Layer, x: torch.Tensor, residual=None, mode: int = SI_FFN_AUTO,
                                ws=None, stream=None) -> dict:
    """T tokens through one layer, each routed on its own: x bf16 [T, H] ->
    {sum, y, routed: bf16 [T, H], ids: int32 [T, k], w: fp32 [T, k]}."""
    T, H = x.shape
    k = layer.spec.top_k
    dev = x.device
    out = {n: torch.empty(T, H, dtype=torch.bfloat16, device=dev) for n in ("sum", "y", "routed")}
    out["ids"] = torch.empty(T, k, dtype=torch.int32, device=dev)
    out["w"] = torch.empty(T, k, dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(layer_batched_workspace_bytes(layer, T), dev)
    res = x if residual is None else residual
    _check(library().si_moe_layer_decode_batched(
        layer.ref, T, mode, _shaped(x, "x", T * H, _BF16), _shaped(res, "residual", T * H, _BF16),
        _cuda(out["sum"], "sum"), _cuda(out["y"], "y"), _cuda(out["ids"], "ids"), _cuda(out["w"], "w"),
        _cuda(out["routed"], "routed"), _cuda(ws, "ws"), ws.numel(), _stream(stream)),
        "si_moe_layer_decode_batched")
    return out


class BatchedStackGraph:
    """T tokens through n_layers layers together (per-token routing), captured
    as one CUDA graph; buffers owned here."""

    def __init__(self, layers, x_in: torch.Tensor, mode: int = SI_FFN_AUTO, want_ids: bool = True):
        self.layers = list(layers)
        arr = (SiMoeLayer * len(self.layers))(*[l.c for l in self.layers])
        self._arr = arr
        T, H = x_in.shape
        if H != self.layers[0].spec.hidden or x_in.dtype != torch.bfloat16:
            raise ValueError(f"x_in must be bf16 [T, {self.layers[0].spec.hidden}]")
        k = self.layers[0].spec.top_k
        dev = x_in.device
        self.x_in = x_in
        self.y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        self.sum = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        self.ids = (torch.empty(len(self.layers), T, k, dtype=torch.int32, device=dev)
                    if want_ids else None)
        nb = int(library().si_moe_stack_batched_workspace_bytes(arr, len(self.layers), T))
        self.ws = workspace(nb, dev)
        h = _vp()
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(torch.cuda.current_stream())
        _check(library().si_moe_stack_graph_create_batched(
            arr, len(self.layers), T, mode, _cuda(x_in, "x_in"), _cuda(self.y, "y"),
            _cuda(self.sum, "sum"), _opt(self.ids, "ids"), _cuda(self.ws, "ws"), self.ws.numel(),
            _stream(cap), ctypes.byref(h)), "si_moe_stack_graph_create_batched")
        self.handle = h
        # one token in the automatic mode: the persistent stack kernel when it takes the layers
        self.persistent = bool(library().si_graph_is_persistent(h))

    def launch(self, stream=None):
        _check(library().si_graph_launch(self.handle, _stream(stream)), "si_graph_launch")

    def close(self):
        if self.handle:
            library().si_graph_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def si_requant_q4_k(src: torch.Tensor, src_type: str, rows: int, cols: int,
                    out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Load-time requant: Q8_0 or Q5_K rows (uint8 [rows, row bytes]) -> Q4_K
    rows (uint8 [rows, cols / 256 * 144])."""
    if out is None:
        out = torch.empty(rows, cols // 256 * 144, dtype=torch.uint8, device=src.device)
    src_rb = int(library().si_row_bytes(DTYPES[src_type], cols))
    _check(library().si_requant_q4_k(_shaped(src, "src", rows * src_rb, _U8), DTYPES[src_type],
                                     rows, cols, _shaped(out, "out", rows * (cols // 256 * 144), _U8),
                                     _stream(stream)), "si_requant_q4_k")
    return out


def si_workspace_status(ws: torch.Tensor, stream=None) -> int:
    v = _i32(0)
    _check(library().si_workspace_status(_cuda(ws, "ws"), _stream(stream), ctypes.byref(v)),
           "si_workspace_status")
    return v.value


def si_test_q4k_block_dots(w: torch.Tensor, rows: int, k: int, a_q8_1: torch.Tensor, stream=None):
    out = torch.empty(rows, k // 32, dtype=torch.int32, device=w.device)
    _check(library().si_test_q4k_block_dots(_shaped(w, "w", rows * (k // 256 * 144), _U8), rows, k,
                                            _shaped(a_q8_1, "a", k // 32 * 36, _U8),
                                            _cuda(out, "out"), _stream(stream)),
           "si_test_q4k_block_dots")
    return out


SI_TEST_DOTS_Q4K_SB, SI_TEST_DOTS_Q4K_HALF, SI_TEST_DOTS_Q5K_HALF = 0, 1, 2
SI_TEST_DOTS_Q4K_SB_TOKENS, SI_TEST_DOTS_Q4K_HALF_TOKENS = 3, 4


def si_test_block_dots(kind: int, w: torch.Tensor, rows: int, k: int, a_q8_1: torch.Tensor,
                       n_vec: int = 1, stream=None):
    """Exact int32 block sums of the library's integer dot helper `kind` ->
    int32 [n_vec, rows, k / 32]."""
    sbb = 176 if kind == SI_TEST_DOTS_Q5K_HALF else 144
    out = torch.empty(n_vec, rows, k // 32, dtype=torch.int32, device=w.device)
    _check(library().si_test_block_dots(kind, _shaped(w, "w", rows * (k // 256 * sbb), _U8), rows, k,
                                        _shaped(a_q8_1, "a", n_vec * (k // 32 * 36), _U8), n_vec,
                                        _cuda(out, "out"), _stream(stream)),
           "si_test_block_dots")
    return out


def si_test_unfused_add_rmsnorm(a, b, c, w_norm, eps: float = 1e-6, stream=None):
    n = a.shape[-1]
    rows = a.numel() // n
    t, s, y = torch.empty_like(a), torch.empty_like(a), torch.empty_like(a)
    _check(library().si_test_unfused_add_rmsnorm(
        _cuda(a, "a"), _cuda(b, "b"), _cuda(c, "c"), _cuda(w_norm, "w_norm"), n, rows, eps,
        _cuda(t, "t"), _cuda(s, "sum"), _cuda(y, "norm"), _stream(stream)),
        "si_test_unfused_add_rmsnorm")
    return s, y


def device_layer(spec, seed: int, layer: int = 0, device="cuda") -> Layer:
    """Generate one layer's synthetic weights on the device and wrap them."""
    import gen
    L = gen.make_layer(spec, seed, layer, device=device)
    t = {k: v for k, v in L.items() if isinstance(v, torch.Tensor)}
    return Layer(spec, t)
