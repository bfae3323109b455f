"""Oracle: the decode-time MoE FFN stage, plain and slow, fp64 accumulation.

TEST INFRASTRUCTURE. Only the tests, the package's smoke check and the CPU
baseline of the benchmark may import this module. It shares no code with the
CUDA path; weights and inputs come from the seeded generator as bytes.

Sources (sparkinfer pull-request pages):
* [R] "perf(qwen3.6): fused router GEMV+top-k + folded residual-norm (decode)"
  (PR #273), Summary item 1: router logits for all experts, top-8 ordered by
  value descending with ties to the lower expert index (the rank-select it
  replaces counts, for each expert, the experts that beat it). Summary item 2:
  routed + shared + residual folded into one 3-input add+RMSNorm, bit-identical
  to the separate residual_add followed by the 2-input add_rmsnorm2.
  "Relation to open PRs": the shared expert's output is gated by a
  sigmoid of a GEMV (gemv_sigmoid).
* [S] "perf(qwen3.6): fuse decode kernel launches - shared-expert + GDN
  conv/L2-norm" (PR #239), Summary item 1: the shared expert's gate and up
  GEMVs and the SwiGLU, h = silu(gate) * up, then a separate down GEMV.
* [Q] "Q4_K shared-expert FFN kernels + Q8_0/Q5_K->Q4_K requant of the MoE FFN
  stage" (PR #359), Summary: expert chain FNQ Q8_1 -> gate/up . silu ->
  quant_h Q8_1 -> down, with int8 dot products against Q4_K / Q8_0 weights.
* Softmax over the 8 selected logits is the statement of the workload
  (the pages do not print where the softmax runs).
"""
from __future__ import annotations

import numpy as np

from . import formats as F


def _bf16_tensor_to_f64(t) -> np.ndarray:
    """bf16 torch tensor -> float64 values, decoded from its bits."""
    import torch
    return F.bf16_from_bits(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _np(t):
    return t.cpu().numpy() if hasattr(t, "cpu") else np.asarray(t)


def as_f64(t) -> np.ndarray:
    """Any generator tensor (bf16, fp32, int) -> exact float64 numpy values."""
    if hasattr(t, "dtype") and str(t.dtype) == "torch.bfloat16":
        return _bf16_tensor_to_f64(t)
    return _np(t).astype(np.float64)


# ----------------------------------------------------------------------------
# Router and top-k  [R] Summary item 1
# ----------------------------------------------------------------------------

def router_logits(x, w_router) -> np.ndarray:
    """l_e = sum_h W_r[e, h] * x[h], fp64 (bf16 / fp32 inputs widen exactly)."""
    return as_f64(w_router) @ as_f64(x)


def topk_sort(logits, k: int = 8) -> list:
    """Experts ordered by logit descending, ties to the lower index; first k."""
    l = [float(v) for v in np.asarray(logits, dtype=np.float64)]
    return sorted(range(len(l)), key=lambda e: (-l[e], e))[:k]


def topk_rank_select(logits, k: int = 8) -> list:
    """The rank scan the fused kernel replaced: rank_e = number of experts j
    with l_j > l_e, or l_j == l_e and j < e; experts with rank < k, in rank
    order. O(E^2)."""
    l = np.asarray(logits, dtype=np.float64)
    e = np.arange(l.size)
    beats = (l[None, :] > l[:, None]) | ((l[None, :] == l[:, None]) & (e[None, :] < e[:, None]))
    rank = beats.sum(axis=1)
    out = [-1] * k
    for ex in range(l.size):
        if rank[ex] < k:
            out[rank[ex]] = ex
    return out


def softmax_selected(logits, ids) -> np.ndarray:
    """w_r = exp(l_r - m) / sum_j exp(l_j - m) over the selected logits only."""
    l = np.asarray(logits, dtype=np.float64)[list(ids)]
    ex = np.exp(l - l.max())
    return ex / ex.sum()


def route(logits, k: int = 8):
    ids = topk_sort(logits, k)
    return ids, softmax_selected(logits, ids)


# ----------------------------------------------------------------------------
# GEMV against encoded weights
# ----------------------------------------------------------------------------

def silu(z):
    return z / (1.0 + np.exp(-z))


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def q4_k_block_dots(w_rows, a: dict) -> np.ndarray:
    """Integer dot of every (row, 32-block): sum_i q_w,i * q_a,i, exact int64.
    w_rows uint8 [rows, K/256*144]; returns int64 [rows, K/32]."""
    _, _, _, _, q = F.q4_k_fields(F.q4_k_rows(w_rows))          # [rows, nsb, 8, 32]
    rows, nsb = q.shape[0], q.shape[1]
    qa = a["q"].reshape(nsb, 8, 32)
    return np.einsum("rsji,sji->rsj", q, qa).reshape(rows, nsb * 8)


def q5_k_block_dots(w_rows, a: dict) -> np.ndarray:
    """The same for Q5_K rows (5-bit codes 0..31): uint8 [rows, K/256*176] ->
    int64 [rows, K/32]."""
    _, _, _, _, q = F.q5_k_fields(F.q5_k_rows(w_rows))          # [rows, nsb, 8, 32]
    rows, nsb = q.shape[0], q.shape[1]
    qa = a["q"].reshape(nsb, 8, 32)
    return np.einsum("rsji,sji->rsj", q, qa).reshape(rows, nsb * 8)


def matvec_q4_k(w_rows, a: dict) -> np.ndarray:
    """Q4_K weights x Q8_1 activations, integer mode. For row r and 32-block b
    (sub-block j of super-block s): acc += d*sc_j*d_a(b)*sum_i q_w q_a
    - dmin*m_j*s_a(b); integer sums exact, combination in fp64."""
    d, dmin, sc, m, _ = F.q4_k_fields(F.q4_k_rows(w_rows))       # [rows, nsb], [rows, nsb, 8]
    rows, nsb = d.shape
    isum = q4_k_block_dots(w_rows, a).reshape(rows, nsb, 8).astype(np.float64)
    da = a["d"].reshape(nsb, 8)
    sa = a["s"].reshape(nsb, 8)
    term = d[..., None] * sc * da[None] * isum - dmin[..., None] * m * sa[None]
    return term.reshape(rows, -1).sum(axis=1)


def matvec_q5_k(w_rows, a: dict) -> np.ndarray:
    """Q5_K weights x Q8_1 activations, integer mode: as matvec_q4_k with
    5-bit codes (the same exact integer block sums, the same combination)."""
    d, dmin, sc, m, q = F.q5_k_fields(F.q5_k_rows(w_rows))
    rows, nsb = d.shape
    qa = a["q"].reshape(nsb, 8, 32)
    isum = np.einsum("rsji,sji->rsj", q, qa).astype(np.float64)
    da = a["d"].reshape(nsb, 8)
    sa = a["s"].reshape(nsb, 8)
    term = d[..., None] * sc * da[None] * isum - dmin[..., None] * m * sa[None]
    return term.reshape(rows, -1).sum(axis=1)


def matvec_q8_0(w_rows, a: dict) -> np.ndarray:
    """Q8_0 weights x Q8_1 activations: acc += d_w(b) * d_a(b) * sum_i q_w q_a."""
    dw, qw = F.q8_0_fields(F.q8_0_rows(w_rows))                  # [rows, nb], [rows, nb, 32]
    isum = np.einsum("rbi,bi->rb", qw, a["q"]).astype(np.float64)
    return (dw * a["d"][None] * isum).sum(axis=1)


def matvec_bf16(w_rows, x) -> np.ndarray:
    """bf16 weights (uint8 little-endian bytes [rows, 2K]) x float64 vector."""
    w = np.ascontiguousarray(_np(w_rows), dtype=np.uint8).view(np.uint16)
    return F.bf16_from_bits(w) @ np.asarray(x, dtype=np.float64)


def matvec(fmt: str, w_rows, act):
    if fmt == "q4_k":
        return matvec_q4_k(_np(w_rows), act)
    if fmt == "q5_k":
        return matvec_q5_k(_np(w_rows), act)
    if fmt == "q8_0":
        return matvec_q8_0(_np(w_rows), act)
    if fmt == "bf16":
        return matvec_bf16(w_rows, act)
    raise ValueError(fmt)


def dequant_rows(fmt: str, w_rows) -> np.ndarray:
    """Encoded rows -> float64 weights [rows, K]."""
    w = _np(w_rows)
    if fmt == "q4_k":
        return F.q4_k_dequant(F.q4_k_rows(w)).reshape(w.shape[0], -1)
    if fmt == "q5_k":
        return F.q5_k_dequant(F.q5_k_rows(w)).reshape(w.shape[0], -1)
    if fmt == "q8_0":
        return F.q8_0_dequant(F.q8_0_rows(w)).reshape(w.shape[0], -1)
    if fmt == "bf16":
        return F.bf16_from_bits(np.ascontiguousarray(w, dtype=np.uint8).view(np.uint16))
    raise ValueError(fmt)


# ----------------------------------------------------------------------------
# Load-time requant ([Q] Summary, bullets 1 and 2)
# ----------------------------------------------------------------------------

def requant_q4_k(fmt: str, w_rows) -> np.ndarray:
    """Q8_0 or Q5_K rows [rows, bytes] -> Q4_K rows: the source weights
    dequantised and rounded to fp32 (each product of the definition is exact in
    fp32, so this is one rounding of the exact value), then q4_k_quantize."""
    w32 = F.fp32(dequant_rows(fmt, w_rows)).astype(np.float32)
    return F.q4_k_quantize(w32)


# ----------------------------------------------------------------------------
# Expert FFN  [S] Summary item 1, [Q] Summary
# ----------------------------------------------------------------------------

def expert_ffn(fmt: str, gate, up, down, x, x_q8_1: dict | None = None,
               down_fmt: str | None = None) -> dict:
    """One expert on one token: h = silu(G x) * (U x); y = D h (D in
    ``down_fmt``, default ``fmt``: the pages' native routed down is Q5_K).

    Quantised weights (integer mode): x enters as its Q8_1 blocks; h is
    rounded to fp32 and quantised to Q8_1 before the down GEMV.
    bf16 weights: fp64 dot products of the exact bf16 values, h unrounded.
    Returns {"g", "u", "h", "y"} in float64.
    """
    if fmt == "bf16":
        g = matvec_bf16(gate, x)
        u = matvec_bf16(up, x)
        h = silu(g) * u
        return {"g": g, "u": u, "h": h, "y": matvec_bf16(down, h)}
    a = x_q8_1 if x_q8_1 is not None else F.q8_1_quantize(F.fp32(x))
    g = matvec(fmt, gate, a)
    u = matvec(fmt, up, a)
    h = silu(g) * u
    ah = F.q8_1_quantize(F.fp32(h))
    return {"g": g, "u": u, "h": h, "h_q8_1": ah, "y": matvec(down_fmt or fmt, down, ah)}


def expert_ffn_float(fmt: str, gate, up, down, x, down_fmt: str | None = None) -> dict:
    """Diagnostic float mode: dequantised weights x unquantised activations."""
    G, U = (dequant_rows(fmt, m) for m in (gate, up))
    D = dequant_rows(down_fmt or fmt, down)
    xx = np.asarray(x, dtype=np.float64)
    g, u = G @ xx, U @ xx
    h = silu(g) * u
    return {"g": g, "u": u, "h": h, "y": D @ h}


def expert_ffn_fp16(fmt: str, gate, up, down, x) -> dict:
    """Tensor-core mode for batched tokens: weights dequantised, rounded to
    fp32 then fp16; x rounded to fp16; h = silu(g)*u rounded to fp16 before the
    down GEMM; products and sums exact (fp64)."""
    G, U, D = (F.fp16(F.fp32(dequant_rows(fmt, m))) for m in (gate, up, down))
    x16 = F.fp16(np.asarray(x, dtype=np.float64))
    g, u = G @ x16, U @ x16
    h = silu(g) * u
    return {"g": g, "u": u, "h": h, "y": D @ F.fp16(h)}


# ----------------------------------------------------------------------------
# Residual fold  [R] Summary item 2
# ----------------------------------------------------------------------------

def add_rmsnorm3(a, b, c, w_norm, eps: float):
    """t = bf16(a + b); sum = bf16(t + c) (c None: sum = t); y = bf16(sum * r * w)
    with r = 1/sqrt(mean(sum^2) + eps) in fp64. Inputs are bf16 values."""
    t = F.bf16(np.asarray(a, np.float64) + np.asarray(b, np.float64))
    s = t if c is None else F.bf16(t + np.asarray(c, np.float64))
    r = 1.0 / np.sqrt(np.mean(s * s) + eps)
    return s, F.bf16(s * r * np.asarray(w_norm, np.float64))


def residual_add(a, b):
    """The separate kernel the fold removed: bf16(a + b)."""
    return F.bf16(np.asarray(a, np.float64) + np.asarray(b, np.float64))


def add_rmsnorm2(a, residual, w_norm, eps: float):
    """The 2-input norm: sum = bf16(a + residual), y = bf16(sum * r * w)."""
    s = F.bf16(np.asarray(a, np.float64) + np.asarray(residual, np.float64))
    r = 1.0 / np.sqrt(np.mean(s * s) + eps)
    return s, F.bf16(s * r * np.asarray(w_norm, np.float64))


def add_rmsnorm_unfused(a, b, c, w_norm, eps: float):
    """residual_add(routed, shared) followed by add_rmsnorm2(., residual)."""
    return add_rmsnorm2(residual_add(a, b), c, w_norm, eps)


# ----------------------------------------------------------------------------
# Whole layer and stack
# ----------------------------------------------------------------------------

def _expert_slot(L, e: int) -> int:
    return L["expert_ids"].index(int(e))


def moe_ffn(L, x, ids, w, mode: str = "int") -> dict:
    """Routed experts combined in rank order, routed = sum_r w_r * y_{e_r},
    and the shared expert shared = sigmoid(w_sg . x) * y_s.

    ``L`` is a generator layer holding (at least) the experts in ``ids``;
    ``mode`` "int" (quantised integer path), "float" or "fp16".
    """
    spec = L["spec"]
    ffn = {"int": expert_ffn, "float": expert_ffn_float, "fp16": expert_ffn_fp16}[mode]
    xx = as_f64(x)
    a = F.q8_1_quantize(F.fp32(xx)) if (spec.expert_type != "bf16" and mode == "int") else None
    ys = []
    down_fmt = getattr(spec, "down_type", None) or spec.expert_type
    for e in ids:
        s = _expert_slot(L, e)
        args = (spec.expert_type, L["gate"][s], L["up"][s], L["down"][s], xx)
        if mode == "int":
            ys.append(ffn(*args, a, down_fmt=down_fmt))
        elif mode == "float":
            ys.append(ffn(*args, down_fmt=down_fmt))
        else:
            ys.append(ffn(*args))
    routed = np.zeros(spec.hidden)
    for r in range(len(ids)):
        routed = routed + w[r] * ys[r]["y"]
    out = {"routed": routed, "experts": ys, "x_q8_1": a}
    if spec.shared_inter > 0:
        gs = sigmoid(float(as_f64(L["w_sg"]) @ xx))
        sargs = (spec.shared_type, L["sh_gate"], L["sh_up"], L["sh_down"], xx)
        if mode == "int" and spec.shared_type != "bf16":
            ys_ = ffn(*sargs, a if a is not None else F.q8_1_quantize(F.fp32(xx)))
        elif mode == "int":
            ys_ = ffn(*sargs)
        else:
            ys_ = ffn(*sargs)
        out.update(shared=gs * ys_["y"], shared_gate=gs, shared_expert=ys_)
    else:
        out.update(shared=np.zeros(spec.hidden), shared_gate=0.0)
    return out


def layer_forward(L, x, residual=None, ids=None, mode: str = "int") -> dict:
    """One layer on one token. x (bf16 [H]) is the FFN input, ``residual``
    (bf16 [H]) defaults to x. ``ids`` overrides the selection (used only where
    the fp32 and fp64 logits disagree on a near-tie). Routed and shared
    outputs are rounded to bf16 where the library stores them."""
    spec = L["spec"]
    xx = as_f64(x)
    res = xx if residual is None else as_f64(residual)
    logits = router_logits(xx, L["w_router"])
    if ids is None:
        ids = topk_sort(logits, spec.top_k)
    w = softmax_selected(logits, ids)
    f = moe_ffn(L, xx, ids, w, mode)
    routed16 = F.bf16(f["routed"])
    shared16 = F.bf16(f["shared"])
    if spec.shared_inter > 0:
        s, y = add_rmsnorm3(routed16, shared16, res, as_f64(L["w_norm"]), spec.eps)
    else:
        s, y = add_rmsnorm2(routed16, res, as_f64(L["w_norm"]), spec.eps)
    return {"logits": logits, "ids": list(ids), "w": w, "routed": f["routed"],
            "routed_bf16": routed16, "shared": f["shared"], "shared_bf16": shared16,
            "shared_gate": f["shared_gate"], "sum": s, "y": y, "ffn": f}
