"""Seeded synthetic inputs for the decode-time MoE FFN stage.

This module feeds both the CUDA path and the CPU oracle. It holds none of the
method's arithmetic (no GEMV, no top-k, no activation quantisation, no norm):
only

* a counter-based random stream: every tensor has a 64-bit key built from
  (seed, layer, role, expert); element i of that tensor is the SplitMix64
  finaliser applied to ``key + (i + 1) * golden_gamma`` (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014);
* a normal approximation with integer-only arithmetic: the sum of the four
  16-bit lanes of one 64-bit draw (Irwin-Hall with n = 4), centred and scaled to
  unit variance. It is bounded at +-3.46 sigma. Using no transcendental
  functions keeps the CPU and GPU evaluations bit-identical;
* the weight *encoders* that turn float weights into the block formats the
  method reads (Q4_K super-blocks, Q8_0 blocks, bf16). The method only ever
  decodes these formats; the encoders are input preparation, in the way a
  model file is prepared before decode starts.

Everything is written with torch integer / fp32 / fp64 elementwise ops so that
the same function, run on CPU (for the oracle) or on CUDA (to fill device
memory with all experts of all layers), produces identical bytes.
"""
from __future__ import annotations

import dataclasses
import math

import torch

MASK64 = (1 << 64) - 1
GOLDEN_GAMMA = 0x9E3779B97F4A7C15
_MIX_M1 = 0xBF58476D1CE4E5B9
_MIX_M2 = 0x94D049BB133111EB
_KEY_ORIGIN = 0x243F6A8885A308D3

# Tensor roles: the third component of every stream key.
ROLE_X = 1
ROLE_ROUTER = 2
ROLE_GATE = 3
ROLE_UP = 4
ROLE_DOWN = 5
ROLE_SH_GATE = 6
ROLE_SH_UP = 7
ROLE_SH_DOWN = 8
ROLE_SH_SIGMOID = 9
ROLE_NORM = 10
ROLE_TIE_W = 11
ROLE_TIE_X = 12
ROLE_TIE_MASK = 13
ROLE_TIE_POOL = 14

WEIGHT_STD = 0.02
NORM_MEAN, NORM_STD = 1.0, 0.1

QK_K = 256          # weights per Q4_K super-block
Q4_K_BYTES = 144    # bytes per Q4_K super-block
Q5_K_BYTES = 176    # bytes per Q5_K super-block
QK8 = 32            # weights per Q8_0 / Q8_1 block
Q8_0_BYTES = 34
Q8_1_BYTES = 36


def _s64(c: int) -> int:
    """Two's-complement int64 value with the same 64 bits as unsigned ``c``."""
    c &= MASK64
    return c - (1 << 64) if c >= (1 << 63) else c


def mix64(z: int) -> int:
    """SplitMix64 finaliser on a Python int (reference for the tensor version)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * _MIX_M1) & MASK64
    z = ((z ^ (z >> 27)) * _MIX_M2) & MASK64
    return z ^ (z >> 31)


def stream_key(*parts: int) -> int:
    """Fold integer parts (seed, layer, role, expert, ...) into one 64-bit key."""
    k = _KEY_ORIGIN
    for p in parts:
        k = mix64(((k ^ (int(p) & MASK64)) + GOLDEN_GAMMA) & MASK64)
    return k


def _lsr(z: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 tensors holding unsigned 64-bit values."""
    return torch.bitwise_and(torch.bitwise_right_shift(z, k), (1 << (64 - k)) - 1)


def _mix64_t(z: torch.Tensor) -> torch.Tensor:
    z = torch.bitwise_xor(z, _lsr(z, 30)) * _s64(_MIX_M1)
    z = torch.bitwise_xor(z, _lsr(z, 27)) * _s64(_MIX_M2)
    return torch.bitwise_xor(z, _lsr(z, 31))


def raw64(keys, n: int, device="cpu") -> torch.Tensor:
    """[len(keys), n] int64 tensor of 64-bit draws; element i of stream k is
    mix64(k + (i + 1) * golden_gamma) mod 2**64."""
    keys = [keys] if isinstance(keys, int) else list(keys)
    kt = torch.tensor([_s64(k) for k in keys], dtype=torch.int64, device=device)
    ctr = (torch.arange(1, n + 1, dtype=torch.int64, device=device) * _s64(GOLDEN_GAMMA))
    return _mix64_t(kt[:, None] + ctr[None, :])


_IH4_SCALE = 1.0 / math.sqrt((65536.0 ** 2 - 1.0) / 3.0)   # 1 / std of a sum of four U{0..65535}
_IH4_MEAN = 2 * 65535                                       # mean of that sum


def normal(keys, n: int, mean: float, std: float, device="cpu") -> torch.Tensor:
    """[len(keys), n] float32 draws of mean + std * z, z the unit-variance
    Irwin-Hall(4) variate of one 64-bit draw. All steps are exact integer ops or
    single IEEE roundings in fp64, then one rounding to fp32."""
    v = raw64(keys, n, device)
    s = (torch.bitwise_and(v, 0xFFFF) + torch.bitwise_and(_lsr(v, 16), 0xFFFF)
         + torch.bitwise_and(_lsr(v, 32), 0xFFFF) + _lsr(v, 48))
    z = (s - _IH4_MEAN).to(torch.float64) * _IH4_SCALE
    return (z * std + mean).to(torch.float32)


def uniform_int(keys, n: int, lo: int, hi: int, device="cpu") -> torch.Tensor:
    """[len(keys), n] int64 uniform integers in [lo, hi] (top 53 bits mod range)."""
    v = _lsr(raw64(keys, n, device), 11)
    return torch.remainder(v, hi - lo + 1) + lo


def _div(a: torch.Tensor, c: float) -> torch.Tensor:
    """IEEE division by a constant on any device. (On CUDA, dividing by a
    Python scalar is evaluated as a multiplication by its reciprocal, which
    can differ from the CPU result in the last bit; dividing by a tensor of
    the same shape is a true division everywhere.)"""
    return a / torch.full_like(a, c)


def to_bf16(w32: torch.Tensor) -> torch.Tensor:
    """Round fp32 to bf16, round-to-nearest-even."""
    return w32.to(torch.bfloat16)


# ----------------------------------------------------------------------------
# Weight encoders (input preparation; the method only decodes these formats)
# ----------------------------------------------------------------------------

def encode_q8_0(w: torch.Tensor) -> torch.Tensor:
    """fp32 [rows, K] -> uint8 [rows, K/32*34]: per 32-block fp16 d = amax/127,
    int8 q = rint(w / d) clamped to [-127, 127]."""
    rows, k = w.shape
    assert k % QK8 == 0
    b = w.reshape(rows, k // QK8, QK8)
    amax = b.abs().amax(-1)
    d16 = _div(amax, 127.0).to(torch.float16)
    df = d16.to(torch.float32)
    safe = torch.where(df > 0, df, torch.ones_like(df))
    q = torch.where(df[..., None] > 0, torch.round(b / safe[..., None]).clamp(-127, 127),
                    torch.zeros_like(b)).to(torch.int8)
    out = torch.empty(rows, k // QK8, Q8_0_BYTES, dtype=torch.uint8, device=w.device)
    out[..., 0:2] = d16.view(torch.uint8).reshape(rows, k // QK8, 2)
    out[..., 2:] = q.view(torch.uint8)
    return out.reshape(rows, (k // QK8) * Q8_0_BYTES)


def q4_k_params(w: torch.Tensor):
    """Plain min/max Q4_K quantiser for synthetic fp32 weights [rows, K].

    Per 32-wide sub-block j of a 256-wide super-block: lo = min(0, min w),
    hi = max w, scale s_j = (hi - lo)/15, offset m'_j = -lo. Super-block
    d = fp16(max_j s_j / 63), dmin = fp16(max_j m'_j / 63); 6-bit
    sc_j = rint(s_j / d), m_j = rint(m'_j / dmin); 4-bit
    q = rint((w + dmin*m_j) / (d*sc_j)), each clamped to its range and 0 where a
    divisor is 0. Returns (d16, dmin16, sc, m, q) with shapes [rows, nsb],
    [rows, nsb], [rows, nsb, 8], [rows, nsb, 8], [rows, nsb, 8, 32].
    """
    rows, k = w.shape
    assert k % QK_K == 0
    nsb = k // QK_K
    x = w.reshape(rows, nsb, 8, 32)
    lo = torch.clamp(x.amin(-1), max=0.0)
    hi = x.amax(-1)
    s = _div(hi - lo, 15.0)
    mneg = -lo
    d16 = _div(s.amax(-1), 63.0).to(torch.float16)
    dmin16 = _div(mneg.amax(-1), 63.0).to(torch.float16)
    df = d16.to(torch.float32)[..., None]
    dmf = dmin16.to(torch.float32)[..., None]
    one = torch.ones_like(df)
    sc = torch.where(df > 0, torch.round(s / torch.where(df > 0, df, one)).clamp(0, 63),
                     torch.zeros_like(s))
    m = torch.where(dmf > 0, torch.round(mneg / torch.where(dmf > 0, dmf, one)).clamp(0, 63),
                    torch.zeros_like(s))
    den = (df * sc)[..., None]                 # exact: 11-bit * 6-bit
    num = x + (dmf * m)[..., None]             # product exact, sum rounded once
    q = torch.where(den > 0, torch.round(num / torch.where(den > 0, den, torch.ones_like(den)))
                    .clamp(0, 15), torch.zeros_like(num))
    return d16, dmin16, sc.to(torch.int64), m.to(torch.int64), q.to(torch.int64)


def pack_q4_k(d16, dmin16, sc, m, q) -> torch.Tensor:
    """Pack Q4_K fields into 144-byte super-blocks, GGUF K-quant byte layout:
    bytes 0-1 fp16 d, 2-3 fp16 dmin, 4-15 the twelve packed 6-bit scale/min
    bytes, 16-143 the 4-bit codes. Scale bytes: b[j] (j<4) = sc_j low 6 bits
    plus bits 4-5 of sc_{j+4} in its top 2 bits; b[j+4] = m_j likewise with
    m_{j+4}; b[j+8] = low nibble of sc_{j+4} | low nibble of m_{j+4} << 4.
    Codes: byte 32p+i holds sub-block 2p element i (low nibble) and sub-block
    2p+1 element i (high nibble)."""
    rows, nsb = d16.shape
    dev = d16.device
    out = torch.empty(rows, nsb, Q4_K_BYTES, dtype=torch.uint8, device=dev)
    out[..., 0:2] = d16.contiguous().view(torch.uint8).reshape(rows, nsb, 2)
    out[..., 2:4] = dmin16.contiguous().view(torch.uint8).reshape(rows, nsb, 2)
    sb = torch.empty(rows, nsb, 12, dtype=torch.int64, device=dev)
    sb[..., 0:4] = (sc[..., 0:4] & 63) | ((sc[..., 4:8] >> 4) << 6)
    sb[..., 4:8] = (m[..., 0:4] & 63) | ((m[..., 4:8] >> 4) << 6)
    sb[..., 8:12] = (sc[..., 4:8] & 15) | ((m[..., 4:8] & 15) << 4)
    out[..., 4:16] = sb.to(torch.uint8)
    qq = q.reshape(rows, nsb, 4, 2, 32)
    codes = qq[:, :, :, 0, :] | (qq[:, :, :, 1, :] << 4)
    out[..., 16:] = codes.reshape(rows, nsb, 128).to(torch.uint8)
    return out.reshape(rows, nsb * Q4_K_BYTES)


def encode_q4_k(w: torch.Tensor) -> torch.Tensor:
    """fp32 [rows, K] -> uint8 [rows, K/256*144] Q4_K super-blocks."""
    return pack_q4_k(*q4_k_params(w))


def q5_k_params(w: torch.Tensor):
    """The min/max quantiser of q4_k_params with 5-bit codes: s_j = (hi - lo)/31,
    q clamped to [0, 31]; the rest (fp16 d/dmin from the largest s/m' over 63,
    6-bit sc/m by rint) as there. Returns (d16, dmin16, sc, m, q)."""
    rows, k = w.shape
    assert k % QK_K == 0
    nsb = k // QK_K
    x = w.reshape(rows, nsb, 8, 32)
    lo = torch.clamp(x.amin(-1), max=0.0)
    hi = x.amax(-1)
    s = _div(hi - lo, 31.0)
    mneg = -lo
    d16 = _div(s.amax(-1), 63.0).to(torch.float16)
    dmin16 = _div(mneg.amax(-1), 63.0).to(torch.float16)
    df = d16.to(torch.float32)[..., None]
    dmf = dmin16.to(torch.float32)[..., None]
    one = torch.ones_like(df)
    sc = torch.where(df > 0, torch.round(s / torch.where(df > 0, df, one)).clamp(0, 63),
                     torch.zeros_like(s))
    m = torch.where(dmf > 0, torch.round(mneg / torch.where(dmf > 0, dmf, one)).clamp(0, 63),
                    torch.zeros_like(s))
    den = (df * sc)[..., None]
    num = x + (dmf * m)[..., None]
    q = torch.where(den > 0, torch.round(num / torch.where(den > 0, den, torch.ones_like(den)))
                    .clamp(0, 31), torch.zeros_like(num))
    return d16, dmin16, sc.to(torch.int64), m.to(torch.int64), q.to(torch.int64)


def pack_q5_k(d16, dmin16, sc, m, q) -> torch.Tensor:
    """Q5_K super-blocks, GGUF layout, 176 bytes: the Q4_K header (d, dmin,
    12 scale bytes), then qh[32] with bit j of byte i = bit 4 of element i of
    sub-block j, then the low 4 bits of the codes in Q4_K's code layout."""
    rows, nsb = d16.shape
    q4 = pack_q4_k(d16, dmin16, sc, m, q & 15).reshape(rows, nsb, Q4_K_BYTES)
    hi = (q >> 4) & 1                                            # [rows, nsb, 8, 32]
    weights = (1 << torch.arange(8, device=q.device, dtype=torch.int64)).reshape(1, 1, 8, 1)
    qh = (hi * weights).sum(dim=2)                               # [rows, nsb, 32]
    out = torch.empty(rows, nsb, Q5_K_BYTES, dtype=torch.uint8, device=d16.device)
    out[..., 0:16] = q4[..., 0:16]
    out[..., 16:48] = qh.to(torch.uint8)
    out[..., 48:176] = q4[..., 16:144]
    return out.reshape(rows, nsb * Q5_K_BYTES)


def encode_q5_k(w: torch.Tensor) -> torch.Tensor:
    """fp32 [rows, K] -> uint8 [rows, K/256*176] Q5_K super-blocks."""
    return pack_q5_k(*q5_k_params(w))


def row_bytes(fmt: str, k: int) -> int:
    if fmt == "q4_k":
        return k // QK_K * Q4_K_BYTES
    if fmt == "q5_k":
        return k // QK_K * Q5_K_BYTES
    if fmt == "q8_0":
        return k // QK8 * Q8_0_BYTES
    if fmt == "bf16":
        return 2 * k
    raise ValueError(fmt)


def encode(w32: torch.Tensor, fmt: str) -> torch.Tensor:
    """Encode fp32 [rows, K] weights into ``fmt``; the result is always a uint8
    tensor [rows, row_bytes(fmt, K)] (bf16 is its little-endian bytes)."""
    if fmt == "q4_k":
        return encode_q4_k(w32)
    if fmt == "q5_k":
        return encode_q5_k(w32)
    if fmt == "q8_0":
        return encode_q8_0(w32)
    if fmt == "bf16":
        return to_bf16(w32).contiguous().view(torch.uint8)
    raise ValueError(fmt)


# ----------------------------------------------------------------------------
# Workload shapes
# ----------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class LayerSpec:
    """Shapes and weight formats of one MoE FFN layer."""
    hidden: int = 2048
    n_experts: int = 256
    top_k: int = 8
    inter: int = 512
    expert_type: str = "q4_k"     # "q4_k" | "bf16"
    shared_inter: int = 512       # 0: no shared expert
    shared_type: str = "q8_0"     # "q8_0" | "q4_k" | "bf16"
    eps: float = 1e-6
    down_type: str = ""           # routed down format; "" = expert_type ("q5_k": Q4_K gate/up)


# One layer, one token, bf16 everywhere, shared expert I=512.
BF16_LAYER = LayerSpec(expert_type="bf16", shared_type="bf16")
# Qwen3.6-35B-A3B-shaped quantised layer: routed Q4_K; shared Q8_0 or Q4_K.
Q4K_LAYER_SHARED_Q8_0 = LayerSpec(expert_type="q4_k", shared_type="q8_0")
Q4K_LAYER_SHARED_Q4_K = LayerSpec(expert_type="q4_k", shared_type="q4_k")
# Qwen3-30B-A3B-shaped layer: 128 experts, I=768, no shared expert.
Q4K_LAYER_128E = LayerSpec(n_experts=128, inter=768, shared_inter=0, shared_type="q4_k")
# The shipped Qwen3.6-35B-A3B formats before the load-time requant: routed
# gate/up Q4_K, routed down Q5_K, shared expert Q8_0.
NATIVE_LAYER_Q5K_DOWN = LayerSpec(expert_type="q4_k", down_type="q5_k", shared_type="q8_0")


def _weights(seed, layer, role, experts, rows, cols, fmt, device, std=WEIGHT_STD, mean=0.0,
             chunk=None):
    """Encoded weights for ``experts`` (list) of one role: uint8 [len, rows, rb]."""
    rb = row_bytes(fmt, cols)
    if chunk is None:   # experts per batch of elementwise ops (a few hundred MB of temporaries)
        chunk = max(1, min(64, (1 << 25) // (rows * cols))) if str(device).startswith("cuda") else 8
    out = torch.empty(len(experts), rows, rb, dtype=torch.uint8, device=device)
    for i in range(0, len(experts), chunk):
        sel = experts[i:i + chunk]
        keys = [stream_key(seed, layer, role, e) for e in sel]
        w = normal(keys, rows * cols, mean, std, device).reshape(len(sel) * rows, cols)
        out[i:i + len(sel)] = encode(w, fmt).reshape(len(sel), rows, rb)
        del w
    return out


def float_weights(seed, layer, role, expert, rows, cols, device="cpu", std=WEIGHT_STD):
    """The fp32 weights of one (role, expert) before encoding (for quantiser pins)."""
    return normal([stream_key(seed, layer, role, expert)], rows * cols, 0.0, std,
                  device).reshape(rows, cols)


def make_layer(spec: LayerSpec, seed: int, layer: int = 0, device="cpu", experts=None):
    """All tensors of one layer.

    ``experts``: None materialises every routed expert (the device side);
    a list materialises only those (the oracle), stored in that order with
    ``expert_ids`` giving their global ids. Routed matrices are uint8
    [n, rows, row_bytes] in the spec's format; bf16 vectors are torch.bfloat16.
    Row-major, K contiguous: gate/up [I x H], down [H x I], router [E x H].
    """
    ids = list(range(spec.n_experts)) if experts is None else [int(e) for e in experts]
    H, I = spec.hidden, spec.inter
    L = {
        "spec": spec, "seed": seed, "layer": layer, "expert_ids": ids,
        "w_router": to_bf16(normal([stream_key(seed, layer, ROLE_ROUTER, 0)],
                                   spec.n_experts * H, 0.0, WEIGHT_STD, device)
                            ).reshape(spec.n_experts, H),
        "gate": _weights(seed, layer, ROLE_GATE, ids, I, H, spec.expert_type, device),
        "up": _weights(seed, layer, ROLE_UP, ids, I, H, spec.expert_type, device),
        "down": _weights(seed, layer, ROLE_DOWN, ids, H, I, spec.down_type or spec.expert_type,
                         device),
        "w_norm": to_bf16(normal([stream_key(seed, layer, ROLE_NORM, 0)], H, NORM_MEAN,
                                 NORM_STD, device)).reshape(H),
    }
    if spec.shared_inter > 0:
        Is = spec.shared_inter
        L["sh_gate"] = _weights(seed, layer, ROLE_SH_GATE, [0], Is, H, spec.shared_type, device)[0]
        L["sh_up"] = _weights(seed, layer, ROLE_SH_UP, [0], Is, H, spec.shared_type, device)[0]
        L["sh_down"] = _weights(seed, layer, ROLE_SH_DOWN, [0], H, Is, spec.shared_type, device)[0]
        L["w_sg"] = to_bf16(normal([stream_key(seed, layer, ROLE_SH_SIGMOID, 0)], H, 0.0,
                                   WEIGHT_STD, device)).reshape(H)
    return L


def make_tokens(seed: int, n_tokens: int, hidden: int = 2048, device="cpu", first: int = 0):
    """Hidden-state inputs x_t ~ N(0, 1) in bf16, [n_tokens, hidden]; token t
    draws from its own stream so any subset can be regenerated alone."""
    keys = [stream_key(seed, 0, ROLE_X, first + t) for t in range(n_tokens)]
    return to_bf16(normal(keys, hidden, 0.0, 1.0, device))


# ----------------------------------------------------------------------------
# Router tie stress: small integers in [-3, 3] stored as fp32
# ----------------------------------------------------------------------------

TIE_FAMILIES = ("uniform", "sparse_x", "duplicate_rows", "zero_x", "constant_rows")


def tie_stress_group(seed: int, group: int, n_experts: int, n_cases: int, hidden: int = 2048,
                     device="cpu"):
    """One group of router tie-stress cases sharing a router matrix.

    Family = TIE_FAMILIES[group % 5]:
      uniform        W, x uniform in [-3, 3];
      sparse_x       W uniform, x zero except ~5% of entries;
      duplicate_rows W's rows drawn from a pool of 4..16 distinct rows, so whole
                     experts tie exactly;
      zero_x         x = 0, every logit is 0 (selection must be experts 0..7);
      constant_rows  row e is a constant c_e in [-3, 3]; logits c_e * sum(x).
    Returns (W fp32 [E, H], X fp32 [n_cases, H], family name).
    """
    fam = TIE_FAMILIES[group % len(TIE_FAMILIES)]
    kw = stream_key(seed, group, ROLE_TIE_W, n_experts)
    xkeys = [stream_key(seed, group, ROLE_TIE_X, n_experts * 100003 + c) for c in range(n_cases)]
    if fam == "duplicate_rows":
        n_pool = 4 + int(uniform_int([stream_key(seed, group, ROLE_TIE_POOL, 0)], 1, 0, 12)[0, 0])
        pool = uniform_int([kw], n_pool * hidden, -3, 3, device).reshape(n_pool, hidden)
        pick = uniform_int([stream_key(seed, group, ROLE_TIE_POOL, 1)], n_experts, 0, n_pool - 1,
                           device)[0]
        W = pool[pick]
    elif fam == "constant_rows":
        c = uniform_int([kw], n_experts, -3, 3, device)[0]
        W = c[:, None].expand(n_experts, hidden).clone()
    else:
        W = uniform_int([kw], n_experts * hidden, -3, 3, device).reshape(n_experts, hidden)
    if fam == "zero_x":
        X = torch.zeros(n_cases, hidden, dtype=torch.int64, device=device)
    else:
        X = uniform_int(xkeys, hidden, -3, 3, device)
        if fam == "sparse_x":
            keep = uniform_int([stream_key(seed, group, ROLE_TIE_MASK, c) for c in range(n_cases)],
                               hidden, 0, 19, device) == 0
            X = torch.where(keep, X, torch.zeros_like(X))
    return W.to(torch.float32), X.to(torch.float32), fam
