"""Oracle: number formats (rounding, Q4_K / Q8_0 decoding, Q8_1 encoding).

TEST INFRASTRUCTURE. Only the tests, the package's smoke check and the CPU
baseline of the benchmark may import this module. It shares no code with the
CUDA path.

Sources (sparkinfer pull-request pages):
* "Q4_K shared-expert FFN kernels + Q8_0/Q5_K->Q4_K requant of the MoE FFN
  stage" (PR #359), Summary, bullets 1 and 2: the routed down projection ships
  as Q5_K and the shared expert as Q8_0; both are requantised to Q4_K once at
  load. The page names the formats but prints neither the Q5_K layout nor the
  requant procedure: the GGUF Q5_K layout is taken, and the requant is read as
  "dequantise to fp32, then quantise to Q4_K with the library's Q4_K
  quantiser" (min/max per 32-wide sub-block; see q4_k_quantize).
* "Q4_K shared-expert FFN kernels + Q8_0/Q5_K->Q4_K requant of the MoE FFN
  stage" (PR #359), Summary: Q8_0 is 34 bytes per 32-weight block; Q4_K cuts
  about 47% of the bytes; activations are quantised to Q8_1 ("FNQ Q8_1",
  "quant_h Q8_1") and dotted with int8 dp4a.
* The Q4_K byte layout and the Q8_1 block layout are not printed on the pages;
  the model is a GGUF Q4_K_M file, so the GGUF K-quant layout is taken (one
  reading; see the design notes). Q8_1 here: 36 bytes {fp16 d, fp16 s, int8
  q[32]}, q = round-half-away(x / d32), d32 = amax / 127 in fp32, s = d32*sum(q).
"""
from __future__ import annotations

import numpy as np

QK_K = 256
Q4_K_BYTES = 144
Q5_K_BYTES = 176
QK8 = 32
Q8_0_BYTES = 34
Q8_1_BYTES = 36


# ----------------------------------------------------------------------------
# Rounding to narrow binary formats, by definition: round-to-nearest-even to a
# binary float with p significant bits and a smallest quantum 2**qmin.
# ----------------------------------------------------------------------------

def _round_sig(v, p: int, qmin: int, emax: int) -> np.ndarray:
    """Round to nearest even on a grid of p significant bits with subnormal
    quantum 2**qmin; a result above the largest finite value (2 - 2**(1-p)) *
    2**emax overflows to infinity of the same sign, as IEEE 754 rounding to
    nearest does."""
    v = np.asarray(v, dtype=np.float64)
    _, e = np.frexp(v)                              # v = m * 2**e, 0.5 <= |m| < 1
    q = np.ldexp(1.0, np.maximum(e - p, qmin))      # spacing of the target grid at v
    r = np.rint(v / q) * q                          # exact scaling; rint is RNE
    big = (2.0 - 2.0 ** (1 - p)) * 2.0 ** emax
    return np.where(np.abs(r) > big, np.copysign(np.inf, v), r)


def bf16(v) -> np.ndarray:
    """Round to bfloat16 (8 significant bits, largest finite (2 - 2**-7) *
    2**127), returned as float64 values."""
    return _round_sig(v, 8, -133, 127)


def fp16(v) -> np.ndarray:
    """Round to IEEE binary16 (11 significant bits, subnormal quantum 2**-24,
    largest finite 65504)."""
    return _round_sig(v, 11, -24, 15)


def fp32(v) -> np.ndarray:
    """Round to IEEE binary32 (numpy's correctly rounded cast), as float64."""
    return np.asarray(v, dtype=np.float64).astype(np.float32).astype(np.float64)


def bf16_from_bits(u16) -> np.ndarray:
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def bf16_bits(v) -> np.ndarray:
    """Bits of the bf16 rounding of v (v must already be exactly representable
    after rounding; the rounding is done here by definition)."""
    r = bf16(v).astype(np.float32)
    return (r.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def fp16_from_bytes(b2) -> np.ndarray:
    """Decode little-endian fp16 from a [..., 2] uint8 array."""
    b2 = np.ascontiguousarray(b2, dtype=np.uint8)
    return b2.view(np.float16)[..., 0].astype(np.float64)


# ----------------------------------------------------------------------------
# Q4_K super-block: 144 bytes per 256 weights
# ----------------------------------------------------------------------------

def q4_k_fields(blocks):
    """Unpack Q4_K super-blocks [..., 144] (uint8).

    Layout: bytes 0-1 fp16 d; 2-3 fp16 dmin; 4-15 twelve bytes of 6-bit
    scales and mins for the 8 sub-blocks of 32; 16-143 the 256 4-bit codes.
      sub-blocks 0-3: scale = byte j low 6 bits, min = byte j+4 low 6 bits;
      sub-blocks 4-7: low 4 bits of scale / min are the low / high nibble of
      byte j+4 (j = 4..7, i.e. bytes 8-11); their top 2 bits are the top 2 bits
      of byte j-4 (scale) and byte j (min).
      codes: within each 32-byte run p (0..3) of the 128 code bytes, byte i
      carries element i of sub-block 2p in its low nibble and element i of
      sub-block 2p+1 in its high nibble.
    Returns d, dmin (float64 [...]), sc, m (int64 [..., 8]), q (int64 [..., 8, 32]).
    """
    blocks = np.asarray(blocks, dtype=np.uint8)
    d = fp16_from_bytes(blocks[..., 0:2])
    dmin = fp16_from_bytes(blocks[..., 2:4])
    s = blocks[..., 4:16].astype(np.int64)
    sc = np.empty(blocks.shape[:-1] + (8,), dtype=np.int64)
    m = np.empty_like(sc)
    for j in range(4):
        sc[..., j] = s[..., j] & 63
        m[..., j] = s[..., j + 4] & 63
    for j in range(4, 8):
        sc[..., j] = (s[..., j + 4] & 0x0F) | ((s[..., j - 4] >> 6) << 4)
        m[..., j] = (s[..., j + 4] >> 4) | ((s[..., j] >> 6) << 4)
    codes = blocks[..., 16:144].astype(np.int64).reshape(blocks.shape[:-1] + (4, 32))
    q = np.empty(blocks.shape[:-1] + (8, 32), dtype=np.int64)
    q[..., 0::2, :] = codes & 0x0F
    q[..., 1::2, :] = codes >> 4
    return d, dmin, sc, m, q


def q4_k_dequant(blocks) -> np.ndarray:
    """Weights of Q4_K super-blocks [..., 144] -> float64 [..., 256]:
    w = d * sc_j * q - dmin * m_j for element q of sub-block j."""
    d, dmin, sc, m, q = q4_k_fields(blocks)
    w = d[..., None, None] * sc[..., None] * q - (dmin[..., None] * m)[..., None]
    return w.reshape(w.shape[:-2] + (QK_K,))


def q4_k_rows(mat) -> np.ndarray:
    """[rows, nsb*144] uint8 -> [rows, nsb, 144]."""
    mat = np.asarray(mat, dtype=np.uint8)
    return mat.reshape(mat.shape[0], -1, Q4_K_BYTES)


def q4_k_pack(d, dmin, sc, m, q) -> np.ndarray:
    """Inverse of q4_k_fields: d, dmin exact fp16 values [...], sc, m ints in
    [0, 63] [..., 8], q ints in [0, 15] [..., 8, 32] -> uint8 [..., 144]."""
    d = np.asarray(d, dtype=np.float64)
    out = np.zeros(d.shape + (Q4_K_BYTES,), dtype=np.uint8)
    out[..., 0:2] = np.ascontiguousarray(d.astype(np.float16)).view(np.uint8).reshape(d.shape + (2,))
    dm = np.asarray(dmin, dtype=np.float64)
    out[..., 2:4] = np.ascontiguousarray(dm.astype(np.float16)).view(np.uint8).reshape(d.shape + (2,))
    sc = np.asarray(sc, dtype=np.int64)
    m = np.asarray(m, dtype=np.int64)
    for j in range(4):
        out[..., 4 + j] = (sc[..., j] & 63) | ((sc[..., j + 4] >> 4) << 6)
        out[..., 8 + j] = (m[..., j] & 63) | ((m[..., j + 4] >> 4) << 6)
        out[..., 12 + j] = (sc[..., j + 4] & 15) | ((m[..., j + 4] & 15) << 4)
    q = np.asarray(q, dtype=np.int64)
    for pp in range(4):
        out[..., 16 + 32 * pp:48 + 32 * pp] = q[..., 2 * pp, :] | (q[..., 2 * pp + 1, :] << 4)
    return out


def q4_k_quantize(w) -> np.ndarray:
    """The library's Q4_K quantiser, on fp32 weights [rows, K] (K % 256 == 0),
    every step an IEEE fp32 operation (numpy float32 arithmetic is correctly
    rounded), rint = round half to even. Per 32-wide sub-block j of a super-block:
      lo = min w if it is negative, else +0; hi = max w if it is positive, else
      +0 (so that the sign of a zero never reaches the bytes);
      s_j = (hi - lo) / 15, m'_j = -lo;
      d = fp16(max_j s_j / 63), dmin = fp16(max_j m'_j / 63);
      sc_j = rint(s_j / d) and m_j = rint(m'_j / dmin), clamped to [0, 63],
      0 where the divisor is 0;
      q = rint((w + dmin * m_j) / (d * sc_j)) clamped to [0, 15], 0 where the
      divisor is 0 (d * sc_j and dmin * m_j are exact in fp32).
    Returns uint8 [rows, K/256*144]."""
    f = np.float32
    w = np.asarray(w, dtype=np.float32)
    rows, k = w.shape
    nsb = k // QK_K
    x = w.reshape(rows, nsb, 8, 32)
    mn, mx = x.min(axis=-1), x.max(axis=-1)
    lo = np.where(mn < 0, mn, f(0)).astype(np.float32)     # +0 unless negative
    hi = np.where(mx > 0, mx, f(0)).astype(np.float32)     # +0 unless positive
    s = (hi - lo) / f(15)
    mneg = -lo
    d16 = (s.max(axis=-1) / f(63)).astype(np.float16)
    dm16 = (mneg.max(axis=-1) / f(63)).astype(np.float16)
    d = d16.astype(np.float32)[..., None]
    dm = dm16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        sc = np.where(d > 0, np.clip(np.rint(s / np.where(d > 0, d, f(1))), 0, 63), 0).astype(np.int64)
        m = np.where(dm > 0, np.clip(np.rint(mneg / np.where(dm > 0, dm, f(1))), 0, 63), 0).astype(np.int64)
        den = (d * sc.astype(np.float32))[..., None]
        num = x + (dm * m.astype(np.float32))[..., None]
        q = np.where(den > 0, np.clip(np.rint(num / np.where(den > 0, den, f(1))), 0, 15), 0)
    out = q4_k_pack(d16.astype(np.float64), dm16.astype(np.float64), sc, m, q.astype(np.int64))
    return out.reshape(rows, nsb * Q4_K_BYTES)


# ----------------------------------------------------------------------------
# Q5_K super-block: 176 bytes per 256 weights
# ----------------------------------------------------------------------------

def q5_k_fields(blocks):
    """Unpack Q5_K super-blocks [..., 176] (uint8), GGUF layout: bytes 0-1 fp16
    d, 2-3 fp16 dmin, 4-15 the 6-bit scales and mins packed as in Q4_K, 16-47
    qh[32] (the fifth bits), 48-175 the low 4 bits of the 256 codes laid out as
    Q4_K's codes. Element i of sub-block j: q = low nibble as in Q4_K
    + 16 * bit j of qh[i]. Returns d, dmin, sc, m, q (q in [0, 31])."""
    blocks = np.asarray(blocks, dtype=np.uint8)
    as_q4 = np.concatenate([blocks[..., 0:16], blocks[..., 48:176]], axis=-1)
    d, dmin, sc, m, q = q4_k_fields(as_q4)
    qh = blocks[..., 16:48].astype(np.int64)                     # [..., 32]
    for j in range(8):
        q[..., j, :] += ((qh >> j) & 1) << 4
    return d, dmin, sc, m, q


def q5_k_dequant(blocks) -> np.ndarray:
    """w = d * sc_j * q - dmin * m_j, float64 [..., 256]."""
    d, dmin, sc, m, q = q5_k_fields(blocks)
    w = d[..., None, None] * sc[..., None] * q - (dmin[..., None] * m)[..., None]
    return w.reshape(w.shape[:-2] + (QK_K,))


def q5_k_rows(mat) -> np.ndarray:
    mat = np.asarray(mat, dtype=np.uint8)
    return mat.reshape(mat.shape[0], -1, Q5_K_BYTES)


# ----------------------------------------------------------------------------
# Q8_0 block: 34 bytes per 32 weights
# ----------------------------------------------------------------------------

def q8_0_fields(blocks):
    """Unpack Q8_0 blocks [..., 34]: fp16 d (bytes 0-1), int8 q[32] (bytes 2-33)."""
    blocks = np.asarray(blocks, dtype=np.uint8)
    d = fp16_from_bytes(blocks[..., 0:2])
    q = np.ascontiguousarray(blocks[..., 2:34]).view(np.int8).astype(np.int64)
    return d, q


def q8_0_dequant(blocks) -> np.ndarray:
    d, q = q8_0_fields(blocks)
    return d[..., None] * q


def q8_0_rows(mat) -> np.ndarray:
    mat = np.asarray(mat, dtype=np.uint8)
    return mat.reshape(mat.shape[0], -1, Q8_0_BYTES)


# ----------------------------------------------------------------------------
# Q8_1 activation blocks: 36 bytes per 32 values, encoded step by step in fp32
# ----------------------------------------------------------------------------

def _round_half_away(v32: np.ndarray) -> np.ndarray:
    """round-half-away-from-zero of fp32 values, evaluated exactly in fp64."""
    v = v32.astype(np.float64)
    return np.where(v >= 0, np.floor(v + 0.5), np.ceil(v - 0.5))


def q8_1_quantize(x) -> dict:
    """Encode an fp32 vector (length a multiple of 32) into Q8_1 blocks.

    Per block, in fp32 exactly as written: amax = max |x_i|;
    d32 = amax / 127 (IEEE division); q_i = round-half-away(x_i / d32)
    clamped to [-127, 127] (all zero when amax = 0); stored d = fp16(d32),
    s = fp16(d32 * float(sum_i q_i)).
    Returns {"d": float64 [nb] (fp16 values), "s": float64 [nb], "q": int64 [nb, 32],
    "d32": float32 [nb]}.
    """
    x32 = np.asarray(x, dtype=np.float32).reshape(-1, QK8)
    amax = np.abs(x32).max(axis=1)
    d32 = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(d32 > 0, d32, np.float32(1.0)).astype(np.float32)
    v = (x32 / safe[:, None]).astype(np.float32)
    q = np.clip(_round_half_away(v), -127, 127).astype(np.int64)
    q[d32 == 0] = 0
    sumq = q.sum(axis=1)
    s32 = (d32 * sumq.astype(np.float32)).astype(np.float32)
    return {"d": fp16(d32.astype(np.float64)), "s": fp16(s32.astype(np.float64)),
            "q": q, "d32": d32}


def q8_1_to_bytes(a: dict) -> np.ndarray:
    """Serialise Q8_1 blocks to [nb, 36] uint8: fp16 d, fp16 s, int8 q[32]."""
    nb = a["q"].shape[0]
    out = np.empty((nb, Q8_1_BYTES), dtype=np.uint8)
    out[:, 0:2] = a["d"].astype(np.float16).reshape(nb, 1).view(np.uint8)
    out[:, 2:4] = a["s"].astype(np.float16).reshape(nb, 1).view(np.uint8)
    out[:, 4:] = a["q"].astype(np.int8).view(np.uint8)
    return out


def q8_1_from_bytes(b) -> dict:
    b = np.asarray(b, dtype=np.uint8).reshape(-1, Q8_1_BYTES)
    return {"d": fp16_from_bytes(b[:, 0:2]), "s": fp16_from_bytes(b[:, 2:4]),
            "q": np.ascontiguousarray(b[:, 4:]).view(np.int8).astype(np.int64)}


def q8_1_dequant(a: dict) -> np.ndarray:
    """Activation values as the stored block represents them: d * q."""
    return (a["d"][:, None] * a["q"]).reshape(-1)
