"""Pins of the oracle's Q5_K decoding, its Q4_K quantiser and the load-time
requant ("Q4_K shared-expert FFN kernels + Q8_0/Q5_K->Q4_K requant of the MoE
FFN stage", PR #359, Summary bullets 1 and 2): a Q5_K block placed by hand,
field bijections, exactness in fp32, the quantiser's error bound and rounding
rule on brute force, and agreement with the generator's independent torch
restatement of the same quantiser. No GPU is needed."""
import numpy as np
import torch

import gen
from oracle import formats as F
from oracle import moe as M


def _q5_block(d=1.0, dmin=0.0, sc=(1,) * 8, m=(0,) * 8, q=None):
    """One Q5_K block assembled byte by byte from the layout's description."""
    blk = np.zeros((1, 176), dtype=np.uint8)
    blk[0, 0:2] = np.array([d], dtype=np.float16).view(np.uint8)
    blk[0, 2:4] = np.array([dmin], dtype=np.float16).view(np.uint8)
    for j in range(4):
        blk[0, 4 + j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        blk[0, 8 + j] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
        blk[0, 12 + j] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    if q is not None:
        for j in range(8):
            for i in range(32):
                v = int(q[j][i])
                blk[0, 16 + i] |= ((v >> 4) & 1) << j
                byte = 48 + 32 * (j // 2) + i
                blk[0, byte] |= (v & 15) << (4 * (j % 2))
    return blk


def test_q5_k_codes_layout_by_hand():
    """Element i of sub-block j: low nibble as in Q4_K, fifth bit = bit j of
    qh[i]; a single 5-bit code placed by hand."""
    blk = np.zeros((1, 176), dtype=np.uint8)
    blk[0, 0:2] = np.array([1.0], dtype=np.float16).view(np.uint8)
    blk[0, 4:8] = 1
    blk[0, 12:16] = 1
    blk[0, 16 + 9] = 1 << 6                     # fifth bit of element 9, sub-block 6
    blk[0, 48 + 32 * 3 + 9] = 0x05              # low nibble of sub-block 6 element 9: 5
    w = F.q5_k_dequant(blk)[0]
    expect = np.zeros(256)
    expect[32 * 6 + 9] = 21.0                   # 16 + 5
    assert np.array_equal(w, expect)


def test_q5_k_random_fields_round_trip():
    g = np.random.default_rng(4)
    for _ in range(40):
        sc = g.integers(0, 64, 8)
        m = g.integers(0, 64, 8)
        q = g.integers(0, 32, (8, 32))
        d, dmin, dsc, dm, dq = F.q5_k_fields(_q5_block(0.0123, 0.00456, sc, m, q))
        assert np.array_equal(dsc[0], sc) and np.array_equal(dm[0], m)
        assert np.array_equal(dq[0], q)


def test_q5_k_dequant_products_exact_in_fp32():
    """d*sc*q needs at most 11 + 6 + 5 = 22 significant bits: exact in fp32."""
    w = gen.float_weights(2, 0, gen.ROLE_DOWN, 0, 16, 512)
    d, dmin, sc, m, q = F.q5_k_fields(F.q5_k_rows(gen.encode_q5_k(w).numpy()))
    a = d[..., None, None] * sc[..., None] * q
    b = dmin[..., None] * m
    assert np.array_equal(F.fp32(a), a) and np.array_equal(F.fp32(b), b)


def test_q5_k_generator_and_oracle_agree_and_error_is_half_a_step():
    w = gen.float_weights(3, 1, gen.ROLE_DOWN, 2, 32, 1024)
    blocks = F.q5_k_rows(gen.encode_q5_k(w).numpy())
    d, dmin, sc, m, q = F.q5_k_fields(blocks)
    assert q.min() >= 0 and q.max() == 31
    wh = F.q5_k_dequant(blocks).reshape(32, 1024)
    bound = 0.5 * d[..., None] * sc + 15.5 * d[..., None] + 0.5 * dmin[..., None]
    bound = np.repeat(bound.reshape(32, -1), 32, axis=1)
    assert np.all(np.abs(w.numpy() - wh) <= bound * (1 + 1e-6) + 1e-12)


def test_q5_k_matvec_is_the_dequantised_product_when_s_is_exact():
    rng = np.random.default_rng(12)
    w = gen.encode_q5_k(gen.float_weights(6, 0, gen.ROLE_DOWN, 1, 24, 512)).numpy()
    x = rng.integers(-127, 128, 512).astype(np.float32) / np.float32(64)
    x[::32] = np.float32(127 / 64)               # amax = 127/64 in every block: d = 1/64 exactly
    a = F.q8_1_quantize(x)
    assert np.all(a["d"] == 1 / 64)
    ref = M.dequant_rows("q5_k", w) @ F.q8_1_dequant(a)
    assert np.allclose(M.matvec_q5_k(w, a), ref, rtol=1e-12, atol=1e-12)


def test_q4_k_pack_inverts_fields():
    g = np.random.default_rng(5)
    for _ in range(40):
        d = np.float64(np.float16(g.uniform(0, 0.01)))
        dmin = np.float64(np.float16(g.uniform(0, 0.01)))
        sc = g.integers(0, 64, 8)
        m = g.integers(0, 64, 8)
        q = g.integers(0, 16, (8, 32))
        blk = F.q4_k_pack(np.array(d), np.array(dmin), sc, m, q)
        dd, ddm, dsc, dm, dq = F.q4_k_fields(blk)
        assert dd == d and ddm == dmin
        assert np.array_equal(dsc, sc) and np.array_equal(dm, m) and np.array_equal(dq, q)


def test_q4_k_quantize_hand_example():
    """A super-block whose sub-block j holds (j + 1) * 2^-10 * (0, 1, ..., 15,
    0, 1, ..., 15): lo = 0, s_j = (j + 1) * 2^-10 exactly, dmin = 0."""
    w = np.zeros((1, 256), dtype=np.float32)
    for j in range(8):
        w[0, 32 * j:32 * j + 32] = np.tile(np.arange(16), 2) * np.float32((j + 1) * 2.0 ** -10)
    blk = F.q4_k_quantize(w)
    d, dmin, sc, m, q = F.q4_k_fields(blk.reshape(1, 1, 144))
    d_expect = np.float64(np.float16(np.float32(8 * 2.0 ** -10) / np.float32(63)))
    assert d[0, 0] == d_expect and dmin[0, 0] == 0.0 and np.all(m == 0)
    s = np.array([(j + 1) * 2.0 ** -10 for j in range(8)], dtype=np.float32)
    assert np.array_equal(sc[0, 0], np.clip(np.rint(s / np.float32(d_expect)), 0, 63))
    # codes: the nearest grid point of each weight, ties to even (brute force)
    grid = d_expect * sc[0, 0][:, None] * np.arange(16)[None, :]           # [8, 16]
    for j in range(8):
        for i in range(32):
            v = np.float32(w[0, 32 * j + i]) / np.float32(d_expect * sc[0, 0, j])
            assert q[0, 0, j, i] == min(15, max(0, int(np.rint(v))))
            assert abs(grid[j, q[0, 0, j, i]] - w[0, 32 * j + i]) <= 0.5 * d_expect * sc[0, 0, j] + 1e-12


def test_q4_k_quantize_matches_the_generators_restatement():
    """Two restatements of the same quantiser (numpy fp32 here, torch fp32 in
    the input generator) give the same bytes."""
    for role, seed in ((gen.ROLE_GATE, 1), (gen.ROLE_SH_DOWN, 7)):
        w = gen.float_weights(seed, 0, role, 0, 48, 1024)
        assert np.array_equal(F.q4_k_quantize(w.numpy()), gen.encode_q4_k(w).numpy())


def test_q4_k_quantize_error_bound_and_zero_block():
    w = gen.float_weights(8, 0, gen.ROLE_UP, 3, 40, 2048).numpy()
    blocks = F.q4_k_rows(F.q4_k_quantize(w))
    d, dmin, sc, m, q = F.q4_k_fields(blocks)
    wh = F.q4_k_dequant(blocks).reshape(40, 2048)
    bound = 0.5 * d[..., None] * sc + 7.5 * d[..., None] + 0.5 * dmin[..., None]
    bound = np.repeat(bound.reshape(40, -1), 32, axis=1)
    assert np.all(np.abs(w - wh) <= bound * (1 + 1e-6) + 1e-12)
    # an all-zero block: every field 0, except that m' = -lo = -0 gives dmin = -0
    # (fp16 bits 0x8000); it decodes to zeros
    z = F.q4_k_quantize(np.zeros((2, 512), dtype=np.float32)).reshape(2, 2, 144)
    assert not z[..., 0:2].any() and np.all(z[..., 2] == 0) and np.all(z[..., 3] == 0x80)
    assert not z[..., 4:].any()
    assert not F.q4_k_dequant(z).any()


def test_requant_of_q8_0_and_q5_k_stays_within_the_q4_k_bound():
    """The requant ([Q] Summary bullets 1, 2): Q4_K of the source's fp32
    weights; the result decodes within the quantiser's bound of them, and
    requantising an already Q4_K-representable source is the identity."""
    w = gen.float_weights(9, 0, gen.ROLE_SH_GATE, 0, 16, 2048)
    for fmt, enc in (("q8_0", gen.encode_q8_0), ("q5_k", gen.encode_q5_k)):
        src = enc(w).numpy()
        x = F.fp32(M.dequant_rows(fmt, src))
        if fmt == "q8_0":
            assert np.array_equal(x, M.dequant_rows(fmt, src))   # d * q is exact in fp32
        out = M.requant_q4_k(fmt, src)
        assert out.shape == (16, 2048 // 256 * 144)
        blocks = F.q4_k_rows(out)
        d, dmin, sc, m, q = F.q4_k_fields(blocks)
        wh = F.q4_k_dequant(blocks).reshape(16, 2048)
        bound = 0.5 * d[..., None] * sc + 7.5 * d[..., None] + 0.5 * dmin[..., None]
        bound = np.repeat(bound.reshape(16, -1), 32, axis=1)
        assert np.all(np.abs(x - wh) <= bound * (1 + 1e-6) + 1e-12)
    q4 = gen.encode_q4_k(w).numpy()
    x4 = F.fp32(M.dequant_rows("q4_k", q4)).astype(np.float32)
    assert np.array_equal(F.q4_k_quantize(x4), F.q4_k_quantize(F.fp32(
        M.dequant_rows("q4_k", F.q4_k_quantize(x4))).astype(np.float32)))


def test_q5_k_block_dots_brute_force():
    """Integer block sums of Q5_K rows, element by element from the bytes:
    code = low or high nibble (sub-block parity) + 16 * bit j of qh[i]."""
    rng = np.random.default_rng(31)
    w = gen.encode_q5_k(gen.float_weights(6, 0, gen.ROLE_DOWN, 1, 3, 512)).numpy()
    a = F.q8_1_quantize(rng.standard_normal(512).astype(np.float32))
    got = M.q5_k_block_dots(w, a)
    for r in range(3):
        for b in range(16):
            sb, j = divmod(b, 8)
            base = sb * 176
            tot = 0
            for i in range(32):
                byte = int(w[r, base + 48 + 32 * (j // 2) + i])
                code = (byte & 15) if j % 2 == 0 else (byte >> 4)
                code += 16 * ((int(w[r, base + 16 + i]) >> j) & 1)
                tot += code * int(a["q"][b, i])
            assert got[r, b] == tot
