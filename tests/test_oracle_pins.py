"""Pins of the CPU oracle against facts other than itself.

Each test ties one oracle function to what the pages print, to a closed form,
to an invariant, to a library routine on a special case, or to brute force on
a tiny input, so that a plausible mistake (a dropped term, a wrong sign or
index, a transposed operand, the wrong rounding rule) fails at least one of
them. No GPU is needed.
"""
import math
import os

import numpy as np
import pytest
import torch

import gen
from oracle import formats as F
from oracle import moe as M

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            out[k] = [float(t) for t in v]
    return out


# ----------------------------------------------------------------------------
# rounding helpers: against library conversions
# ----------------------------------------------------------------------------

def test_bf16_rounding_matches_torch_conversion():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.005859375, -1.005859375]]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(F.bf16(v.astype(np.float64)), ref)


def test_fp16_rounding_matches_numpy_cast():
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(20000) * 10.0 ** rng.integers(-8, 4, 20000)).astype(np.float32)
    ref = v.astype(np.float16).astype(np.float64)
    assert np.array_equal(F.fp16(v.astype(np.float64)), ref)


def test_fp16_and_bf16_overflow_like_the_library_casts():
    """Past the largest finite value the rounding overflows to infinity:
    65504 is the largest binary16, 65520 (halfway to 2**16) rounds up to inf."""
    v = np.concatenate([np.linspace(65000.0, 66000.0, 4001), [65519.99, 65520.0, 1e6, 3e38]])
    v = np.concatenate([v, -v]).astype(np.float32)
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).astype(np.float64)
    got = F.fp16(v.astype(np.float64))
    assert np.array_equal(got, ref)
    assert F.fp16(65519.0) == 65504.0 and F.fp16(65520.0) == np.inf and F.fp16(-7e4) == -np.inf
    big = np.float32(3.3895313892515355e38)                 # (2 - 2**-7) * 2**127
    w = np.array([big, np.nextafter(big, np.float32(np.inf)), np.finfo(np.float32).max,
                  -np.finfo(np.float32).max, 3.39e38, 3.4e38], dtype=np.float32)
    ref16 = torch.from_numpy(w).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(F.bf16(w.astype(np.float64)), ref16)


def test_fp16_ties_to_even():
    # 1 + 2^-11 is halfway between 1 and 1 + 2^-10: nearest-even gives 1.
    assert F.fp16(1.0 + 2.0 ** -11) == 1.0
    assert F.fp16(1.0 + 3 * 2.0 ** -11) == 1.0 + 2.0 ** -9
    assert F.bf16(1.0 + 2.0 ** -8) == 1.0


# ----------------------------------------------------------------------------
# block formats
# ----------------------------------------------------------------------------

def test_format_sizes_match_pages():
    g = _golden("format_sizes.txt")
    assert F.Q8_0_BYTES == g["q8_0_block_bytes"][0] and F.QK8 == g["q8_0_block_weights"][0]
    fewer = 1.0 - (F.Q4_K_BYTES / F.QK_K) / (F.Q8_0_BYTES / F.QK8)
    assert abs(fewer - g["q4_k_fewer_bytes_fraction"][0]) <= g["q4_k_fewer_bytes_tolerance"][0]
    # the generator writes blocks of the same sizes
    assert gen.row_bytes("q4_k", 2048) == 8 * 144 and gen.row_bytes("q8_0", 2048) == 64 * 34


def _pack(sc, m, q=None, d=1.0, dmin=1.0):
    sc = torch.tensor(sc, dtype=torch.int64).reshape(1, 1, 8)
    m = torch.tensor(m, dtype=torch.int64).reshape(1, 1, 8)
    q = torch.zeros(1, 1, 8, 32, dtype=torch.int64) if q is None else q
    d16 = torch.tensor([[d]], dtype=torch.float16)
    dm16 = torch.tensor([[dmin]], dtype=torch.float16)
    return gen.pack_q4_k(d16, dm16, sc, m, q).numpy().reshape(1, 144)


def test_q4_k_scale_fields_are_a_bijection():
    """Every 6-bit scale and min of every sub-block decodes back alone."""
    for j in range(8):
        for v in range(64):
            sc = [0] * 8
            sc[j] = v
            dsc, dm = F.q4_k_fields(_pack(sc, [0] * 8))[2:4]
            assert dsc[0].tolist() == sc and dm[0].tolist() == [0] * 8
            m = [0] * 8
            m[j] = v
            dsc, dm = F.q4_k_fields(_pack([0] * 8, m))[2:4]
            assert dsc[0].tolist() == [0] * 8 and dm[0].tolist() == m


def test_q4_k_random_fields_round_trip():
    g = torch.Generator().manual_seed(3)
    for _ in range(50):
        sc = torch.randint(0, 64, (8,), generator=g).tolist()
        m = torch.randint(0, 64, (8,), generator=g).tolist()
        q = torch.randint(0, 16, (1, 1, 8, 32), generator=g)
        d, dmin, dsc, dm, dq = F.q4_k_fields(_pack(sc, m, q, d=0.0123, dmin=0.00456))
        assert dsc[0].tolist() == sc and dm[0].tolist() == m
        assert np.array_equal(dq[0], q[0, 0].numpy())
        assert d[0] == np.float64(np.float16(0.0123)) and dmin[0] == np.float64(np.float16(0.00456))


def test_q4_k_codes_layout_by_hand():
    """Sub-block 2p element i is the low nibble of code byte 32p+i, sub-block
    2p+1 element i its high nibble: a single code placed by hand."""
    blk = np.zeros((1, 144), dtype=np.uint8)
    blk[0, 0:2] = np.array([1.0], dtype=np.float16).view(np.uint8)   # d = 1
    blk[0, 4:8] = 1                                                # sc_0..3 = 1
    blk[0, 8:12] = 1                                               # sc_4..7 low nibble = 1
    blk[0, 16 + 32 * 1 + 5] = 0x70                                 # p=1, i=5: high nibble 7
    w = F.q4_k_dequant(blk)[0]
    expect = np.zeros(256)
    expect[32 * 3 + 5] = 7.0                                       # sub-block 3, element 5
    assert np.array_equal(w, expect)


def test_q4_k_dequant_within_quantiser_error_bound():
    """Encoding the generator's fp32 weights and decoding them must land
    within |w - w^| <= d*sc_j/2 + 7.5 d + dmin/2 for every weight."""
    for role, seed in ((gen.ROLE_GATE, 0), (gen.ROLE_DOWN, 5), (gen.ROLE_SH_UP, 9)):
        w = gen.float_weights(seed, 0, role, 3, 64, 2048)
        enc = gen.encode_q4_k(w).numpy()
        blocks = F.q4_k_rows(enc)
        d, dmin, sc, m, q = F.q4_k_fields(blocks)
        wh = F.q4_k_dequant(blocks).reshape(64, 2048)
        bound = (0.5 * d[..., None] * sc + 7.5 * d[..., None] + 0.5 * dmin[..., None])
        bound = np.repeat(bound.reshape(64, -1), 32, axis=1)
        err = np.abs(w.numpy().astype(np.float64) - wh)
        assert np.all(err <= bound * (1 + 1e-6) + 1e-12)
        # and the quantiser is not trivially loose: mean error well under the step
        assert err.mean() < 0.35 * np.mean(d[..., None] * sc)


def test_q4_k_dequant_products_exact_in_fp32():
    w = gen.float_weights(1, 0, gen.ROLE_UP, 0, 32, 2048)
    d, dmin, sc, m, q = F.q4_k_fields(F.q4_k_rows(gen.encode_q4_k(w).numpy()))
    a = d[..., None, None] * sc[..., None] * q
    b = dmin[..., None] * m
    assert np.array_equal(F.fp32(a), a) and np.array_equal(F.fp32(b), b)


def test_q8_0_round_trip_bound():
    w = gen.float_weights(2, 0, gen.ROLE_SH_GATE, 0, 32, 2048).numpy().astype(np.float64)
    enc = gen.encode_q8_0(torch.from_numpy(w.astype(np.float32))).numpy()
    d, q = F.q8_0_fields(F.q8_0_rows(enc))
    wh = F.q8_0_dequant(F.q8_0_rows(enc)).reshape(32, 2048)
    bound = np.repeat(d, 32, axis=1) * 0.5 * (1 + 2.0 ** -9)   # fp16 d rounding of amax/127
    assert np.all(np.abs(w - wh) <= bound + 1e-12)
    assert np.abs(q).max() == 127


# ----------------------------------------------------------------------------
# Q8_1 encoding
# ----------------------------------------------------------------------------

def test_q8_1_worked_example():
    g = _golden("q8_1_worked_example.txt")
    x = np.zeros(32)
    x[:len(g["x64"])] = np.array(g["x64"]) / 64.0
    a = F.q8_1_quantize(x)
    q = np.zeros(32, dtype=np.int64)
    q[:len(g["q"])] = g["q"]
    assert np.array_equal(a["q"][0], q)
    assert a["d"][0] == g["d"][0] and a["s"][0] == g["s"][0]
    b = F.q8_1_to_bytes(a)
    back = F.q8_1_from_bytes(b)
    assert np.array_equal(back["q"], a["q"]) and back["d"][0] == a["d"][0]


def test_q8_1_properties():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(32 * 500) * 10.0 ** rng.integers(-3, 3, 32 * 500)).astype(np.float32)
    x[32 * 7:32 * 8] = 0.0
    a = F.q8_1_quantize(x)
    xb = x.reshape(-1, 32).astype(np.float64)
    d32 = a["d32"].astype(np.float64)
    err = np.abs(xb - d32[:, None] * a["q"])
    assert np.all(err <= d32[:, None] * (0.5 + 1e-6))
    amax_pos = np.abs(xb).argmax(axis=1)
    live = d32 > 0
    assert np.all(np.abs(a["q"][np.arange(len(d32)), amax_pos][live]) == 127)
    assert np.all(a["q"][7] == 0) and a["d"][7] == 0 and a["s"][7] == 0
    neg = F.q8_1_quantize(-x)
    assert np.array_equal(neg["q"], -a["q"])


# ----------------------------------------------------------------------------
# router, top-k, softmax
# ----------------------------------------------------------------------------

def test_topk_hand_example():
    # values: e0=1, e1=3, e2=3, e3=2, e4=-0.0, e5=+0.0, e6=3, e7=-1, e8=2, e9=0.5
    l = [1.0, 3.0, 3.0, 2.0, -0.0, 0.0, 3.0, -1.0, 2.0, 0.5]
    # 3s tie -> 1,2,6; 2s -> 3,8; then 1 -> 0; 0.5 -> 9; -0.0 == +0.0 -> 4 before 5
    expect = [1, 2, 6, 3, 8, 0, 9, 4]
    assert M.topk_sort(l) == expect
    assert M.topk_rank_select(l) == expect


@pytest.mark.parametrize("n_experts", [256, 128])
def test_topk_sort_equals_rank_select_on_tie_stress(n_experts):
    for group in range(10):
        W, X, fam = gen.tie_stress_group(11, group, n_experts, 20)
        logits = X.double().numpy() @ W.double().numpy().T
        for t in range(X.shape[0]):
            a = M.topk_sort(logits[t])
            assert a == M.topk_rank_select(logits[t]), fam
            if fam == "zero_x":
                assert a == list(range(8))


def test_router_logits_integer_exact():
    W, X, _ = gen.tie_stress_group(4, 0, 128, 3)
    for t in range(3):
        l = M.router_logits(X[t], W)
        brute = [sum(int(W[e, h]) * int(X[t, h]) for h in range(2048)) for e in range(0, 128, 17)]
        assert [int(v) for v in l[0:128:17]] == brute


def test_softmax_selected_pins():
    from scipy.special import softmax
    rng = np.random.default_rng(5)
    l = rng.standard_normal(256) * 2
    ids, w = M.route(l)
    full = softmax(l)
    assert np.allclose(w, full[ids] / full[ids].sum(), rtol=1e-13, atol=0)
    assert abs(w.sum() - 1.0) < 1e-15
    assert np.all(np.diff(w) <= 0)
    # two-valued closed form: four logits a, four b, rest far below
    l2 = np.full(64, -50.0)
    l2[[3, 9, 20, 40]] = 1.5
    l2[[5, 6, 7, 8]] = -0.5
    ids2, w2 = M.route(l2)
    assert ids2 == [3, 9, 20, 40, 5, 6, 7, 8]
    wa = math.exp(1.5) / (4 * math.exp(1.5) + 4 * math.exp(-0.5))
    wb = math.exp(-0.5) / (4 * math.exp(1.5) + 4 * math.exp(-0.5))
    assert np.allclose(w2, [wa] * 4 + [wb] * 4, rtol=1e-14)


def test_x_zero_routes_to_first_eight_uniformly():
    L = gen.make_layer(gen.Q4K_LAYER_SHARED_Q8_0, 0, experts=list(range(8)))
    x = torch.zeros(2048, dtype=torch.bfloat16)
    o = M.layer_forward(L, x)
    assert o["ids"] == list(range(8)) and np.allclose(o["w"], 1 / 8)
    assert np.all(o["routed"] == 0) and np.all(o["y"] == 0) and o["shared_gate"] == 0.5


# ----------------------------------------------------------------------------
# integer dots and GEMVs
# ----------------------------------------------------------------------------

def _exact_activations(rng, n):
    """Q8_1-exact activations: per block amax 127/64 and small |sum q|, so that
    d = 1/64 and s = d * sum(q) are exact in fp16."""
    q = rng.integers(-40, 41, size=(n // 32, 32))
    q[:, 0] = 127
    return (q / 64.0).reshape(-1)


def test_q4_k_block_dots_brute_force():
    rng = np.random.default_rng(9)
    w = gen.encode_q4_k(gen.float_weights(3, 0, gen.ROLE_GATE, 1, 3, 512)).numpy()
    a = F.q8_1_quantize(rng.standard_normal(512).astype(np.float32))
    got = M.q4_k_block_dots(w, a)
    for r in range(3):
        for b in range(16):                        # 32-block b of the row
            sb, j = divmod(b, 8)                   # super-block, sub-block
            base = sb * 144 + 16 + 32 * (j // 2)
            tot = 0
            for i in range(32):
                byte = int(w[r, base + i])
                code = (byte & 15) if j % 2 == 0 else (byte >> 4)
                tot += code * int(a["q"][b, i])
            assert got[r, b] == tot


def test_q4_k_matvec_equals_dequantised_product_when_s_is_exact():
    rng = np.random.default_rng(10)
    w = gen.encode_q4_k(gen.float_weights(4, 0, gen.ROLE_UP, 2, 48, 2048)).numpy()
    x = _exact_activations(rng, 2048)
    a = F.q8_1_quantize(x)
    assert np.all(a["d"] == 1 / 64) and np.allclose(a["s"], a["d"] * a["q"].sum(1), rtol=0, atol=0)
    ref = M.dequant_rows("q4_k", w) @ F.q8_1_dequant(a)
    got = M.matvec_q4_k(w, a)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_q8_0_matvec_equals_dequantised_product():
    rng = np.random.default_rng(11)
    w = gen.encode_q8_0(gen.float_weights(5, 0, gen.ROLE_SH_DOWN, 0, 40, 512)).numpy()
    a = F.q8_1_quantize(rng.standard_normal(512).astype(np.float32))
    ref = M.dequant_rows("q8_0", w) @ F.q8_1_dequant(a)
    assert np.allclose(M.matvec_q8_0(w, a), ref, rtol=1e-12, atol=1e-12)


def test_expert_ffn_tiny_literal():
    """H=2, I=1, bf16: G=[[1,0]], U=[[0,2]], D=[[1],[3]], x=[1,1]:
    g=1, u=2, h=silu(1)*2 = 2/(1+e^-1), y = [h, 3h]."""
    def rows(vals):
        return torch.tensor(vals, dtype=torch.bfloat16).contiguous().view(torch.uint8).numpy()
    G, U, D = rows([[1.0, 0.0]]), rows([[0.0, 2.0]]), rows([[1.0], [3.0]])
    o = M.expert_ffn("bf16", G, U, D, np.array([1.0, 1.0]))
    h = 2.0 / (1.0 + math.exp(-1.0))
    assert o["h"][0] == pytest.approx(h, rel=1e-15)
    assert np.allclose(o["y"], [h, 3 * h], rtol=1e-15)


def test_routed_combination_is_convex_over_identical_experts():
    """With every selected expert holding the same weights, the routed
    output equals that one expert's output (the weights sum to one)."""
    L = gen.make_layer(gen.Q4K_LAYER_SHARED_Q4_K, 2, experts=[0])
    L8 = dict(L)
    L8["expert_ids"] = list(range(8))
    for k in ("gate", "up", "down"):
        L8[k] = L[k].expand(8, *L[k].shape[1:])
    x = M.as_f64(gen.make_tokens(2, 1)[0])
    ids = list(range(8))
    w = M.softmax_selected(np.linspace(1, 0, 8), ids)
    f = M.moe_ffn(L8, x, ids, w)
    assert np.allclose(f["routed"], f["experts"][0]["y"], rtol=1e-13, atol=1e-15)


def test_shared_gate_is_sigmoid_of_dot():
    L = gen.make_layer(gen.Q4K_LAYER_SHARED_Q8_0, 3, experts=[0])
    x = M.as_f64(gen.make_tokens(3, 1)[0])
    f = M.moe_ffn(L, x, [0], np.array([1.0]))
    z = float(np.dot(M.as_f64(L["w_sg"]), x))
    assert f["shared_gate"] == pytest.approx(1 / (1 + math.exp(-z)), rel=1e-15)
    assert np.allclose(f["shared"], f["shared_gate"] * f["shared_expert"]["y"], rtol=1e-15)


# ----------------------------------------------------------------------------
# residual fold
# ----------------------------------------------------------------------------

def test_add_rmsnorm3_equals_unfused_chain_bit_exact():
    rng = np.random.default_rng(12)
    for _ in range(20):
        a, b, c = (F.bf16(rng.standard_normal(2048) * s) for s in (0.1, 0.2, 1.0))
        w = F.bf16(1 + 0.1 * rng.standard_normal(2048))
        s1, y1 = M.add_rmsnorm3(a, b, c, w, 1e-6)
        s2, y2 = M.add_rmsnorm_unfused(a, b, c, w, 1e-6)
        assert np.array_equal(s1, s2) and np.array_equal(y1, y2)


def test_rmsnorm_constant_vector_closed_form():
    for cval in (0.75, -3.0, 1e-4):
        a = np.full(2048, cval)
        z = np.zeros(2048)
        w = F.bf16(np.linspace(0.5, 1.5, 2048))
        s, y = M.add_rmsnorm3(a, z, z, w, 1e-6)
        assert np.all(s == F.bf16(cval))
        cv = F.bf16(cval)
        assert np.array_equal(y, F.bf16(w * cv / math.sqrt(cv * cv + 1e-6)))


def test_rmsnorm_output_has_unit_rms_with_unit_weights():
    rng = np.random.default_rng(13)
    c = F.bf16(rng.standard_normal(2048) * 3)
    s, y = M.add_rmsnorm3(np.zeros(2048), np.zeros(2048), c, np.ones(2048), 0.0)
    assert abs(math.sqrt(np.mean(y * y)) - 1.0) < 4e-3
