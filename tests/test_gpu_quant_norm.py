"""Q8_1 quantiser and residual norm on the GPU against the oracle."""
import numpy as np
import pytest
import torch

import gen
import moe_decode_ffn_gb300 as m
from oracle import formats as F
from oracle import moe as M
from oracle import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    m.build()
    m.library()


def _activation_vector(n, seed):
    x = gen.normal([gen.stream_key(seed, n, 77)], n, 0.0, 1.0)[0]
    scale = gen.uniform_int([gen.stream_key(seed, n, 78)], n // 32, -8, 6)[0].to(torch.float32)
    x = x * torch.pow(torch.tensor(10.0), scale).repeat_interleave(32) / 10
    nb = n // 32
    if nb > 3:
        x[0:32] = 0.0                                           # all-zero block
        x[32:64] = torch.arange(-16, 16, dtype=torch.float32) / 64 + 0.0078125   # exact halves
        x[64:96] = torch.tensor([127.0] + [-62.5, 0.5, 2.5, -0.25] * 7 + [1, 2, 3]) / 64
    return x


# 32 * 393217: more groups of 8 values than one pass of the grid-stride
# quantiser covers on a 152-SM part, ending in a partial warp
@pytest.mark.parametrize("n", [32, 256, 2048, 32 * 1001, 1 << 20, 32 * 393217])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quantize_q8_1_bit_exact(n, dtype):
    x = _activation_vector(n, 5).to(dtype)
    got = m.si_quantize_q8_1(x.cuda()).cpu().numpy().reshape(-1, 36)
    ref = F.q8_1_to_bytes(F.q8_1_quantize(x.float().numpy()))
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:5]


@pytest.mark.parametrize("offset", [4, 8, 12])
def test_quantize_q8_1_output_only_4_byte_aligned(offset):
    """An output that starts 4 bytes past a 16-byte boundary (the minimum
    alignment the call accepts): the same bytes, none written outside it."""
    n = 32 * 8192 + 32 * 37          # 32 full chunks of 256 blocks, then a partial one
    x = _activation_vector(n, 6).to(torch.bfloat16)
    buf = torch.full((n // 32 * 36 + 32,), 0xA5, dtype=torch.uint8, device="cuda")
    out = buf[offset:offset + n // 32 * 36]
    m.si_quantize_q8_1(x.cuda(), out=out)
    got = buf.cpu().numpy()
    ref = F.q8_1_to_bytes(F.q8_1_quantize(x.float().numpy())).reshape(-1)
    assert np.array_equal(got[offset:offset + ref.size], ref)
    assert (got[:offset] == 0xA5).all() and (got[offset + ref.size:] == 0xA5).all()


def _near_half_quotients(n_blocks, seed):
    """Blocks whose quotients x / d sit on, or within a few 1e-5 of, the
    half-integer rounding boundaries (and others well inside), for scales d
    that are not powers of two, plus blocks of subnormal and tiny amax."""
    rng = np.random.default_rng(seed)
    out = np.zeros((n_blocks, 32), dtype=np.float32)
    offsets = np.array([0.0, 1e-7, -1e-7, 1e-6, -1e-6, 1e-5, -1e-5, 2.2e-5, -2.2e-5, 2.9e-5,
                        -2.9e-5, 3.1e-5, -3.1e-5, 5e-5, -5e-5, 0.25])
    for b in range(n_blocks):
        amax = np.float32(rng.uniform(0.01, 100.0) * 10.0 ** rng.integers(-30, 30))
        if b % 17 == 0:
            amax = np.float32(rng.uniform(1.0, 1000.0) * 1e-42)   # subnormal scale
        d = np.float32(amax / np.float32(127.0))
        out[b, 0] = amax if b % 2 else -amax
        for i in range(1, 32):
            k = rng.integers(-127, 127)
            t = k + 0.5 + offsets[rng.integers(len(offsets))]
            v = np.float32(np.float64(t) * np.float64(d))
            if abs(v) > amax:
                v = np.float32(np.sign(v) * amax)
            if rng.integers(4) == 0:   # the neighbours of the product
                v = np.nextafter(v, np.float32(np.inf) if rng.integers(2) else np.float32(-np.inf))
                if abs(v) > amax:
                    v = np.float32(np.sign(v) * amax)
            out[b, i] = v
    return out.reshape(-1)


def test_quantize_q8_1_codes_at_rounding_boundaries():
    """Codes decided by quotients on or next to a half-integer: bit-exact
    against the oracle's IEEE fp32 division (also through the norm's fused
    Q8_1 output path's encoder, which is the same)."""
    x = torch.from_numpy(_near_half_quotients(4096, 11))
    got = m.si_quantize_q8_1(x.cuda()).cpu().numpy().reshape(-1, 36)
    ref = F.q8_1_to_bytes(F.q8_1_quantize(x.numpy()))
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:5]


def _norm_inputs(rows, n, seed, scales=(0.1, 0.2, 1.0)):
    keys = [gen.stream_key(seed, i, rows, n) for i in range(4)]
    vs = [gen.to_bf16(gen.normal([keys[i]], rows * n, 0.0, s)[0].reshape(rows, n))
          for i, s in enumerate(scales)]
    w = gen.to_bf16(gen.normal([keys[3]], n, 1.0, 0.1)[0])
    return vs, w


@pytest.mark.parametrize("rows,n", [(1, 2048), (3, 256), (5, 4096), (2, 16384)])
def test_add_rmsnorm3_against_oracle(rows, n):
    (a, b, c), w = _norm_inputs(rows, n, 9)
    s, y, q8 = m.si_add_rmsnorm3(a.cuda(), b.cuda(), c.cuda(), w.cuda(), 1e-6, want_q8=True)
    s, y, q8 = s.cpu(), y.cpu(), q8.cpu().numpy().reshape(rows, -1, 36)
    for r in range(rows):
        rs, ry = M.add_rmsnorm3(M.as_f64(a[r]), M.as_f64(b[r]), M.as_f64(c[r]), M.as_f64(w), 1e-6)
        assert np.array_equal(M.as_f64(s[r]), rs)              # two fp32 adds: exact
        ok, rep = P.float_parity(M.as_f64(y[r]), ry)
        assert ok, rep
        # the fused Q8_1 output equals the quantiser applied to the kernel's own y
        assert np.array_equal(q8[r], F.q8_1_to_bytes(F.q8_1_quantize(M.as_f64(y[r]))))


def test_add_rmsnorm3_equals_unfused_chain_on_gpu():
    (a, b, c), w = _norm_inputs(4, 2048, 11)
    s1, y1, _ = m.si_add_rmsnorm3(a.cuda(), b.cuda(), c.cuda(), w.cuda(), 1e-6)
    s2, y2 = m.si_test_unfused_add_rmsnorm(a.cuda(), b.cuda(), c.cuda(), w.cuda(), 1e-6)
    assert torch.equal(s1, s2) and torch.equal(y1, y2)


def test_add_rmsnorm_two_input_mode():
    (a, b, _), w = _norm_inputs(2, 2048, 12)
    s, y, _ = m.si_add_rmsnorm3(a.cuda(), b.cuda(), None, w.cuda(), 1e-6)
    for r in range(2):
        rs, ry = M.add_rmsnorm2(M.as_f64(a[r]), M.as_f64(b[r]), M.as_f64(w), 1e-6)
        assert np.array_equal(M.as_f64(s[r].cpu()), rs)
        ok, rep = P.float_parity(M.as_f64(y[r].cpu()), ry)
        assert ok, rep


def test_rmsnorm_zero_and_constant_rows():
    n = 2048
    a = torch.zeros(2, n, dtype=torch.bfloat16)
    a[1] = 0.75
    z = torch.zeros_like(a)
    w = gen.to_bf16(torch.linspace(0.5, 1.5, n))
    s, y, _ = m.si_add_rmsnorm3(a.cuda(), z.cuda(), z.cuda(), w.cuda(), 1e-6)
    y = M.as_f64(y.cpu())
    assert np.all(y[0] == 0)
    ref = F.bf16(M.as_f64(w) * 0.75 / np.sqrt(0.75 ** 2 + 1e-6))
    assert np.all(np.abs(y[1] - ref) <= P.ulp_bf16(ref))
