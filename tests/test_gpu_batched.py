"""Batched tokens with per-token routing (grouped experts) against the oracle,
on the Qwen3-30B-A3B-shaped layer (128 experts, top-8, H=2048, I=768, Q4_K,
no shared expert)."""
import functools

import numpy as np
import pytest
import torch

import gen
import moe_decode_ffn_gb300 as m
from oracle import formats as F
from oracle import moe as M
from oracle import parity as P
from tests.gpu_common import bf16_np, device_layer

pytestmark = pytest.mark.gpu

SPEC = gen.Q4K_LAYER_128E
SEED = 500


@pytest.fixture(scope="module", autouse=True)
def _lib():
    m.build()
    m.library()


@functools.lru_cache(maxsize=2)
def host_layer_all(spec, seed, layer):
    """Every expert's bytes on the host (generated on the device; the generator
    is device independent)."""
    L = gen.make_layer(spec, seed, layer, device="cuda")
    return {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in L.items()}


def routing(seed, T, spec=SPEC, same=False):
    """Seeded distinct ids per token and softmax weights in rank order."""
    ids, ws = [], []
    for t in range(T):
        keys = gen.raw64([gen.stream_key(seed, 0 if same else t, 777)], spec.n_experts)[0]
        ids.append(torch.argsort(keys)[: spec.top_k].to(torch.int32))
        z = gen.normal([gen.stream_key(seed, t, 778)], spec.top_k, 0.0, 1.0)[0].double()
        ws.append(torch.softmax(torch.sort(z, descending=True).values, 0).to(torch.float32))
    return torch.stack(ids), torch.stack(ws)


def check_tokens(routed, x, ids, w, tokens):
    host = host_layer_all(SPEC, SEED, 0)
    for t in tokens:
        f = M.moe_ffn(host, M.as_f64(x[t]), ids[t].tolist(), w[t].double().numpy())
        ok, rep = P.float_parity(bf16_np(routed[t]), F.bf16(f["routed"]))
        assert ok, f"token {t}: {rep}"


@pytest.mark.parametrize("T", [1, 4, 16, 64])
def test_batched_int8_against_oracle(T):
    dev = device_layer(SPEC, SEED, 0)
    ids, w = routing(T, T)
    x = gen.make_tokens(900 + T, T)
    routed = m.si_moe_ffn_batched(dev, x.cuda(), ids.cuda(), w.cuda(), m.SI_FFN_INT8)
    torch.cuda.synchronize()
    tokens = range(T) if T <= 16 else range(0, T, 9)
    check_tokens(routed.cpu(), x, ids, w, tokens)


def test_batched_tokens_sharing_experts_spill_over_chunks():
    """All 40 tokens pick the same 8 experts: 40 tokens per expert, more than
    one chunk of resident token tiles."""
    T = 40
    dev = device_layer(SPEC, SEED, 0)
    ids, w = routing(7, T, same=True)
    x = gen.make_tokens(901, T)
    routed = m.si_moe_ffn_batched(dev, x.cuda(), ids.cuda(), w.cuda(), m.SI_FFN_INT8)
    torch.cuda.synchronize()
    check_tokens(routed.cpu(), x, ids, w, [0, 17, 39])


def test_batched_one_token_equals_single_token_path():
    dev = device_layer(SPEC, SEED, 0)
    ids, w = routing(3, 1)
    x = gen.make_tokens(902, 1).cuda()
    routed_b = m.si_moe_ffn_batched(dev, x, ids.cuda(), w.cuda(), m.SI_FFN_INT8)
    routed_d, _ = m.si_moe_ffn_decode(dev, x[0], ids[0].cuda(), w[0].cuda())
    assert torch.equal(routed_b[0], routed_d)


def test_batched_deterministic_and_status_clean():
    dev = device_layer(SPEC, SEED, 0)
    ids, w = routing(11, 16)
    x = gen.make_tokens(903, 16).cuda()
    ws = m.workspace(m.ffn_batched_workspace_bytes(dev, 16))
    a = m.si_moe_ffn_batched(dev, x, ids.cuda(), w.cuda(), m.SI_FFN_INT8, ws=ws)
    b = m.si_moe_ffn_batched(dev, x, ids.cuda(), w.cuda(), m.SI_FFN_INT8, ws=ws)
    assert torch.equal(a, b)
    assert m.si_workspace_status(ws) == m.SI_OK


# A wider layer: two super-blocks of each gate/up row per lane (H=4096) and
# eight half-super-block pieces per down row (I=1024).
WIDE = gen.LayerSpec(hidden=4096, n_experts=16, top_k=4, inter=1024, shared_inter=0,
                     expert_type="q4_k", shared_type="q4_k")


@pytest.mark.parametrize("T", [3, 12])
def test_batched_int8_wide_layer_against_oracle(T):
    dev = device_layer(WIDE, SEED, 0)
    ids, w = routing(40 + T, T, spec=WIDE)
    x = gen.make_tokens(950 + T, T, hidden=WIDE.hidden)
    routed = m.si_moe_ffn_batched(dev, x.cuda(), ids.cuda(), w.cuda(), m.SI_FFN_INT8)
    torch.cuda.synchronize()
    host = host_layer_all(WIDE, SEED, 0)
    for t in range(T):
        f = M.moe_ffn(host, M.as_f64(x[t]), ids[t].tolist(), w[t].double().numpy())
        ok, rep = P.float_parity(bf16_np(routed.cpu()[t]), F.bf16(f["routed"]))
        assert ok, f"token {t}: {rep}"


def test_batched_rejects_unsupported():
    dev = device_layer(SPEC, SEED, 0)
    ids, w = routing(1, 2)
    x = gen.make_tokens(904, 2).cuda()
    with pytest.raises(m.SiError) as e:
        m.si_moe_ffn_batched(dev, x, ids.cuda(), w.cuda(), 7)
    assert e.value.status == m.SI_ERR_INVALID_ARG
    shared_layer = device_layer(gen.Q4K_LAYER_SHARED_Q4_K, 100, 0)
    assert m.ffn_batched_workspace_bytes(shared_layer, 2) == 0


# ---------------------------------------------------------------------------
# tensor-core mode
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n,k", [(16, 16), (32, 64), (64, 256), (48, 128)])
def test_umma_f16_block_exact(n, k):
    """Small integers: every product and sum is exact in fp32, so the tensor
    core result must equal the integer matrix product exactly."""
    g = torch.Generator().manual_seed(n * 1000 + k)
    a = torch.randint(-4, 5, (128, k), generator=g).to(torch.float16)
    b = torch.randint(-4, 5, (n, k), generator=g).to(torch.float16)
    out = torch.empty(128, n, dtype=torch.float32, device="cuda")
    ws = m.workspace(256)
    da, db = a.cuda(), b.cuda()      # keep the device copies alive until the kernel has run
    st = m.library().si_test_umma_f16(da.data_ptr(), db.data_ptr(), n, k, out.data_ptr(),
                                      ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == m.SI_OK
    assert m.si_workspace_status(ws) == m.SI_OK
    ref = a.double().numpy() @ b.double().numpy().T
    assert np.array_equal(out.cpu().double().numpy(), ref)


def check_tokens_fp16(routed, x, ids, w, tokens):
    host = host_layer_all(SPEC, SEED, 0)
    for t in tokens:
        f = M.moe_ffn(host, M.as_f64(x[t]), ids[t].tolist(), w[t].double().numpy(), mode="fp16")
        ok, rep = P.float_parity(bf16_np(routed[t]), F.bf16(f["routed"]))
        assert ok, f"token {t}: {rep}"


@pytest.mark.parametrize("T", [16, 64])
def test_batched_tensor_against_oracle_fp16_mode(T):
    dev = device_layer(SPEC, SEED, 0)
    ids, w = routing(T + 100, T)
    x = gen.make_tokens(950 + T, T)
    routed = m.si_moe_ffn_batched(dev, x.cuda(), ids.cuda(), w.cuda(), m.SI_FFN_TENSOR)
    torch.cuda.synchronize()
    check_tokens_fp16(routed.cpu(), x, ids, w, range(0, T, 5))


def test_batched_tensor_tokens_sharing_experts():
    T = 40
    dev = device_layer(SPEC, SEED, 0)
    ids, w = routing(8, T, same=True)
    x = gen.make_tokens(951, T)
    ws = m.workspace(m.ffn_batched_workspace_bytes(dev, T))
    routed = m.si_moe_ffn_batched(dev, x.cuda(), ids.cuda(), w.cuda(), m.SI_FFN_TENSOR, ws=ws)
    torch.cuda.synchronize()
    assert m.si_workspace_status(ws) == m.SI_OK
    check_tokens_fp16(routed.cpu(), x, ids, w, [0, 21, 39])


def test_batched_auto_mode_is_the_integer_path():
    dev = device_layer(SPEC, SEED, 0)
    ids, w = routing(9, 16)
    x = gen.make_tokens(952, 16).cuda()
    auto = m.si_moe_ffn_batched(dev, x, ids.cuda(), w.cuda(), m.SI_FFN_AUTO)
    int8 = m.si_moe_ffn_batched(dev, x, ids.cuda(), w.cuda(), m.SI_FFN_INT8)
    assert torch.equal(auto, int8)
