"""Expert FFNs (routed + shared) on the GPU against the oracle, full-size
256-expert layers generated on the device."""
import numpy as np
import pytest
import torch

import gen
import moe_decode_ffn_gb300 as m
from oracle import formats as F
from oracle import moe as M
from oracle import parity as P
from tests.gpu_common import bf16_np, device_layer, host_layer_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    m.build()
    m.library()


@pytest.mark.parametrize("rows,k", [(64, 2048), (48, 512), (5, 768)])
def test_q4k_block_dots_bit_exact(rows, k):
    w = gen.encode_q4_k(gen.float_weights(7, 0, gen.ROLE_GATE, rows, rows, k))
    x = gen.normal([gen.stream_key(8, k)], k, 0.0, 1.0)[0]
    a = F.q8_1_quantize(x.numpy())
    a_bytes = torch.from_numpy(F.q8_1_to_bytes(a).reshape(-1))
    got = m.si_test_q4k_block_dots(w.cuda(), rows, k, a_bytes.cuda()).cpu().numpy()
    assert np.array_equal(got, M.q4_k_block_dots(w.numpy(), a))


# (kind, format, rows, k, vectors): the full gate/up (H = 2048) and down
# (I = 512 and 768) shapes of the studied layers, for every integer helper.
BLOCK_DOT_CASES = [
    (m.SI_TEST_DOTS_Q4K_SB, "q4_k", 512, 2048, 2),
    (m.SI_TEST_DOTS_Q4K_SB, "q4_k", 768, 2048, 1),
    (m.SI_TEST_DOTS_Q4K_HALF, "q4_k", 2048, 512, 2),
    (m.SI_TEST_DOTS_Q4K_HALF, "q4_k", 2048, 768, 1),
    (m.SI_TEST_DOTS_Q5K_HALF, "q5_k", 2048, 512, 2),
    (m.SI_TEST_DOTS_Q5K_HALF, "q5_k", 2048, 768, 1),
    (m.SI_TEST_DOTS_Q4K_SB_TOKENS, "q4_k", 768, 2048, 8),
    (m.SI_TEST_DOTS_Q4K_SB_TOKENS, "q4_k", 512, 2048, 3),
    (m.SI_TEST_DOTS_Q4K_HALF_TOKENS, "q4_k", 2048, 768, 8),
    (m.SI_TEST_DOTS_Q4K_HALF_TOKENS, "q4_k", 2048, 512, 5),
]


@pytest.mark.parametrize("kind,fmt,rows,k,nv", BLOCK_DOT_CASES)
def test_integer_block_dots_of_every_helper_bit_exact(kind, fmt, rows, k, nv):
    """Every integer dot helper (gate/up super-blocks, down halves, Q5_K
    halves, the batched forms that reuse a super-block's code words for
    several tokens) gives the oracle's exact int32 block sums."""
    w = gen.encode(gen.float_weights(17, kind, gen.ROLE_DOWN, rows, rows, k), fmt)
    # activations of both signs with a few blocks at full scale and one all-zero block
    x = gen.normal([gen.stream_key(18, kind, k, v) for v in range(nv)], k, 0.0, 1.0)
    x[:, 32:64] = 0.0
    acts = [F.q8_1_quantize(x[v].numpy()) for v in range(nv)]
    a_bytes = torch.from_numpy(np.concatenate([F.q8_1_to_bytes(a).reshape(-1) for a in acts]))
    got = m.si_test_block_dots(kind, w.cuda(), rows, k, a_bytes.cuda(), nv).cpu().numpy()
    dots = M.q5_k_block_dots if fmt == "q5_k" else M.q4_k_block_dots
    for v in range(nv):
        assert np.array_equal(got[v], dots(w.numpy(), acts[v])), v


def _routing(seed, spec):
    """Seeded distinct expert ids and softmax weights (inputs of the FFN call)."""
    keys = gen.raw64([gen.stream_key(seed, 999)], spec.n_experts)[0]
    ids = torch.argsort(keys)[: spec.top_k].to(torch.int32)
    z = gen.normal([gen.stream_key(seed, 998)], spec.top_k, 0.0, 1.0)[0].double()
    w = torch.softmax(torch.sort(z, descending=True).values, 0).to(torch.float32)
    return ids, w


SPECS = {
    "q4k_shared_q8_0": gen.Q4K_LAYER_SHARED_Q8_0,
    "q4k_shared_q4k": gen.Q4K_LAYER_SHARED_Q4_K,
    "bf16": gen.BF16_LAYER,
    "q4k_128e_i768": gen.Q4K_LAYER_128E,
    # bf16 shapes that take the other branches of the bf16 kernels: two
    # 2048-wide chunks per gate/up row and two 512-wide chunks per down row
    # (H=4096, I=1024) with a shared width that ends mid-chunk (768); a
    # hidden size that ends mid-chunk (2304); down rows narrower than one
    # chunk and no shared expert (I=256)
    "bf16_h4096_i1024": gen.LayerSpec(hidden=4096, n_experts=16, top_k=4, inter=1024,
                                      expert_type="bf16", shared_inter=768, shared_type="bf16"),
    "bf16_h2304_i512": gen.LayerSpec(hidden=2304, n_experts=8, top_k=2, inter=512,
                                     expert_type="bf16", shared_inter=256, shared_type="bf16"),
    "bf16_no_shared_i256": gen.LayerSpec(hidden=2048, n_experts=8, top_k=2, inter=256,
                                         expert_type="bf16", shared_inter=0, shared_type="bf16"),
}


@pytest.mark.parametrize("name", list(SPECS))
@pytest.mark.parametrize("seed", [0, 1])
def test_ffn_decode_against_oracle(name, seed):
    spec = SPECS[name]
    dev = device_layer(spec, 100, 0)
    ids, w = _routing(seed, spec)
    x = gen.make_tokens(500 + seed, 1, hidden=spec.hidden)[0]
    ws = m.workspace(m.ffn_workspace_bytes(dev))
    routed, shared = m.si_moe_ffn_decode(dev, x.cuda(), ids.cuda(), w.cuda(), ws=ws)
    assert m.si_workspace_status(ws) == m.SI_OK
    host = host_layer_for(spec, 100, 0, ids.tolist())
    f = M.moe_ffn(host, M.as_f64(x), ids.tolist(), w.double().numpy())
    ok, rep = P.float_parity(bf16_np(routed), F.bf16(f["routed"]))
    assert ok, "routed " + rep
    if spec.shared_inter:
        ok, rep = P.float_parity(bf16_np(shared), F.bf16(f["shared"]))
        assert ok, "shared " + rep


def test_ffn_given_q8_1_input_matches_internal_quantisation():
    spec = gen.Q4K_LAYER_SHARED_Q8_0
    dev = device_layer(spec, 100, 0)
    ids, w = _routing(3, spec)
    x = gen.make_tokens(503, 1)[0].cuda()
    xq = m.si_quantize_q8_1(x)
    r1, s1 = m.si_moe_ffn_decode(dev, x, ids.cuda(), w.cuda())
    r2, s2 = m.si_moe_ffn_decode(dev, x, ids.cuda(), w.cuda(), x_q8_1=xq)
    assert torch.equal(r1, r2) and torch.equal(s1, s2)


def test_ffn_h_codes_follow_the_oracle():
    """The gate/up kernel's Q8_1 codes of h: almost all equal to the oracle's
    (h is fp32 on both sides; rounding-order differences may move a value
    across a code boundary by one)."""
    spec = gen.Q4K_LAYER_SHARED_Q4_K
    dev = device_layer(spec, 100, 0)
    ids, w = _routing(4, spec)
    x = gen.make_tokens(504, 1)[0]
    ws = m.workspace(m.ffn_workspace_bytes(dev))
    m.si_moe_ffn_decode(dev, x.cuda(), ids.cuda(), w.cuda(), ws=ws)
    torch.cuda.synchronize()
    nq = spec.top_k * spec.inter + spec.shared_inter
    hq = ws[256:256 + nq].cpu().view(torch.int8).numpy().astype(np.int64)
    host = host_layer_for(spec, 100, 0, ids.tolist())
    f = M.moe_ffn(host, M.as_f64(x), ids.tolist(), w.double().numpy())
    ref = np.concatenate([e["h_q8_1"]["q"].reshape(-1) for e in f["experts"]] +
                         [f["shared_expert"]["h_q8_1"]["q"].reshape(-1)])
    diff = np.abs(hq - ref)
    assert diff.max() <= 1 and (diff != 0).mean() < 2e-3


def test_ffn_rejects_bad_arguments():
    spec = gen.Q4K_LAYER_SHARED_Q8_0
    dev = device_layer(spec, 100, 0)
    ids, w = _routing(0, spec)
    x = gen.make_tokens(1, 1)[0].cuda()
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(m.SiError) as e:
        m.si_moe_ffn_decode(dev, x, ids.cuda(), w.cuda(), ws=small)
    assert e.value.status == m.SI_ERR_WORKSPACE


def test_binding_rejects_buffers_of_the_wrong_size():
    """The C ABI takes raw pointers; the binding checks element counts and
    dtypes so that a short buffer never reaches a kernel."""
    spec = gen.Q4K_LAYER_SHARED_Q8_0
    dev = device_layer(spec, 100, 0)
    ids, w = _routing(0, spec)
    x = gen.make_tokens(1, 1)[0].cuda()
    with pytest.raises(ValueError):
        m.si_moe_ffn_decode(dev, x[:1024], ids.cuda(), w.cuda())
    with pytest.raises(ValueError):
        m.si_moe_ffn_decode(dev, x, ids[:4].cuda(), w.cuda())
    with pytest.raises(ValueError):
        m.si_moe_ffn_decode(dev, x.float(), ids.cuda(), w.cuda())
    with pytest.raises(ValueError):
        m.si_moe_layer_decode(dev, x, x[:2047])


def test_ffn_out_of_range_expert_is_reported_not_faulted():
    spec = gen.Q4K_LAYER_SHARED_Q8_0
    dev = device_layer(spec, 100, 0)
    _, w = _routing(0, spec)
    ids = torch.tensor([0, 1, 2, 3, 4, 5, 6, 100000], dtype=torch.int32)
    x = gen.make_tokens(1, 1)[0].cuda()
    ws = m.workspace(m.ffn_workspace_bytes(dev))
    m.si_moe_ffn_decode(dev, x, ids.cuda(), w.cuda(), ws=ws)
    assert m.si_workspace_status(ws) == m.SI_ERR_INVALID_ARG


@pytest.mark.parametrize("fmt", ["q4_k", "q8_0", "bf16"])
def test_generator_bytes_identical_on_cpu_and_gpu(fmt):
    """Device-generated weights are the bytes the oracle regenerates on the CPU."""
    for role, e in ((gen.ROLE_GATE, 0), (gen.ROLE_DOWN, 77), (gen.ROLE_SH_UP, 0)):
        cpu = gen._weights(5, 1, role, [e, e + 1], 512, 2048, fmt, "cpu")
        dev = gen._weights(5, 1, role, [e, e + 1], 512, 2048, fmt, "cuda")
        assert torch.equal(cpu, dev.cpu()), (fmt, role)
    assert torch.equal(gen.make_tokens(9, 4), gen.make_tokens(9, 4, device="cuda").cpu())
