"""The C-ABI library builds, loads and exports every declared symbol; host
argument validation (no device work)."""
import ctypes
import os
import re

import pytest

import moe_decode_ffn_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    m.build()
    return m.library()


def declared_symbols():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(si_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 18
    for n in names:
        assert hasattr(lib, n), n
        assert n in m.SIGNATURES, f"binding lacks {n}"


def test_status_strings_and_version(lib):
    for code in range(7):
        assert m.status_string(code).startswith("SI_")
    assert m.status_string(99) == "unknown si_status"
    assert lib.si_version() >> 16 == 1


def test_row_bytes(lib):
    assert lib.si_row_bytes(m.SI_Q4_K, 2048) == 8 * 144
    assert lib.si_row_bytes(m.SI_Q8_0, 2048) == 64 * 34
    assert lib.si_row_bytes(m.SI_Q8_1, 2048) == 64 * 36
    assert lib.si_row_bytes(m.SI_BF16, 2048) == 4096
    assert lib.si_row_bytes(m.SI_Q4_K, 100) == 0


def test_workspace_queries(lib):
    a = lib.si_moe_router_workspace_bytes(256, 2048, 1)
    b = lib.si_moe_router_workspace_bytes(256, 2048, 100)
    assert 0 < a < b and a % 256 == 0 and b % 256 == 0
    assert lib.si_moe_router_workspace_bytes(0, 2048, 1) == 0


def test_invalid_arguments_are_rejected_before_any_launch(lib):
    assert lib.si_quantize_q8_1(None, m.SI_F32, 32, None, None) == m.SI_ERR_INVALID_ARG
    assert lib.si_quantize_q8_1(16, m.SI_F32, 33, 16, None) == m.SI_ERR_INVALID_ARG
    assert lib.si_quantize_q8_1(16, m.SI_Q4_K, 32, 16, None) == m.SI_ERR_UNSUPPORTED
    r = lib.si_moe_router_topk(16, m.SI_BF16, 16, m.SI_BF16, 2048, 300, 8, 1, 16, 16, None, 256,
                               1 << 20, None)
    assert r == m.SI_ERR_INVALID_ARG                 # too many experts
    r = lib.si_moe_router_topk(16, m.SI_BF16, 16, m.SI_BF16, 2048, 256, 8, 1, 16, 16, None, 256,
                               16, None)
    assert r == m.SI_ERR_WORKSPACE                   # workspace too small
    r = lib.si_moe_router_topk(16, m.SI_BF16, 16, m.SI_BF16, 2048, 256, 9, 1, 16, 16, None, 256,
                               1 << 20, None)
    assert r == m.SI_ERR_INVALID_ARG                 # top_k > 8
    assert lib.si_add_rmsnorm3(16, 16, None, 16, 100, 1, 1e-6, 16, 16, None, None) == m.SI_ERR_INVALID_ARG
    L = m.SiMoeLayer()
    assert lib.si_moe_ffn_decode(ctypes.byref(L), 1, 16, None, 16, 16, 16, None, 256, 1 << 20,
                                 None) == m.SI_ERR_INVALID_ARG
    assert lib.si_graph_launch(None, None) == m.SI_ERR_INVALID_ARG
    assert lib.si_graph_is_persistent(None) == -1
    h = ctypes.c_void_p()
    assert lib.si_moe_stack_graph_create_mode(ctypes.byref(L), 1, 1, 16, 16, None, None, 256,
                                              1 << 20, 7, None, ctypes.byref(h)) == m.SI_ERR_INVALID_ARG


def test_empty_inputs_are_rejected_or_are_no_ops(lib):
    """Zero tokens, rows or values: every call answers before touching the
    device (an error, or for the load-time requant a no-op)."""
    assert lib.si_quantize_q8_1(16, m.SI_F32, 0, 16, None) == m.SI_ERR_INVALID_ARG
    r = lib.si_moe_router_topk(16, m.SI_BF16, 16, m.SI_BF16, 2048, 256, 8, 0, 16, 16, None, 256,
                               1 << 20, None)
    assert r == m.SI_ERR_INVALID_ARG
    assert lib.si_add_rmsnorm3(16, 16, None, 16, 2048, 0, 1e-6, 16, 16, None, None) == m.SI_ERR_INVALID_ARG
    assert lib.si_requant_q4_k(16, m.SI_Q8_0, 0, 2048, 16, None) == m.SI_OK
    L = m.SiMoeLayer()
    L.hidden, L.n_experts, L.top_k, L.inter = 2048, 128, 8, 768
    L.expert_type = m.SI_Q4_K
    L.w_gate = L.w_up = L.w_down = 256
    assert lib.si_moe_ffn_batched_workspace_bytes(ctypes.byref(L), 0) == 0
    assert lib.si_moe_ffn_batched(ctypes.byref(L), 0, 1, 16, 16, 16, 16, 256, 1 << 20,
                                  None) == m.SI_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert lib.si_moe_stack_graph_create_mode(ctypes.byref(L), 1, 0, 16, 16, None, None, 256,
                                              1 << 20, 0, None, ctypes.byref(h)) == m.SI_ERR_INVALID_ARG
    assert lib.si_moe_stack_graph_create_mode(ctypes.byref(L), 0, 1, 16, 16, None, None, 256,
                                              1 << 20, 0, None, ctypes.byref(h)) == m.SI_ERR_INVALID_ARG


def test_layer_descriptor_validation(lib):
    L = m.SiMoeLayer()
    L.hidden, L.n_experts, L.top_k, L.inter = 2048, 256, 8, 512
    L.expert_type = m.SI_Q4_K
    L.w_gate = L.w_up = L.w_down = 256
    L.shared_inter, L.shared_type = 512, m.SI_Q8_0
    L.ws_gate = L.ws_up = L.ws_down = L.w_shared_sigmoid = 256
    L.w_router, L.router_type, L.w_norm, L.eps = 256, m.SI_BF16, 256, 1e-6
    assert lib.si_moe_ffn_workspace_bytes(ctypes.byref(L), 1) > 0
    assert lib.si_moe_layer_workspace_bytes(ctypes.byref(L)) > 0
    L.shared_type = m.SI_BF16          # bf16 shared with Q4_K routed: not built
    assert lib.si_moe_layer_workspace_bytes(ctypes.byref(L)) == 0
    L.shared_type = m.SI_Q4_K
    L.inter = 500                      # not a multiple of 256
    assert lib.si_moe_layer_workspace_bytes(ctypes.byref(L)) == 0
    L.inter = 512
    L.w_gate = 257                     # misaligned
    assert lib.si_moe_layer_workspace_bytes(ctypes.byref(L)) == 0


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(m, "_lib", None)
    monkeypatch.setattr(m, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        m.library()
