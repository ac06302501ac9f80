"""The C-ABI library loads, exports every symbol include/edge0.h declares, and
rejects bad arguments on the host before launching anything (no GPU needed)."""
import ctypes as C
import os
import re

import pytest

from int4_routed_expert_prerouter_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "edge0.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(edge0_[A-Za-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_operations():
    syms = declared_symbols()
    for name in ("edge0_prerouter_topk", "edge0_moe_int4_forward", "edge0_lora_delta",
                 "edge0_decode_layer"):
        assert name in syms


def test_every_declared_symbol_is_exported(lib):
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, missing
    assert sorted(binding.EXPORTED) == declared_symbols()


def test_status_strings(lib):
    for code in range(5):
        assert binding.status_string(code)
    assert binding.status_string(0) == "ok"


def test_sizes(lib):
    # packed sizes equal the canonical sizes when rows are a multiple of 16:
    # 1,769,472 bytes per 35B-tier expert (gate + up + down at d=2048, I=512)
    gu = lib.edge0_q4_gate_up_packed_bytes(1, 512, 2048)
    dn = lib.edge0_q4_down_packed_bytes(1, 2048, 512)
    assert gu == 2 * (512 * 2048 // 2 + 512 * 32 * 4)
    assert gu + dn == 1769472
    assert lib.edge0_q4_gate_up_packed_bytes(256, 512, 2048) == 256 * gu
    assert lib.edge0_q4_down_packed_bytes(1, 512, 100) == 0     # in % 64
    assert lib.edge0_f16_packed_bytes(512, 2048) == 512 * 2048 * 2
    assert lib.edge0_f16_packed_bytes(4, 128) == 16 * 128 * 2   # rows padded to 16
    assert binding.workspace_bytes(40, 1, 2048, 256) > 0
    assert lib.edge0_workspace_bytes(0, 1, 2048, 256) == 0


def test_host_validation_rejects_bad_arguments(lib):
    E = binding.EDGE0_EINVAL
    assert lib.edge0_pack_q4_gate_up(None, None, None, None, None, None, 1, 64, 64, None, None) == E
    assert lib.edge0_pack_q4_down(None, None, None, 1, 16, 64, None, None) == E
    assert lib.edge0_pack_f16(None, 16, 64, 64, None, None) == E
    assert lib.edge0_pack_f16_kmajor(None, 16, 64, 64, None, None) == E
    assert lib.edge0_pack_cols_T(None, 16, 64, 0, 8, None, None) == E
    assert lib.edge0_moe_int4_forward(None, None, None, None, 1, None, None, 0, None) == E
    assert lib.edge0_prerouter_topk(None, None, None, None, 1, None, None, None, None, 0, None) == E
    assert lib.edge0_lora_delta(None, None, 1, None, None) == E
    assert lib.edge0_decode_layer(None, None, None, 1, 0, None) == E
    assert lib.edge0_decode_step(None, 0, None, None, 1, 0, None) == E
    st = binding.RouteState()
    assert lib.edge0_state_init(C.byref(st), None) == E
    # a MoE descriptor with an input width that is not a multiple of the group
    moe = binding.MoeDesc(100, 16, 2, 128, 128, 16, 16, None, None, None, 0)
    x = C.c_void_p(16)
    assert lib.edge0_moe_int4_forward(C.byref(moe), x, x, x, 1, x, x, 1 << 20, None) == E
    # K > E
    moe = binding.MoeDesc(256, 16, 17, 128, 128, 16, 16, None, None, None, 0)
    assert lib.edge0_moe_int4_forward(C.byref(moe), x, x, x, 1, x, x, 1 << 20, None) == E
    # batch above the limit
    moe = binding.MoeDesc(256, 16, 2, 128, 128, 16, 16, None, None, None, 0)
    assert lib.edge0_moe_int4_forward(C.byref(moe), x, x, x, 99, x, x, 1 << 20, None) == E
    # misaligned input pointer
    assert lib.edge0_moe_int4_forward(C.byref(moe), C.c_void_p(18), x, x, 1, x, x, 1 << 20, None) == E
    # workspace too small
    assert lib.edge0_moe_int4_forward(C.byref(moe), x, x, x, 1, x, x, 64, None) == E


def test_batched_path_sizes_and_host_validation(lib):
    from int4_routed_expert_prerouter_gb300 import configs
    c = configs.STACK8
    size = lambda B: lib.edge0_decode_workspace_bytes(c.L, B, c.d, c.E, c.K, c.I, c.Is, c.H)
    # B <= 4: the persistent engine's workspace
    assert size(4) == lib.edge0_workspace_bytes(c.L, 4, c.d, c.E)
    # B > 4: at least the layer output, x of every layer and act of every
    # (token, expert) pair of the batched path
    B = 64
    assert size(B) >= 256 + B * c.d * 4 + c.L * B * c.d * 2 + (B * c.K + B) * c.I * 4
    assert size(256) > size(64) > 0
    assert size(257) == 0
    # decode calls on the batched path that the host rejects before any launch
    E = binding.EDGE0_EINVAL
    p = C.c_void_p(256)
    layer = binding.LayerDesc()
    layer.moe = binding.MoeDesc(c.d, c.E, c.K, c.I, c.Is, p, p, None, None, None, 0)
    layer.router = p

    def state(B, nbytes):
        return binding.RouteState(c.L, B, c.K, p, p, p, p, nbytes)

    st = state(257, 1 << 40)
    assert lib.edge0_decode_step(C.byref(layer), 1, p, C.byref(st), 257, 0, None) == E   # B above the limit
    st = state(64, 1 << 40)
    assert lib.edge0_decode_step(C.byref(layer), 1, p, C.byref(st), 64, -1, None) == E   # step counter: engine only
    st = state(64, 4096)
    assert lib.edge0_decode_step(C.byref(layer), 1, p, C.byref(st), 64, 0, None) == E    # workspace too small
