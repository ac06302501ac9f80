"""The allocation-free MoE forward (edge0_moe_int4_forward_noalloc).

It serves callers that cannot allocate memory when they run the MoE block (an
allocator-free part of a serving loop, a memory budget fixed at start-up, a host
that only hands over buffers it already owns): its scratch is a fixed array
inside the library.  These tests call it through the C ABI twice in a row and
check each result against edge0_moe_int4_forward (which takes a caller-owned
workspace) and against the CPU oracle, within the parity tolerance the other
tests use; they cover a layer without a shared expert, a slot table over a
smaller slot stack, and the device-side status that edge0_noalloc_error reads.
The file is named to be collected last.
"""
import ctypes as C

import pytest
import torch

import oracle
from int4_routed_expert_prerouter_gb300 import binding, configs, inputs
from parity_util import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _stream():
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _noalloc(moe, x, ids, w):
    y = torch.empty_like(x)
    rc = binding.lib().edge0_moe_int4_forward_noalloc(C.byref(moe), C.c_void_p(x.data_ptr()),
                                                      C.c_void_p(ids.data_ptr()), C.c_void_p(w.data_ptr()),
                                                      x.shape[0], C.c_void_p(y.data_ptr()), _stream())
    assert rc == 0, binding.status_string(rc)
    return y


def _device_status():
    code = C.c_int(-1)
    rc = binding.lib().edge0_noalloc_error(_stream(), C.byref(code))
    assert rc == 0, binding.status_string(rc)
    return code.value


def _oracle_y(cfg, lw, x, ids, w):
    _, y = oracle.moe_forward(cfg, lw, x.cpu(), ids.cpu(), w.cpu())
    return y


CASES = [configs.STACK35.with_(L=1, E=32, B=2, head_owner_last=-1, prerouted=()),
         configs.TOY.with_(B=3, head_owner_last=-1, prerouted=())]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: f"{c.name}-B{c.B}")
def test_noalloc_matches_the_workspace_entry_point_two_calls_in_a_row(cfg):
    model = inputs.make_model(cfg.with_(L=1), seed=41)
    dm = binding.DeviceModel(model, DEV)
    ws = torch.zeros(binding.workspace_bytes(1, cfg.B, cfg.d, cfg.E), dtype=torch.uint8, device=DEV)
    for call in range(2):
        x = torch.stack([oracle.rmsnorm(h) for h in inputs.hidden(cfg, 10 + call, seed=41)]).to(DEV)
        ids, w = inputs.routing(cfg, 41, call)
        ids, w = ids.to(DEV), w.to(DEV)
        y_ref = binding.moe_int4_forward(dm, 0, x, ids, w, ws)
        y = _noalloc(dm.layers[0].moe, x, ids, w)
        torch.cuda.synchronize()
        assert _device_status() == 0
        assert_close(y, y_ref.double(), f"call {call} vs the workspace entry point")
        assert_close(y, _oracle_y(cfg, model.layers[0], x, ids, w), f"call {call} vs the oracle")


def test_noalloc_without_a_shared_expert():
    cfg = CASES[0]
    model = inputs.make_model(cfg.with_(L=1), seed=43)
    dm = binding.DeviceModel(model, DEV)
    moe = binding.MoeDesc.from_buffer_copy(dm.layers[0].moe)
    moe.sh_gate_up = moe.sh_down = None
    ws = torch.zeros(binding.workspace_bytes(1, cfg.B, cfg.d, cfg.E), dtype=torch.uint8, device=DEV)
    lw = model.layers[0]
    # the oracle's view of the same layer without its shared expert: zero weights
    # (nibbles and biases 0) contribute nothing
    zero = lambda trip: tuple(torch.zeros_like(t) for t in trip)
    lw0 = inputs.LayerWeights(lw.gate, lw.up, lw.down, zero(lw.sh_gate), zero(lw.sh_up), zero(lw.sh_down),
                              lw.router, lw.gamma, lw.lora, lw.bias, lw.head, lw.prerouted)
    for call in range(2):
        x = torch.stack([oracle.rmsnorm(h) for h in inputs.hidden(cfg, 20 + call, seed=43)]).to(DEV)
        ids, w = inputs.routing(cfg, 43, call)
        ids, w = ids.to(DEV), w.to(DEV)
        y = _noalloc(moe, x, ids, w)
        y_ref = torch.empty_like(x)
        rc = binding.lib().edge0_moe_int4_forward(C.byref(moe), C.c_void_p(x.data_ptr()),
                                                  C.c_void_p(ids.data_ptr()), C.c_void_p(w.data_ptr()), cfg.B,
                                                  C.c_void_p(y_ref.data_ptr()), C.c_void_p(ws.data_ptr()),
                                                  ws.numel(), _stream())
        assert rc == 0
        torch.cuda.synchronize()
        assert _device_status() == 0
        assert_close(y, y_ref.double(), f"call {call} vs the workspace entry point")
        assert_close(y, _oracle_y(cfg, lw0, x, ids, w), f"call {call} vs the oracle")


def _slot_stacks(dm, cfg, resident):
    """Device slot stacks holding the experts `resident` (slot i = resident[i])
    and the slot table of all E experts (-1: not resident)."""
    gu, dn = dm.stacks[0]
    gu_s = gu.view(cfg.E, -1)[resident].contiguous()
    dn_s = dn.view(cfg.E, -1)[resident].contiguous()
    table = torch.full((cfg.E,), -1, dtype=torch.int32)
    table[resident] = torch.arange(len(resident), dtype=torch.int32)
    return gu_s, dn_s, table.to(DEV)


def test_noalloc_with_a_slot_table_over_fewer_slots():
    cfg = CASES[0]
    model = inputs.make_model(cfg.with_(L=1), seed=45)
    dm = binding.DeviceModel(model, DEV)
    resident = torch.arange(cfg.E - 1, -1, -2)          # odd experts, reversed: 16 slots of 32
    gu_s, dn_s, table = _slot_stacks(dm, cfg, resident)
    moe = binding.MoeDesc.from_buffer_copy(dm.layers[0].moe)
    moe.gate_up, moe.down = gu_s.data_ptr(), dn_s.data_ptr()
    moe.slot_table, moe.n_slots = table.data_ptr(), len(resident)
    ws = torch.zeros(binding.workspace_bytes(1, cfg.B, cfg.d, cfg.E), dtype=torch.uint8, device=DEV)
    g = torch.Generator().manual_seed(45)
    for call in range(2):
        x = torch.stack([oracle.rmsnorm(h) for h in inputs.hidden(cfg, 30 + call, seed=45)]).to(DEV)
        ids = torch.stack([resident[torch.randperm(len(resident), generator=g)[:cfg.K]]
                           for _ in range(cfg.B)]).to(torch.int32)
        w = torch.softmax(torch.randn(cfg.B, cfg.K, generator=g), -1)
        ids, w = ids.to(DEV), w.to(DEV)
        y = _noalloc(moe, x, ids, w)
        y_ref = torch.empty_like(x)
        rc = binding.lib().edge0_moe_int4_forward(C.byref(moe), C.c_void_p(x.data_ptr()),
                                                  C.c_void_p(ids.data_ptr()), C.c_void_p(w.data_ptr()), cfg.B,
                                                  C.c_void_p(y_ref.data_ptr()), C.c_void_p(ws.data_ptr()),
                                                  ws.numel(), _stream())
        assert rc == 0
        torch.cuda.synchronize()
        assert _device_status() == 0
        assert_close(y, y_ref.double(), f"call {call} vs the workspace entry point")
        assert_close(y, _oracle_y(cfg, model.layers[0], x, ids, w), f"call {call} vs the oracle")


def test_noalloc_reports_a_slot_outside_the_stack_then_recovers():
    # an id whose slot-table entry is n_slots: the kernel's own check records
    # EDGE0_EINVAL (no copy is made from it); edge0_noalloc_error reads and clears it
    cfg = CASES[0]
    model = inputs.make_model(cfg.with_(L=1), seed=47)
    dm = binding.DeviceModel(model, DEV)
    resident = torch.arange(0, cfg.E, 2)
    gu_s, dn_s, table = _slot_stacks(dm, cfg, resident)
    table[1] = len(resident)                             # outside [0, n_slots)
    moe = binding.MoeDesc.from_buffer_copy(dm.layers[0].moe)
    moe.gate_up, moe.down = gu_s.data_ptr(), dn_s.data_ptr()
    moe.slot_table, moe.n_slots = table.data_ptr(), len(resident)
    x = torch.stack([oracle.rmsnorm(h) for h in inputs.hidden(cfg, 40, seed=47)]).to(DEV)
    bad = torch.tensor([[1, 0, 2, 4]] * cfg.B, dtype=torch.int32, device=DEV)
    w = torch.full((cfg.B, cfg.K), 0.25, device=DEV)
    _noalloc(moe, x, bad, w)
    torch.cuda.synchronize()
    assert _device_status() == binding.EDGE0_EINVAL
    assert _device_status() == 0
    good = torch.tensor([[6, 0, 2, 4]] * cfg.B, dtype=torch.int32, device=DEV)
    y = _noalloc(moe, x, good, w)
    torch.cuda.synchronize()
    assert _device_status() == 0
    assert_close(y, _oracle_y(cfg, model.layers[0], x, good, w), "after the reported error")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = binding.lib()
    x = C.c_void_p(256)
    # d = 4096 with 512 experts at B = 4 needs 512 + 10 B d + 16 B E + 384 B = 198,656
    # bytes of scratch, more than the fixed array holds
    moe = binding.MoeDesc(4096, 512, 8, 512, 512, 256, 256, None, None, None, 0)
    rc = lib.edge0_moe_int4_forward_noalloc(C.byref(moe), x, x, x, 4, x, None)
    assert rc == binding.EDGE0_EUNSUPPORTED
