"""The allocation-free MoE forward (edge0_moe_int4_forward_noalloc).

It serves callers that cannot allocate memory when they run the MoE block (an
allocator-free part of a serving loop, a memory budget fixed at start-up, a host
that only hands over buffers it already owns): its scratch is a fixed array
inside the library.  This test calls it through the C ABI twice in a row and
checks each result against edge0_moe_int4_forward (which takes a caller-owned
workspace) within the parity tolerance the other tests use.  It lives in its own
file, named to be collected last.
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


@pytest.mark.parametrize("cfg", [configs.STACK35.with_(L=1, E=32, B=2, head_owner_last=-1, prerouted=()),
                                 configs.TOY.with_(B=3, head_owner_last=-1, prerouted=())],
                         ids=lambda c: f"{c.name}-B{c.B}")
def test_noalloc_matches_the_workspace_entry_point_two_calls_in_a_row(cfg):
    model = inputs.make_model(cfg.with_(L=1), seed=41)
    dm = binding.DeviceModel(model, DEV)
    ws = torch.zeros(binding.workspace_bytes(1, cfg.B, cfg.d, cfg.E),
                     dtype=torch.uint8, device=DEV)
    lib = binding.lib()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        x = torch.stack([oracle.rmsnorm(h) for h in inputs.hidden(cfg, 10 + call, seed=41)]).to(DEV)
        ids, w = inputs.routing(cfg, 41, call)
        ids, w = ids.to(DEV), w.to(DEV)
        y_ref = binding.moe_int4_forward(dm, 0, x, ids, w, ws)
        y = torch.empty_like(x)
        rc = lib.edge0_moe_int4_forward_noalloc(C.byref(dm.layers[0].moe), C.c_void_p(x.data_ptr()),
                                                C.c_void_p(ids.data_ptr()), C.c_void_p(w.data_ptr()),
                                                cfg.B, C.c_void_p(y.data_ptr()), stream)
        assert rc == 0, binding.status_string(rc)
        torch.cuda.synchronize()
        assert_close(y, y_ref.double(), f"call {call}")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = binding.lib()
    x = C.c_void_p(256)
    # d = 4096 with 512 experts at B = 4 needs 512 + 10 B d + 16 B E + 384 B = 198,656
    # bytes of scratch, more than the fixed array holds
    moe = binding.MoeDesc(4096, 512, 8, 512, 512, 256, 256, None, None, None, 0)
    assert binding.lib().edge0_workspace_bytes(1, 4, 4096, 512) - 160 * 4096 * 8 > 128 * 1024
    rc = lib.edge0_moe_int4_forward_noalloc(C.byref(moe), x, x, x, 4, x, None)
    assert rc == binding.EDGE0_EUNSUPPORTED
