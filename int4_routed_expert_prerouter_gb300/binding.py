"""ctypes binding of libedge0 (include/edge0.h): argument marshalling only.

PyTorch provides device memory and streams; every step of the decode path runs
in the library's CUDA kernels.  Importing this module loads the compiled
library and raises if it is missing -- there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np
import torch

from . import build as _build
from .configs import SIGMOID_GROUP, Config

P = C.c_void_p
EDGE0_OK, EDGE0_EINVAL, EDGE0_ECUDA, EDGE0_ETIMEOUT, EDGE0_EUNSUPPORTED = 0, 1, 2, 3, 4
MAX_LAYERS, MAX_BATCH, MAX_BATCHED = 48, 4, 256

_lib = None


class Edge0Error(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


def lib():
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libedge0 is not built ({path}); run __graft_entry__.build()")
        _lib = C.CDLL(path)
        _declare(_lib)
    return _lib


# ------------------------------------------------------------- structs ----
class Route(C.Structure):
    _fields_ = [("kind", C.c_int), ("n_groups", C.c_int), ("topk_groups", C.c_int),
                ("scale", C.c_float), ("bias", P)]


class MoeDesc(C.Structure):
    _fields_ = [("d", C.c_int), ("E", C.c_int), ("K", C.c_int), ("I", C.c_int), ("Is", C.c_int),
                ("gate_up", P), ("down", P), ("sh_gate_up", P), ("sh_down", P),
                ("slot_table", P), ("n_slots", C.c_int), ("host_gate_up", P), ("host_down", P),
                ("down_rows", P), ("sh_down_rows", P), ("tier_counts", P)]


class LoraDesc(C.Structure):
    _fields_ = [("r", C.c_int), ("in_", C.c_int), ("out", C.c_int), ("alpha", C.c_float),
                ("A", P), ("A_T", P), ("B", P)]


class HeadDesc(C.Structure):
    _fields_ = [("d", C.c_int), ("E", C.c_int), ("H", C.c_int), ("K", C.c_int),
                ("fc1_dense", P), ("fc1_oh_T", P), ("fc2", P), ("linit_dense", P),
                ("linit_oh_T", P), ("route", Route)]


class LayerDesc(C.Structure):
    _fields_ = [("moe", MoeDesc), ("lora_gate", LoraDesc), ("lora_up", LoraDesc),
                ("lora_down", LoraDesc), ("router", P), ("route", Route), ("gamma", P),
                ("eps", C.c_float), ("prerouted", C.c_int), ("has_head", C.c_int),
                ("head", HeadDesc), ("head_target", C.c_int), ("index", C.c_int), ("ready", P)]


class RouteState(C.Structure):
    _fields_ = [("L", C.c_int), ("B", C.c_int), ("K", C.c_int),
                ("pred_ids", P), ("pred_w", P), ("exec_ids", P), ("workspace", P),
                ("workspace_bytes", C.c_size_t), ("record_h", P), ("record_logits", P)]


def _declare(L):
    L.edge0_status_string.argtypes = [C.c_int]
    L.edge0_status_string.restype = C.c_char_p
    L.edge0_q4_gate_up_packed_bytes.argtypes = [C.c_int] * 3
    L.edge0_q4_gate_up_packed_bytes.restype = C.c_size_t
    L.edge0_pack_q4_gate_up.argtypes = [P, P, P, P, P, P, C.c_int, C.c_int, C.c_int, P, P]
    L.edge0_q4_down_packed_bytes.argtypes = [C.c_int] * 3
    L.edge0_q4_down_packed_bytes.restype = C.c_size_t
    L.edge0_pack_q4_down.argtypes = [P, P, P, C.c_int, C.c_int, C.c_int, P, P]
    L.edge0_pack_q4_rows.argtypes = [P, P, P, C.c_int, C.c_int, C.c_int, P, P]
    L.edge0_f16_packed_bytes.argtypes = [C.c_int] * 2
    L.edge0_f16_packed_bytes.restype = C.c_size_t
    L.edge0_pack_f16.argtypes = [P, C.c_int, C.c_int, C.c_int, P, P]
    L.edge0_pack_f16_kmajor.argtypes = [P, C.c_int, C.c_int, C.c_int, P, P]
    L.edge0_pack_cols_T.argtypes = [P, C.c_int, C.c_int, C.c_int, C.c_int, P, P]
    L.edge0_workspace_bytes.argtypes = [C.c_int] * 4
    L.edge0_workspace_bytes.restype = C.c_size_t
    L.edge0_decode_workspace_bytes.argtypes = [C.c_int] * 8
    L.edge0_decode_workspace_bytes.restype = C.c_size_t
    L.edge0_pool_create.argtypes = [C.c_int, C.c_int, C.c_int, C.c_size_t, C.c_size_t, C.POINTER(P)]
    L.edge0_pool_set_layer.argtypes = [P, C.c_int, P, P, P, P, P]
    L.edge0_pool_plan.argtypes = [P, C.c_int, P, C.c_int, P, P, C.POINTER(C.c_int)]
    L.edge0_pool_host_prefetch.argtypes = [P, P, C.c_int]
    L.edge0_pool_host_copy.argtypes = [P]
    L.edge0_pool_device_init.argtypes = [P]
    L.edge0_pool_prefetch_async.argtypes = [P, P, C.c_int, P, P]
    L.edge0_pool_inject.argtypes = [P, C.c_int, C.c_ulonglong]
    L.edge0_pool_wait.argtypes = [P, C.c_ulonglong]
    L.edge0_pool_stats_ex.argtypes = [P, P, C.c_int]
    L.edge0_pool_stats.argtypes = [P, C.POINTER(C.c_longlong), C.POINTER(C.c_longlong)]
    L.edge0_pool_resident.argtypes = [P, C.c_int, P]
    L.edge0_pool_destroy.argtypes = [P]
    L.edge0_pool_destroy.restype = None
    L.edge0_state_init.argtypes = [C.POINTER(RouteState), P]
    L.edge0_state_error.argtypes = [C.POINTER(RouteState), P, C.POINTER(C.c_int)]
    L.edge0_state_set_wait_limit.argtypes = [C.POINTER(RouteState), C.c_ulonglong, P]
    L.edge0_prerouter_topk.argtypes = [C.POINTER(HeadDesc), P, P, P, C.c_int, P, P, P, P,
                                       C.c_size_t, P]
    L.edge0_moe_int4_forward.argtypes = [C.POINTER(MoeDesc), P, P, P, C.c_int, P, P, C.c_size_t, P]
    L.edge0_moe_int4_forward_noalloc.argtypes = [C.POINTER(MoeDesc), P, P, P, C.c_int, P, P]
    L.edge0_noalloc_error.argtypes = [P, C.POINTER(C.c_int)]
    L.edge0_tc_gemm_f16.argtypes = [P, P, P, C.c_int, C.c_int, C.c_int, P, P]
    L.edge0_prefill_workspace_bytes.argtypes = [C.c_int] * 6
    L.edge0_prefill_workspace_bytes.restype = C.c_size_t
    L.edge0_prefill.argtypes = [C.POINTER(LayerDesc), C.c_int, P, C.c_int, P, C.c_uint, P, C.c_size_t, P]
    L.edge0_lora_delta.argtypes = [C.POINTER(LoraDesc), P, C.c_int, P, P]
    L.edge0_decode_layer.argtypes = [C.POINTER(LayerDesc), P, C.POINTER(RouteState), C.c_int,
                                     C.c_int, P]
    L.edge0_decode_step.argtypes = [C.POINTER(LayerDesc), C.c_int, P, C.POINTER(RouteState),
                                    C.c_int, C.c_int, P]
    for name in ("edge0_pack_q4_gate_up", "edge0_pack_q4_down", "edge0_pack_q4_rows", "edge0_pack_f16",
                 "edge0_pack_f16_kmajor", "edge0_pack_cols_T", "edge0_state_init",
                 "edge0_state_error", "edge0_prerouter_topk", "edge0_moe_int4_forward",
                 "edge0_lora_delta", "edge0_decode_layer", "edge0_decode_step",
                 "edge0_moe_int4_forward_noalloc", "edge0_state_set_wait_limit", "edge0_noalloc_error",
                 "edge0_prefill", "edge0_tc_gemm_f16"):
        getattr(L, name).restype = C.c_int


EXPORTED = ["edge0_status_string", "edge0_q4_gate_up_packed_bytes", "edge0_pack_q4_gate_up",
            "edge0_q4_down_packed_bytes", "edge0_pack_q4_down", "edge0_pack_q4_rows", "edge0_f16_packed_bytes",
            "edge0_pack_f16", "edge0_pack_f16_kmajor", "edge0_pack_cols_T",
            "edge0_workspace_bytes", "edge0_decode_workspace_bytes", "edge0_state_init",
            "edge0_state_error", "edge0_state_set_wait_limit", "edge0_prerouter_topk", "edge0_moe_int4_forward",
            "edge0_lora_delta", "edge0_decode_layer", "edge0_decode_step",
            "edge0_moe_int4_forward_noalloc", "edge0_noalloc_error", "edge0_prefill_workspace_bytes",
            "edge0_prefill", "edge0_tc_gemm_f16", "edge0_pool_create", "edge0_pool_set_layer",
            "edge0_pool_plan", "edge0_pool_host_prefetch", "edge0_pool_host_copy", "edge0_pool_device_init",
            "edge0_pool_prefetch_async", "edge0_pool_wait", "edge0_pool_inject", "edge0_pool_stats_ex", "edge0_pool_stats",
            "edge0_pool_resident", "edge0_pool_destroy"]


def status_string(code: int) -> str:
    return lib().edge0_status_string(code).decode()


def _check(code, what):
    if code != EDGE0_OK:
        raise Edge0Error(code, what)


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


# ------------------------------------------------------------ packing ----
def pack_q4_gate_up(gate, up, stream=None) -> torch.Tensor:
    """gate, up: (q [E, I, d/8] int32, s, b [E, I, d/64] fp16) on the device ->
    packed interleaved gate/up (uint8)."""
    qg, sg, bg = (t.contiguous() for t in gate)
    qu, su, bu = (t.contiguous() for t in up)
    E, I, w8 = qg.shape
    d = w8 * 8
    n = lib().edge0_q4_gate_up_packed_bytes(E, I, d)
    dst = torch.empty(n, dtype=torch.uint8, device=qg.device)
    _check(lib().edge0_pack_q4_gate_up(_ptr(qg), _ptr(sg), _ptr(bg), _ptr(qu), _ptr(su), _ptr(bu),
                                       E, I, d, _ptr(dst), _stream(stream)), "edge0_pack_q4_gate_up")
    return dst


def pack_q4_down(trip, stream=None) -> torch.Tensor:
    """(q [E, out, in/8] int32, s, b [E, out, in/64] fp16) -> packed K-major int4 (uint8)."""
    q, s, b = (t.contiguous() for t in trip)
    E, out, w8 = q.shape
    inp = w8 * 8
    n = lib().edge0_q4_down_packed_bytes(E, out, inp)
    dst = torch.empty(n, dtype=torch.uint8, device=q.device)
    _check(lib().edge0_pack_q4_down(_ptr(q), _ptr(s), _ptr(b), E, out, inp, _ptr(dst), _stream(stream)),
           "edge0_pack_q4_down")
    return dst


def pack_q4_rows(trip, stream=None) -> torch.Tensor:
    """(q [E, out, in/8] int32, s, b [E, out, in/64] fp16) -> row-tile major int4 units (uint8)."""
    q, s, b = (t.contiguous() for t in trip)
    E, out, w8 = q.shape
    inp = w8 * 8
    n = lib().edge0_q4_down_packed_bytes(E, out, inp)
    dst = torch.empty(n, dtype=torch.uint8, device=q.device)
    _check(lib().edge0_pack_q4_rows(_ptr(q), _ptr(s), _ptr(b), E, out, inp, _ptr(dst), _stream(stream)),
           "edge0_pack_q4_rows")
    return dst


def pack_f16(W, cols=None, stream=None, kmajor=False) -> torch.Tensor:
    """W [out, ld] fp16 (device); packs W[:, :cols] row-tile major (or K-major)."""
    W = W.contiguous()
    out, full = W.shape
    inp = cols if cols is not None else full
    n = lib().edge0_f16_packed_bytes(out, inp)
    dst = torch.empty(n, dtype=torch.uint8, device=W.device)
    fn = lib().edge0_pack_f16_kmajor if kmajor else lib().edge0_pack_f16
    _check(fn(_ptr(W), out, inp, full, _ptr(dst), _stream(stream)), "edge0_pack_f16")
    return dst


def pack_cols_T(W, col0, ncols, stream=None) -> torch.Tensor:
    W = W.contiguous()
    out, ld = W.shape
    dst = torch.empty(ncols, out, dtype=torch.float16, device=W.device)
    _check(lib().edge0_pack_cols_T(_ptr(W), out, ld, col0, ncols, _ptr(dst), _stream(stream)),
           "edge0_pack_cols_T")
    return dst


def workspace_bytes(L, B, d, E) -> int:
    return int(lib().edge0_workspace_bytes(L, B, d, E))


def decode_workspace_bytes(cfg: Config, B: int) -> int:
    """Workspace of a decode state for B sequences (either path)."""
    return int(lib().edge0_decode_workspace_bytes(cfg.L, B, cfg.d, cfg.E, cfg.K, cfg.I, cfg.Is, cfg.H))


# ------------------------------------------------------------ the model ----
def _route(cfg: Config, bias) -> Route:
    if cfg.route_kind == SIGMOID_GROUP:
        return Route(SIGMOID_GROUP, cfg.n_groups, cfg.topk_groups, cfg.route_scale, _ptr(bias))
    return Route(0, 1, 1, 1.0, _ptr(bias))


class DeviceModel:
    """A model's weights packed on the GPU plus the layer descriptors that point at them."""

    def __init__(self, model, device="cuda", stream=None):
        cfg = model.cfg
        self.cfg = cfg
        self.device = torch.device(device)
        self.keep = []
        dev = self.device
        self.layers = (LayerDesc * cfg.L)()
        self.stacks = [None] * cfg.L   # packed routed (gate/up, down) stacks per layer
        self.biases = []
        for l, lw in enumerate(model.layers):
            self.biases.append(None if lw.bias is None else lw.bias.to(dev, torch.float32).contiguous())
        for l, lw in enumerate(model.layers):
            self.layers[l] = self._layer(cfg, l, lw, model, stream)
        torch.cuda.synchronize(dev)

    def _k(self, t):
        self.keep.append(t)
        return _ptr(t)

    def _layer(self, cfg, l, lw, model, stream):
        dev = self.device
        d, E, K, I, Is, H, r = cfg.d, cfg.E, cfg.K, cfg.I, cfg.Is, cfg.H, cfg.r
        g = lambda t: t.to(dev)
        L = LayerDesc()
        gt = lambda trip: tuple(g(t) for t in trip)
        self.stacks[l] = (pack_q4_gate_up(gt(lw.gate), gt(lw.up), stream), pack_q4_down(gt(lw.down), stream))
        L.moe = MoeDesc(d, E, K, I, Is,
                        _ptr(self.stacks[l][0]),
                        _ptr(self.stacks[l][1]),
                        self._k(pack_q4_gate_up(gt(lw.sh_gate), gt(lw.sh_up), stream)),
                        self._k(pack_q4_down(gt(lw.sh_down), stream)),
                        None, 0, None, None,
                        # down by output row tiles, for the batch-1 decode kernel
                        self._k(pack_q4_rows(gt(lw.down), stream)),
                        self._k(pack_q4_rows(gt(lw.sh_down), stream)))
        lo = lw.lora
        alpha = float(cfg.alpha)
        lora = lambda A, Bm, inp, out: LoraDesc(
            r, inp, out, alpha, self._k(pack_f16(g(A), stream=stream)),
            self._k(g(A).t().contiguous()), self._k(g(Bm).contiguous()))
        L.lora_gate = lora(lo["Ag"], lo["Bg"], d, Is)
        L.lora_up = lora(lo["Au"], lo["Bu"], d, Is)
        L.lora_down = lora(lo["Ad"], lo["Bd"], Is, d)
        L.router = self._k(pack_f16(g(lw.router), stream=stream))
        L.route = _route(cfg, self.biases[l])
        L.gamma = self._k(g(lw.gamma).contiguous())
        L.eps = cfg.eps
        L.prerouted = 1 if lw.prerouted else 0
        L.index = l
        if lw.head is not None:
            hd = lw.head
            fc1, fc2, linit = g(hd["fc1"]), g(hd["fc2"]), g(hd["linit"])
            tgt = hd["target"]
            L.has_head = 1
            L.head_target = tgt
            L.head = HeadDesc(d, E, H, K, self._k(pack_f16(fc1, cols=d, stream=stream)),
                              self._k(pack_cols_T(fc1, d, 2 * E, stream)),
                              self._k(pack_f16(fc2, stream=stream, kmajor=True)),
                              self._k(pack_f16(linit, cols=d, stream=stream)),
                              self._k(pack_cols_T(linit, d, 2 * E, stream)),
                              _route(cfg, self.biases[tgt]))
        return L


class DecodeState:
    """Routing state + workspace for B sequences over a model's L layers."""

    def __init__(self, cfg: Config, B=None, device="cuda", stream=None):
        B = cfg.B if B is None else B
        dev = torch.device(device)
        self.B = B
        self.d, self.E = cfg.d, cfg.E
        self.rec_h = self.rec_logits = None
        self.pred_ids = torch.zeros(2, cfg.L, B, cfg.K, dtype=torch.int32, device=dev)
        self.pred_w = torch.zeros(2, cfg.L, B, cfg.K, dtype=torch.float32, device=dev)
        self.exec_ids = torch.zeros(2, cfg.L, B, cfg.K, dtype=torch.int32, device=dev)
        nbytes = decode_workspace_bytes(cfg, B)
        assert nbytes > 0, f"no decode path for B = {B}"
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        self.st = RouteState(cfg.L, B, cfg.K, _ptr(self.pred_ids), _ptr(self.pred_w),
                             _ptr(self.exec_ids), _ptr(self.workspace), nbytes, None, None)
        _check(lib().edge0_state_init(C.byref(self.st), _stream(stream)), "edge0_state_init")

    def record(self, on=True):
        """Batch-1 calls record each layer's output h ([L, d] fp16) and each head's
        logits ([L, E] fp32, at the owner layer's row) into self.rec_h /
        self.rec_logits (None: off)."""
        dev = self.workspace.device
        if on:
            self.rec_h = torch.zeros(self.st.L, self.d, dtype=torch.float16, device=dev)
            self.rec_logits = torch.full((self.st.L, self.E), float("nan"), dtype=torch.float32, device=dev)
            self.st.record_h, self.st.record_logits = _ptr(self.rec_h), _ptr(self.rec_logits)
        else:
            self.rec_h = self.rec_logits = None
            self.st.record_h = self.st.record_logits = None

    def set_wait_limit(self, wait_ns, stream=None):
        _check(lib().edge0_state_set_wait_limit(C.byref(self.st), int(wait_ns), _stream(stream)),
               "edge0_state_set_wait_limit")

    def hold_first_barrier(self, n):
        """Test hook (workspace header field `hold`): the next launch's first grid
        barrier waits for n arrivals beyond the grid, so it cannot complete."""
        torch.cuda.synchronize(self.workspace.device)
        self.workspace[28:32].copy_(torch.tensor([int(n)], dtype=torch.int32).view(torch.uint8))
        torch.cuda.synchronize(self.workspace.device)

    TRACE_CTAS, TRACE_SLOTS, TRACE_PRODUCER = 160, 4096, 3072

    def set_trace(self, on):
        """Switch the engine's per-layer trace on/off (workspace header flag)."""
        torch.cuda.synchronize(self.workspace.device)
        flag = torch.tensor([1 if on else 0], dtype=torch.int32)
        self.workspace[24:28].copy_(flag.view(torch.uint8))
        if on:
            self.workspace[-self.TRACE_CTAS * self.TRACE_SLOTS * 8:].zero_()
        torch.cuda.synchronize(self.workspace.device)

    def read_trace(self):
        """(consumer, producer): [CTAs, events, 3] int64 (tag, globaltimer ns, SM clock)
        triples; consumer tags are layer << 8 | point (0 start, 1 x built, 2 routed,
        3 gate/up done, 4 exchange done, 5 act done, 6 down done + barrier arrival,
        7 head done, 8 gate/up data seen, 9 down data seen, 10-12 inside act/down),
        producer tags layer << 8 | 0x80 + point (table started, built, routing
        known, items issued)."""
        torch.cuda.synchronize(self.workspace.device)
        raw = self.workspace[-self.TRACE_CTAS * self.TRACE_SLOTS * 8:].cpu().view(torch.int64)
        raw = raw.view(self.TRACE_CTAS, self.TRACE_SLOTS)
        cons = raw[:, :self.TRACE_PRODUCER // 3 * 3].reshape(self.TRACE_CTAS, -1, 3)
        prod = raw[:, self.TRACE_PRODUCER:self.TRACE_PRODUCER + (self.TRACE_SLOTS - self.TRACE_PRODUCER) // 3 * 3].reshape(self.TRACE_CTAS, -1, 3)
        return cons, prod

    def error(self, stream=None) -> int:
        code = C.c_int(0)
        _check(lib().edge0_state_error(C.byref(self.st), _stream(stream), C.byref(code)),
               "edge0_state_error")
        return code.value


class ExpertPool:
    """Host tier for a DeviceModel's routed experts (edge0_pool_*, device mode):
    every layer's packed experts move to pinned host memory the device can read,
    and the layer keeps `n_slots` device slots, filled from the prerouter's
    prediction one token ahead by the pool's device planner and copy kernel.
    The model's descriptors are pointed at the slots, the published slot table,
    the host stacks and a pair of residency counters; the full device stacks are
    released."""

    STATS = ("requests", "hits", "planned", "published", "failed", "skipped", "bytes", "bad_ids")

    def __init__(self, dm: "DeviceModel", n_slots: int, copy_stream=None):
        cfg = dm.cfg
        self.dm, self.n_slots = dm, n_slots
        dev = dm.device
        self.gu_bytes = int(lib().edge0_q4_gate_up_packed_bytes(1, cfg.I, cfg.d))
        self.dn_bytes = int(lib().edge0_q4_down_packed_bytes(1, cfg.d, cfg.I))
        self.pool = C.c_void_p()
        _check(lib().edge0_pool_create(cfg.L, cfg.E, n_slots, self.gu_bytes, self.dn_bytes,
                                       C.byref(self.pool)), "edge0_pool_create")
        self.copy_stream = copy_stream or torch.cuda.Stream(dev)
        # per layer [0]: active routed experts summed over steps, [1]: of them read from host memory
        self.tier_counts = torch.zeros(cfg.L, 2, dtype=torch.int64, device=dev)
        self.keep = []
        for l in range(cfg.L):
            gu, dn = dm.stacks[l]
            hg = torch.empty(gu.numel(), dtype=torch.uint8, pin_memory=True)
            hd = torch.empty(dn.numel(), dtype=torch.uint8, pin_memory=True)
            hg.copy_(gu)
            hd.copy_(dn)
            sg = torch.empty(n_slots * self.gu_bytes, dtype=torch.uint8, device=dev)
            sd = torch.empty(n_slots * self.dn_bytes, dtype=torch.uint8, device=dev)
            tb = torch.full((cfg.E,), -1, dtype=torch.int32, device=dev)
            _check(lib().edge0_pool_set_layer(self.pool, l, _ptr(hg), _ptr(hd), _ptr(sg), _ptr(sd), _ptr(tb)),
                   "edge0_pool_set_layer")
            m = dm.layers[l].moe
            m.gate_up, m.down, m.slot_table, m.n_slots = _ptr(sg), _ptr(sd), _ptr(tb), n_slots
            m.host_gate_up, m.host_down = _ptr(hg), _ptr(hd)
            m.tier_counts = C.c_void_p(self.tier_counts[l].data_ptr())
            self.keep += [hg, hd, sg, sd, tb]
            dm.stacks[l] = None
        self.slots = [(self.keep[5 * l + 2], self.keep[5 * l + 3], self.keep[5 * l + 4]) for l in range(cfg.L)]
        self.host = [(self.keep[5 * l], self.keep[5 * l + 1]) for l in range(cfg.L)]
        torch.cuda.synchronize(dev)
        _check(lib().edge0_pool_device_init(self.pool), "edge0_pool_device_init")

    def prefetch(self, st: "DecodeState", t: int, predicted=(), cached=(), stream=None):
        """Enqueue, after step t's work on `stream`, the residency plan of each
        layer in `predicted` from the experts its prediction for step t + 1 names
        (union over the batch), and of each layer in `cached` from the experts
        step t ran (least-recently-used caching, for layers without a
        prediction); the copies go on the copy stream.  Nothing waits: no host
        read-back, and the next step reads experts whose copies are still in
        flight from host memory."""
        L = self.dm.cfg.L
        ids = (C.c_void_p * L)()
        for l in cached:
            ids[l] = st.exec_ids[t & 1, l].data_ptr()
        for l in predicted:
            ids[l] = st.pred_ids[t & 1, l].data_ptr()
        _check(lib().edge0_pool_prefetch_async(self.pool, ids, st.B * self.dm.cfg.K, _stream(stream),
                                               C.c_void_p(self.copy_stream.cuda_stream)),
               "edge0_pool_prefetch_async")

    def wait(self, timeout_ns) -> int:
        """Bounded host poll for the last copy pass: EDGE0_OK or EDGE0_ETIMEOUT."""
        rc = lib().edge0_pool_wait(self.pool, int(timeout_ns))
        if rc not in (EDGE0_OK, EDGE0_ETIMEOUT):
            _check(rc, "edge0_pool_wait")
        return rc

    def inject(self, fail_every=0, delay_ns=0):
        _check(lib().edge0_pool_inject(self.pool, int(fail_every), int(delay_ns)), "edge0_pool_inject")

    def stats(self) -> dict:
        """The pool's counters (waits for the device)."""
        out = (C.c_longlong * 8)()
        _check(lib().edge0_pool_stats_ex(self.pool, out, 8), "edge0_pool_stats_ex")
        return dict(zip(self.STATS, list(out)))

    def tiers(self) -> np.ndarray:
        """[L, 2]: per layer, active routed experts and those of them read from
        host memory, summed over the steps run so far (waits for the device)."""
        torch.cuda.synchronize(self.tier_counts.device)
        return self.tier_counts.cpu().numpy().copy()

    def resident(self, l: int) -> np.ndarray:
        """The published map of layer l: slot of each expert, -1 for the host tier
        (waits for the device)."""
        out = np.empty(self.dm.cfg.E, dtype=np.int32)
        _check(lib().edge0_pool_resident(self.pool, l, C.c_void_p(out.ctypes.data)), "edge0_pool_resident")
        return out

    def __del__(self):
        if getattr(self, "pool", None):
            lib().edge0_pool_destroy(self.pool)
            self.pool = None


# ---------------------------------------------------------- operations ----
def decode_step(dm: DeviceModel, st: DecodeState, h: torch.Tensor, step: int, stream=None):
    """All layers of one decode step on h [B, d] fp16 (device, in place)."""
    assert h.is_cuda and h.dtype == torch.float16 and h.is_contiguous()
    _check(lib().edge0_decode_step(dm.layers, dm.cfg.L, _ptr(h), C.byref(st.st), st.B, step,
                                   _stream(stream)), "edge0_decode_step")


def tc_gemm_f16(A: torch.Tensor, B: torch.Tensor, stream=None) -> torch.Tensor:
    """A [M, K] fp16 x B [N, K]^T fp16 -> fp32 [M, N] on tcgen05 (device tensors)."""
    A, B = A.contiguous(), B.contiguous()
    M, K = A.shape
    N = B.shape[0]
    D = torch.empty(M, N, dtype=torch.float32, device=A.device)
    status = torch.zeros(1, dtype=torch.int32, device=A.device)
    _check(lib().edge0_tc_gemm_f16(_ptr(A), _ptr(B), _ptr(D), M, N, K, _ptr(status), _stream(stream)),
           "edge0_tc_gemm_f16")
    torch.cuda.synchronize(A.device)
    code = int(status.item())
    if code:
        raise RuntimeError(f"edge0_tc_gemm_f16: {status_string(code)}")
    return D


def prefill_workspace_bytes(cfg: Config, T: int) -> int:
    return int(lib().edge0_prefill_workspace_bytes(T, cfg.d, cfg.E, cfg.K, cfg.I, cfg.Is))


PREFILL_TCGEN05_GATE_UP = 1


def prefill(dm: DeviceModel, h: torch.Tensor, workspace: torch.Tensor, ids_out=None, layers=None, flags=0,
            stream=None):
    """The model's layers (or layers[a:b] given as a slice) over a prompt h [T, d]
    fp16 (device, in place); every layer on its own router.  ids_out: None or
    [L][T][K] int32 (device); flags: PREFILL_TCGEN05_GATE_UP for the tcgen05
    gate/up kernel."""
    assert h.is_cuda and h.dtype == torch.float16 and h.is_contiguous() and h.dim() == 2
    arr, L = dm.layers, dm.cfg.L
    if layers is not None:
        idx = list(range(L))[layers]
        arr = (LayerDesc * len(idx))(*[dm.layers[i] for i in idx])
        L = len(idx)
    _check(lib().edge0_prefill(arr, L, _ptr(h), h.shape[0], _ptr(ids_out), flags, _ptr(workspace),
                               workspace.numel(), _stream(stream)), "edge0_prefill")


def decode_layer(dm: DeviceModel, l: int, st: DecodeState, h: torch.Tensor, step: int, stream=None):
    assert h.is_cuda and h.dtype == torch.float16 and h.is_contiguous()
    _check(lib().edge0_decode_layer(C.byref(dm.layers[l]), _ptr(h), C.byref(st.st), st.B, step,
                                    _stream(stream)), "edge0_decode_layer")


def moe_int4_forward(dm: DeviceModel, l: int, x, ids, w, workspace, stream=None) -> torch.Tensor:
    B = x.shape[0]
    y = torch.empty_like(x)
    _check(lib().edge0_moe_int4_forward(C.byref(dm.layers[l].moe), _ptr(x), _ptr(ids), _ptr(w), B,
                                        _ptr(y), _ptr(workspace), workspace.numel(),
                                        _stream(stream)), "edge0_moe_int4_forward")
    return y


def prerouter_topk(dm: DeviceModel, l: int, x, exec_ids, prev_ids, workspace, stream=None):
    cfg = dm.cfg
    B = x.shape[0]
    ids = torch.empty(B, cfg.K, dtype=torch.int32, device=x.device)
    w = torch.empty(B, cfg.K, dtype=torch.float32, device=x.device)
    logits = torch.empty(B, cfg.E, dtype=torch.float32, device=x.device)
    _check(lib().edge0_prerouter_topk(C.byref(dm.layers[l].head), _ptr(x), _ptr(exec_ids),
                                      _ptr(prev_ids), B, _ptr(ids), _ptr(w), _ptr(logits),
                                      _ptr(workspace), workspace.numel(), _stream(stream)),
           "edge0_prerouter_topk")
    return ids, w, logits


def lora_delta(desc: LoraDesc, v, y, stream=None):
    B = v.shape[0]
    _check(lib().edge0_lora_delta(C.byref(desc), _ptr(v), B, _ptr(y), _stream(stream)),
           "edge0_lora_delta")
    return y
