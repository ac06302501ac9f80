"""CPU oracle for the prerouted int4 MoE decode path -- TEST INFRASTRUCTURE ONLY.

A plain single-threaded C++ restatement (``oracle.cpp``) of what the path
computes, in fp64, loaded through ctypes.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it; the
CUDA library never links or calls it, and it shares no code with it.

Every routine in ``oracle.cpp`` names the page section it restates.  Pins (the
tests that tie the oracle to what the pages and the mathematics fix) live in
``tests/test_oracle_*.py``.  Parity unpinned: none.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_HDR = os.path.join(_HERE, "oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with the host C++ compiler (portable C++17, -O2)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_SO)
             or os.path.getmtime(_SO) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-o", tmp, _SRC])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = C.CDLL(build())
            _declare(_lib)
    return _lib


# ------------------------------------------------------------------ ctypes ----
P = C.c_void_p


class Q4(C.Structure):
    _fields_ = [("q", P), ("s", P), ("b", P), ("out", C.c_int), ("in_", C.c_int)]


class Route(C.Structure):
    _fields_ = [("kind", C.c_int), ("n_groups", C.c_int), ("topk_groups", C.c_int),
                ("scale", C.c_float), ("bias", P)]


class Moe(C.Structure):
    _fields_ = [("d", C.c_int), ("I", C.c_int), ("Is", C.c_int), ("E", C.c_int), ("K", C.c_int),
                ("gate_q", P), ("up_q", P), ("down_q", P),
                ("gate_s", P), ("gate_b", P), ("up_s", P), ("up_b", P), ("down_s", P), ("down_b", P),
                ("sh_gate_q", P), ("sh_up_q", P), ("sh_down_q", P),
                ("sh_gate_s", P), ("sh_gate_b", P), ("sh_up_s", P), ("sh_up_b", P),
                ("sh_down_s", P), ("sh_down_b", P)]


class Layer(C.Structure):
    _fields_ = [("moe", Moe),
                ("lora_Ag", P), ("lora_Bg", P), ("lora_Au", P), ("lora_Bu", P), ("lora_Ad", P),
                ("lora_Bd", P), ("r", C.c_int), ("alpha", C.c_double),
                ("router", P), ("gamma", P), ("eps", C.c_double), ("route", Route),
                ("prerouted", C.c_int), ("fc1", P), ("fc2", P), ("linit", P), ("H", C.c_int),
                ("head_target", C.c_int)]


class State(C.Structure):
    _fields_ = [("L", C.c_int), ("B", C.c_int), ("K", C.c_int),
                ("pred_ids", P), ("pred_w", P), ("exec_ids", P)]


class Record(C.Structure):
    _fields_ = [("x", P), ("ids", P), ("w", P), ("hout", P), ("head_logits", P),
                ("router_logits", P)]


def _declare(L):
    L.orc_half_to_double.argtypes = [C.c_uint16]
    L.orc_half_to_double.restype = C.c_double
    L.orc_double_to_half.argtypes = [C.c_double]
    L.orc_double_to_half.restype = C.c_uint16
    L.orc_gelu_erf.argtypes = [C.c_double]
    L.orc_gelu_erf.restype = C.c_double
    L.orc_silu.argtypes = [C.c_double]
    L.orc_silu.restype = C.c_double
    L.orc_int4_unpack.argtypes = [P, C.c_long, P]
    L.orc_int4_pack.argtypes = [P, C.c_long, P]
    L.orc_int4_dequant.argtypes = [C.POINTER(Q4), P]
    L.orc_int4_matvec.argtypes = [C.POINTER(Q4), P, P]
    L.orc_f16_matvec.argtypes = [P, C.c_int, C.c_int, C.c_int, P, P]
    L.orc_expert_swiglu.argtypes = [C.POINTER(Q4)] * 3 + [P, P]
    L.orc_lora_delta.argtypes = [P, P, C.c_int, C.c_int, C.c_int, C.c_double, P, P]
    L.orc_topk.argtypes = [P, C.c_int, C.c_int, P]
    L.orc_route_softmax_topk.argtypes = [P, P, C.c_int, C.c_int, P, P]
    L.orc_route_sigmoid_group.argtypes = [P, P, C.c_int, C.c_int, C.c_int, C.c_int, C.c_float, P, P]
    L.orc_prerouter_logits.argtypes = [P, P, P, C.c_int, C.c_int, C.c_int, P, P, P, C.c_int, P]
    L.orc_rmsnorm.argtypes = [P, P, C.c_int, C.c_double, P]
    L.orc_moe_forward.argtypes = [C.POINTER(Moe), P, P, P, C.c_int, P, P]
    L.orc_decode_layer.argtypes = [C.POINTER(Layer), C.c_int, C.POINTER(State), P, C.c_int,
                                   C.POINTER(Record)]
    L.orc_decode_step.argtypes = [C.POINTER(Layer), C.POINTER(State), P, C.c_int, C.POINTER(Record)]


# --------------------------------------------------------------- helpers -----
def _cpu(t: torch.Tensor) -> torch.Tensor:
    assert t.device.type == "cpu", "the oracle takes host tensors"
    return t.contiguous()


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _bits16(t: torch.Tensor) -> torch.Tensor:
    return _cpu(t).view(torch.int16)


def half_to_double(h: int) -> float:
    return lib().orc_half_to_double(h & 0xFFFF)


def double_to_half(v: float) -> int:
    return lib().orc_double_to_half(float(v))


def gelu_erf(z: float) -> float:
    return lib().orc_gelu_erf(float(z))


def silu(z: float) -> float:
    return lib().orc_silu(float(z))


def int4_unpack(packed: torch.Tensor) -> torch.Tensor:
    p = _cpu(packed).view(torch.int32)
    out = torch.empty(p.numel() * 8, dtype=torch.uint8)
    lib().orc_int4_unpack(_ptr(p), p.numel(), _ptr(out))
    return out


def int4_pack(nibbles: torch.Tensor) -> torch.Tensor:
    n = _cpu(nibbles).to(torch.uint8)
    assert n.numel() % 8 == 0
    out = torch.empty(n.numel() // 8, dtype=torch.int32)
    lib().orc_int4_pack(_ptr(n), out.numel(), _ptr(out))
    return out


def _q4(q, s, b, out, inp, keep):
    q, s, b = _cpu(q), _cpu(s), _cpu(b)
    keep += [q, s, b]
    return Q4(q.data_ptr(), s.data_ptr(), b.data_ptr(), out, inp)


def int4_dequant(q, s, b, out, inp) -> torch.Tensor:
    keep = []
    m = _q4(q, s, b, out, inp, keep)
    w = torch.empty(out, inp, dtype=torch.float64)
    lib().orc_int4_dequant(C.byref(m), _ptr(w))
    return w


def int4_matvec(q, s, b, out, inp, v) -> torch.Tensor:
    keep = []
    m = _q4(q, s, b, out, inp, keep)
    v = _cpu(v).to(torch.float64)
    y = torch.empty(out, dtype=torch.float64)
    lib().orc_int4_matvec(C.byref(m), _ptr(v), _ptr(y))
    return y


def f16_matvec(W, v) -> torch.Tensor:
    W = _cpu(W)
    out, inp = W.shape
    v = _cpu(v).to(torch.float64)
    y = torch.empty(out, dtype=torch.float64)
    lib().orc_f16_matvec(_ptr(W), out, inp, inp, _ptr(v), _ptr(y))
    return y


def expert_swiglu(gate, up, down, x) -> torch.Tensor:
    """gate/up/down: (q, s, b) of one expert with q [out, in/8]."""
    keep = []
    I, d = gate[0].shape[-2], gate[0].shape[-1] * 8
    g = _q4(*[t.reshape(t.shape[-2], t.shape[-1]) for t in gate], I, d, keep)
    u = _q4(*[t.reshape(t.shape[-2], t.shape[-1]) for t in up], I, d, keep)
    dn = _q4(*[t.reshape(t.shape[-2], t.shape[-1]) for t in down], d, I, keep)
    x = _cpu(x).to(torch.float64)
    y = torch.empty(d, dtype=torch.float64)
    lib().orc_expert_swiglu(C.byref(g), C.byref(u), C.byref(dn), _ptr(x), _ptr(y))
    return y


def lora_delta(A, B, alpha, v) -> torch.Tensor:
    A, B = _cpu(A), _cpu(B)
    r, inp = A.shape
    out = B.shape[0]
    v = _cpu(v).to(torch.float64)
    dy = torch.empty(out, dtype=torch.float64)
    lib().orc_lora_delta(_ptr(A), _ptr(B), r, inp, out, float(alpha), _ptr(v), _ptr(dy))
    return dy


def topk(score, k) -> torch.Tensor:
    s = _cpu(score).to(torch.float32)
    idx = torch.empty(k, dtype=torch.int32)
    lib().orc_topk(_ptr(s), s.numel(), k, _ptr(idx))
    return idx


def route_softmax_topk(logits, K, bias=None):
    lg = _cpu(logits).to(torch.float32)
    bias = None if bias is None else _cpu(bias).to(torch.float32)
    ids = torch.empty(K, dtype=torch.int32)
    w = torch.empty(K, dtype=torch.float32)
    lib().orc_route_softmax_topk(_ptr(lg), _ptr(bias), lg.numel(), K, _ptr(ids), _ptr(w))
    return ids, w


def route_sigmoid_group(logits, K, n_groups, G, scale, bias=None):
    lg = _cpu(logits).to(torch.float32)
    bias = None if bias is None else _cpu(bias).to(torch.float32)
    ids = torch.empty(K, dtype=torch.int32)
    w = torch.empty(K, dtype=torch.float32)
    lib().orc_route_sigmoid_group(_ptr(lg), _ptr(bias), lg.numel(), K, n_groups, G, float(scale),
                                  _ptr(ids), _ptr(w))
    return ids, w


def prerouter_logits(fc1, fc2, linit, x, exec_ids, prev_ids, d, E, H, K):
    fc1, fc2, linit, x = _cpu(fc1), _cpu(fc2), _cpu(linit), _cpu(x)
    ex = _cpu(exec_ids).to(torch.int32)
    pv = None if prev_ids is None else _cpu(prev_ids).to(torch.int32)
    out = torch.empty(E, dtype=torch.float32)
    lib().orc_prerouter_logits(_ptr(fc1), _ptr(fc2), _ptr(linit), d, E, H, _ptr(x), _ptr(ex),
                               _ptr(pv), K, _ptr(out))
    return out


def rmsnorm(h, gamma=None, eps=1e-6):
    h = _cpu(h)
    gamma = None if gamma is None else _cpu(gamma)
    x = torch.empty_like(h)
    lib().orc_rmsnorm(_ptr(h), _ptr(gamma), h.numel(), float(eps), _ptr(x))
    return x


def _moe_struct(cfg, lw, keep) -> Moe:
    def c(t):
        t = _cpu(t)
        keep.append(t)
        return t.data_ptr()
    g, u, dn = lw.gate, lw.up, lw.down
    sg, su, sdn = lw.sh_gate, lw.sh_up, lw.sh_down
    return Moe(cfg.d, cfg.I, cfg.Is, cfg.E, cfg.K,
               c(g[0]), c(u[0]), c(dn[0]), c(g[1]), c(g[2]), c(u[1]), c(u[2]), c(dn[1]), c(dn[2]),
               c(sg[0]), c(su[0]), c(sdn[0]), c(sg[1]), c(sg[2]), c(su[1]), c(su[2]),
               c(sdn[1]), c(sdn[2]))


def moe_forward(cfg, lw, x, ids, w):
    """Routed + shared experts without LoRA.  Returns (y fp16 [B,d], y fp64 [B,d])."""
    keep = []
    m = _moe_struct(cfg, lw, keep)
    x, ids, w = _cpu(x), _cpu(ids).to(torch.int32), _cpu(w).to(torch.float32)
    B = x.shape[0]
    y16 = torch.empty(B, cfg.d, dtype=torch.float16)
    y = torch.empty(B, cfg.d, dtype=torch.float64)
    lib().orc_moe_forward(C.byref(m), _ptr(x), _ptr(ids), _ptr(w), B, _ptr(y16), _ptr(y))
    return y16, y


class Stack:
    """The oracle's view of a model plus its routing state, for decode steps."""

    def __init__(self, model, B=None):
        cfg = model.cfg
        self.cfg = cfg
        self.B = B if B is not None else cfg.B
        self._keep = []
        arr = (Layer * cfg.L)()
        for l, lw in enumerate(model.layers):
            L_ = arr[l]
            L_.moe = _moe_struct(cfg, lw, self._keep)
            for name in ("Ag", "Bg", "Au", "Bu", "Ad", "Bd"):
                t = _cpu(lw.lora[name])
                self._keep.append(t)
                setattr(L_, "lora_" + name, t.data_ptr())
            L_.r, L_.alpha = cfg.r, float(cfg.alpha)
            for name, t in (("router", lw.router), ("gamma", lw.gamma)):
                t = _cpu(t)
                self._keep.append(t)
                setattr(L_, name, t.data_ptr())
            L_.eps = cfg.eps
            bias = None
            if lw.bias is not None:
                bias = _cpu(lw.bias).to(torch.float32)
                self._keep.append(bias)
            L_.route = Route(cfg.route_kind, cfg.n_groups, cfg.topk_groups, cfg.route_scale,
                             None if bias is None else bias.data_ptr())
            L_.prerouted = 1 if lw.prerouted else 0
            if lw.head is not None:
                for name in ("fc1", "fc2", "linit"):
                    t = _cpu(lw.head[name])
                    self._keep.append(t)
                    setattr(L_, name, t.data_ptr())
                L_.H = cfg.H
                L_.head_target = lw.head["target"]
        self.layers = arr
        L, B, K = cfg.L, self.B, cfg.K
        self.pred_ids = torch.zeros(2, L, B, K, dtype=torch.int32)
        self.pred_w = torch.zeros(2, L, B, K, dtype=torch.float32)
        self.exec_ids = torch.zeros(2, L, B, K, dtype=torch.int32)
        self.state = State(L, B, K, self.pred_ids.data_ptr(), self.pred_w.data_ptr(),
                           self.exec_ids.data_ptr())

    def step(self, h: torch.Tensor, t: int, record: bool = True, layers=None):
        """Run decode step t on h [B, d] fp16 (updated in place).  Returns the
        per-layer record dict when ``record``."""
        cfg = self.cfg
        h = _cpu(h)
        assert h.dtype == torch.float16 and h.shape == (self.B, cfg.d)
        rec = None
        out = None
        if record:
            L, B, K, d, E = cfg.L, self.B, cfg.K, cfg.d, cfg.E
            out = dict(x=torch.zeros(L, B, d, dtype=torch.float16),
                       ids=torch.zeros(L, B, K, dtype=torch.int32),
                       w=torch.zeros(L, B, K, dtype=torch.float32),
                       hout=torch.zeros(L, B, d, dtype=torch.float16),
                       head_logits=torch.full((L, B, E), float("nan"), dtype=torch.float32),
                       router_logits=torch.full((L, B, E), float("nan"), dtype=torch.float32))
            rec = Record(*[out[k].data_ptr() for k in ("x", "ids", "w", "hout", "head_logits",
                                                       "router_logits")])
        if layers is None:
            lib().orc_decode_step(self.layers, C.byref(self.state), _ptr(h), t,
                                  None if rec is None else C.byref(rec))
        else:
            for l in layers:
                lib().orc_decode_layer(self.layers, l, C.byref(self.state), _ptr(h), t,
                                       None if rec is None else C.byref(rec))
        return out
