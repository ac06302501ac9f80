"""Seeded synthetic inputs for the prerouted int4 MoE decode path.

This module only draws random numbers; it computes nothing the method computes.
Both the CPU oracle and the CUDA path consume the tensors it returns, in the
canonical layouts the pages describe:

* int4 expert weights as MLX affine group-64: packed uint32 ``[E, out, in/8]``
  (stored as int32 bit patterns; nibble i of word j is input 8j+i) with fp16
  scales and biases ``[E, out, in/64]`` ("Inside Edge0-35B", "Architectural
  Deep Dive"; "Edge0 streams a 35B MoE off SSD", "Counting the bytes");
* dense fp16 weights in ``nn.Linear`` layout ``[out, in]``.

Recipe (seed 0 unless stated; every tensor has its own substream keyed by
(seed, layer, tensor id)):

* nibbles q ~ U{0..15} (uniform random bytes, two nibbles each);
* zero-point z ~ U{0..15}; scale s = U[0.5, 1.5) / (8 sqrt(in)) rounded to fp16;
  bias b = fp16(-s z);
* router, fc1, fc2, linear_init ~ N(0, 1/fan_in) in fp16;
* LoRA A, B ~ N(0, 0.02^2) in fp16;
* hidden states ~ N(0, 1) in fp16, one substream per decode step;
* RMSNorm gain 1 (``gamma="random"`` draws 1 + N(0, 0.1^2) for unit tests);
* Zipf(a) router-logit bias: -a ln(rank) with rank a seeded permutation of 1..E.

Large int4 stacks may be drawn on a CUDA device (``device="cuda"``): the values
then come from torch's CUDA generator and differ from a CPU draw with the same
seed, so a run always draws once and hands the same tensors to both sides.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

from .configs import GROUP, Config

# tensor ids of the substreams
_T_GATE, _T_UP, _T_DOWN = 1, 2, 3
_T_SH_GATE, _T_SH_UP, _T_SH_DOWN = 4, 5, 6
_T_ROUTER, _T_FC1, _T_FC2, _T_LINIT = 7, 8, 9, 10
_T_AG, _T_BG, _T_AU, _T_BU, _T_AD, _T_BD = 11, 12, 13, 14, 15, 16
_T_GAMMA, _T_ZIPF, _T_HIDDEN = 17, 18, 19
_SUB_Q, _SUB_S, _SUB_Z = 0, 1, 2


def _gen(seed: int, layer: int, tid: int, sub: int, device) -> torch.Generator:
    key = np.random.SeedSequence([seed, layer + 1, tid, sub]).generate_state(1, np.uint64)[0]
    g = torch.Generator(device=device)
    g.manual_seed(int(key) & ((1 << 63) - 1))
    return g


def int4_stack(seed: int, layer: int, tid: int, E: int, out: int, inp: int, device="cpu"):
    """(q, s, b) for E experts of one [out, inp] int4 matrix, canonical layout."""
    assert inp % GROUP == 0
    dev = torch.device(device)
    nbytes = E * out * inp // 2
    q = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=dev,
                      generator=_gen(seed, layer, tid, _SUB_Q, dev))
    q = q.view(torch.int32).view(E, out, inp // 8)
    ng = E * out * (inp // GROUP)
    u = torch.rand(ng, dtype=torch.float32, device=dev, generator=_gen(seed, layer, tid, _SUB_S, dev))
    s = ((u + 0.5) / (8.0 * math.sqrt(inp))).to(torch.float16)
    z = torch.randint(0, 16, (ng,), dtype=torch.int32, device=dev,
                      generator=_gen(seed, layer, tid, _SUB_Z, dev))
    b = (-(s.float() * z.float())).to(torch.float16)
    return q, s.view(E, out, inp // GROUP), b.view(E, out, inp // GROUP)


def normal_f16(seed: int, layer: int, tid: int, shape, std: float, device="cpu"):
    dev = torch.device(device)
    v = torch.randn(*shape, dtype=torch.float32, device=dev, generator=_gen(seed, layer, tid, 0, dev))
    return (v * std).to(torch.float16)


def zipf_bias(seed: int, layer: int, E: int, a: float) -> torch.Tensor:
    g = _gen(seed, layer, _T_ZIPF, 0, "cpu")
    rank = torch.randperm(E, generator=g).to(torch.float64) + 1.0
    return (-a * torch.log(rank)).to(torch.float32)


def hidden(cfg: Config, step: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """h_0 of one decode step: [B, d] fp16 ~ N(0, 1)."""
    return normal_f16(seed, 100000 + step, _T_HIDDEN, (cfg.B, cfg.d), 1.0, device)


@dataclass
class LayerWeights:
    gate: tuple
    up: tuple
    down: tuple
    sh_gate: tuple
    sh_up: tuple
    sh_down: tuple
    router: torch.Tensor
    gamma: torch.Tensor
    lora: dict                      # Ag, Bg, Au, Bu, Ad, Bd
    bias: torch.Tensor | None       # routing selection bias [E] fp32
    head: dict | None               # fc1, fc2, linit, target
    prerouted: bool


@dataclass
class Model:
    cfg: Config
    seed: int
    layers: list = field(default_factory=list)


def make_layer(cfg: Config, l: int, seed: int = 0, device="cpu", small_device="cpu",
               gamma: str = "unit") -> LayerWeights:
    d, E, I, Is, H, r = cfg.d, cfg.E, cfg.I, cfg.Is, cfg.H, cfg.r
    gate = int4_stack(seed, l, _T_GATE, E, I, d, device)
    up = int4_stack(seed, l, _T_UP, E, I, d, device)
    down = int4_stack(seed, l, _T_DOWN, E, d, I, device)
    sh_gate = int4_stack(seed, l, _T_SH_GATE, 1, Is, d, device)
    sh_up = int4_stack(seed, l, _T_SH_UP, 1, Is, d, device)
    sh_down = int4_stack(seed, l, _T_SH_DOWN, 1, d, Is, device)
    sd = small_device
    router = normal_f16(seed, l, _T_ROUTER, (E, d), 1.0 / math.sqrt(d), sd)
    if gamma == "random":
        gm = (1.0 + normal_f16(seed, l, _T_GAMMA, (d,), 0.1, sd).float()).to(torch.float16)
    else:
        gm = torch.ones(d, dtype=torch.float16, device=sd)
    lora = dict(
        Ag=normal_f16(seed, l, _T_AG, (r, d), 0.02, sd),
        Bg=normal_f16(seed, l, _T_BG, (Is, r), 0.02, sd),
        Au=normal_f16(seed, l, _T_AU, (r, d), 0.02, sd),
        Bu=normal_f16(seed, l, _T_BU, (Is, r), 0.02, sd),
        Ad=normal_f16(seed, l, _T_AD, (r, Is), 0.02, sd),
        Bd=normal_f16(seed, l, _T_BD, (d, r), 0.02, sd),
    )
    bias = zipf_bias(seed, l, E, cfg.zipf).to(sd) if cfg.zipf else None
    head = None
    owners = cfg.head_owners()
    if l in owners:
        f_in = cfg.f_in
        head = dict(
            fc1=normal_f16(seed, l, _T_FC1, (H, f_in), 1.0 / math.sqrt(f_in), sd),
            fc2=normal_f16(seed, l, _T_FC2, (E, H), 1.0 / math.sqrt(H), sd),
            linit=normal_f16(seed, l, _T_LINIT, (E, f_in), 1.0 / math.sqrt(f_in), sd),
            target=cfg.head_target(l),
        )
    return LayerWeights(gate, up, down, sh_gate, sh_up, sh_down, router, gm, lora, bias, head,
                        l in cfg.prerouted)


def make_model(cfg: Config, seed: int = 0, device="cpu", small_device="cpu",
               gamma: str = "unit") -> Model:
    m = Model(cfg, seed)
    for l in range(cfg.L):
        m.layers.append(make_layer(cfg, l, seed, device, small_device, gamma))
    return m


def routing(cfg: Config, seed: int, tag: int, device="cpu"):
    """Random routing (ids, w) [B, K] for the standalone MoE entry point:
    K distinct experts per token and weights drawn from U[0.05, 1.05)."""
    g = _gen(seed, 200000 + tag, 0, 0, "cpu")
    ids = torch.stack([torch.randperm(cfg.E, generator=g)[: cfg.K] for _ in range(cfg.B)])
    w = torch.rand(cfg.B, cfg.K, generator=g) + 0.05
    return ids.to(torch.int32).to(device), w.to(torch.float32).to(device)
