"""Workload presets for the prerouted int4 MoE decode path.

Shapes follow "The Other Half of the Memory Wall" (S3.1 "Problem": 256 experts,
40 layers; S3.2 "Head": f_in = d_model + 2E, hidden 512, heads owned by layers
6-38 consumed at 7-38 on the 35B tier, 8B input 1536 + 2x128; App. A: 8B tier
routes sigmoid-group with n=8, G=4, s=2.5, K=8) and the byte counts of
"Edge0 streams a 35B MoE off SSD" ("Counting the bytes": 1,327,104 B per 8B
expert, which with the 35B tier's 1.77 MB per expert fixes intermediate 512).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

SOFTMAX_TOPK = 0
SIGMOID_GROUP = 1
GROUP = 64  # affine quantisation group (int4 group-64)


@dataclass(frozen=True)
class Config:
    name: str
    L: int            # MoE layers
    d: int            # d_model
    E: int            # routed experts
    K: int            # experts per token
    I: int            # routed expert intermediate
    Is: int           # shared expert intermediate
    H: int            # prerouter hidden width
    r: int            # LoRA rank
    alpha: float      # LoRA alpha
    B: int            # sequences decoded together
    steps: int        # decode steps
    route_kind: int = SOFTMAX_TOPK
    n_groups: int = 1
    topk_groups: int = 1
    route_scale: float = 1.0
    zipf: float | None = None          # Zipf exponent of the router logit bias
    head_owner_first: int = 0          # heads owned by layers [first, last]
    head_owner_last: int = -1
    ring: bool = False                 # single layer whose head predicts itself
    prerouted: tuple = ()              # layers that consume a prediction (t > 0)
    pool_frac: float | None = None     # HBM expert pool as a fraction of all experts
    eps: float = 1e-6
    description: str = ""

    @property
    def f_in(self) -> int:
        return self.d + 2 * self.E

    def head_owners(self) -> list[int]:
        return list(range(self.head_owner_first, self.head_owner_last + 1))

    def head_target(self, owner: int) -> int:
        return owner if self.ring else owner + 1

    def with_(self, **kw) -> "Config":
        return replace(self, **kw)


def q4_bytes(out: int, inp: int) -> int:
    """Bytes of one int4 matrix: packed nibbles + one fp16 scale and bias per 64 inputs."""
    return out * inp // 2 + out * (inp // GROUP) * 2 * 2


def expert_bytes(d: int, I: int) -> int:
    """gate [I, d] + up [I, d] + down [d, I], int4 group-64."""
    return 2 * q4_bytes(I, d) + q4_bytes(d, I)


TOY = Config(
    name="toy", L=2, d=256, E=16, K=2, I=128, Is=128, H=64, r=4, alpha=8.0, B=1, steps=8,
    head_owner_first=0, head_owner_last=0, prerouted=(1,),
    description="toy prerouted MoE decode: 2 layers, d=256, E=16, K=2, I=Is=128, H=64, "
                "LoRA r=4 alpha=8, batch 1, 8 steps",
)

LAYER35 = Config(
    name="35b_layer", L=1, d=2048, E=256, K=4, I=512, Is=512, H=512, r=16, alpha=32.0, B=1,
    steps=256, head_owner_first=0, head_owner_last=0, ring=True, prerouted=(0,),
    description="35B-tier single MoE layer decode: d=2048, E=256, K=4, I=Is=512, H=512, "
                "LoRA r=16 alpha=32, batch 1, 256 steps (the layer's head predicts itself)",
)

STACK35 = Config(
    name="35b_stack", L=40, d=2048, E=256, K=4, I=512, Is=512, H=512, r=16, alpha=32.0, B=1,
    steps=512, head_owner_first=6, head_owner_last=38, prerouted=tuple(range(7, 39)),
    description="35B-tier 40-layer stack: heads on layers 6-38, layers 7-38 prerouted, "
                "layers 0-6 and 39 on their own router, batch 1, 512 steps",
)

STACK8 = Config(
    name="8b_stack", L=40, d=1536, E=128, K=8, I=512, Is=512, H=512, r=16, alpha=32.0, B=64,
    steps=256, route_kind=SIGMOID_GROUP, n_groups=8, topk_groups=4, route_scale=2.5, zipf=1.1,
    head_owner_first=7, head_owner_last=38, prerouted=tuple(range(8, 40)),
    description="8B-tier 40-layer stack: d=1536, E=128, K=8, sigmoid-group n=8 G=4 s=2.5, "
                "Zipf(1.1) logit bias, 64 sequences, 256 steps",
)

HOST35 = Config(
    name="35b_host_tier", L=40, d=2048, E=256, K=4, I=512, Is=512, H=512, r=16, alpha=32.0,
    B=256, steps=256, zipf=1.1, head_owner_first=6, head_owner_last=38,
    prerouted=tuple(range(7, 39)), pool_frac=0.25,
    description="35B-tier batched decode, 256 sequences, HBM expert pool capped at 25% of "
                "experts, the rest in pinned host memory, Zipf(1.1) logit bias, 256 steps",
)

CONFIGS = {c.name: c for c in (TOY, LAYER35, STACK35, STACK8, HOST35)}
