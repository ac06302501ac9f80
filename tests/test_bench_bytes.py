"""The algorithmic bytes behind bench.py's roofline numerator, pinned to the
numbers the pages print (tests/golden/pages_numbers.json) and to a hand count."""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from int4_routed_expert_prerouter_gb300 import configs  # noqa: E402

GOLDEN = json.load(open(os.path.join(ROOT, "tests", "golden", "pages_numbers.json")))


def test_expert_bytes_match_the_pages():
    # "Counting the bytes": 1,327,104 B per 8B-tier expert; "Problem": ~1.77 MB per 35B-tier expert
    assert configs.expert_bytes(1536, 512) == GOLDEN["expert_bytes_8b"]["value"]
    assert round(configs.expert_bytes(2048, 512) / 1e6, 2) == GOLDEN["expert_mb_35b"]["value_mb"]


def test_head_parameters_match_the_pages():
    c = configs.STACK35
    f_in = c.d + 2 * c.E
    assert f_in == GOLDEN["f_in_35b"]["value"]
    params = c.H * f_in + c.E * c.H + c.E * f_in        # fc1, fc2, linear_init
    assert params == GOLDEN["head_params"]["value"]
    assert len(c.head_owners()) * params * 2 == GOLDEN["heads_bytes_35b"]["value"]


def test_batch1_step_bytes():
    # one decode step of the 35B-tier stack: 40 layers x (4 routed + shared
    # expert + LoRA), 33 heads (dense parts + 2K gathered one-hot columns), 8
    # routers of the layers that route themselves
    c = configs.STACK35
    own = c.L - len(c.prerouted)
    assert own == 8
    expert = 1_769_472
    head = (512 * 2048 + 256 * 2048 + 256 * 512) * 2 + 2 * 4 * (512 + 256) * 2
    lora = 2 * (16 * 2048 + 512 * 16) * 2 + (16 * 512 + 2048 * 16) * 2
    assert (head, lora) == (3_420_160, 245_760)
    want = 40 * (4 * expert + expert + lora) + 33 * head + 8 * 256 * 2048 * 2
    assert want == 484_978_688
    assert bench.algorithmic_bytes_per_token(c, own) == want


def test_batched_step_bytes_count_each_active_expert_once():
    c = configs.STACK8.with_(L=3, B=4, head_owner_first=0, head_owner_last=1, prerouted=(1, 2))
    ex = np.zeros((c.L, c.B, c.K), dtype=np.int32)
    for l in range(c.L):
        for b in range(c.B):
            ex[l, b] = np.arange(c.K) + (b % 2) * 3      # tokens share experts
    distinct = [len(np.unique(ex[l])) for l in range(c.L)]
    assert distinct == [c.K + 3] * c.L
    expert = configs.expert_bytes(c.d, c.I)
    lora = (2 * (c.r * c.d + c.Is * c.r) + (c.r * c.Is + c.d * c.r)) * 2
    head = (c.H * c.d + c.E * c.d + c.E * c.H) * 2 + c.B * 2 * c.K * (c.H + c.E) * 2
    want = sum(n * expert + expert + lora for n in distinct) + 2 * head + 1 * c.E * c.d * 2
    assert bench.batched_bytes_per_step(c, ex, 1) == want
