"""Host-tier expert pool: the planner's policy (no GPU needed).  A requested
expert that is not resident takes a free slot, else the least recently
requested slot whose expert is not requested now; requested experts left
without a slot stay in the host tier."""
import ctypes as C
import random

import numpy as np
import pytest

from int4_routed_expert_prerouter_gb300 import binding, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


class Pool:
    def __init__(self, lib, L, E, n_slots):
        self.lib, self.E = lib, E
        self.p = C.c_void_p()
        assert lib.edge0_pool_create(L, E, n_slots, 1024, 1024, C.byref(self.p)) == 0

    def plan(self, l, ids):
        a = np.array(ids, dtype=np.int32)
        oe = np.zeros(self.E, dtype=np.int32)
        os_ = np.zeros(self.E, dtype=np.int32)
        n = C.c_int(0)
        rc = self.lib.edge0_pool_plan(self.p, l, a.ctypes.data_as(C.c_void_p), len(ids),
                                      oe.ctypes.data_as(C.c_void_p), os_.ctypes.data_as(C.c_void_p), C.byref(n))
        return rc, list(zip(oe[:n.value].tolist(), os_[:n.value].tolist()))

    def stats(self):
        h, c = C.c_longlong(0), C.c_longlong(0)
        assert self.lib.edge0_pool_stats(self.p, C.byref(h), C.byref(c)) == 0
        return h.value, c.value

    def resident(self, l):
        out = np.zeros(self.E, dtype=np.int32)
        assert self.lib.edge0_pool_resident(self.p, l, out.ctypes.data_as(C.c_void_p)) == 0
        return out.tolist()

    def __del__(self):
        self.lib.edge0_pool_destroy(self.p)


def test_pool_lru_hand_case(lib):
    p = Pool(lib, 1, 8, 3)
    assert p.plan(0, [1, 2]) == (0, [(1, 0), (2, 1)])          # free slots in order
    assert p.plan(0, [2, 3, 3]) == (0, [(3, 2)])              # 2 hits; duplicates count once
    assert p.plan(0, [4]) == (0, [(4, 0)])                    # LRU victim: expert 1 (slot 0)
    assert p.plan(0, [1, 4, 2, 3]) == (0, [])                 # all slots requested now: 1 stays on host
    assert p.stats() == (1 + 3, 4)
    assert p.plan(0, [1]) == (0, [(1, 0)])                    # slots 0-2 tie in recency: lowest index
    assert p.plan(0, [8])[0] == binding.EDGE0_EINVAL           # id outside [0, E)


def _reference(n_slots, requests):
    """The same policy restated: slot contents and last-request times."""
    expert_in = [-1] * n_slots
    used = [0] * n_slots
    out = []
    for clock, req in enumerate(requests, start=1):
        want = sorted(set(req))
        resident = {e: s for s, e in enumerate(expert_in) if e >= 0}
        for e in want:
            if e in resident:
                used[resident[e]] = clock
        copies = []
        for e in want:
            if e in resident:
                continue
            cand = [s for s in range(n_slots) if used[s] != clock]
            if not cand:
                break
            free = [s for s in cand if expert_in[s] < 0]
            s = free[0] if free else min(cand, key=lambda s: (used[s], s))
            expert_in[s] = e
            used[s] = clock
            resident = {e2: s2 for s2, e2 in enumerate(expert_in) if e2 >= 0}
            copies.append((e, s))
        out.append(copies)
    return out


@pytest.mark.parametrize("E,n_slots", [(16, 4), (64, 16), (256, 64)])
def test_pool_matches_a_plain_lru_restatement(lib, E, n_slots):
    rng = random.Random(E)
    # Zipf-like requests: a few hot experts and a long tail
    w = [1.0 / (i + 1) ** 1.1 for i in range(E)]
    reqs = [rng.choices(range(E), weights=w, k=rng.randint(1, 3 * n_slots // 2)) for _ in range(60)]
    p = Pool(lib, 2, E, n_slots)
    ref = _reference(n_slots, reqs)
    slot_of = [-1] * E
    for req, exp in zip(reqs, ref):
        rc, got = p.plan(1, req)
        assert rc == 0 and got == exp
        # the resident map follows the copies: a copied expert evicts the slot's
        # previous one
        for e, sl in got:
            for e2 in range(E):
                if slot_of[e2] == sl:
                    slot_of[e2] = -1
            slot_of[e] = sl
        assert p.resident(1) == slot_of
    # layer 0 untouched by layer 1's plans
    assert p.resident(0) == [-1] * E
    assert p.plan(0, [0])[1] == [(0, 0)]


def test_pool_rejects_bad_arguments(lib):
    E = binding.EDGE0_EINVAL
    out = C.c_void_p()
    assert lib.edge0_pool_create(0, 8, 2, 1, 1, C.byref(out)) == E
    assert lib.edge0_pool_create(1, 8, 9, 1, 1, C.byref(out)) == E     # more slots than experts
    assert lib.edge0_pool_create(1, 8, 2, 0, 1, C.byref(out)) == E
    p = Pool(lib, 1, 8, 2)
    assert lib.edge0_pool_set_layer(p.p, 0, None, None, None, None, None) == E
    assert lib.edge0_pool_prefetch(p.p, 0, None, 0, None, None) == E     # no device side set
    assert lib.edge0_pool_plan(p.p, 1, None, 0, None, None, None) == E
