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
    ids = (C.c_void_p * 1)()
    assert lib.edge0_pool_prefetch_async(p.p, ids, 1, None, None) == E   # no device state
    assert lib.edge0_pool_wait(p.p, 0) == E
    assert lib.edge0_pool_host_prefetch(p.p, ids, 1) == E                # layer 0 not set
    assert lib.edge0_pool_host_copy(p.p) == E
    assert lib.edge0_pool_inject(p.p, -1, 0) == E
    assert lib.edge0_pool_inject(p.p, 0, 2_000_000_000) == E             # delays are bounded (1 s)
    assert lib.edge0_pool_plan(p.p, 1, None, 0, None, None, None) == E
    assert lib.edge0_pool_create(1, 8, 2, 24, 16, C.byref(out)) == E    # sizes are multiples of 16


# ------------------------------------------- the copy protocol, on the host ----
# edge0_pool_host_prefetch / edge0_pool_host_copy run the device pool's planner
# and publication steps over host buffers (a fake copy engine): plans evict at
# planning time, copies publish only when complete, a layer with copies in
# flight skips its next plan, injected failures leave the expert unpublished
# and free the slot at the next plan.

def _aligned(nbytes, dtype=np.uint8):
    raw = np.zeros(nbytes + 64, dtype=np.uint8)
    off = (-raw.ctypes.data) % 64
    return raw[off:off + nbytes].view(dtype)


class HostPool:
    def __init__(self, lib, L, E, S, gu=32, dn=16, seed=0):
        self.lib, self.L, self.E, self.S, self.gu, self.dn = lib, L, E, S, gu, dn
        self.p = C.c_void_p()
        assert lib.edge0_pool_create(L, E, S, gu, dn, C.byref(self.p)) == 0
        rng = np.random.default_rng(seed)
        self.host_gu = [_aligned(E * gu) for _ in range(L)]
        self.host_dn = [_aligned(E * dn) for _ in range(L)]
        for a in self.host_gu + self.host_dn:
            a[:] = rng.integers(0, 256, a.size, dtype=np.uint8)
        self.slot_gu = [_aligned(S * gu) for _ in range(L)]
        self.slot_dn = [_aligned(S * dn) for _ in range(L)]
        self.table = [_aligned(E * 4, np.int32) for _ in range(L)]
        for l in range(L):
            self.table[l][:] = -1
            ptr = lambda a: C.c_void_p(a.ctypes.data)
            assert lib.edge0_pool_set_layer(self.p, l, ptr(self.host_gu[l]), ptr(self.host_dn[l]),
                                            ptr(self.slot_gu[l]), ptr(self.slot_dn[l]), ptr(self.table[l])) == 0

    def prefetch(self, ids_by_layer, n):
        keep = []
        arr = (C.c_void_p * self.L)()
        for l, ids in ids_by_layer.items():
            a = np.array(ids, dtype=np.int32)
            assert a.size == n
            keep.append(a)
            arr[l] = a.ctypes.data
        assert self.lib.edge0_pool_host_prefetch(self.p, arr, n) == 0

    def copy(self):
        assert self.lib.edge0_pool_host_copy(self.p) == 0

    def inject(self, fail_every):
        assert self.lib.edge0_pool_inject(self.p, fail_every, 0) == 0

    def stats(self):
        out = (C.c_longlong * 8)()
        assert self.lib.edge0_pool_stats_ex(self.p, out, 8) == 0
        return dict(zip(binding.ExpertPool.STATS, list(out)))

    def check_published(self):
        """Every published entry's slot holds that expert's bytes."""
        for l in range(self.L):
            for e, s in enumerate(self.table[l].tolist()):
                if s < 0:
                    continue
                assert 0 <= s < self.S
                assert np.array_equal(self.slot_gu[l][s * self.gu:(s + 1) * self.gu],
                                      self.host_gu[l][e * self.gu:(e + 1) * self.gu]), (l, e, s)
                assert np.array_equal(self.slot_dn[l][s * self.dn:(s + 1) * self.dn],
                                      self.host_dn[l][e * self.dn:(e + 1) * self.dn]), (l, e, s)
            pub = [s for s in self.table[l].tolist() if s >= 0]
            assert len(pub) == len(set(pub)), f"layer {l}: a slot published twice"

    def __del__(self):
        self.lib.edge0_pool_destroy(self.p)


def test_protocol_publishes_only_completed_copies(lib):
    p = HostPool(lib, 2, 8, 3)
    p.prefetch({0: [1, 2, 1]}, 3)
    assert p.table[0].tolist() == [-1] * 8                   # planned, not yet copied
    assert p.stats()["planned"] == 2
    p.copy()
    assert p.table[0].tolist() == [-1, 0, 1, -1, -1, -1, -1, -1]
    assert p.table[1].tolist() == [-1] * 8                   # layer 1 had no request
    p.check_published()
    # a new expert evicts the least recently requested one at planning time
    p.prefetch({0: [2, 5, 5]}, 3)                             # 2 hits, 5 takes free slot 2
    p.copy()
    p.prefetch({0: [6, 6, 6]}, 3)                             # victim: slot 0 (expert 1)
    assert p.table[0][1] == -1 and p.table[0][6] == -1         # evicted at once, new one not yet
    p.copy()
    assert p.table[0][6] == 0
    p.check_published()
    st = p.stats()
    assert (st["requests"], st["hits"], st["planned"], st["published"]) == (2 + 2 + 1, 1, 4, 4)
    assert st["bytes"] == 4 * (32 + 16)


def test_protocol_layer_with_copies_in_flight_skips_its_plan(lib):
    p = HostPool(lib, 1, 8, 2)
    p.prefetch({0: [3, 4]}, 2)
    p.prefetch({0: [5, 6]}, 2)                                # previous copies in flight
    st = p.stats()
    assert st["skipped"] == 1 and st["planned"] == 2
    p.copy()
    assert sorted(p.table[0].tolist()) == [-1] * 6 + [0, 1]
    p.prefetch({0: [5, 6]}, 2)
    p.copy()
    assert p.table[0][5] >= 0 and p.table[0][6] >= 0 and p.table[0][3] == -1 and p.table[0][4] == -1
    p.check_published()


def test_protocol_failed_copies_stay_unpublished_and_free_their_slot(lib):
    p = HostPool(lib, 1, 8, 4)
    p.inject(2)                                               # copies 1, 3, 5, ... fail
    p.prefetch({0: [0, 1, 2, 3]}, 4)
    p.copy()
    st = p.stats()
    assert st["failed"] == 2 and st["published"] == 2
    t = p.table[0].tolist()
    assert t[0] >= 0 and t[1] == -1 and t[2] >= 0 and t[3] == -1
    p.check_published()
    p.inject(0)
    p.prefetch({0: [0, 1, 2, 3]}, 4)                          # 0, 2 hits; 1, 3 copied again
    st2 = p.stats()
    assert st2["hits"] == 2 and st2["planned"] == 6
    p.copy()
    assert min(p.table[0][:4].tolist()) >= 0
    p.check_published()


def test_protocol_more_requests_than_slots(lib):
    p = HostPool(lib, 1, 16, 3)
    p.prefetch({0: [9, 1, 4, 7, 2, 2]}, 6)                    # 5 distinct, 3 slots
    p.copy()
    t = p.table[0]
    assert sorted(e for e in range(16) if t[e] >= 0) == [1, 2, 4]   # id order, then out of slots
    assert p.stats()["requests"] == 5
    p.check_published()


class _ProtocolModel:
    """The protocol restated: planner map, published table, busy layers,
    failures, counters."""

    def __init__(self, L, E, S):
        self.L, self.E, self.S = L, E, S
        self.expert_in = [[-1] * S for _ in range(L)]
        self.used = [[0] * S for _ in range(L)]
        self.fail = [[0] * S for _ in range(L)]
        self.clk = [0] * L
        self.busy = [False] * L
        self.jobs = [[] for _ in range(L)]
        self.seq0 = [0] * L
        self.table = [[-1] * E for _ in range(L)]
        self.st = dict.fromkeys(binding.ExpertPool.STATS, 0)

    def prefetch(self, ids_by_layer):
        for l, ids in ids_by_layer.items():
            if self.busy[l]:
                self.st["skipped"] += 1
                continue
            ei, used, fail = self.expert_in[l], self.used[l], self.fail[l]
            for s in range(self.S):
                if fail[s]:
                    ei[s], used[s], fail[s] = -1, 0, 0
            self.clk[l] += 1
            now = self.clk[l]
            want = sorted(set(ids))
            self.st["requests"] += len(want)
            where = {e: s for s, e in enumerate(ei) if e >= 0}
            for e in want:
                if e in where:
                    used[where[e]] = now
                    self.st["hits"] += 1
            jobs = []
            for e in want:
                if e in where:
                    continue
                cand = [s for s in range(self.S) if used[s] != now]
                if not cand:
                    break
                free = [s for s in cand if ei[s] < 0]
                s = free[0] if free else min(cand, key=lambda s: (used[s], s))
                if ei[s] >= 0:
                    self.table[l][ei[s]] = -1
                    del where[ei[s]]
                ei[s], used[s] = e, now
                where[e] = s
                jobs.append((e, s))
            self.jobs[l] = jobs
            self.seq0[l] = self.st["planned"]
            self.st["planned"] += len(jobs)
            self.busy[l] = True

    def copy(self, fail_every, nbytes):
        for l in range(self.L):
            if not self.busy[l]:
                continue
            for k, (e, s) in enumerate(self.jobs[l]):
                if fail_every and (self.seq0[l] + k) % fail_every == fail_every - 1:
                    self.fail[l][s] = 1
                    self.st["failed"] += 1
                else:
                    self.table[l][e] = s
                    self.st["published"] += 1
                    self.st["bytes"] += nbytes
            self.busy[l] = False


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_protocol_matches_a_restatement_under_random_operations(lib, seed):
    rng = random.Random(seed)
    L, E, S, n = 3, 32, 6, 12
    p = HostPool(lib, L, E, S, gu=48, dn=32, seed=seed)
    m = _ProtocolModel(L, E, S)
    w = [1.0 / (i + 1) ** 1.1 for i in range(E)]
    fail_every = 0
    for _ in range(120):
        op = rng.random()
        if op < 0.5:
            req = {l: rng.choices(range(E), weights=w, k=n) for l in range(L) if rng.random() < 0.8}
            p.prefetch(req, n)
            m.prefetch(req)
        elif op < 0.9:
            p.copy()
            m.copy(fail_every, 48 + 32)
        else:
            fail_every = rng.choice([0, 0, 2, 3, 5])
            p.inject(fail_every)
        for l in range(L):
            assert p.table[l].tolist() == m.table[l], f"layer {l}"
        assert p.stats() == m.st
        p.check_published()


def test_device_init_without_a_gpu_leaves_the_host_model_usable(lib):
    # no GPU here: the device state cannot be allocated; the call reports it
    # and the pool stays on the host model
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present (the host buffers below are not device memory)")
    p = HostPool(lib, 1, 8, 2)
    assert lib.edge0_pool_device_init(p.p) == binding.EDGE0_ECUDA
    p.prefetch({0: [1, 2]}, 2)
    p.copy()
    assert sorted(e for e in range(8) if p.table[0][e] >= 0) == [1, 2]
    p.check_published()
