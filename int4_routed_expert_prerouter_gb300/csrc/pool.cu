// Expert pool with a host tier: a fixed number of device slots per layer in front
// of every expert's packed weights held in pinned host memory, filled by
// copy-engine prefetch from the prerouter's prediction one token ahead ("The
// Other Half of the Memory Wall", S3.1 "SSD Streaming Expert Layers", S3.2
// "Motivation": the prediction made at token t selects the loads that overlap
// token t+1's forward pass; S5.3 "The Advantage of the Prerouter": prefetch
// against least-recently-used residency).  On GB300 the tiers are HBM and the
// host memory behind the host link; an expert whose slot-table entry is -1 is
// read by the kernels directly from host memory.
//
// Host code only.  The planner keeps, per layer, which expert sits in each slot
// and when each slot was last requested; the device slot table is a copy of
// that map, written by the prefetch after its weight copies.
#include <string.h>

#include <vector>

#include "internal.cuh"

struct edge0_pool {
    int L, E, n_slots;
    size_t gu_bytes, dn_bytes;
    struct Layer {
        const char* host_gu = nullptr;
        const char* host_dn = nullptr;
        char* dev_gu = nullptr;
        char* dev_dn = nullptr;
        int32_t* dev_table = nullptr;
        std::vector<int> slot_of;       // expert -> slot or -1
        std::vector<int> expert_in;     // slot -> expert or -1
        std::vector<long long> used;    // slot -> last request (planner clock)
        std::vector<int32_t> table;     // staging copy of slot_of for the device
    };
    std::vector<Layer> layers;
    long long clock = 0, hits = 0, copies = 0;
};

namespace {

// Plan: mark the experts of ids[0..n) (duplicates allowed) as requested now;
// assign each requested expert that is not resident a slot: a free one, else the
// least recently used slot holding an expert outside the request; stop when no
// slot is left (the rest stay in the host tier).  Fills the copies to make.
int plan(edge0_pool* P, int l, const int32_t* ids, int n, int32_t* out_expert, int32_t* out_slot, int* n_copy) {
    edge0_pool::Layer& Ly = P->layers[l];
    const long long now = ++P->clock;
    std::vector<char> want(P->E, 0);
    for (int i = 0; i < n; ++i) {
        const int e = ids[i];
        if (e < 0 || e >= P->E) return EDGE0_EINVAL;
        want[e] = 1;
    }
    // resident requested experts are hits: their slots are protected this round
    for (int e = 0; e < P->E; ++e)
        if (want[e] && Ly.slot_of[e] >= 0) {
            Ly.used[Ly.slot_of[e]] = now;
            ++P->hits;
        }
    int nc = 0;
    for (int e = 0; e < P->E; ++e) {
        if (!want[e] || Ly.slot_of[e] >= 0) continue;
        int victim = -1;
        for (int s = 0; s < P->n_slots; ++s) {
            if (Ly.used[s] == now) continue;   // requested this round
            if (Ly.expert_in[s] < 0) { victim = s; break; }
            if (victim < 0 || Ly.used[s] < Ly.used[victim]) victim = s;
        }
        if (victim < 0) break;                 // pool full of requested experts
        const int old = Ly.expert_in[victim];
        if (old >= 0) Ly.slot_of[old] = -1;
        Ly.expert_in[victim] = e;
        Ly.slot_of[e] = victim;
        Ly.used[victim] = now;
        out_expert[nc] = e;
        out_slot[nc] = victim;
        ++nc;
        ++P->copies;
    }
    *n_copy = nc;
    return EDGE0_OK;
}

}  // namespace

extern "C" int edge0_pool_create(int L, int E, int n_slots, size_t gu_bytes, size_t dn_bytes, edge0_pool** out) {
    if (!out || L <= 0 || E <= 0 || E > EDGE0_MAX_E || n_slots <= 0 || n_slots > E || !gu_bytes || !dn_bytes)
        return EDGE0_EINVAL;
    edge0_pool* P = new edge0_pool;
    P->L = L;
    P->E = E;
    P->n_slots = n_slots;
    P->gu_bytes = gu_bytes;
    P->dn_bytes = dn_bytes;
    P->layers.resize(L);
    for (auto& Ly : P->layers) {
        Ly.slot_of.assign(E, -1);
        Ly.expert_in.assign(n_slots, -1);
        Ly.used.assign(n_slots, 0);
        Ly.table.assign(E, -1);
    }
    *out = P;
    return EDGE0_OK;
}

extern "C" void edge0_pool_destroy(edge0_pool* P) { delete P; }

extern "C" int edge0_pool_set_layer(edge0_pool* P, int l, const void* host_gu, const void* host_dn, void* dev_gu,
                                    void* dev_dn, int32_t* dev_table) {
    if (!P || l < 0 || l >= P->L || !host_gu || !host_dn || !dev_gu || !dev_dn || !dev_table) return EDGE0_EINVAL;
    if (((uintptr_t)dev_gu | (uintptr_t)dev_dn | (uintptr_t)host_gu | (uintptr_t)host_dn) & 15) return EDGE0_EINVAL;
    auto& Ly = P->layers[l];
    Ly.host_gu = (const char*)host_gu;
    Ly.host_dn = (const char*)host_dn;
    Ly.dev_gu = (char*)dev_gu;
    Ly.dev_dn = (char*)dev_dn;
    Ly.dev_table = dev_table;
    return EDGE0_OK;
}

extern "C" int edge0_pool_plan(edge0_pool* P, int l, const int32_t* ids, int n, int32_t* out_expert,
                               int32_t* out_slot, int* n_copy) {
    if (!P || l < 0 || l >= P->L || n < 0 || (n && !ids) || !out_expert || !out_slot || !n_copy) return EDGE0_EINVAL;
    return plan(P, l, ids, n, out_expert, out_slot, n_copy);
}

extern "C" int edge0_pool_prefetch(edge0_pool* P, int l, const int32_t* ids, int n, cudaStream_t stream,
                                   int* copied) {
    if (!P || l < 0 || l >= P->L || n < 0 || (n && !ids)) return EDGE0_EINVAL;
    auto& Ly = P->layers[l];
    if (!Ly.dev_table) return EDGE0_EINVAL;
    std::vector<int32_t> ce(P->E), cs(P->E);
    int nc = 0;
    int rc = plan(P, l, ids, n, ce.data(), cs.data(), &nc);
    if (rc) return rc;
    for (int i = 0; i < nc; ++i) {
        if (cudaMemcpyAsync(Ly.dev_gu + (size_t)cs[i] * P->gu_bytes, Ly.host_gu + (size_t)ce[i] * P->gu_bytes,
                            P->gu_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
            cudaMemcpyAsync(Ly.dev_dn + (size_t)cs[i] * P->dn_bytes, Ly.host_dn + (size_t)ce[i] * P->dn_bytes,
                            P->dn_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
            return EDGE0_ECUDA;
    }
    // the table after the copies (from pageable memory: staged at the call)
    for (int e = 0; e < P->E; ++e) Ly.table[e] = Ly.slot_of[e];
    if (cudaMemcpyAsync(Ly.dev_table, Ly.table.data(), (size_t)P->E * 4, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
        return EDGE0_ECUDA;
    if (copied) *copied = nc;
    return EDGE0_OK;
}

extern "C" int edge0_pool_resident(const edge0_pool* P, int l, int32_t* slot_of) {
    if (!P || l < 0 || l >= P->L || !slot_of) return EDGE0_EINVAL;
    for (int e = 0; e < P->E; ++e) slot_of[e] = P->layers[l].slot_of[e];
    return EDGE0_OK;
}

extern "C" int edge0_pool_stats(const edge0_pool* P, long long* hits, long long* copies) {
    if (!P) return EDGE0_EINVAL;
    if (hits) *hits = P->hits;
    if (copies) *copies = P->copies;
    return EDGE0_OK;
}
