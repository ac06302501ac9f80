// Residency planner of the host-tier expert pool, shared by the device planner
// kernel, the host planner and the host model of the copy protocol ("The Other
// Half of the Memory Wall", S3.1 "SSD Streaming Expert Layers": a layer keeps a
// fixed number of staged expert slots; S3.2 "Motivation": the prediction made at
// token t names the experts to load for token t+1; S5.3: prefetch against
// least-recently-used residency).
//
// Per layer the planner owns slot_of[E] (its map: slot of an expert, or -1),
// expert_in[S] and used[S] (planner clock of the slot's last request).  The
// published map table[E], which the expert kernels read, follows slot_of with a
// delay: an evicted expert leaves table at planning time, a copied expert
// enters it only once its copy is complete.  fail[S] marks a slot whose copy
// did not complete; the next plan frees it.
#pragma once
#include <stdint.h>

namespace edge0 {
namespace pool {

enum Stat : int {
    ST_REQUESTS = 0,   // requested (layer, expert) pairs, duplicates within a request counted once
    ST_HITS,           // requested pairs found in the planner's map
    ST_PLANNED,        // copies planned
    ST_PUBLISHED,      // copies completed and entered into the published map
    ST_FAILED,         // copies that did not complete (slot freed at the next plan)
    ST_SKIPPED,        // layer plans skipped: the layer's previous copies still in flight
    ST_BYTES,          // bytes of the published copies
    ST_BAD_IDS,        // requested ids outside [0, E) (ignored)
    ST_COUNT
};

enum Meta : int {
    MT_NJ = 0,      // copies of the layer's last plan
    MT_GEN,         // plan generation that wrote them
    MT_BUSY,        // 1 from a plan until the copy pass of its generation has ended
    MT_CLK,         // planner clock of the layer
    MT_SEQ0,        // sequence number of the plan's first copy (fault injection)
    MT_COUNT = 8
};

struct LayerState {
    int* slot_of;     // [E]
    int* expert_in;   // [S]
    int* used;        // [S]
    int* fail;        // [S]
    int* job_e;       // [S] expert of each planned copy
    int* job_s;       // [S] its slot
};

// Slots whose copy failed: free again, their expert back in the host tier.
__host__ __device__ inline void reclaim_failed(const LayerState& L, int S) {
    for (int s = 0; s < S; ++s)
        if (L.fail[s]) {
            if (L.expert_in[s] >= 0) L.slot_of[L.expert_in[s]] = -1;
            L.expert_in[s] = -1;
            L.used[s] = 0;
            L.fail[s] = 0;
        }
}

// One request at planner clock `now`: want[e] != 0 for the requested experts.
// Requested experts already in the map are hits and protect their slots for
// this request.  Every other requested expert, in id order, takes a free slot,
// else the least recently requested slot whose expert is not requested now
// (lowest index on equal recency); when no such slot is left the rest stay in
// the host tier.  An evicted expert leaves `table` (if given) at once.  Writes
// the copies to make to L.job_e / L.job_s and returns their number.
__host__ __device__ inline int plan_request(const unsigned char* want, int E, int S, const LayerState& L, int now,
                                            int32_t* table, long long* requests, long long* hits) {
    long long rq = 0, h = 0;
    for (int e = 0; e < E; ++e)
        if (want[e]) {
            ++rq;
            if (L.slot_of[e] >= 0) {
                L.used[L.slot_of[e]] = now;
                ++h;
            }
        }
    int nj = 0;
    for (int e = 0; e < E; ++e) {
        if (!want[e] || L.slot_of[e] >= 0) continue;
        int victim = -1;
        for (int s = 0; s < S; ++s) {
            if (L.used[s] == now) continue;            // requested now
            if (L.expert_in[s] < 0) { victim = s; break; }
            if (victim < 0 || L.used[s] < L.used[victim]) victim = s;
        }
        if (victim < 0) break;                          // every slot requested now
        const int old = L.expert_in[victim];
        if (old >= 0) {
            L.slot_of[old] = -1;
            if (table) table[old] = -1;
        }
        L.expert_in[victim] = e;
        L.slot_of[e] = victim;
        L.used[victim] = now;
        L.job_e[nj] = e;
        L.job_s[nj] = victim;
        ++nj;
    }
    *requests += rq;
    *hits += h;
    return nj;
}

// Fault injection: copy number `seq` (counted over the pool's plans) fails when
// fail_every > 0 and seq % fail_every == fail_every - 1.
__host__ __device__ inline bool injected_failure(long long seq, int fail_every) {
    return fail_every > 0 && seq % fail_every == fail_every - 1;
}

}  // namespace pool
}  // namespace edge0
