// Device helpers shared by the persistent engine and the batched decode path:
// the int4 nibble masks of the tensor-core fragments and the routing rule.
#pragma once
#include "internal.cuh"

namespace edge0 {

// A fragments of one 16-input step of a 16-row tile from one 32-bit word of the
// packed int4 layout: nibbles become fp16 subnormals q 2^-24 (the second nibble
// of a byte is q 2^-20, i.e. x16, undone by the caller's scale)
__device__ __forceinline__ void q4_masks(uint32_t w, uint32_t A[4]) {
    const uint32_t w8 = w >> 8;
    A[0] = w & 0x000F000Fu;    // row g,   k 2t | 2t+1
    A[1] = w & 0x00F000F0u;    // row g+8, k 2t | 2t+1   (x16)
    A[2] = w8 & 0x000F000Fu;   // row g,   k 2t+8 | 2t+9
    A[3] = w8 & 0x00F000F0u;   // row g+8, k 2t+8 | 2t+9 (x16)
}

// ---------------------------------------------------------- routing -----
// top-K over `score` (E values, E <= 512) by one warp, value descending, lower
// index first on ties; masked entries are -inf.  Lane l owns entries l + 32 i.
static __device__ __noinline__ void warp_topk(const float* score, int E, int K, int* ids, int lane) {
    unsigned taken = 0;   // bit i: entry lane + 32 i already selected
    for (int k = 0; k < K; ++k) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int i = 0, e = lane; e < E; ++i, e += 32) {
            if ((taken >> i) & 1u) continue;
            const float v = score[e];
            if (v > bv) { bv = v; bi = e; }   // e increases: ties keep the lower index
        }
        for (int s = 16; s; s >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, s);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, s);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (bi == 0x7fffffff) bi = 0;   // fewer than K candidates (not reachable for valid shapes)
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == 0) ids[k] = bi;
    }
    __syncwarp();
}

// Routing rule of App. A, one token per warp.  logits: E fp32 in shared memory;
// scratch: 2 E floats of shared memory for this warp.
static __device__ __noinline__ void warp_route(const float* logits, int E, int K, int kind, int n_groups,
                                        int G, float scale, const float* bias, float* scratch,
                                        int* ids, float* w, int lane) {
    float* sel = scratch;
    float* sig = scratch + E;
    const bool group = kind == EDGE0_ROUTE_SIGMOID_GROUP;
    for (int e = lane; e < E; e += 32) {
        const float l = logits[e];
        const float s = group ? 1.0f / (1.0f + expf(-l)) : l;
        sig[e] = s;
        sel[e] = bias ? s + bias[e] : s;
    }
    __syncwarp();
    if (group) {
        const int per = E / n_groups;
        // group score: sum of the two largest selection scores of the group
        float gscore = -INFINITY;
        if (lane < n_groups) {
            float a = -INFINITY, b = -INFINITY;
            for (int j = 0; j < per; ++j) {
                const float v = sel[lane * per + j];
                if (v > a) { b = a; a = v; }
                else if (v > b) { b = v; }
            }
            gscore = a + b;
        }
        // keep the best G groups (lower group index on ties)
        unsigned keep = 0;
        for (int k = 0; k < G; ++k) {
            const bool cand = lane < n_groups && !((keep >> lane) & 1u);
            float bv = cand ? gscore : -INFINITY;
            int bi = cand ? lane : 0x7fffffff;
            for (int s = 16; s; s >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, s);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, s);
                if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
            }
            if (bi < 32) keep |= 1u << bi;
        }
        for (int e = lane; e < E; e += 32)
            if (!((keep >> (e / per)) & 1u)) sel[e] = -INFINITY;
        __syncwarp();
    }
    warp_topk(sel, E, K, ids, lane);
    if (lane == 0) {
        if (group) {
            float sum = 0.0f;
            for (int k = 0; k < K; ++k) sum += sig[ids[k]];
            for (int k = 0; k < K; ++k) w[k] = scale * sig[ids[k]] / (sum + 1e-20f);
        } else {
            const float mx = sel[ids[0]];
            float sum = 0.0f;
            for (int k = 0; k < K; ++k) sum += expf(sel[ids[k]] - mx);
            for (int k = 0; k < K; ++k) w[k] = expf(sel[ids[k]] - mx) / sum;
        }
    }
    __syncwarp();
}


}  // namespace edge0
