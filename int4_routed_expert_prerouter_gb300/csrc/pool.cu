// Expert pool with a host tier: a fixed number of device slots per layer in front
// of every expert's packed weights held in pinned host memory, filled from the
// prerouter's prediction one token ahead ("The Other Half of the Memory Wall",
// S3.1 "SSD Streaming Expert Layers", S3.2 "Motivation": the prediction made at
// token t selects the loads that overlap token t+1's forward pass; S5.3 "The
// Advantage of the Prerouter": prefetch against least-recently-used
// residency).  On GB300 the tiers are HBM and the host memory behind the host
// link; an expert whose published slot-table entry is -1 is read by the
// kernels directly from host memory.
//
// The pool runs on the device.  After the work that wrote a step's
// predictions, one planner CTA per layer turns them into copies (pool_plan.cuh)
// on the compute stream: evicted experts leave the published map before any
// later kernel of that stream reads it.  A copy kernel on a second stream then
// moves the planned experts from host memory into their slots and publishes
// each one (release store of its table entry) once all of its bytes are in
// place.  Nothing waits: the compute stream never waits for a copy (an expert
// whose copy is still in flight is read from the host tier), and a layer whose
// previous copies are still in flight skips its next plan.  Faults are
// injected on the host side of this protocol (copies that are marked failed,
// a delayed copy pass), never by a faulting access.
//
// The same planner and publication steps also run on the host over host
// buffers (edge0_pool_plan, edge0_pool_host_prefetch, edge0_pool_host_copy),
// which lets the protocol be exercised without a GPU.
#include <string.h>

#include <chrono>
#include <thread>
#include <vector>

#include "internal.cuh"
#include "pool_plan.cuh"

using edge0::pool::LayerState;

namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyVec = 16;                                    // uint4 per thread and chunk
constexpr int kCopyChunk = kCopyThreads * kCopyVec * 16;       // 64 KB
// few copy CTAs: a resident copy CTA keeps an expert kernel's CTA off its SM
// (the expert kernels take whole SMs), so the copies run on 8 SMs at a time;
// they still end long before the next step (~370 MB per step)
constexpr int kCopyCtas = 8;
constexpr unsigned long long kMaxDelayNs = 1000000000ull;

struct PoolLayerDev {
    const char* host_gu;
    const char* host_dn;
    char* dev_gu;
    char* dev_dn;
    int32_t* table;
};

// device state of the pool (one allocation), passed to the kernels by value
struct PoolDevP {
    PoolLayerDev* ly;                  // [L]
    int* meta;                         // [L][MT_COUNT]
    int *slot_of, *expert_in, *used, *fail, *job_e, *job_s;   // [L][E] / [L][S]
    unsigned* done;                    // [L][S] chunks of each planned copy done
    unsigned long long* stat;          // [ST_COUNT]
    unsigned* exit_cnt;                // CTAs of the running copy pass that have ended
    int L, E, S;
    long long gu_bytes, dn_bytes;
};

struct IdsP {
    const int32_t* p[EDGE0_MAX_LAYERS];
};

}  // namespace

struct edge0_pool {
    int L, E, n_slots;
    size_t gu_bytes, dn_bytes;
    struct Layer {
        const char* host_gu = nullptr;
        const char* host_dn = nullptr;
        char* dev_gu = nullptr;
        char* dev_dn = nullptr;
        int32_t* dev_table = nullptr;
        std::vector<int> slot_of, expert_in, used, fail, job_e, job_s;
        int meta[edge0::pool::MT_COUNT] = {0};
        LayerState state() {
            return LayerState{slot_of.data(), expert_in.data(), used.data(), fail.data(), job_e.data(), job_s.data()};
        }
    };
    std::vector<Layer> layers;
    long long stat[edge0::pool::ST_COUNT] = {0};
    int gen = 0;                       // plans made over the whole pool
    int fail_every = 0;
    unsigned long long delay_ns = 0;
    // device mode
    bool device = false;
    void* dmem = nullptr;
    PoolDevP dp{};
    cudaEvent_t planned = nullptr;
    cudaEvent_t copied = nullptr;      // after the last copy pass enqueued
};

namespace {

using namespace edge0;
using namespace edge0::pool;

__device__ __forceinline__ unsigned long long gtime_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ LayerState dev_state(const PoolDevP& p, int l) {
    const long long e = (long long)l * p.E, s = (long long)l * p.S;
    return LayerState{p.slot_of + e, p.expert_in + s, p.used + s, p.fail + s, p.job_e + s, p.job_s + s};
}

// One CTA per layer: the layer's requested experts (ids[l][0..n), or none when
// ids[l] is null) become a plan.
__global__ void __launch_bounds__(256) k_pool_plan(PoolDevP p, IdsP ids, int n, int gen) {
    extern __shared__ unsigned char want[];
    __shared__ int skip, bad;
    const int l = blockIdx.x, tid = threadIdx.x;
    const int32_t* src = ids.p[l];
    if (!src) return;
    int* meta = p.meta + l * MT_COUNT;
    if (tid == 0) {
        skip = (int)ld_acquire_u32(reinterpret_cast<const unsigned*>(meta + MT_BUSY));
        bad = 0;
        if (skip) atomicAdd(&p.stat[ST_SKIPPED], 1ull);
    }
    for (int e = tid; e < p.E; e += blockDim.x) want[e] = 0;
    __syncthreads();
    if (skip) return;
    for (int i = tid; i < n; i += blockDim.x) {
        const int e = src[i];
        if (e >= 0 && e < p.E)
            want[e] = 1;
        else
            atomicAdd(&bad, 1);
    }
    __syncthreads();
    if (tid != 0) return;
    if (bad) atomicAdd(&p.stat[ST_BAD_IDS], (unsigned long long)bad);
    const LayerState L = dev_state(p, l);
    reclaim_failed(L, p.S);
    const int now = ++meta[MT_CLK];
    long long rq = 0, h = 0;
    const int nj = plan_request(want, p.E, p.S, L, now, p.ly[l].table, &rq, &h);
    atomicAdd(&p.stat[ST_REQUESTS], (unsigned long long)rq);
    atomicAdd(&p.stat[ST_HITS], (unsigned long long)h);
    const unsigned long long seq0 = atomicAdd(&p.stat[ST_PLANNED], (unsigned long long)nj);
    for (int k = 0; k < nj; ++k) p.done[l * p.S + k] = 0;
    meta[MT_NJ] = nj;
    meta[MT_SEQ0] = (int)(seq0 & 0x7FFFFFFF);
    meta[MT_GEN] = gen;
    meta[MT_BUSY] = 1;
}

// One 64 KB piece of a copy (len a multiple of 16 bytes): every thread's loads
// in flight before its stores.
__device__ __forceinline__ void copy_chunk(const char* src, char* dst, long long len) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    const int n16 = (int)(len >> 4);
    uint4 v[kCopyVec];
#pragma unroll
    for (int i = 0; i < kCopyVec; ++i) {
        const int j = threadIdx.x + i * kCopyThreads;
        if (j < n16) v[i] = s4[j];
    }
#pragma unroll
    for (int i = 0; i < kCopyVec; ++i) {
        const int j = threadIdx.x + i * kCopyThreads;
        if (j < n16) d4[j] = v[i];
    }
}

// The copies of plan generation `gen`, in layer order, 64 KB pieces dealt to
// the CTAs in turn.  The CTA that completes a copy's last piece publishes it;
// the last CTA to end clears the planned layers' busy flags.
__global__ void __launch_bounds__(kCopyThreads) k_pool_copy(PoolDevP p, int gen, int fail_every,
                                                            unsigned long long delay_ns) {
    __shared__ int pre[EDGE0_MAX_LAYERS + 1];
    const int tid = threadIdx.x;
    if (tid == 0) {
        pre[0] = 0;
        for (int l = 0; l < p.L; ++l) {
            const int* m = p.meta + l * MT_COUNT;
            pre[l + 1] = pre[l] + (m[MT_GEN] == gen ? m[MT_NJ] : 0);
        }
        if (delay_ns) {   // injected delay of the copy pass (bounded: at most 1 s)
            const unsigned long long t0 = gtime_ns();
            while (gtime_ns() - t0 < delay_ns) __nanosleep(4096);
        }
    }
    __syncthreads();
    const int cg = (int)((p.gu_bytes + kCopyChunk - 1) / kCopyChunk);
    const int cj = cg + (int)((p.dn_bytes + kCopyChunk - 1) / kCopyChunk);
    const long long total = (long long)pre[p.L] * cj;
    for (long long u = blockIdx.x; u < total; u += gridDim.x) {   // CTA-uniform
        const int job = (int)(u / cj), c = (int)(u - (long long)job * cj);
        int l = 0;
        while (pre[l + 1] <= job) ++l;
        const int k = job - pre[l];
        const int e = p.job_e[l * p.S + k], s = p.job_s[l * p.S + k];
        const long long seq = (long long)p.meta[l * MT_COUNT + MT_SEQ0] + k;
        const bool failed = injected_failure(seq, fail_every);
        if (!failed) {
            const PoolLayerDev Y = p.ly[l];
            if (c < cg) {
                const long long off = (long long)c * kCopyChunk;
                const long long len = p.gu_bytes - off < kCopyChunk ? p.gu_bytes - off : kCopyChunk;
                copy_chunk(Y.host_gu + (long long)e * p.gu_bytes + off, Y.dev_gu + (long long)s * p.gu_bytes + off,
                           len);
            } else {
                const long long off = (long long)(c - cg) * kCopyChunk;
                const long long len = p.dn_bytes - off < kCopyChunk ? p.dn_bytes - off : kCopyChunk;
                copy_chunk(Y.host_dn + (long long)e * p.dn_bytes + off, Y.dev_dn + (long long)s * p.dn_bytes + off,
                           len);
            }
        }
        __threadfence();
        __syncthreads();
        if (tid == 0 && atomicAdd(&p.done[l * p.S + k], 1u) == (unsigned)cj - 1) {
            __threadfence();
            if (failed) {
                p.fail[l * p.S + s] = 1;
                atomicAdd(&p.stat[ST_FAILED], 1ull);
            } else {
                st_release_u32(reinterpret_cast<unsigned*>(p.ly[l].table + e), (unsigned)s);
                atomicAdd(&p.stat[ST_PUBLISHED], 1ull);
                atomicAdd(&p.stat[ST_BYTES], (unsigned long long)(p.gu_bytes + p.dn_bytes));
            }
        }
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(p.exit_cnt, 1u) == gridDim.x - 1) {
            __threadfence();
            for (int l = 0; l < p.L; ++l)
                if (p.meta[l * MT_COUNT + MT_GEN] == gen)
                    st_release_u32(reinterpret_cast<unsigned*>(p.meta + l * MT_COUNT + MT_BUSY), 0u);
            *p.exit_cnt = 0;
        }
    }
}

bool layers_set(const edge0_pool* P) {
    for (const auto& Ly : P->layers)
        if (!Ly.dev_table) return false;
    return true;
}

}  // namespace

extern "C" int edge0_pool_create(int L, int E, int n_slots, size_t gu_bytes, size_t dn_bytes, edge0_pool** out) {
    if (!out || L <= 0 || L > EDGE0_MAX_LAYERS || E <= 0 || E > EDGE0_MAX_E || n_slots <= 0 || n_slots > E ||
        !gu_bytes || !dn_bytes || gu_bytes % 16 || dn_bytes % 16)
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
        Ly.fail.assign(n_slots, 0);
        Ly.job_e.assign(n_slots, -1);
        Ly.job_s.assign(n_slots, -1);
    }
    *out = P;
    return EDGE0_OK;
}

extern "C" void edge0_pool_destroy(edge0_pool* P) {
    if (!P) return;
    if (P->device) {
        cudaDeviceSynchronize();   // no copy pass may still use the state
        cudaFree(P->dmem);
        cudaEventDestroy(P->planned);
        cudaEventDestroy(P->copied);
    }
    delete P;
}

extern "C" int edge0_pool_set_layer(edge0_pool* P, int l, const void* host_gu, const void* host_dn, void* dev_gu,
                                    void* dev_dn, int32_t* dev_table) {
    if (!P || P->device || l < 0 || l >= P->L || !host_gu || !host_dn || !dev_gu || !dev_dn || !dev_table)
        return EDGE0_EINVAL;
    if (((uintptr_t)dev_gu | (uintptr_t)dev_dn | (uintptr_t)host_gu | (uintptr_t)host_dn) & 15) return EDGE0_EINVAL;
    auto& Ly = P->layers[l];
    Ly.host_gu = (const char*)host_gu;
    Ly.host_dn = (const char*)host_dn;
    Ly.dev_gu = (char*)dev_gu;
    Ly.dev_dn = (char*)dev_dn;
    Ly.dev_table = dev_table;
    return EDGE0_OK;
}

// ------------------------------------------------------------ host mode ----
extern "C" int edge0_pool_plan(edge0_pool* P, int l, const int32_t* ids, int n, int32_t* out_expert,
                               int32_t* out_slot, int* n_copy) {
    if (!P || P->device || l < 0 || l >= P->L || n < 0 || (n && !ids) || !out_expert || !out_slot || !n_copy)
        return EDGE0_EINVAL;
    auto& Ly = P->layers[l];
    std::vector<unsigned char> want(P->E, 0);
    for (int i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= P->E) return EDGE0_EINVAL;
        want[ids[i]] = 1;
    }
    const LayerState S = Ly.state();
    reclaim_failed(S, P->n_slots);
    const int now = ++Ly.meta[MT_CLK];
    long long rq = 0, h = 0;
    const int nj = plan_request(want.data(), P->E, P->n_slots, S, now, nullptr, &rq, &h);
    P->stat[ST_REQUESTS] += rq;
    P->stat[ST_HITS] += h;
    P->stat[ST_PLANNED] += nj;
    for (int k = 0; k < nj; ++k) {
        out_expert[k] = Ly.job_e[k];
        out_slot[k] = Ly.job_s[k];
    }
    *n_copy = nj;
    return EDGE0_OK;
}

extern "C" int edge0_pool_host_prefetch(edge0_pool* P, const int32_t* const* ids, int n) {
    if (!P || P->device || !ids || n < 0 || !layers_set(P)) return EDGE0_EINVAL;
    const int gen = ++P->gen;
    std::vector<unsigned char> want(P->E);
    for (int l = 0; l < P->L; ++l) {
        if (!ids[l]) continue;
        auto& Ly = P->layers[l];
        if (Ly.meta[MT_BUSY]) {
            ++P->stat[ST_SKIPPED];
            continue;
        }
        std::fill(want.begin(), want.end(), 0);
        for (int i = 0; i < n; ++i) {
            const int e = ids[l][i];
            if (e >= 0 && e < P->E)
                want[e] = 1;
            else
                ++P->stat[ST_BAD_IDS];
        }
        const LayerState S = Ly.state();
        reclaim_failed(S, P->n_slots);
        const int now = ++Ly.meta[MT_CLK];
        long long rq = 0, h = 0;
        const int nj = plan_request(want.data(), P->E, P->n_slots, S, now, Ly.dev_table, &rq, &h);
        P->stat[ST_REQUESTS] += rq;
        P->stat[ST_HITS] += h;
        Ly.meta[MT_SEQ0] = (int)(P->stat[ST_PLANNED] & 0x7FFFFFFF);
        P->stat[ST_PLANNED] += nj;
        Ly.meta[MT_NJ] = nj;
        Ly.meta[MT_GEN] = gen;
        Ly.meta[MT_BUSY] = 1;
    }
    return EDGE0_OK;
}

extern "C" int edge0_pool_host_copy(edge0_pool* P) {
    if (!P || P->device || !layers_set(P)) return EDGE0_EINVAL;
    for (auto& Ly : P->layers) {
        if (!Ly.meta[MT_BUSY]) continue;
        for (int k = 0; k < Ly.meta[MT_NJ]; ++k) {
            const int e = Ly.job_e[k], s = Ly.job_s[k];
            if (injected_failure((long long)Ly.meta[MT_SEQ0] + k, P->fail_every)) {
                Ly.fail[s] = 1;
                ++P->stat[ST_FAILED];
                continue;
            }
            memcpy(Ly.dev_gu + (size_t)s * P->gu_bytes, Ly.host_gu + (size_t)e * P->gu_bytes, P->gu_bytes);
            memcpy(Ly.dev_dn + (size_t)s * P->dn_bytes, Ly.host_dn + (size_t)e * P->dn_bytes, P->dn_bytes);
            Ly.dev_table[e] = s;
            ++P->stat[ST_PUBLISHED];
            P->stat[ST_BYTES] += (long long)(P->gu_bytes + P->dn_bytes);
        }
        Ly.meta[MT_BUSY] = 0;
    }
    return EDGE0_OK;
}

// ---------------------------------------------------------- device mode ----
extern "C" int edge0_pool_device_init(edge0_pool* P) {
    if (!P || P->device || !layers_set(P)) return EDGE0_EINVAL;
    const int L = P->L, E = P->E, S = P->n_slots;
    auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
    size_t o = 0;
    const size_t o_stat = o;  o += al(ST_COUNT * 8 + 16);
    const size_t o_ly = o;    o += al(sizeof(PoolLayerDev) * L);
    const size_t o_meta = o;  o += al((size_t)L * MT_COUNT * 4);
    const size_t o_slot = o;  o += al((size_t)L * E * 4);
    const size_t o_arr = o;   o += al((size_t)L * S * 4) * 7;   // expert_in, used, fail, job_e, job_s, done
    char* base = nullptr;
    if (cudaMalloc(&base, o) != cudaSuccess) return EDGE0_ECUDA;
    std::vector<char> img(o, 0);
    std::vector<PoolLayerDev> ly(L);
    for (int l = 0; l < L; ++l) {
        const auto& Y = P->layers[l];
        ly[l] = PoolLayerDev{Y.host_gu, Y.host_dn, Y.dev_gu, Y.dev_dn, Y.dev_table};
    }
    memcpy(img.data() + o_ly, ly.data(), sizeof(PoolLayerDev) * L);
    // empty pool: every map entry -1
    memset(img.data() + o_slot, 0xFF, (size_t)L * E * 4);
    const size_t arr = al((size_t)L * S * 4);
    memset(img.data() + o_arr, 0xFF, arr);   // expert_in
    std::vector<int32_t> empty(E, -1);
    int rc = EDGE0_OK;
    if (cudaMemcpy(base, img.data(), o, cudaMemcpyHostToDevice) != cudaSuccess) rc = EDGE0_ECUDA;
    for (int l = 0; l < L && rc == EDGE0_OK; ++l)
        if (cudaMemcpy(P->layers[l].dev_table, empty.data(), (size_t)E * 4, cudaMemcpyHostToDevice) != cudaSuccess)
            rc = EDGE0_ECUDA;
    if (rc == EDGE0_OK && (cudaEventCreateWithFlags(&P->planned, cudaEventDisableTiming) != cudaSuccess ||
                           cudaEventCreateWithFlags(&P->copied, cudaEventDisableTiming) != cudaSuccess))
        rc = EDGE0_ECUDA;
    if (rc != EDGE0_OK) {
        if (P->planned) cudaEventDestroy(P->planned);
        P->planned = nullptr;
        cudaFree(base);
        return rc;
    }
    PoolDevP& d = P->dp;
    d.stat = reinterpret_cast<unsigned long long*>(base + o_stat);
    d.exit_cnt = reinterpret_cast<unsigned*>(base + o_stat + ST_COUNT * 8);
    d.ly = reinterpret_cast<PoolLayerDev*>(base + o_ly);
    d.meta = reinterpret_cast<int*>(base + o_meta);
    d.slot_of = reinterpret_cast<int*>(base + o_slot);
    d.expert_in = reinterpret_cast<int*>(base + o_arr);
    d.used = reinterpret_cast<int*>(base + o_arr + arr);
    d.fail = reinterpret_cast<int*>(base + o_arr + 2 * arr);
    d.job_e = reinterpret_cast<int*>(base + o_arr + 3 * arr);
    d.job_s = reinterpret_cast<int*>(base + o_arr + 4 * arr);
    d.done = reinterpret_cast<unsigned*>(base + o_arr + 5 * arr);
    d.L = L;
    d.E = E;
    d.S = S;
    d.gu_bytes = (long long)P->gu_bytes;
    d.dn_bytes = (long long)P->dn_bytes;
    P->dmem = base;
    P->device = true;
    for (auto& Ly : P->layers) {   // the host copies of the state are no longer used
        std::fill(Ly.slot_of.begin(), Ly.slot_of.end(), -1);
        std::fill(Ly.expert_in.begin(), Ly.expert_in.end(), -1);
    }
    memset(P->stat, 0, sizeof(P->stat));
    return EDGE0_OK;
}

extern "C" int edge0_pool_prefetch_async(edge0_pool* P, const int32_t* const* ids, int n, cudaStream_t stream,
                                         cudaStream_t copy_stream) {
    if (!P || !P->device || !ids || n <= 0) return EDGE0_EINVAL;
    IdsP q;
    memset(&q, 0, sizeof(q));
    for (int l = 0; l < P->L; ++l) q.p[l] = ids[l];
    const int gen = ++P->gen;
    k_pool_plan<<<P->L, 256, (size_t)P->E, stream>>>(P->dp, q, n, gen);
    if (cudaGetLastError() != cudaSuccess) return EDGE0_ECUDA;
    if (cudaEventRecord(P->planned, stream) != cudaSuccess ||
        cudaStreamWaitEvent(copy_stream, P->planned, 0) != cudaSuccess)
        return EDGE0_ECUDA;
    k_pool_copy<<<kCopyCtas, kCopyThreads, 0, copy_stream>>>(P->dp, gen, P->fail_every, P->delay_ns);
    if (cudaGetLastError() != cudaSuccess || cudaEventRecord(P->copied, copy_stream) != cudaSuccess)
        return EDGE0_ECUDA;
    return EDGE0_OK;
}

extern "C" int edge0_pool_wait(edge0_pool* P, unsigned long long timeout_ns) {
    if (!P || !P->device) return EDGE0_EINVAL;
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        const cudaError_t q = cudaEventQuery(P->copied);
        if (q == cudaSuccess) return EDGE0_OK;
        if (q != cudaErrorNotReady) return EDGE0_ECUDA;
        const auto ns = std::chrono::duration_cast<std::chrono::nanoseconds>(std::chrono::steady_clock::now() - t0);
        if ((unsigned long long)ns.count() >= timeout_ns) return EDGE0_ETIMEOUT;
        std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
}

extern "C" int edge0_pool_inject(edge0_pool* P, int fail_every, unsigned long long delay_ns) {
    if (!P || fail_every < 0 || delay_ns > kMaxDelayNs) return EDGE0_EINVAL;
    P->fail_every = fail_every;
    P->delay_ns = delay_ns;
    return EDGE0_OK;
}

// ------------------------------------------------------------- read-out ----
extern "C" int edge0_pool_stats_ex(const edge0_pool* P, long long* out, int n) {
    if (!P || !out || n < ST_COUNT) return EDGE0_EINVAL;
    if (!P->device) {
        for (int i = 0; i < ST_COUNT; ++i) out[i] = P->stat[i];
        return EDGE0_OK;
    }
    unsigned long long v[ST_COUNT];
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(v, P->dp.stat, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
        return EDGE0_ECUDA;
    for (int i = 0; i < ST_COUNT; ++i) out[i] = (long long)v[i];
    return EDGE0_OK;
}

extern "C" int edge0_pool_stats(const edge0_pool* P, long long* hits, long long* copies) {
    long long v[ST_COUNT];
    const int rc = edge0_pool_stats_ex(P, v, ST_COUNT);
    if (rc) return rc;
    if (hits) *hits = v[ST_HITS];
    if (copies) *copies = v[ST_PLANNED];
    return EDGE0_OK;
}

extern "C" int edge0_pool_resident(const edge0_pool* P, int l, int32_t* slot_of) {
    if (!P || l < 0 || l >= P->L || !slot_of) return EDGE0_EINVAL;
    if (!P->device) {
        for (int e = 0; e < P->E; ++e) slot_of[e] = P->layers[l].slot_of[e];
        return EDGE0_OK;
    }
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(slot_of, P->layers[l].dev_table, (size_t)P->E * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        return EDGE0_ECUDA;
    return EDGE0_OK;
}
