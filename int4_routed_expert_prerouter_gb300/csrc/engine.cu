// Persistent decode engine: one CTA per SM, 16 consumer warps + 1 producer warp.
//
// A decode step is a sequence of phases separated by grid barriers:
//   R (own-routed layers, or step 0): router GEMV -> logits
//   A: gate/up of the routed experts and the shared expert, LoRA A x, head
//      fc1[:, :d] x and linear_init[:, :d] x
//   B: down of the routed experts (weighted by w) and the shared expert (+ LoRA
//      down), head fc2 gelu(z) (+ linear_init and the one-hot columns)
// Every phase's work is a list of "segments" (one packed matrix, or one expert's
// matrix) cut into 576-byte int4 / 2048-byte fp16 units; each CTA takes a
// contiguous byte range of the phase.  The producer warp builds each phase's
// segment and chunk list once, publishes it to the consumers through a ring of
// list slots, and streams the CTA's units (and small auxiliary tensors) into a
// ring of shared-memory stages with bulk copies as soon as the routing that
// selects them is known -- for prerouted layers that is at step start, so
// weight traffic runs ahead across grid barriers.  Consumer warps read each unit
// once from shared memory and do the dot products on the tensor cores
// (m16n8k16, fp32 accumulate) with the int4 nibbles turned into fp16 subnormals
// by a single mask (q * 2^-24); each warp adds its partial sums into a per-phase
// shared-memory accumulator without CTA-wide synchronisation, and the CTA flushes
// it to fp32 accumulators in global memory once per phase.
#include "internal.cuh"

namespace edge0 {

enum PhaseKind : int { PH_R = 0, PH_A = 1, PH_B = 2 };
enum SrcKind : int { SRC_X = 0, SRC_ACT = 1, SRC_ACTSH = 2, SRC_GELU = 3 };
enum OutKind : int {
    OUT_GUG, OUT_GUU, OUT_GUSG, OUT_GUSU, OUT_AG, OUT_AU, OUT_Z, OUT_LIN, OUT_Y, OUT_LOGR, OUT_LOGH
};
enum ExtraKind : int { EX_NONE = 0, EX_LORA_DOWN = 1, EX_HEAD = 2 };
enum AuxKind : int { AUX_UNITS = 0, AUX_BG, AUX_BU, AUX_AD, AUX_BD, AUX_FC1OH, AUX_LINOH };

struct Seg {
    const char* base;
    int off;           // byte offset of the segment in the phase
    int kind;          // 0 int4, 1 fp16
    int n_rt, n_g, rows, ub;
    int src, out, expert, extra;
    int cu0, cu1;      // this CTA's units of the segment
};

struct Chunk {
    int aux, seg, u0, u1, tok, bytes;
    int sacc;          // unit chunks: first accumulator row of the chunk
};

constexpr int kMaxChunk = 48;
constexpr int kListSlots = 4;
constexpr int kSaccRowsPhase = 1024;   // accumulator rows of one CTA in one phase
constexpr int kBdBytes = 8192;         // LoRA-down B rows of one CTA in one phase
constexpr unsigned long long kTimeoutNs = 2000000000ull;   // bounded waits: 2 s

// one phase's work of this CTA, built by the producer and read by the consumers
struct PhaseList {
    int seq;           // phase index + 1 once published
    int nseg, nch, sacc_rows;
    int has_sh, has_head, bd_row0, bd_rows;
    Seg seg[kMaxSeg];
    Chunk ch[kMaxChunk];
};

// ------------------------------------------------------------ smem plan ----
struct Plan {
    int stage, full, empty, xf, xsum, actf, actsum, ashf, ashsum, gf, gsum, ash32, gsh, ush, aacc,
        v, zsm, linsm, lx, hs, rscr, sacc, bd, lists, ids, wts, ready, red, ctl, total;
};

__host__ __device__ inline int al(int x, int a) { return (x + a - 1) / a * a; }

__host__ __device__ inline Plan make_plan(int L, int B, int K, int d, int E, int I, int Is, int H,
                                          int r) {
    Plan p;
    const int R16 = ceil_div(r, 16) * 16;
    int o = 0;
    p.stage = o;  o += kStages * kStageBytes;
    p.full = o;   o += 8 * kStages;
    p.empty = o;  o += 8 * kStages;
    o = al(o, 16);
    p.xf = o;     o += al(B * d * 2, 16);
    p.xsum = o;   o += al(B * (d / kGroup) * 4, 16);
    // activation sources keep a hi and a lo fragment array (see put_group)
    p.actf = o;   o += al(2 * B * K * I * 2, 16);
    p.actsum = o; o += al(2 * B * K * (I / kGroup) * 4, 16);
    p.ashf = o;   o += al(2 * B * Is * 2, 16);
    p.ashsum = o; o += al(2 * B * (Is / kGroup) * 4, 16);
    p.gf = o;     o += al(2 * B * H * 2, 16);
    p.gsum = o;   o += al(2 * B * (H / kGroup) * 4, 16);
    p.ash32 = o;  o += al(B * Is * 4, 16);
    p.gsh = o;    o += al(B * Is * 4, 16);
    p.ush = o;    o += al(B * Is * 4, 16);
    p.aacc = o;   o += al(B * 2 * R16 * 4, 16);
    p.v = o;      o += al(B * R16 * 4, 16);
    p.zsm = o;    o += al(B * H * 4, 16);
    p.linsm = o;  o += al(B * E * 4, 16);
    p.lx = o;     o += al(B * E * 4, 16);
    p.hs = o;     o += al(B * d * 2, 16);
    p.rscr = o;   o += al(B * 2 * E * 4, 16);
    p.sacc = o;   o += al(kSaccRowsPhase * B * 4, 16);
    p.bd = o;     o += kBdBytes;
    p.lists = o;  o += al(kListSlots * (int)sizeof(PhaseList), 16);
    p.ids = o;    o += al(L * B * K * 4, 16);
    p.wts = o;    o += al(L * B * K * 4, 16);
    p.ready = o;  o += al(L * 4, 16);
    p.red = o;    o += al(B * kConsumerWarps * 4 + 64, 16);
    p.ctl = o;    o += 64;
    p.total = o;
    return p;
}

// ------------------------------------------------------------ helpers -----
__device__ __forceinline__ unsigned long long now_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// shared control words
struct Ctl {
    int trace;        // record phase timestamps
    int tslot;        // next trace slot
    int abort;        // CTA-local: give up
    int step;
    unsigned pc0;
    int issued;       // chunks issued by the producer
    int cdone;        // phases the consumers have finished
};

__device__ void raise_error(WsHeader* hdr, Ctl* ctl, int code) {
    atomicCAS(&hdr->error, 0, code);
    atomicExch(&hdr->abort, 1);
    ctl->abort = 1;
}

__device__ __forceinline__ bool should_abort(WsHeader* hdr, Ctl* ctl) {
    return *(volatile int*)&ctl->abort || ld_volatile_s32(&hdr->abort);
}

// wait on an mbarrier phase with a time bound; false on abort/timeout
__device__ bool mbar_wait(uint64_t* bar, uint32_t parity, WsHeader* hdr, Ctl* ctl) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = now_ns();
    for (unsigned it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 63) {
            if (should_abort(hdr, ctl)) return false;
            if (now_ns() - t0 > kTimeoutNs) {
                raise_error(hdr, ctl, EDGE0_ETIMEOUT);
                return false;
            }
        }
    }
}

// spin until *flag >= want (shared memory, written by the other role); bounded
__device__ bool wait_flag(volatile int* flag, int want, WsHeader* hdr, Ctl* ctl) {
    if (*flag >= want) return true;
    const unsigned long long t0 = now_ns();
    for (unsigned it = 0; *flag < want; ++it) {
        __nanosleep(32);
        if ((it & 63) == 63) {
            if (should_abort(hdr, ctl)) return false;
            if (now_ns() - t0 > kTimeoutNs) {
                raise_error(hdr, ctl, EDGE0_ETIMEOUT);
                return false;
            }
        }
    }
    return true;
}

// ---------------------------------------------------------- routing -----
// top-K over `score` (E values in shared/global memory) by one warp, value
// descending, lower index first on ties; masked entries are -inf.
__device__ void warp_topk(const float* score, int E, int K, int* ids, int lane) {
    unsigned taken[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) taken[i] = 0;
    for (int k = 0; k < K; ++k) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int i = 0; i < 16; ++i) {
            const int e = lane + 32 * i;
            if (e >= E || taken[i]) continue;
            const float v = score[e];
            if (v > bv || (v == bv && e < bi)) { bv = v; bi = e; }
        }
#pragma unroll
        for (int s = 16; s; s >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, s);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, s);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (bi == 0x7fffffff) bi = 0;   // fewer than K candidates (not reachable for valid shapes)
        if ((bi & 31) == lane) taken[bi >> 5] = 1;
        if (lane == 0) ids[k] = bi;
        __syncwarp();
    }
}

// Routing rule of App. A, one token per warp.  logits: E fp32 (global or shared);
// scratch: 2 * E floats of shared memory for this warp.
__device__ void warp_route(const float* logits, int E, int K, int kind, int n_groups, int G,
                           float scale, const float* bias, float* scratch, int* ids, float* w,
                           int lane) {
    float* sel = scratch;
    float* sig = scratch + E;
    if (kind == EDGE0_ROUTE_SIGMOID_GROUP) {
        for (int e = lane; e < E; e += 32) {
            const float s = 1.0f / (1.0f + expf(-logits[e]));
            sig[e] = s;
            sel[e] = bias ? s + bias[e] : s;
        }
        __syncwarp();
        const int per = E / n_groups;
        // group scores: sum of the two largest selection scores of each group
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
        unsigned gtaken = 0;
        for (int k = 0; k < G; ++k) {
            float bv = (lane < n_groups && !((gtaken >> lane) & 1)) ? gscore : -INFINITY;
            int bi = (lane < n_groups && !((gtaken >> lane) & 1)) ? lane : 0x7fffffff;
#pragma unroll
            for (int s = 16; s; s >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, s);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, s);
                if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
            }
            if (bi < 32) { gtaken |= 1u << bi; keep |= 1u << bi; }
        }
        __syncwarp();
        for (int e = lane; e < E; e += 32)
            if (!((keep >> (e / per)) & 1)) sel[e] = -INFINITY;
        __syncwarp();
        warp_topk(sel, E, K, ids, lane);
        __syncwarp();
        if (lane == 0) {
            float sum = 0.0f;
            for (int k = 0; k < K; ++k) sum += sig[ids[k]];
            for (int k = 0; k < K; ++k) w[k] = scale * sig[ids[k]] / (sum + 1e-20f);
        }
    } else {
        for (int e = lane; e < E; e += 32) sel[e] = bias ? logits[e] + bias[e] : logits[e];
        __syncwarp();
        warp_topk(sel, E, K, ids, lane);
        __syncwarp();
        if (lane == 0) {
            const float mx = sel[ids[0]];
            float sum = 0.0f;
            for (int k = 0; k < K; ++k) sum += expf(sel[ids[k]] - mx);
            for (int k = 0; k < K; ++k) w[k] = expf(sel[ids[k]] - mx) / sum;
        }
    }
    __syncwarp();
}

// ------------------------------------------------------------ context -----
struct Ctx {
    const Prog* p;
    char* sm;
    Plan pl;
    WsHeader* hdr;
    Ctl* ctl;
    AccLayout acc;
    int nct, cta;
    int step;
    int R16;
};

__device__ __forceinline__ float* acc_set(const Ctx& c, unsigned pc) {
    return reinterpret_cast<float*>(c.p->ws + kWsHeaderBytes) + (long long)(pc % 3) * c.acc.total;
}
__device__ __forceinline__ __half* hbuf(const Ctx& c, int i) {
    return reinterpret_cast<__half*>(c.p->ws + kWsHeaderBytes + 3 * c.acc.total * 4) +
           (long long)i * c.p->B * c.p->d;
}

// optional phase trace: slot i of this CTA <- globaltimer (thread 0 only)
__device__ __forceinline__ unsigned long long* trace_area(const Ctx& c) {
    const char* base = c.p->ws + kWsHeaderBytes + 3 * c.acc.total * 4 + 2LL * c.p->B * c.p->d * 2 + 256;
    return reinterpret_cast<unsigned long long*>(const_cast<char*>(base)) + (long long)c.cta * kTraceSlots;
}

// record (tag, globaltimer) when tracing is on; consumer thread 0 only
__device__ __forceinline__ void stamp(const Ctx& c, int tag) {
    if (threadIdx.x != 0 || !c.ctl->trace) return;
    if (c.ctl->trace >= 2 && (tag & 0xF0000) == 0 && (tag & 0xF) > 4) return;
    const int s = c.ctl->tslot;
    if (s + 2 > kTraceSlots) return;
    unsigned long long* a = trace_area(c);
    a[s] = (unsigned long long)tag;
    a[s + 1] = now_ns();
    c.ctl->tslot = s + 2;
}

// detailed stamps for one two-layer window (trace mode >= 2: window starts at layer mode - 2)
__device__ __forceinline__ void dstamp(const Ctx& c, int l, int tag) {
    const int m = c.ctl->trace;
    if (m >= 2 && l >= m - 2 && l <= m - 1) stamp(c, tag);
}

__device__ __forceinline__ int* sm_ids(const Ctx& c, int l) {
    return reinterpret_cast<int*>(c.sm + c.pl.ids) + l * c.p->B * c.p->K;
}
__device__ __forceinline__ float* sm_w(const Ctx& c, int l) {
    return reinterpret_cast<float*>(c.sm + c.pl.wts) + l * c.p->B * c.p->K;
}
__device__ __forceinline__ PhaseList* list_slot(const Ctx& c, int pi) {
    return reinterpret_cast<PhaseList*>(c.sm + c.pl.lists) + (pi % kListSlots);
}

__device__ __forceinline__ bool has_router_phase(const Prog& p, int l, int step) {
    return p.mode == MODE_DECODE && (!(p.layers[l].flags & LF_PREROUTED) || step == 0);
}

__device__ __forceinline__ int expert_slot(const LayerP& Ly, int e) {
    return Ly.slot_table ? Ly.slot_table[e] : e;
}

__device__ __forceinline__ int units_of(int kind, int bytes) {   // ceil(bytes / unit)
    return kind ? (bytes + kF16Unit - 1) >> 11 : (bytes + kQ4Unit - 1) / kQ4Unit;
}

// Build the segment list of phase `ph` of layer l into L->seg (deterministic).
// Returns the phase's byte total, or -1 for an expert id or slot out of range.
__device__ int build_segments(const Ctx& c, int l, int ph, const int* ids, PhaseList* Lp) {
    const Prog& p = *c.p;
    const LayerP& Ly = p.layers[l];
    const int B = p.B, K = p.K, d = p.d, E = p.E, I = p.I, Is = p.Is, H = p.H, r = p.r;
    int n = 0;
    int off = 0;
    Seg* S = Lp->seg;
    auto add = [&](const char* base, int kind, int rows, int in, int src, int out, int expert,
                   int extra) {
        if (n >= kMaxSeg) return;
        Seg& s = S[n++];
        s.base = base;
        s.kind = kind;
        s.n_rt = ceil_div(rows, kRowTile);
        s.n_g = in / kGroup;
        s.rows = rows;
        s.ub = kind ? kF16Unit : kQ4Unit;
        s.src = src;
        s.out = out;
        s.expert = expert;
        s.extra = extra;
        s.off = off;
        off += s.n_rt * s.n_g * s.ub;
    };
    const bool moe_phase = p.mode != MODE_HEAD;
    const bool head = (p.mode == MODE_HEAD) || (p.mode == MODE_DECODE && (Ly.flags & LF_HEAD));
    const bool lora = p.mode == MODE_DECODE && (Ly.flags & LF_LORA);
    const bool shared = moe_phase && (Ly.flags & LF_SHARED);
    if (ph == PH_R) {
        add(Ly.router, 1, E, d, SRC_X, OUT_LOGR, -1, EX_NONE);
    } else {
        // distinct routed experts in order of first appearance over (b, k)
        if (moe_phase) {
            for (int i = 0; i < B * K; ++i) {
                const int e = ids[i];
                bool seen = false;
                for (int j = 0; j < i; ++j) seen |= (ids[j] == e);
                if (seen) continue;
                if (e < 0 || e >= E) return -1;
                const long long slot = expert_slot(Ly, e);
                if (slot < 0 || slot >= Ly.n_slots) return -1;
                if (ph == PH_A) {
                    add(Ly.gate + slot * q4_bytes(I, d), 0, I, d, SRC_X, OUT_GUG, e, EX_NONE);
                    add(Ly.up + slot * q4_bytes(I, d), 0, I, d, SRC_X, OUT_GUU, e, EX_NONE);
                } else {
                    add(Ly.down + slot * q4_bytes(d, I), 0, d, I, SRC_ACT, OUT_Y, e, EX_NONE);
                }
            }
        }
        if (ph == PH_A) {
            if (shared) {
                add(Ly.sh_gate, 0, Is, d, SRC_X, OUT_GUSG, -1, EX_NONE);
                add(Ly.sh_up, 0, Is, d, SRC_X, OUT_GUSU, -1, EX_NONE);
            }
            if (shared && lora) {
                add(Ly.lora_Ag, 1, r, d, SRC_X, OUT_AG, -1, EX_NONE);
                add(Ly.lora_Au, 1, r, d, SRC_X, OUT_AU, -1, EX_NONE);
            }
            if (head) {
                add(Ly.fc1, 1, H, d, SRC_X, OUT_Z, -1, EX_NONE);
                add(Ly.linit, 1, E, d, SRC_X, OUT_LIN, -1, EX_NONE);
            }
        } else {
            if (shared)
                add(Ly.sh_down, 0, d, Is, SRC_ACTSH, OUT_Y, -1, lora ? EX_LORA_DOWN : EX_NONE);
            if (head) add(Ly.fc2, 1, E, H, SRC_GELU, OUT_LOGH, -1, EX_HEAD);
        }
    }
    Lp->nseg = n;
    return off;
}

// Build this CTA's chunk list of a phase (after build_segments).  Auxiliary
// chunks precede the segment that needs them.  n_prev: rows of the previous
// token's mask (0 or K).  Returns 0, or an EDGE0_* status.
__device__ int build_chunks(const Ctx& c, int total, int n_prev, PhaseList* Lp) {
    const Prog& p = *c.p;
    const int lo = (int)((long long)total * c.cta / c.nct);
    const int hi = (int)((long long)total * (c.cta + 1) / c.nct);
    int n = 0, rows = 0;
    bool over = false;
    // every chunk is written once, whole
    auto push = [&](int aux, int seg, int u0, int u1, int tok, int bytes, int sacc_row) {
        if (n >= kMaxChunk) { over = true; return; }
        Chunk v;
        v.aux = aux; v.seg = seg; v.u0 = u0; v.u1 = u1; v.tok = tok; v.bytes = bytes;
        v.sacc = sacc_row;
        Lp->ch[n] = v;
        ++n;
    };
    Lp->has_sh = 0;
    Lp->has_head = 0;
    Lp->bd_row0 = 0;
    Lp->bd_rows = 0;
    for (int s = 0; s < Lp->nseg; ++s) {
        Seg& S = Lp->seg[s];
        const int nu = S.n_rt * S.n_g;
        int a = lo - S.off, b = hi - S.off;
        a = a <= 0 ? 0 : units_of(S.kind, a);
        b = b <= 0 ? 0 : units_of(S.kind, b);
        const int u0 = a < nu ? a : nu, u1 = b < nu ? b : nu;
        S.cu0 = u0;
        S.cu1 = u1;
        if (u0 >= u1) continue;
        if (S.src == SRC_ACTSH) Lp->has_sh = 1;
        if (S.src == SRC_GELU) Lp->has_head = 1;
        if (S.extra == EX_LORA_DOWN) {
            push(AUX_BG, s, 0, 0, 0, p.Is * p.r * 2, 0);
            push(AUX_BU, s, 0, 0, 0, p.Is * p.r * 2, 0);
            push(AUX_AD, s, 0, 0, 0, (int)f16_bytes(p.r, p.Is), 0);
            // B_d rows of the row tiles whose group-0 unit belongs to this CTA
            const int ng = S.n_g;
            const int rt_a = (u0 + ng - 1) / ng, rt_b = (u1 - 1) / ng;   // inclusive
            if (rt_a <= rt_b) {
                const int row0 = rt_a * kRowTile;
                int row1 = (rt_b + 1) * kRowTile;
                if (row1 > p.d) row1 = p.d;
                if ((row1 - row0) * p.r * 2 > kBdBytes) return EDGE0_EUNSUPPORTED;
                Lp->bd_row0 = row0;
                Lp->bd_rows = row1 - row0;
                push(AUX_BD, s, rt_a, rt_b + 1, 0, (row1 - row0) * p.r * 2, 0);
            }
        }
        if (S.extra == EX_HEAD) {
            for (int t = 0; t < p.B; ++t) push(AUX_FC1OH, s, 0, 0, t, (p.K + n_prev) * p.H * 2, 0);
            for (int t = 0; t < p.B; ++t) push(AUX_LINOH, s, 0, 0, t, (p.K + n_prev) * p.E * 2, 0);
        }
        int cap = kStageBytes / S.ub;
        if (cap > 30 * S.n_g) cap = 30 * S.n_g;     // a chunk spans at most 32 row tiles
        for (int x = u0; x < u1; x += cap) {
            const int y = x + cap < u1 ? x + cap : u1;
            push(AUX_UNITS, s, x, y, 0, (y - x) * S.ub, rows);
            rows += ((y - 1) / S.n_g - x / S.n_g + 1) * kRowTile;
        }
    }
    if (over || rows > kSaccRowsPhase) return EDGE0_EUNSUPPORTED;
    Lp->nch = n;
    Lp->sacc_rows = rows;
    return EDGE0_OK;
}

// ------------------------------------------------------------ producer -----
__device__ void producer(Ctx& c) {
    const Prog& p = *c.p;
    Ctl* ctl = c.ctl;
    uint64_t* full = reinterpret_cast<uint64_t*>(c.sm + c.pl.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(c.sm + c.pl.empty);
    volatile int* ready = reinterpret_cast<volatile int*>(c.sm + c.pl.ready);
    const uint64_t pol = policy_evict_first();
    const int step = c.step;
    int stage = 0;
    uint32_t round = 0;
    int issued = 0;
    int pi = 0;

    for (int l = 0; l < p.L; ++l) {
        const LayerP& Ly = p.layers[l];
        for (int ph = PH_R; ph <= PH_B; ++ph) {
            if (ph == PH_R && !has_router_phase(p, l, step)) continue;
            // the list slot is free once the consumers finished phase pi - kListSlots
            if (!wait_flag(&ctl->cdone, pi - kListSlots + 1, c.hdr, ctl)) return;
            if (ph != PH_R) {
                if (!wait_flag(&ready[l], 1, c.hdr, ctl)) return;
                __threadfence_block();
            }
            PhaseList* Lp = list_slot(c, pi);
            const int* ids = sm_ids(c, l);
            const int total = build_segments(c, l, ph, ids, Lp);
            if (total < 0) { raise_error(c.hdr, ctl, EDGE0_EINVAL); return; }
            // previous-token mask rows for the head's one-hot columns
            const int32_t* prev = nullptr;
            if (p.mode == MODE_HEAD) prev = p.prev_in;
            else if (p.mode == MODE_DECODE && step > 0)
                prev = p.exec_ids + (((long long)((step - 1) & 1) * p.Ls + Ly.sidx) * p.B) * p.K;
            const int n_prev = prev ? p.K : 0;
            for (int i = 0; i < n_prev * p.B; ++i)
                if (prev[i] < 0 || prev[i] >= p.E) { raise_error(c.hdr, ctl, EDGE0_EINVAL); return; }
            if (ph != PH_R)
                for (int i = 0; i < p.K * p.B; ++i)
                    if (ids[i] < 0 || ids[i] >= p.E) { raise_error(c.hdr, ctl, EDGE0_EINVAL); return; }
            const int rc = build_chunks(c, total, n_prev, Lp);
            if (rc) { raise_error(c.hdr, ctl, rc); return; }
            __threadfence_block();
            *(volatile int*)&Lp->seq = pi + 1;
            for (int i = 0; i < Lp->nch; ++i) {
                const Chunk& x = Lp->ch[i];
                if (!mbar_wait(&empty[stage], (round & 1) ^ 1, c.hdr, ctl)) return;
                char* dst = c.sm + c.pl.stage + stage * kStageBytes;
                mbar_arrive_expect_tx(&full[stage], (uint32_t)x.bytes);
                const Seg& s = Lp->seg[x.seg];
                switch (x.aux) {
                    case AUX_UNITS:
                        bulk_g2s(dst, s.base + (long long)x.u0 * s.ub, x.bytes, &full[stage], pol);
                        break;
                    case AUX_BG:
                        bulk_g2s(dst, Ly.lora_Bg, x.bytes, &full[stage], pol);
                        break;
                    case AUX_BU:
                        bulk_g2s(dst, Ly.lora_Bu, x.bytes, &full[stage], pol);
                        break;
                    case AUX_AD:
                        bulk_g2s(dst, Ly.lora_Ad, x.bytes, &full[stage], pol);
                        break;
                    case AUX_BD:
                        bulk_g2s(dst, Ly.lora_Bd + (long long)x.u0 * kRowTile * p.r, x.bytes,
                                 &full[stage], pol);
                        break;
                    case AUX_FC1OH:
                    case AUX_LINOH: {
                        const bool f = x.aux == AUX_FC1OH;
                        const int rowlen = f ? p.H : p.E;
                        const __half* tab = f ? Ly.fc1_oh : Ly.linit_oh;
                        const int* ex = ids + x.tok * p.K;
                        for (int k = 0; k < p.K; ++k)
                            bulk_g2s(dst + k * rowlen * 2, tab + (long long)ex[k] * rowlen,
                                     rowlen * 2, &full[stage], pol);
                        for (int k = 0; k < n_prev; ++k)
                            bulk_g2s(dst + (p.K + k) * rowlen * 2,
                                     tab + (long long)(p.E + prev[x.tok * p.K + k]) * rowlen,
                                     rowlen * 2, &full[stage], pol);
                        break;
                    }
                }
                ++issued;
                *(volatile int*)&ctl->issued = issued;
                if (++stage == kStages) { stage = 0; ++round; }
            }
            ++pi;
        }
    }
}

// ------------------------------------------------------------ consumers ----
__device__ __forceinline__ void cbar() { named_bar_sync(1, kConsumerThreads); }

__device__ __forceinline__ bool aborted(const Ctx& c) { return *(volatile int*)&c.ctl->abort != 0; }

// grid-wide barrier among the consumer warps of all CTAs
__device__ bool grid_barrier(Ctx& c, unsigned long long& target) {
    cbar();
    bool ok = true;
    if (threadIdx.x == 0) {
        __threadfence();
        red_release_add_u64(&c.hdr->barrier, 1ull);
        target += (unsigned long long)c.nct;
        if (ld_acquire_u64(&c.hdr->barrier) < target) {
            const unsigned long long t0 = now_ns();
            for (unsigned it = 0; ld_acquire_u64(&c.hdr->barrier) < target; ++it) {
                if ((it & 15) == 15) {
                    if (should_abort(c.hdr, c.ctl)) { ok = false; break; }
                    if (now_ns() - t0 > kTimeoutNs) { raise_error(c.hdr, c.ctl, EDGE0_ETIMEOUT); ok = false; break; }
                }
            }
        }
        if (!ok) c.ctl->abort = 1;
    }
    cbar();
    return !aborted(c);
}

// B-fragment / sum pointers of tensor-core column n of segment s (null when
// inactive).  Column n carries token n / 2: its hi part (n even) or its lo part
// (n odd, activation sources only; x is exactly fp16 and has no lo part).
__device__ __forceinline__ void col_src(const Ctx& c, const Seg& s, int l, int n, const __half** f,
                                        const float** sum) {
    const Prog& p = *c.p;
    *f = nullptr;
    *sum = nullptr;
    const int b = n >> 1, part = n & 1;
    if (b >= p.B) return;
    const char* sm = c.sm;
    switch (s.src) {
        case SRC_X:
            if (part) return;
            *f = reinterpret_cast<const __half*>(sm + c.pl.xf) + (long long)b * p.d;
            *sum = reinterpret_cast<const float*>(sm + c.pl.xsum) + b * (p.d / kGroup);
            break;
        case SRC_ACT: {
            const int* ids = sm_ids(c, l) + b * p.K;
            const long long npair = (long long)p.B * p.K;
            for (int k = 0; k < p.K; ++k)
                if (ids[k] == s.expert) {
                    const long long pr = b * p.K + k + part * npair;
                    *f = reinterpret_cast<const __half*>(sm + c.pl.actf) + pr * p.I;
                    *sum = reinterpret_cast<const float*>(sm + c.pl.actsum) + pr * (p.I / kGroup);
                    break;
                }
            break;
        }
        case SRC_ACTSH: {
            const long long r = b + part * p.B;
            *f = reinterpret_cast<const __half*>(sm + c.pl.ashf) + r * p.Is;
            *sum = reinterpret_cast<const float*>(sm + c.pl.ashsum) + r * (p.Is / kGroup);
            break;
        }
        default: {
            const long long r = b + part * p.B;
            *f = reinterpret_cast<const __half*>(sm + c.pl.gf) + r * p.H;
            *sum = reinterpret_cast<const float*>(sm + c.pl.gsum) + r * (p.H / kGroup);
            break;
        }
    }
}

// k slot of token b for routed segment s (-1: token does not use this expert)
__device__ __forceinline__ int col_kslot(const Ctx& c, const Seg& s, int l, int b) {
    if (s.expert < 0) return 0;
    const int* ids = sm_ids(c, l) + b * c.p->K;
    for (int k = 0; k < c.p->K; ++k)
        if (ids[k] == s.expert) return k;
    return -1;
}

__device__ __forceinline__ float* out_ptr(const Ctx& c, const Seg& s, float* F, int row, int b, int k) {
    const Prog& p = *c.p;
    const AccLayout& a = c.acc;
    switch (s.out) {
        case OUT_GUG: return F + a.gu + ((long long)(b * p.K + k) * 2 + 0) * p.I + row;
        case OUT_GUU: return F + a.gu + ((long long)(b * p.K + k) * 2 + 1) * p.I + row;
        case OUT_GUSG: return F + a.gus + ((long long)b * 2 + 0) * p.Is + row;
        case OUT_GUSU: return F + a.gus + ((long long)b * 2 + 1) * p.Is + row;
        case OUT_AG: return F + a.aacc + ((long long)b * 2 + 0) * c.R16 + row;
        case OUT_AU: return F + a.aacc + ((long long)b * 2 + 1) * c.R16 + row;
        case OUT_Z: return F + a.z + (long long)b * p.H + row;
        case OUT_LIN: return F + a.lin + (long long)b * p.E + row;
        case OUT_Y: return F + a.y + (long long)b * p.d + row;
        case OUT_LOGR: return F + a.logr + (long long)b * p.E + row;
        default: return F + a.logh + (long long)b * p.E + row;
    }
}

// ----------------------------------------------------------- prologues -----
// x = fp16(h rsqrt(mean h^2 + eps) gamma) for all tokens, written as B fragments.
// hsrc: fp16 [B, d]; ysrc: fp32 [B, d] added first (h = fp16(hsrc + ysrc)), or null.
// hdst: where CTA 0 stores the updated h (or null).  norm=false: x = hsrc.
__device__ void build_x(Ctx& c, const __half* hsrc, const float* ysrc, __half* hdst,
                        const __half* gamma, float eps, bool norm) {
    const Prog& p = *c.p;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int B = p.B, d = p.d;
    __half* xf = reinterpret_cast<__half*>(c.sm + c.pl.xf);
    float* xsum = reinterpret_cast<float*>(c.sm + c.pl.xsum);
    float* red = reinterpret_cast<float*>(c.sm + c.pl.red);
    __half* hs = reinterpret_cast<__half*>(c.sm + c.pl.hs);   // the (updated) h, fp16
    float ss[EDGE0_MAX_BATCH];
#pragma unroll
    for (int b = 0; b < EDGE0_MAX_BATCH; ++b) ss[b] = 0.f;
    for (int i = tid; i < B * d; i += kConsumerThreads) {
        float v = __half2float(hsrc[i]);
        if (ysrc) v += ysrc[i];
        const __half hv = __float2half_rn(v);
        hs[i] = hv;
        if (hdst && c.cta == 0) hdst[i] = hv;
        const float f = __half2float(hv);
        const int b = i / d;
#pragma unroll
        for (int bb = 0; bb < EDGE0_MAX_BATCH; ++bb)
            if (bb == b) ss[bb] += f * f;
    }
    if (norm) {
        for (int b = 0; b < B; ++b) {
            float s = ss[b];
#pragma unroll
            for (int k = 16; k; k >>= 1) s += __shfl_xor_sync(0xffffffffu, s, k);
            if (lane == 0) red[b * kConsumerWarps + wid] = s;
        }
    }
    cbar();
    float* rs = red + B * kConsumerWarps;
    if (norm && tid < B) {
        float s = 0.f;
        for (int w = 0; w < kConsumerWarps; ++w) s += red[tid * kConsumerWarps + w];
        rs[tid] = rsqrtf(s / (float)d + eps);
    }
    cbar();
    const int ng = d / kGroup;
    for (int it = wid; it < B * ng; it += kConsumerWarps) {
        const int b = it / ng, grp = it - b * ng;
        const int i0 = grp * kGroup + lane, i1 = i0 + 32;
        float v0 = __half2float(hs[b * d + i0]), v1 = __half2float(hs[b * d + i1]);
        if (norm) {
            const float r = rs[b];
            v0 = __half2float(__float2half_rn(v0 * r * (gamma ? __half2float(gamma[i0]) : 1.0f)));
            v1 = __half2float(__float2half_rn(v1 * r * (gamma ? __half2float(gamma[i1]) : 1.0f)));
        }
        put_group(xf + (long long)b * d + grp * kGroup, xsum + b * ng + grp, v0, v1, lane);
    }
    cbar();
}

// zero this CTA's slice of accumulator set (pc % 3)
__device__ void zero_set_slice(const Ctx& c, unsigned pc) {
    float* F = acc_set(c, pc);
    const long long n = c.acc.total;
    const long long a = n * c.cta / c.nct, b = n * (c.cta + 1) / c.nct;
    for (long long i = a + threadIdx.x; i < b; i += kConsumerThreads) F[i] = 0.f;
}

// top-K of a finished head: logits in set `pc`, written to pred[step & 1][target]
__device__ void head_topk(Ctx& c, int l, unsigned pc) {
    const Prog& p = *c.p;
    const LayerP& Ly = p.layers[l];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    float* F = acc_set(c, pc);
    float* scr = reinterpret_cast<float*>(c.sm + c.pl.rscr);   // 2E floats per token
    for (int b = wid; b < p.B; b += kConsumerWarps) {
        __shared__ int tids[EDGE0_MAX_BATCH][EDGE0_MAX_K];
        __shared__ float tw[EDGE0_MAX_BATCH][EDGE0_MAX_K];
        warp_route(F + c.acc.logh + (long long)b * p.E, p.E, p.K, Ly.head_route_kind, Ly.head_n_groups,
                   Ly.head_topk_groups, Ly.head_route_scale, Ly.head_bias,
                   scr + (long long)b * 2 * p.E, tids[b], tw[b], lane);
        if (lane < p.K) {
            if (p.mode == MODE_HEAD) {
                p.out_ids[b * p.K + lane] = tids[b][lane];
                p.out_w[b * p.K + lane] = tw[b][lane];
            } else {
                const long long o = (((long long)(c.step & 1) * p.Ls + Ly.head_target) * p.B + b) * p.K + lane;
                p.pred_ids[o] = tids[b][lane];
                p.pred_w[o] = tw[b][lane];
            }
        }
        __syncwarp();
    }
}

// One warp computes units [ua, ub) of segment s held in `stage` (chunk starting
// at unit cu0) and adds its per-row partial sums into the accumulator rows sacc
// (relative to row tile rt0, B columns).
__device__ void warp_units(const Ctx& c, const Seg& s, int l, const char* stage, int cu0, int ua,
                           int ub, float* sacc, int rt0) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int B = c.p->B;
    const __half* bf;
    const float* dummy;
    col_src(c, s, l, g, &bf, &dummy);
    const float* sum0;
    const float* sum1;
    const __half* f0;
    const __half* f1;
    col_src(c, s, l, 2 * t, &f0, &sum0);
    col_src(c, s, l, 2 * t + 1, &f1, &sum1);
    const bool q4 = s.kind == 0;
    const int ng = s.n_g;
    int cur = -1;
    float y[4] = {0.f, 0.f, 0.f, 0.f};
    float lo[4] = {0.f, 0.f, 0.f, 0.f}, hi[4] = {0.f, 0.f, 0.f, 0.f};
    auto flush = [&](int rt) {
        float vg, vg8;   // token t: hi column + lo column
        if (!q4) {
#pragma unroll
            for (int i = 0; i < 4; ++i) { y[i] = lo[i] + 16.0f * hi[i]; lo[i] = 0.f; hi[i] = 0.f; }
            vg = y[0] + kLoInv * y[1];
            vg8 = y[2] + kLoInv * y[3];
        } else {
            vg = y[0] + y[1];
            vg8 = y[2] + y[3];
        }
        const int r0 = (rt - rt0) * kRowTile + g;
        if (t < B) {
            atomicAdd(&sacc[r0 * B + t], vg);
            atomicAdd(&sacc[(r0 + 8) * B + t], vg8);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) y[i] = 0.f;
    };
    int rt = ua / ng, grp = ua - rt * ng;
    for (int u = ua; u < ub; ++u) {
        if (rt != cur) {
            if (cur >= 0) flush(cur);
            cur = rt;
        }
        const char* unit = stage + (u - cu0) * s.ub;
        uint4 b0 = make_uint4(0, 0, 0, 0), b1 = make_uint4(0, 0, 0, 0);
        if (bf) {
            const uint4* bp = reinterpret_cast<const uint4*>(bf + (grp * 4 + t) * 16);
            b0 = bp[0];
            b1 = bp[1];
        }
        if (q4) {
            const uint4 wv = *reinterpret_cast<const uint4*>(unit + 16 * lane);
            const uint2 sc = *reinterpret_cast<const uint2*>(unit + 512 + 8 * g);
            float a4[4] = {0.f, 0.f, 0.f, 0.f};
            constexpr uint32_t M0 = 0x000F000Fu, M1 = 0x00F000F0u;
            const uint32_t x8 = wv.x >> 8, z8 = wv.z >> 8, y8 = wv.y >> 8, w8 = wv.w >> 8;
            uint32_t a[4];
            a[0] = wv.x & M0; a[1] = wv.z & M0; a[2] = x8 & M0; a[3] = z8 & M0;
            mma_16816(a4, a, b0.x, b0.y);
            a[0] = wv.x & M1; a[1] = wv.z & M1; a[2] = x8 & M1; a[3] = z8 & M1;
            mma_16816(a4, a, b0.z, b0.w);
            a[0] = wv.y & M0; a[1] = wv.w & M0; a[2] = y8 & M0; a[3] = w8 & M0;
            mma_16816(a4, a, b1.x, b1.y);
            a[0] = wv.y & M1; a[1] = wv.w & M1; a[2] = y8 & M1; a[3] = w8 & M1;
            mma_16816(a4, a, b1.z, b1.w);
            const __half2 sb0 = *reinterpret_cast<const __half2*>(&sc.x);
            const __half2 sb1 = *reinterpret_cast<const __half2*>(&sc.y);
            const float sg = __low2float(sb0) * 16777216.0f, bg = __high2float(sb0);
            const float sg8 = __low2float(sb1) * 16777216.0f, bg8 = __high2float(sb1);
            const float xs0 = sum0 ? sum0[grp] : 0.f, xs1 = sum1 ? sum1[grp] : 0.f;
            // column 2t: hi part of token t; column 2t+1: lo part (scaled by 2^11)
            y[0] += sg * a4[0] + bg * xs0;
            y[1] += sg * kLoInv * a4[1] + bg * xs1;
            y[2] += sg8 * a4[2] + bg8 * xs0;
            y[3] += sg8 * kLoInv * a4[3] + bg8 * xs1;
        } else {
            const uint4 a0 = *reinterpret_cast<const uint4*>(unit + 0 * 512 + 16 * lane);
            const uint4 a1 = *reinterpret_cast<const uint4*>(unit + 1 * 512 + 16 * lane);
            const uint4 a2 = *reinterpret_cast<const uint4*>(unit + 2 * 512 + 16 * lane);
            const uint4 a3 = *reinterpret_cast<const uint4*>(unit + 3 * 512 + 16 * lane);
            uint32_t a[4];
            a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
            mma_16816(lo, a, b0.x, b0.y);
            a[0] = a1.x; a[1] = a1.y; a[2] = a1.z; a[3] = a1.w;
            mma_16816(hi, a, b0.z, b0.w);
            a[0] = a2.x; a[1] = a2.y; a[2] = a2.z; a[3] = a2.w;
            mma_16816(lo, a, b1.x, b1.y);
            a[0] = a3.x; a[1] = a3.y; a[2] = a3.z; a[3] = a3.w;
            mma_16816(hi, a, b1.z, b1.w);
        }
        if (++grp == ng) { grp = 0; ++rt; }
    }
    if (cur >= 0) flush(cur);
}

// act = silu(g) u of every routed pair whose down segment has units in this CTA
__device__ void build_act(Ctx& c, int l, const PhaseList* Lp, unsigned pcA) {
    const Prog& p = *c.p;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const float* F = acc_set(c, pcA);
    __half* actf = reinterpret_cast<__half*>(c.sm + c.pl.actf);
    float* actsum = reinterpret_cast<float*>(c.sm + c.pl.actsum);
    const int ng = p.I / kGroup;
    const int* ids = sm_ids(c, l);
    const long long npair = (long long)p.B * p.K;
    for (int it = wid; it < p.B * p.K * ng; it += kConsumerWarps) {
        const int pair = it / ng, grp = it - pair * ng;
        const int e = ids[pair];
        bool need = false;
        for (int s = 0; s < Lp->nseg; ++s)
            if (Lp->seg[s].out == OUT_Y && Lp->seg[s].expert == e)
                need = Lp->seg[s].cu0 < Lp->seg[s].cu1;
        if (!need) continue;
        const float* gp = F + c.acc.gu + (long long)pair * 2 * p.I;
        const int i0 = grp * kGroup + lane, i1 = i0 + 32;
        const float a0 = silu_f(gp[i0]) * gp[p.I + i0];
        const float a1 = silu_f(gp[i1]) * gp[p.I + i1];
        put_group(actf + (long long)pair * p.I + grp * kGroup, actsum + pair * ng + grp, a0, a1, lane,
                  actf + (pair + npair) * p.I + grp * kGroup, actsum + (pair + npair) * ng + grp);
    }
}

// ------------------------------------------------------------ the kernel ---
__global__ void __launch_bounds__(kThreads, 1) engine_kernel(const __grid_constant__ Prog prog) {
    extern __shared__ __align__(128) char smem[];
    Ctx c;
    c.sm = smem;
    c.pl = make_plan(prog.L, prog.B, prog.K, prog.d, prog.E, prog.I, prog.Is, prog.H, prog.r);
    c.p = &prog;
    c.hdr = reinterpret_cast<WsHeader*>(prog.ws);
    c.ctl = reinterpret_cast<Ctl*>(smem + c.pl.ctl);
    c.acc = acc_layout(prog.B, prog.K, prog.I, prog.Is, prog.r, prog.H, prog.E, prog.d);
    c.nct = gridDim.x;
    c.cta = blockIdx.x;
    c.R16 = ceil_div(prog.r, 16) * 16;
    const int tid = threadIdx.x;
    const Prog& p = *c.p;

    if (tid == 0) {
        c.ctl->abort = 0;
        c.ctl->issued = 0;
        c.ctl->cdone = 0;
        c.ctl->step = p.step >= 0 ? p.step : ld_volatile_s32(&c.hdr->step);
        c.ctl->pc0 = *(volatile unsigned*)&c.hdr->pc;
        c.ctl->trace = c.cta < kTraceCtas ? ld_volatile_s32(&c.hdr->trace) : 0;
        c.ctl->tslot = 0;
        uint64_t* full = reinterpret_cast<uint64_t*>(smem + c.pl.full);
        uint64_t* empty = reinterpret_cast<uint64_t*>(smem + c.pl.empty);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_mbar_init();
    }
    {
        int* ready = reinterpret_cast<int*>(smem + c.pl.ready);
        for (int l = tid; l < p.L; l += kThreads) ready[l] = 0;
        for (int i = tid; i < kListSlots; i += kThreads)
            reinterpret_cast<PhaseList*>(smem + c.pl.lists)[i].seq = 0;
        float* sacc = reinterpret_cast<float*>(smem + c.pl.sacc);
        for (int i = tid; i < kSaccRowsPhase * p.B; i += kThreads) sacc[i] = 0.f;
    }
    __syncthreads();
    c.step = c.ctl->step;
    // routing known at launch: predictions (prerouted layers, step > 0) or inputs
    {
        int* ready = reinterpret_cast<int*>(smem + c.pl.ready);
        const int BK = p.B * p.K;
        for (int l = 0; l < p.L; ++l) {
            const LayerP& Ly = p.layers[l];
            const int* src_i = nullptr;
            const float* src_w = nullptr;
            if (p.mode == MODE_DECODE && (Ly.flags & LF_PREROUTED) && c.step > 0) {
                const long long o = (((long long)((c.step - 1) & 1) * p.Ls + Ly.sidx) * p.B) * p.K;
                src_i = p.pred_ids + o;
                src_w = p.pred_w + o;
            } else if (p.mode == MODE_MOE) {
                src_i = p.ids_in;
                src_w = p.w_in;
            } else if (p.mode == MODE_HEAD) {
                src_i = p.exec_in;
            }
            if (!src_i) continue;
            for (int i = tid; i < BK; i += kThreads) {
                sm_ids(c, l)[i] = src_i[i];
                sm_w(c, l)[i] = src_w ? src_w[i] : 0.f;
            }
            if (tid == 0) ready[l] = 1;
        }
    }
    __syncthreads();

    if (tid >= kConsumerThreads) {
        if (tid == kConsumerThreads) producer(c);
        return;
    }

    // ------------------------------------------------------ consumer side --
    const int lane = tid & 31, wid = tid >> 5;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + c.pl.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + c.pl.empty);
    float* sacc = reinterpret_cast<float*>(smem + c.pl.sacc);
    volatile int* ready = reinterpret_cast<volatile int*>(smem + c.pl.ready);
    const int B = p.B;
    unsigned long long bar_target = 0;
    if (tid == 0) {
        const unsigned long long v = ld_acquire_u64(&c.hdr->barrier);
        bar_target = v - v % (unsigned long long)c.nct;
    }
    unsigned pc = c.ctl->pc0;
    int stage = 0;
    uint32_t round = 0;
    int consumed = 0;
    int pi = 0;
    unsigned pc_prevB = 0;        // phase of the previous layer's B (y, head logits)
    bool prev_head = false;        // previous layer's head logits await top-K
    int prev_layer = -1;
    cbar();

    for (int l = 0; l < p.L && !aborted(c); ++l) {
        const LayerP& Ly = p.layers[l];
        const bool decode = p.mode == MODE_DECODE;
        unsigned pcR = 0;
        const bool rphase = has_router_phase(p, l, c.step);
        for (int ph = PH_R; ph <= PH_B; ++ph) {
            if (ph == PH_R && !rphase) continue;
            // ---------------- prologue
            const int ttag = (l << 8) | (ph << 4);
            stamp(c, ttag | 0);
            zero_set_slice(c, pc + 1);
            dstamp(c, l, 0x10000 | ttag | 1);
            const bool first_of_layer = (ph == PH_R) || (ph == PH_A && !rphase);
            if (first_of_layer) {
                if (decode) {
                    const __half* hs = (l <= 1) ? p.h_io : hbuf(c, (l - 1) & 1);
                    const float* ys = l == 0 ? nullptr : acc_set(c, pc_prevB) + c.acc.y;
                    build_x(c, hs, ys, l == 0 ? nullptr : hbuf(c, l & 1), Ly.gamma, Ly.eps, true);
                } else {
                    build_x(c, p.x_in, nullptr, nullptr, nullptr, 0.f, false);
                }
                if (prev_head && c.cta == c.nct - 1) head_topk(c, prev_layer, pc_prevB);
                prev_head = false;
            }
            dstamp(c, l, 0x10000 | ttag | 2);
            if (ph == PH_R) pcR = pc;
            if (ph == PH_A && rphase) {
                // own routing from the router logits of phase R
                const float* F = acc_set(c, pcR);
                float* scr = reinterpret_cast<float*>(smem + c.pl.rscr);
                for (int b = wid; b < B; b += kConsumerWarps) {
                    __shared__ int rid[EDGE0_MAX_BATCH][EDGE0_MAX_K];
                    __shared__ float rw[EDGE0_MAX_BATCH][EDGE0_MAX_K];
                    warp_route(F + c.acc.logr + (long long)b * p.E, p.E, p.K, Ly.route_kind, Ly.n_groups,
                               Ly.topk_groups, Ly.route_scale, Ly.bias, scr + (long long)b * 2 * p.E,
                               rid[b], rw[b], lane);
                    if (lane < p.K) {
                        sm_ids(c, l)[b * p.K + lane] = rid[b][lane];
                        sm_w(c, l)[b * p.K + lane] = rw[b][lane];
                    }
                }
                cbar();
                if (tid == 0) {
                    __threadfence_block();
                    ready[l] = 1;
                }
            }
            if (ph == PH_A && decode && c.cta == 0) {
                for (int i = tid; i < B * p.K; i += kConsumerThreads)
                    p.exec_ids[(((long long)(c.step & 1) * p.Ls + Ly.sidx) * B) * p.K + i] = sm_ids(c, l)[i];
            }
            // this phase's list, published by the producer
            PhaseList* Lp = list_slot(c, pi);
            dstamp(c, l, 0x10000 | ttag | 3);
            if (tid == 0) wait_flag(&Lp->seq, pi + 1, c.hdr, c.ctl);
            cbar();
            dstamp(c, l, 0x10000 | ttag | 4);
            if (aborted(c)) break;
            if (Lp->seq != pi + 1) break;
            float* F = acc_set(c, pc);
            const float* FA = acc_set(c, pc - 1);     // phase A results (valid in phase B)
            if (ph == PH_B) {
                build_act(c, l, Lp, pc - 1);
                if (Lp->has_sh) {
                    float* gsh = reinterpret_cast<float*>(smem + c.pl.gsh);
                    float* ush = reinterpret_cast<float*>(smem + c.pl.ush);
                    float* aacc = reinterpret_cast<float*>(smem + c.pl.aacc);
                    for (int i = tid; i < B * p.Is; i += kConsumerThreads) {
                        const int b = i / p.Is, j = i - b * p.Is;
                        gsh[i] = FA[c.acc.gus + ((long long)b * 2) * p.Is + j];
                        ush[i] = FA[c.acc.gus + ((long long)b * 2 + 1) * p.Is + j];
                    }
                    for (int i = tid; i < B * 2 * c.R16; i += kConsumerThreads) aacc[i] = FA[c.acc.aacc + i];
                    const bool lora = decode && (Ly.flags & LF_LORA);
                    if (!lora) {
                        cbar();
                        __half* ashf = reinterpret_cast<__half*>(smem + c.pl.ashf);
                        float* ashsum = reinterpret_cast<float*>(smem + c.pl.ashsum);
                        const int ng = p.Is / kGroup;
                        for (int it = wid; it < B * ng; it += kConsumerWarps) {
                            const int b = it / ng, grp = it - b * ng;
                            const int i0 = b * p.Is + grp * kGroup + lane, i1 = i0 + 32;
                            put_group(ashf + (long long)b * p.Is + grp * kGroup, ashsum + b * ng + grp,
                                      silu_f(gsh[i0]) * ush[i0], silu_f(gsh[i1]) * ush[i1], lane,
                                      ashf + (long long)(b + B) * p.Is + grp * kGroup,
                                      ashsum + (b + B) * ng + grp);
                        }
                    }
                }
                if (Lp->has_head) {
                    float* zsm = reinterpret_cast<float*>(smem + c.pl.zsm);
                    float* linsm = reinterpret_cast<float*>(smem + c.pl.linsm);
                    for (int i = tid; i < B * p.H; i += kConsumerThreads) zsm[i] = FA[c.acc.z + i];
                    for (int i = tid; i < B * p.E; i += kConsumerThreads) linsm[i] = FA[c.acc.lin + i];
                }
                cbar();
            }
            // ---------------- chunk loop
            stamp(c, ttag | 1);
            const __half* held_bg = nullptr;
            int held_bg_stage = -1;
            for (int i = 0; i < Lp->nch; ++i) {
                const Chunk x = Lp->ch[i];
                const int st = stage;
                if (!mbar_wait(&full[st], round & 1, c.hdr, c.ctl)) { c.ctl->abort = 1; break; }
                dstamp(c, l, 0x20000 | (i << 8) | (ph << 4) | x.aux);
                const char* buf = smem + c.pl.stage + st * kStageBytes;
                const Seg& s = Lp->seg[x.seg];
                bool release = true;
                if (x.aux == AUX_UNITS) {
                    // each warp takes a contiguous share of the chunk's units; no CTA sync
                    const int n = x.u1 - x.u0;
                    const int ua = x.u0 + (n * wid) / kConsumerWarps;
                    const int ub2 = x.u0 + (n * (wid + 1)) / kConsumerWarps;
                    if (ua < ub2)
                        warp_units(c, s, l, buf, x.u0, ua, ub2, sacc + x.sacc * B, x.u0 / s.n_g);
                    __syncwarp();
                } else if (x.aux == AUX_BG) {
                    held_bg = reinterpret_cast<const __half*>(buf);
                    held_bg_stage = st;
                    release = false;
                } else if (x.aux == AUX_BU) {
                    // act_s = silu(g + (a/r) Bg ag) * (u + (a/r) Bu au), fp32 copy + fragments
                    cbar();
                    const __half* Bu = reinterpret_cast<const __half*>(buf);
                    const float* gsh = reinterpret_cast<const float*>(smem + c.pl.gsh);
                    const float* ush = reinterpret_cast<const float*>(smem + c.pl.ush);
                    const float* aacc = reinterpret_cast<const float*>(smem + c.pl.aacc);
                    float* ash32 = reinterpret_cast<float*>(smem + c.pl.ash32);
                    for (int j = tid; j < B * p.Is; j += kConsumerThreads) {
                        const int b = j / p.Is, row = j - b * p.Is;
                        const float* ag = aacc + (b * 2) * c.R16;
                        const float* au = aacc + (b * 2 + 1) * c.R16;
                        float dg = 0.f, du = 0.f;
                        for (int q = 0; q < p.r; ++q) {
                            dg += __half2float(held_bg[row * p.r + q]) * ag[q];
                            du += __half2float(Bu[row * p.r + q]) * au[q];
                        }
                        const float gg = gsh[j] + Ly.lora_scale * dg;
                        const float uu = ush[j] + Ly.lora_scale * du;
                        ash32[j] = silu_f(gg) * uu;
                    }
                    cbar();
                    __half* ashf = reinterpret_cast<__half*>(smem + c.pl.ashf);
                    float* ashsum = reinterpret_cast<float*>(smem + c.pl.ashsum);
                    const int ng = p.Is / kGroup;
                    for (int it = wid; it < B * ng; it += kConsumerWarps) {
                        const int b = it / ng, grp = it - b * ng;
                        const int i0 = b * p.Is + grp * kGroup + lane;
                        put_group(ashf + (long long)b * p.Is + grp * kGroup, ashsum + b * ng + grp,
                                  ash32[i0], ash32[i0 + 32], lane,
                                  ashf + (long long)(b + B) * p.Is + grp * kGroup,
                                  ashsum + (b + B) * ng + grp);
                    }
                    cbar();
                    if (lane == 0) mbar_arrive(&empty[held_bg_stage]);
                    held_bg = nullptr;
                } else if (x.aux == AUX_AD) {
                    // v = A_d act_s (r rows), warp 0 on the tensor cores
                    float* v = reinterpret_cast<float*>(smem + c.pl.v);
                    float* tmp = reinterpret_cast<float*>(smem + c.pl.rscr);   // 16 x B scratch
                    if (wid == 0) {
                        Seg sa;
                        sa.base = nullptr; sa.off = 0; sa.kind = 1;
                        sa.n_rt = ceil_div(p.r, kRowTile); sa.n_g = p.Is / kGroup; sa.rows = p.r;
                        sa.ub = kF16Unit; sa.src = SRC_ACTSH; sa.out = 0; sa.expert = -1; sa.extra = 0;
                        sa.cu0 = 0; sa.cu1 = 0;
                        for (int q = lane; q < kRowTile * sa.n_rt * B; q += 32) tmp[q] = 0.f;
                        __syncwarp();
                        warp_units(c, sa, l, buf, 0, 0, sa.n_rt * sa.n_g, tmp, 0);
                        __syncwarp();
                        for (int q = lane; q < c.R16 * B; q += 32) {
                            const int row = q / B, b = q - row * B;
                            v[b * c.R16 + row] = row < p.r ? tmp[q] : 0.f;
                        }
                    }
                    cbar();
                } else if (x.aux == AUX_BD) {
                    // this CTA's B_d rows, kept for the phase-end flush
                    const uint4* src = reinterpret_cast<const uint4*>(buf);
                    uint4* dst = reinterpret_cast<uint4*>(smem + c.pl.bd);
                    for (int q = tid; q < x.bytes / 16; q += kConsumerThreads) dst[q] = src[q];
                    cbar();
                } else if (x.aux == AUX_FC1OH) {
                    // gelu(z + one-hot columns) fragments for token x.tok
                    const __half* rows = reinterpret_cast<const __half*>(buf);
                    const int nrows = x.bytes / (p.H * 2);
                    const float* zsm = reinterpret_cast<const float*>(smem + c.pl.zsm) + x.tok * p.H;
                    __half* gf = reinterpret_cast<__half*>(smem + c.pl.gf) + (long long)x.tok * p.H;
                    float* gsum = reinterpret_cast<float*>(smem + c.pl.gsum) + x.tok * (p.H / kGroup);
                    __half* gfl = gf + (long long)B * p.H;
                    float* gsuml = gsum + B * (p.H / kGroup);
                    for (int grp = wid; grp < p.H / kGroup; grp += kConsumerWarps) {
                        const int i0 = grp * kGroup + lane, i1 = i0 + 32;
                        float z0 = zsm[i0], z1 = zsm[i1];
                        for (int q = 0; q < nrows; ++q) {
                            z0 += __half2float(rows[q * p.H + i0]);
                            z1 += __half2float(rows[q * p.H + i1]);
                        }
                        const float g0 = 0.5f * z0 * (1.0f + erff(z0 * 0.70710678118654752f));
                        const float g1 = 0.5f * z1 * (1.0f + erff(z1 * 0.70710678118654752f));
                        put_group(gf + grp * kGroup, gsum + grp, g0, g1, lane, gfl + grp * kGroup,
                                  gsuml + grp);
                    }
                    cbar();
                } else if (x.aux == AUX_LINOH) {
                    const __half* rows = reinterpret_cast<const __half*>(buf);
                    const int nrows = x.bytes / (p.E * 2);
                    const float* linsm = reinterpret_cast<const float*>(smem + c.pl.linsm) + x.tok * p.E;
                    float* lx = reinterpret_cast<float*>(smem + c.pl.lx) + x.tok * p.E;
                    for (int e = tid; e < p.E; e += kConsumerThreads) {
                        float v = linsm[e];
                        for (int q = 0; q < nrows; ++q) v += __half2float(rows[q * p.E + e]);
                        lx[e] = v;
                    }
                    cbar();
                }
                if (release && lane == 0) mbar_arrive(&empty[st]);
                dstamp(c, l, 0x30000 | (i << 8) | (ph << 4) | x.aux);
                if (++stage == kStages) { stage = 0; ++round; }
                ++consumed;
            }
            cbar();
            if (aborted(c)) break;
            // ---------------- flush this phase's accumulator rows to global memory
            stamp(c, ttag | 2);
            float wcol[EDGE0_MAX_BATCH];
            int kcol[EDGE0_MAX_BATCH];
            for (int i = 0; i < Lp->nch; ++i) {
                const Chunk& x = Lp->ch[i];
                if (x.aux != AUX_UNITS) continue;
                const Seg& s = Lp->seg[x.seg];
                const int rt0 = x.u0 / s.n_g, rt1 = (x.u1 - 1) / s.n_g;
                const int nrows = (rt1 - rt0 + 1) * kRowTile;
                for (int b = 0; b < B; ++b) {
                    kcol[b] = col_kslot(c, s, l, b);
                    wcol[b] = (s.out == OUT_Y && s.expert >= 0 && kcol[b] >= 0) ? sm_w(c, l)[b * p.K + kcol[b]] : 1.f;
                }
                float* sa = sacc + x.sacc * B;
                for (int q = tid; q < nrows * B; q += kConsumerThreads) {
                    const int rl = q / B, b = q - rl * B;
                    const int rt = rt0 + (rl >> 4);
                    const int row = rt * kRowTile + (rl & 15);
                    float val = sa[q];
                    sa[q] = 0.f;
                    if (row >= s.rows || kcol[b] < 0) continue;
                    const bool own0 = (rt * s.n_g >= x.u0) && (rt * s.n_g < x.u1);
                    if (own0 && s.extra == EX_LORA_DOWN) {
                        const __half* bd = reinterpret_cast<const __half*>(smem + c.pl.bd) +
                                           (long long)(row - Lp->bd_row0) * p.r;
                        const float* v = reinterpret_cast<const float*>(smem + c.pl.v) + b * c.R16;
                        float dsum = 0.f;
                        for (int j = 0; j < p.r; ++j) dsum += __half2float(bd[j]) * v[j];
                        val += Ly.lora_scale * dsum;
                    }
                    if (own0 && s.extra == EX_HEAD)
                        val += reinterpret_cast<const float*>(smem + c.pl.lx)[b * p.E + row];
                    red_add_f32(out_ptr(c, s, F, row, b, kcol[b]), val * wcol[b]);
                }
            }
            dstamp(c, l, 0x10000 | ttag | 5);
            cbar();
            if (tid == 0) *(volatile int*)&c.ctl->cdone = pi + 1;
            // ---------------- end of phase
            stamp(c, ttag | 3);
            if (!grid_barrier(c, bar_target)) break;
            stamp(c, ttag | 4);
            if (ph == PH_B) {
                pc_prevB = pc;
                prev_head = (p.mode != MODE_MOE) && (p.mode == MODE_HEAD || (Ly.flags & LF_HEAD));
                prev_layer = l;
            }
            ++pc;
            ++pi;
        }
    }

    if (!aborted(c)) {
        // ---------------- tail
        const float* Y = acc_set(c, pc_prevB) + c.acc.y;
        if (p.mode == MODE_DECODE) {
            const __half* hs = (p.L <= 1) ? p.h_io : hbuf(c, (p.L - 1) & 1);
            const long long n = (long long)B * p.d;
            const long long a = n * c.cta / c.nct, b = n * (c.cta + 1) / c.nct;
            // h_L = fp16(h_{L-1} + y); h_{L-1} of a single-layer call is h_io itself
            for (long long i = a + tid; i < b; i += kConsumerThreads)
                p.h_io[i] = __float2half_rn(__half2float(hs[i]) + Y[i]);
        } else if (p.mode == MODE_MOE) {
            const long long n = (long long)B * p.d;
            const long long a = n * c.cta / c.nct, b = n * (c.cta + 1) / c.nct;
            for (long long i = a + tid; i < b; i += kConsumerThreads) p.y_out[i] = __float2half_rn(Y[i]);
        }
        if (p.mode == MODE_HEAD && p.out_logits) {
            const float* Lg = acc_set(c, pc_prevB) + c.acc.logh;
            const long long n = (long long)B * p.E;
            const long long a = n * c.cta / c.nct, b = n * (c.cta + 1) / c.nct;
            for (long long i = a + tid; i < b; i += kConsumerThreads) p.out_logits[i] = Lg[i];
        }
        if (prev_head && c.cta == c.nct - 1) head_topk(c, prev_layer, pc_prevB);
        if (c.cta == 0 && tid == 0) {
            c.hdr->pc = pc;
            if (p.step < 0) c.hdr->step = c.step + 1;
        }
    } else if (tid == 0) {
        // drain copies still in flight before the CTA exits (bounded)
        const int issued = *(volatile int*)&c.ctl->issued;
        const unsigned long long t0 = now_ns();
        for (int k = consumed; k < issued; ++k) {
            while (!mbar_try_wait(&full[stage], round & 1))
                if (now_ns() - t0 > 100000000ull) break;
            if (++stage == kStages) { stage = 0; ++round; }
        }
    }
}

int engine_smem_bytes(const Prog& p) {
    return make_plan(p.L, p.B, p.K, p.d, p.E, p.I, p.Is, p.H, p.r).total;
}

}  // namespace edge0
