// Persistent decode engine: one CTA per SM in clusters of two ("pairs"); 16
// consumer warps + 1 producer warp per CTA.
//
// Dependencies of one decode layer ("The Other Half of the Memory Wall", S3.1
// "Math contract", S3.2 "Head", S3.3):
//   x = RMSNorm(h)                         needs all of the previous layer's y
//   gate/up rows of each expert            need all of x
//   down rows                              need all of act = silu(gate) * up
//   y = sum_k w_k down_k act_k + shared    -> next layer
//   head(x, executed, previous) -> top-K   needed only at the next token
// The engine takes ONE grid-wide synchronisation per layer (plus one after the
// router on own-routed layers):
//   * every expert (and the shared expert) is cut into half-row tiles of 8
//     act rows ("hr"); the packed gate/up tile of an hr interleaves its 8 gate
//     rows with its 8 up rows, so one tensor-core row tile yields gate and up of
//     the same act rows in the same lane;
//   * each CTA pair owns a contiguous run of hr over the flattened (shared,
//     routed slot 0, 1, ...) list; the two CTAs split d in halves, compute
//     partial gate/up sums for all of the pair's rows, swap them through
//     distributed shared memory (st.async + mbarrier), then each forms act for
//     all the pair's rows and applies the matching 16-column slices of down
//     (packed K-major) to its half of the output rows, adding w-weighted
//     partial sums into y with vector reductions;
//   * the shared expert's LoRA runs inside the pairs that own shared rows: A x
//     and v = A_down act are summed in small global accumulators, and the
//     same pairs apply B_down (split over the output rows) once v is complete;
//   * every prerouter head of the step runs in one flush after the last layer
//     (a head's prediction is consumed one token later); its logits accumulate
//     in global memory and the last CTA to finish its tasks computes the top-K.
// The producer warp streams each CTA's weight slices into a byte ring of shared
// memory with bulk copies as soon as the routing that selects them is known
// (prerouted layers: at step start, so the stream runs ahead across barriers).
// int4 nibbles enter m16n8k16 tensor-core steps as fp16 subnormals (q * 2^-24)
// through single masks; activations travel as hi + lo fp16 columns.
#include <string.h>

#include <mutex>

#include "internal.cuh"
#include "common.cuh"

namespace edge0 {

constexpr int kMaxSegs = 4;        // expert runs in one pair's share of a layer
constexpr int kMaxItems = 64;      // copy items of one CTA in one layer
constexpr int kItemMax = 16384;    // bytes of one copy item (copies of 16 KB reach full HBM rate)
constexpr int kSlots = 256;        // item barriers (>= 2 x kMaxItems)
constexpr int kTables = 3;         // layer tables in flight
constexpr int kMaxChunks = 4;      // 4-element chunks of [B, d] per consumer thread
constexpr int kVWarp = 15;         // consumer warp that forms the LoRA v of a CTA with shared rows
constexpr int kMaxD = 2048;
constexpr int kMinRing = 2 * kItemMax;

// Copy items.  Unit items (router, gate/up, LoRA A, fc1, linear_init) copy a run
// of n consecutive units of the CTA's half of the input groups, from unit b of
// the half (the run may cross row tiles).  Down items copy n consecutive 16-row
// steps (from step b of group a) over the CTA's half of the output rows (DQ),
// those followed by the group's scales (DQS, when the run ends at step 3), or the
// scales alone (DSC).
enum ItemKind : int {
    IT_ROUTER = 0, IT_GU, IT_LA, IT_LU, IT_BG, IT_BU, IT_DSC, IT_DQ, IT_DQS, IT_ADT, IT_BD, IT_FC1,
    IT_FC2, IT_LINIT
};
__host__ __device__ inline bool unit_kind(int k) {
    return k == IT_ROUTER || k == IT_GU || k == IT_LA || k == IT_LU || k == IT_FC1 || k == IT_LINIT;
}

// ------------------------------------------------------------------ plan ----
struct Seg {
    int slot;     // -1: shared expert; else routed slot (index into the layer's distinct experts)
    int hr0, hr1; // half-row tiles [hr0, hr1) of the expert
    int hoff;     // half-row tiles of the pair before this segment
    int q0, q1;   // 16-row act quarters [q0, q1) the segment touches
    int qoff;     // quarters of the pair before this segment
};

struct PairPlan {
    int nseg, over;
    Seg seg[kMaxSegs];
    int n_hr, n_q;
    int has_sh;   // the pair owns shared-expert rows
    int hd0, hd1; // head tasks (tables of the head flush)
    int ru0, ru1; // router units (in this rank's half of d)
    int la0, la1; // LoRA A units (A_gate then A_up groups of this rank's half of d)
    int bd0, bd1; // LoRA B_down row tiles (of this rank's half of the output rows)
};

// [n i / parts, n (i + 1) / parts): 32-bit arithmetic (n * parts < 2^31 for
// every split the engine makes; the host checks the shapes)
__host__ __device__ inline void split_range(int n, int parts, int i, int* a, int* b) {
    *a = n * i / parts;
    *b = n * (i + 1) / parts;
}

struct Shape {
    int d, I, Is, E, H, r;
    int n_slots;                // routed expert slots (0: none)
    int shared, lora, router;   // parts present in the layer
    int ps;                     // pairs that own shared-expert rows
};

// The shared expert's LoRA runs once per layer, not repeated by each pair that
// owns shared rows: those pairs compute A_gate x and A_up x (split over d) into a
// small global accumulator, wait for it to be complete before their act, and add
// v = A_down act of their rows into a second one (one warp, while the others run
// the down rows); after their down rows they apply B_down (split over the output
// rows) to the complete v.  The routed pairs carry no LoRA work.

__host__ __device__ inline int shared_pairs(int P, int n_sh, int n_rt, bool lora) {
    if (n_sh <= 0) return 0;
    if (n_rt <= 0) return P;
    // cost in int4-unit equivalents per CTA: an hr is 16 gate/up units + half a
    // 16-row down slice over half of d; shared pairs carry the LoRA A and v terms
    // and the wait for the A sums and the B_down rows
    int best = 0x7fffffff, pick = 1;
    for (int ps = 1; ps < P; ++ps) {
        const int cs = ceil_div(n_sh, ps) * 24 + (lora ? 20 : 0);
        const int cr = ceil_div(n_rt, P - ps) * 24;
        const int cmax = cs > cr ? cs : cr;
        if (cmax <= best) { best = cmax; pick = ps; }   // ties: more shared pairs
    }
    return pick;
}

__host__ __device__ inline int half_lo(int n, int rank) { return rank ? n / 2 : 0; }
__host__ __device__ inline int half_hi(int n, int rank) { return rank ? n : n / 2; }

__host__ __device__ inline void pair_plan(const Shape& S, int P, int pair, int rank, PairPlan& pp) {
    pp.nseg = 0;
    pp.over = 0;
    pp.n_hr = 0;
    pp.n_q = 0;
    pp.has_sh = 0;
    pp.hd0 = pp.hd1 = 0;
    pp.ru0 = pp.ru1 = 0;
    pp.la0 = pp.la1 = 0;
    pp.bd0 = pp.bd1 = 0;
    const int hpe = S.I / kHalfRow;
    const int n_sh = S.shared ? S.Is / kHalfRow : 0;
    const int n_rt = S.n_slots * hpe;
    const int Ps = S.ps;
    int a, b;
    if (pair < Ps) {
        split_range(n_sh, Ps, pair, &a, &b);
        if (a < b) {
            Seg& s = pp.seg[pp.nseg++];
            s.slot = -1; s.hr0 = a; s.hr1 = b; s.hoff = 0; s.q0 = a / 2; s.q1 = (b + 1) / 2; s.qoff = 0;
            pp.n_hr = b - a;
            pp.n_q = s.q1 - s.q0;
            pp.has_sh = 1;
        }
    } else if (P > Ps) {
        split_range(n_rt, P - Ps, pair - Ps, &a, &b);
        while (a < b) {
            const int slot = a / hpe;
            const int end = (slot + 1) * hpe < b ? (slot + 1) * hpe : b;
            if (pp.nseg >= kMaxSegs) { pp.over = 1; break; }
            Seg& s = pp.seg[pp.nseg++];
            s.slot = slot;
            s.hr0 = a - slot * hpe;
            s.hr1 = end - slot * hpe;
            s.hoff = pp.n_hr;
            s.q0 = s.hr0 / 2;
            s.q1 = (s.hr1 + 1) / 2;
            s.qoff = pp.n_q;
            pp.n_hr += s.hr1 - s.hr0;
            pp.n_q += s.q1 - s.q0;
            a = end;
        }
    }
    // LoRA (implies a shared expert, so Ps >= 1): A units and B_down rows on the
    // shared pairs
    if (S.lora && pair < Ps) {
        const int n_gd = S.d / kGroup, ngh = half_hi(n_gd, rank) - half_lo(n_gd, rank);
        const int n_rtd = S.d / kRowTile, nrt = half_hi(n_rtd, rank) - half_lo(n_rtd, rank);
        split_range(2 * ngh, Ps, pair, &pp.la0, &pp.la1);
        split_range(nrt, Ps, pair, &pp.bd0, &pp.bd1);
    }
    if (S.router) {
        const int n_gd = S.d / kGroup;
        const int ngh = half_hi(n_gd, rank) - half_lo(n_gd, rank);
        split_range((S.E / kRowTile) * ngh, P, pair, &pp.ru0, &pp.ru1);
    }
}

// ---- head flush.  A head depends only on its layer's x and routing, and its
// prediction is consumed one token later, so every head of a launch runs in one
// phase after the last layer (one flush per decode step).  The heads' tasks (per
// head: H/16 fc1 row tiles with their fc2 columns, then E/16 linear_init row
// tiles) form one list, split contiguously over the CTAs; each CTA does its tasks
// over all of d (no pair exchange), in tables of at most p.ft tasks of one head.
__host__ __device__ inline bool is_head_layer(const Prog& p, int l) {
    return p.mode == MODE_HEAD || (p.mode == MODE_DECODE && (p.layers[l].flags & LF_HEAD));
}
__host__ __device__ inline int n_heads(const Prog& p) {
    if (p.mode == MODE_HEAD) return 1;
    int n = 0;
    for (int l = 0; l < p.L; ++l) n += is_head_layer(p, l) ? 1 : 0;
    return n;
}
__host__ __device__ inline int head_layer(const Prog& p, int hi) {
    for (int l = 0; l < p.L; ++l)
        if (is_head_layer(p, l) && hi-- == 0) return l;
    return 0;
}
__host__ __device__ inline int head_tasks(const Prog& p) { return p.H / kRowTile + p.E / kRowTile; }
// table j of CTA `cta` of an nct grid: head layer *hl, tasks [*t0, *t1); false
// past the CTA's last table
__host__ __device__ inline bool flush_table(const Prog& p, int nct, int cta, int j, int* hl, int* t0, int* t1) {
    const int nt = head_tasks(p);
    int g, g1;
    split_range(n_heads(p) * nt, nct, cta, &g, &g1);
    for (int i = 0; g < g1; ++i) {
        const int hi = g / nt, t = g - hi * nt;
        int e = t + p.ft < nt ? t + p.ft : nt;
        if (hi * nt + e > g1) e = g1 - hi * nt;
        if (i == j) {
            *hl = head_layer(p, hi);
            *t0 = t;
            *t1 = e;
            return true;
        }
        g = hi * nt + e;
    }
    return false;
}
// layers of the launch that have item tables before the flush
__host__ __device__ inline int n_layer_tabs(const Prog& p) { return p.mode == MODE_HEAD ? 0 : p.L; }

// one copy of a contiguous global region into the ring
struct Item {
    int kind, seg;
    int bytes, off;   // size, ring offset
    int lin;          // linear ring position (off = lin mod ring size)
    int a, b, n;      // kind-specific position and count
};

// one K-group of down rows a segment touches: where its 16-row steps and scales
// sit in the ring (offsets of row tile 0 of this CTA's half) and which act
// quarters they multiply
constexpr int kMaxDg = 12;
struct DGroup {
    int seg, nq, ql0;   // segment, steps, act quarter (in the pair's list) of the first step
    int soff;           // ring offset of the scales
    int qoff[4];        // ring offset of each step
};

struct LayerTab {
    int seq;          // table index + 1 once published
    int hl;           // head layer of a flush table, -1 for a layer table
    int k0, n;        // global index of the first item; items
    int p1, p2, p3;   // first item of P1 (gate/up), P2 (down), P3 (head); router items from 0
    int ndg;          // down groups
    int ibg, ibu, iadt, ibd;   // first item of the LoRA B_gate, B_up, A_down^T, B_down rows (or -1)
    PairPlan pl;
    DGroup dg[kMaxDg];
    Item it[kMaxItems];
};

// this CTA's halves
struct Halves {
    int gh0, gh1;   // groups of d
    int rt0, rt1;   // row tiles of d
    int e0, e1;     // row tiles of E
};
__host__ __device__ inline Halves halves(int d, int E, int rank) {
    Halves h;
    h.gh0 = half_lo(d / kGroup, rank);
    h.gh1 = half_hi(d / kGroup, rank);
    h.rt0 = half_lo(d / kRowTile, rank);
    h.rt1 = half_hi(d / kRowTile, rank);
    h.e0 = half_lo(E / kRowTile, rank);
    h.e1 = half_hi(E / kRowTile, rank);
    return h;
}

// appends one item (or, for a run of units, as many items of at most kItemMax
// bytes as it takes) to T, placing it in the ring at the running position `lin`
struct ItemSink {
    LayerTab* T;
    int n, lin, pos, ring;   // pos = lin mod ring
    bool ok;
};
__host__ __device__ __forceinline__ void push_item(ItemSink& k, int kind, int seg, int bytes, int a, int b,
                                                   int cnt) {
    if (bytes <= 0) return;
    if (k.n >= kMaxItems || bytes > kItemMax || bytes > k.ring) { k.ok = false; return; }
    if (k.pos + bytes > k.ring) { k.lin += k.ring - k.pos; k.pos = 0; }   // no item wraps
    Item& it = k.T->it[k.n++];
    it.kind = kind; it.seg = seg; it.bytes = bytes; it.off = k.pos; it.lin = k.lin;
    it.a = a; it.b = b; it.n = cnt;
    k.lin += bytes;
    k.pos += bytes;
}
__host__ __device__ __forceinline__ void push_units(ItemSink& k, int kind, int seg, int a, int first,
                                                    int units, int ub) {
    const int per = kItemMax / ub;
    for (int j = 0; j < units; j += per) {
        const int m = units - j < per ? units - j : per;
        push_item(k, kind, seg, m * ub, a, first + j, m);
    }
}

// Builds one CTA's copy items of one layer into T (deterministic: the producer
// issues them, the consumers read them from the published table, the host uses
// it to check limits).  `lin` is the running linear ring position.  Returns
// false if a limit is exceeded.
__host__ __device__ __noinline__ bool build_items(const Shape& Sh, int P, int pair, int rank, int ring,
                                                  LayerTab* T, int& lin) {
    PairPlan& pl = T->pl;
    pair_plan(Sh, P, pair, rank, pl);
    if (pl.over) return false;
    const Halves hv = halves(Sh.d, Sh.E, rank);
    ItemSink k{T, 0, lin, lin % ring, ring, true};
    T->ndg = 0;
    T->hl = -1;
    T->ibg = T->ibu = T->iadt = T->ibd = -1;
    const int ngh = hv.gh1 - hv.gh0, nrt = hv.rt1 - hv.rt0;
    const int r = Sh.r;
    // router units: this pair's share of (E row tiles) x (this rank's groups)
    push_units(k, IT_ROUTER, 0, 0, pl.ru0, pl.ru1 - pl.ru0, kF16Unit);
    T->p1 = k.n;
    // LoRA A units first (every shared pair waits for the sums of all of them):
    // A_gate groups [la0, la1) n [0, ngh), then A_up groups
    if (pl.la0 < ngh && pl.la0 < pl.la1) {
        const int e = pl.la1 < ngh ? pl.la1 : ngh;
        push_units(k, IT_LA, 0, 0, pl.la0, e - pl.la0, kF16Unit);
    }
    if (pl.la1 > ngh) {
        const int b0 = pl.la0 > ngh ? pl.la0 : ngh;
        push_units(k, IT_LU, 0, 0, b0 - ngh, pl.la1 - b0, kF16Unit);
    }
    for (int s = 0; s < pl.nseg; ++s) {
        const Seg& g = pl.seg[s];
        push_units(k, IT_GU, s, 0, g.hr0 * ngh, (g.hr1 - g.hr0) * ngh, kQ4Unit);
        if (g.slot < 0 && Sh.lora) {
            const int rows = (g.hr1 - g.hr0) * kHalfRow;
            T->ibg = k.n;
            push_item(k, IT_BG, s, rows * r * 2, g.hr0 * kHalfRow, 0, rows);
            T->ibu = k.n;
            push_item(k, IT_BU, s, rows * r * 2, g.hr0 * kHalfRow, 0, rows);
            T->iadt = k.n;
            push_item(k, IT_ADT, s, rows * r * 2, g.hr0 * kHalfRow, 0, rows);
        }
    }
    T->p2 = k.n;
    for (int s = 0; s < pl.nseg; ++s) {
        const Seg& g = pl.seg[s];
        const int qbytes = nrt * kQ4Quarter, sbytes = nrt * kQ4Scales;
        const int qper = kItemMax / qbytes > 0 ? kItemMax / qbytes : 1;
        for (int gg = g.q0 / 4; gg <= (g.q1 - 1) / 4; ++gg) {
            const int qa = g.q0 > 4 * gg ? g.q0 : 4 * gg, qb = g.q1 < 4 * gg + 4 ? g.q1 : 4 * gg + 4;
            DGroup* D = nullptr;
            if (T->ndg < kMaxDg) {
                D = &T->dg[T->ndg++];
                D->seg = s;
                D->nq = qb - qa;
                D->ql0 = g.qoff + qa - g.q0;
            } else {
                k.ok = false;
            }
            // runs of steps (at most kItemMax bytes), the scales merged into the last
            // run when the group's steps and scales are adjacent and fit
            for (int q = qa; q < qb; q += qper) {
                const int m = qb - q < qper ? qb - q : qper;
                const bool last = q + m == qb;
                const int n0 = k.n;
                if (last && qb == 4 * gg + 4 && m * qbytes + sbytes <= kItemMax) {
                    push_item(k, IT_DQS, s, m * qbytes + sbytes, gg, q - 4 * gg, m);
                    if (D && k.n > n0) D->soff = T->it[n0].off + m * qbytes;
                } else {
                    push_item(k, IT_DQ, s, m * qbytes, gg, q - 4 * gg, m);
                    if (last) {
                        push_item(k, IT_DSC, s, sbytes, gg, 0, nrt);
                        if (D && k.n > n0 + 1) D->soff = T->it[n0 + 1].off;
                    }
                }
                if (D && k.n > n0)
                    for (int qi = 0; qi < m; ++qi) D->qoff[q - qa + qi] = T->it[n0].off + qi * qbytes;
            }
        }
    }
    // LoRA B_down rows: row tiles [bd0, bd1) of this rank's half
    if (pl.bd1 > pl.bd0) {
        T->ibd = k.n;
        const int per = kItemMax / (r * 2);
        for (int row = (hv.rt0 + pl.bd0) * kRowTile; row < (hv.rt0 + pl.bd1) * kRowTile; row += per) {
            const int m = (hv.rt0 + pl.bd1) * kRowTile - row < per ? (hv.rt0 + pl.bd1) * kRowTile - row : per;
            push_item(k, IT_BD, 0, m * r * 2, row, 0, m);
        }
    }
    T->p3 = k.n;
    T->n = k.n;
    lin = k.lin;
    return k.ok;
}

// Items of one head-flush table (tasks [t0, t1) of head layer hl, over all of
// d): the fc1 and linear_init units of both halves of d (seg = half).  The fc2
// column blocks are small and read directly from global memory (held in the
// ring they would halve its streaming depth).  p1 = 0, p2 = p3 = n.
__host__ __device__ __noinline__ bool build_flush_items(const Prog& p, int hl, int t0, int t1, int ring,
                                                        LayerTab* T, int& lin) {
    ItemSink k{T, 0, lin, lin % ring, ring, true};
    PairPlan& pl = T->pl;
    pl.nseg = 0; pl.over = 0; pl.n_hr = 0; pl.n_q = 0; pl.has_sh = 0;
    pl.ru0 = pl.ru1 = pl.la0 = pl.la1 = pl.bd0 = pl.bd1 = 0;
    pl.hd0 = t0;
    pl.hd1 = t1;
    T->hl = hl;
    T->ndg = 0;
    T->ibg = T->ibu = T->iadt = T->ibd = -1;
    T->p1 = 0;
    const int nH = p.H / kRowTile, hn0 = p.d / kGroup / 2, nE = p.E / kRowTile;
    for (int t = t0; t < t1; ++t)
        for (int h = 0; h < 2; ++h) {
            if (t < nH) push_units(k, IT_FC1, h, t, t * hn0, hn0, kF16Unit);
            else push_units(k, IT_LINIT, h, t - nH, (t - nH) * hn0, hn0, kF16Unit);
        }
    T->p2 = k.n;
    T->p3 = k.n;
    T->n = k.n;
    lin = k.lin;
    (void)nE;
    return k.ok;
}

// ------------------------------------------------------------ smem plan ----
struct Ctl {
    int trace, tslot, abort, step, cdone, issued, last, ptslot;
    unsigned long long bar_seen;   // grid-barrier count right after this CTA's last arrival
    unsigned long long tmo;        // limit of every bounded wait (ns)
};
constexpr int kTraceProducer = 3072;   // first trace word of the producer's stamps

struct Plan {
    int ring, full, empty, xch, lin, tabs, xf, xsum, hs, gam, part, recv, act32, af, qsum, vlo, zpart,
        gf, ids, wts, dist, ndist, prv, nprv, ready, rscr, red, ctl, total;
};

__host__ __device__ inline int al16(int x) { return (x + 15) & ~15; }
// head-flush tasks per table: at most 12, and one consumer thread per (task, row, token)
__host__ __device__ inline int flush_tasks_max(int B) {
    const int t = kConsumerThreads / (kRowTile * B);
    return t < 12 ? t : 12;
}

__host__ __device__ inline int msg_floats(const Prog& p) { return p.hr_max * 16 * p.B; }

// base: bytes at the start of shared memory taken by the parameter copy and the context
__host__ __device__ inline Plan make_plan(const Prog& p, int base) {
    Plan s;
    const int B = p.B, K = p.K, L = p.L;
    const int n_gd = p.d / kGroup, ngh = n_gd - n_gd / 2;
    const int ft = flush_tasks_max(B);
    int o = base;
    s.full = o;   o += kSlots * 8;
    s.empty = o;  o += kSlots * 8;
    s.xch = o;    o += 2 * 8;
    o = al16(o);
    s.lin = o;    o += kSlots * 4;
    s.tabs = o;   o += al16(kTables * (int)sizeof(LayerTab));
    s.xf = o;     o += al16(n_gd * 4 * B * 4 * 8);   // all of d (head flush), else this CTA's half
    s.xsum = o;   o += al16(ngh * B * 4);
    s.hs = o;     o += al16(B * p.d * 2);
    s.gam = o;    o += al16(p.d * 2);   // RMSNorm gain of the next decode layer
    s.part = o;   o += al16(msg_floats(p) * 4);
    s.recv = o;   o += al16(msg_floats(p) * 4);
    s.act32 = o;  o += al16(p.hr_max * 8 * B * 4);
    s.af = o;     o += al16(p.q_max * B * 2 * 4 * 8);
    s.qsum = o;   o += al16(p.q_max * B * 4);
    s.vlo = o;    o += al16(32 * B * 4);
    s.zpart = o;  o += al16(ft * 16 * B * 4);
    s.gf = o;     o += al16(ft * B * 2 * 4 * 8);
    s.ids = o;    o += al16(L * B * K * 4);
    s.wts = o;    o += al16(L * B * K * 4);
    s.dist = o;   o += al16(L * (p.slots_max > 0 ? p.slots_max : 1) * 4);
    s.ndist = o;  o += al16(L * 4);
    s.prv = o;    o += al16(L * B * K * 4);
    s.nprv = o;   o += al16(L * 4);
    s.ready = o;  o += al16(L * 4);
    s.rscr = o;   o += al16(B * 3 * p.E * 4);
    s.red = o;    o += al16((B * kConsumerWarps + 64) * 4);
    s.ctl = o;    o += al16((int)sizeof(Ctl));
    o = (o + 127) & ~127;
    s.ring = o;
    s.total = o + p.ring_bytes;
    return s;
}

// ------------------------------------------------------------- context ----
// Per-CTA context.  It and a copy of the kernel parameters live at fixed places
// at the start of dynamic shared memory (every function reads them there: no
// context is passed around, nothing of it is kept in local memory).
struct Ctx {
    Plan pl;
    WsHeader* hdr;
    Ctl* ctl;
    WsLayout ws;
    Halves hv;
    int nct, cta, pair, rank, P;
    int step, par;
};

extern __shared__ __align__(128) char g_smem[];
constexpr int kProgOff = 0;
constexpr int kCtxOff = (int)((sizeof(Prog) + 127) / 128 * 128);
constexpr int kCtxBytes = (int)((sizeof(Ctx) + 127) / 128 * 128);
__device__ __forceinline__ Ctx& ctx() { return *reinterpret_cast<Ctx*>(g_smem + kCtxOff); }
__device__ __forceinline__ const Prog& prg() { return *reinterpret_cast<const Prog*>(g_smem + kProgOff); }

__device__ __forceinline__ unsigned long long now_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __noinline__ void raise_error(int code) {
    const Ctx& c = ctx();
    atomicCAS(&c.hdr->error, 0, code);
    atomicExch(&c.hdr->abort, 1);
    *(volatile int*)&c.ctl->abort = 1;
}
__device__ __forceinline__ bool should_abort() {
    const Ctx& c = ctx();
    return *(volatile int*)&c.ctl->abort || ld_volatile_s32(&c.hdr->abort);
}
__device__ __forceinline__ bool aborted() {
    const Ctx& c = ctx(); return *(volatile int*)&c.ctl->abort != 0; }

// wait on an mbarrier phase with a time bound; false on abort/timeout
__device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity) {
    const Ctx& c = ctx();
    const unsigned long long t0 = now_ns();
    for (unsigned it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 63) {
            if (should_abort()) return false;
            if (now_ns() - t0 > ctx().ctl->tmo) { raise_error(EDGE0_ETIMEOUT); return false; }
        }
    }
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    const Ctx& c = ctx();
    return mbar_try_wait(bar, parity) || mbar_wait_slow(bar, parity);
}

// spin until *flag >= want (shared memory, written by the other role); bounded
__device__ __noinline__ bool wait_flag(volatile int* flag, int want) {
    const Ctx& c = ctx();
    if (*flag >= want) return true;
    const unsigned long long t0 = now_ns();
    for (unsigned it = 0; *flag < want; ++it) {
        __nanosleep(32);
        if ((it & 63) == 63) {
            if (should_abort()) return false;
            if (now_ns() - t0 > ctx().ctl->tmo) { raise_error(EDGE0_ETIMEOUT); return false; }
        }
    }
    return true;
}

template <class T>
__device__ __forceinline__ T* SM(int off) {
    const Ctx& c = ctx(); return reinterpret_cast<T*>(g_smem + off); }

__device__ __forceinline__ uint64_t* full_bar(int k) {
    const Ctx& c = ctx(); return SM<uint64_t>(c.pl.full) + (k % kSlots); }
__device__ __forceinline__ uint64_t* empty_bar(int k) {
    const Ctx& c = ctx(); return SM<uint64_t>(c.pl.empty) + (k % kSlots); }
__device__ __forceinline__ uint32_t item_parity(int k) { return (uint32_t)((k / kSlots) & 1); }
__device__ __forceinline__ LayerTab* tab_of(int l) {
    const Ctx& c = ctx(); return SM<LayerTab>(c.pl.tabs) + (l % kTables); }
__device__ __forceinline__ int* ids_of(int l) {
    const Ctx& c = ctx(); return SM<int>(c.pl.ids) + l * prg().B * prg().K; }
__device__ __forceinline__ float* w_of(int l) {
    const Ctx& c = ctx(); return SM<float>(c.pl.wts) + l * prg().B * prg().K; }
__device__ __forceinline__ int* dist_of(int l) {
    const Ctx& c = ctx();
    return SM<int>(c.pl.dist) + l * (prg().slots_max > 0 ? prg().slots_max : 1);
}
__device__ __forceinline__ int* prev_of(int l) {
    const Ctx& c = ctx(); return SM<int>(c.pl.prv) + l * prg().B * prg().K; }
__device__ __forceinline__ const char* ring_at(const Item& it) {
    const Ctx& c = ctx(); return g_smem + c.pl.ring + it.off; }

__device__ __forceinline__ float* ws_f(long long off) {
    const Ctx& c = ctx(); return reinterpret_cast<float*>(prg().ws + off); }
__device__ __forceinline__ float* y_buf(int par, int sidx) {
    const Ctx& c = ctx();
    return ws_f(c.ws.y) + ((long long)par * prg().Ls + sidx) * prg().B * prg().d;
}
__device__ __forceinline__ float* logr_buf(int par, int sidx) {
    const Ctx& c = ctx();
    return ws_f(c.ws.logr) + ((long long)par * prg().Ls + sidx) * prg().B * prg().E;
}
__device__ __forceinline__ float* logh_buf(int par, int sidx) {
    const Ctx& c = ctx();
    return ws_f(c.ws.logh) + ((long long)par * prg().Ls + sidx) * prg().B * prg().E;
}
// the LoRA sums of a layer: A_gate x at [q B + b], A_up x at [(16 + q) B + b],
// v = A_down act at [(32 + q) B + b]
__device__ __forceinline__ float* lora_buf(int par, int sidx) {
    const Ctx& c = ctx();
    return ws_f(c.ws.lora) + ((long long)par * prg().Ls + sidx) * prg().B * kLoraAcc;
}
// x of a head layer (fp16 [B][d]), kept for the head flush
__device__ __forceinline__ __half* xs_buf(int sidx) {
    const Ctx& c = ctx();
    return reinterpret_cast<__half*>(prg().ws + c.ws.xs) + (long long)sidx * prg().B * prg().d;
}
__device__ __forceinline__ unsigned* cnt_buf(int par, int sidx, int which) {
    const Ctx& c = ctx();
    return reinterpret_cast<unsigned*>(prg().ws + c.ws.cnt) + (par * prg().Ls + sidx) * kLayerCounters + which;
}

// optional trace: (tag, globaltimer) pairs per CTA, written by consumer thread 0
__device__ __noinline__ void stamp_slow(int tag) {
    const Ctx& c = ctx();
    const int s = c.ctl->tslot;
    if (s + 3 > kTraceProducer) return;
    unsigned long long* a =
        reinterpret_cast<unsigned long long*>(prg().ws + c.ws.trace) + (long long)c.cta * kTraceSlots;
    a[s] = (unsigned long long)tag;
    a[s + 1] = now_ns();
    a[s + 2] = clock64();
    c.ctl->tslot = s + 3;
}
__device__ __forceinline__ void stamp(int tag) {
    const Ctx& c = ctx();
    if (threadIdx.x == 0 && c.ctl->trace) stamp_slow(tag);
}
// a value in place of the time (thread 0, when tracing)
__device__ __noinline__ void stamp_value(int tag, unsigned long long v) {
    const Ctx& c = ctx();
    if (threadIdx.x != 0 || !c.ctl->trace) return;
    const int s = c.ctl->tslot;
    if (s + 3 > kTraceProducer) return;
    unsigned long long* a =
        reinterpret_cast<unsigned long long*>(prg().ws + c.ws.trace) + (long long)c.cta * kTraceSlots;
    a[s] = (unsigned long long)tag;
    a[s + 1] = v;
    a[s + 2] = clock64();
    c.ctl->tslot = s + 3;
}
// the producer's stamps (slots from kTraceProducer on)
__device__ __noinline__ void stamp_producer(int tag) {
    const Ctx& c = ctx();
    if (!c.ctl->trace) return;
    const int s = c.ctl->ptslot;
    if (s + 3 > kTraceSlots) return;
    unsigned long long* a =
        reinterpret_cast<unsigned long long*>(prg().ws + c.ws.trace) + (long long)c.cta * kTraceSlots;
    a[s] = (unsigned long long)tag;
    a[s + 1] = now_ns();
    a[s + 2] = clock64();
    c.ctl->ptslot = s + 3;
}

__host__ __device__ inline bool has_router_phase(const Prog& p, int l, int step) {
    return p.mode == MODE_DECODE && (!(p.layers[l].flags & LF_PREROUTED) || step == 0);
}

__host__ __device__ inline Shape layer_shape(const Prog& p, int l, bool router) {
    const LayerP& Ly = p.layers[l];
    Shape S;
    S.d = p.d; S.I = p.I; S.Is = p.Is; S.E = p.E; S.H = p.H; S.r = p.r;
    S.n_slots = p.mode == MODE_HEAD ? 0 : p.slots_max;
    S.shared = (p.mode != MODE_HEAD && (Ly.flags & LF_SHARED)) ? 1 : 0;
    S.lora = (S.shared && p.mode == MODE_DECODE && (Ly.flags & LF_LORA)) ? 1 : 0;
    S.router = router ? 1 : 0;
    S.ps = S.shared ? p.ps[S.lora] : 0;
    return S;
}

__device__ __forceinline__ void cbar() { named_bar_sync(1, kConsumerThreads); }
// consumer barrier that also returns the OR of `v` over the consumer threads
__device__ __forceinline__ bool cbar_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n"
        " selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(kConsumerThreads)
        : "memory");
    return r != 0;
}

// distinct experts of a layer's routing in order of first appearance; false if
// an id is out of range (single thread)
__device__ bool make_dist(int l) {
    const Ctx& c = ctx();
    const Prog& p = prg();
    const int* ids = ids_of(l);
    int* dist = dist_of(l);
    int n = 0;
    bool ok = true;
    for (int i = 0; i < p.B * p.K; ++i) {
        const int e = ids[i];
        if (e < 0 || e >= p.E) { ok = false; continue; }
        bool seen = false;
        for (int j = 0; j < n; ++j) seen |= dist[j] == e;
        if (!seen && n < p.slots_max) dist[n++] = e;
    }
    SM<int>(c.pl.ndist)[l] = n;
    return ok;
}

// make_dist by one warp (B K <= 32 ids, lane i holding id i): an id is new if
// no lower lane holds it; its slot is its rank among the new ids
__device__ bool make_dist_warp(int l, int lane) {
    const Ctx& c = ctx();
    const Prog& p = prg();
    const int n = p.B * p.K;
    const int e = lane < n ? ids_of(l)[lane] : -1;
    const bool bad = lane < n && (e < 0 || e >= p.E);
    const unsigned act = __ballot_sync(0xffffffffu, lane < n && !bad);
    const unsigned same = __match_any_sync(0xffffffffu, lane < n && !bad ? e : -1);
    const bool first = lane < n && !bad && (__ffs(same & act) - 1) == lane;
    const unsigned firsts = __ballot_sync(0xffffffffu, first);
    if (first) dist_of(l)[__popc(firsts & ((1u << lane) - 1u))] = e;
    if (lane == 0) SM<int>(c.pl.ndist)[l] = __popc(firsts);
    return !__any_sync(0xffffffffu, bad);
}

// ------------------------------------------------------------ producer -----
// global source of an item; null: nothing to copy (a routed slot no token uses);
// (const char*)1: an expert slot outside the stacks
__device__ __noinline__ const char* item_src(int l, const LayerTab* T, const Item& it) {
    const Ctx& c = ctx();
    const Prog& p = prg();
    const LayerP& Ly = p.layers[l];
    const int n_gd = p.d / kGroup, r = p.r, n_rtd = p.d / kRowTile;
    const int h = c.rank, hn0 = n_gd / 2;
    // first unit of this CTA's half of a row-tile-major matrix with `tiles` row tiles
    auto half0 = [&](int tiles) { return (long long)h * tiles * hn0; };
    const char* gu = nullptr;
    const char* dn = nullptr;
    int I = p.I;
    if (it.kind == IT_GU || it.kind == IT_DSC || it.kind == IT_DQ || it.kind == IT_DQS) {
        const Seg& g = T->pl.seg[it.seg];
        if (g.slot < 0) {
            gu = Ly.sh_gu;
            dn = Ly.sh_down;
            I = p.Is;
        } else {
            if (g.slot >= SM<int>(c.pl.ndist)[l]) return nullptr;
            const int e = dist_of(l)[g.slot];
            const int slot = Ly.slot_table ? Ly.slot_table[e] : e;
            if (slot < 0 || slot >= Ly.n_slots) return reinterpret_cast<const char*>(1);
            gu = Ly.gu + (long long)slot * q4_bytes(2 * p.I, p.d);
            dn = Ly.down + (long long)slot * q4_bytes(p.d, p.I);
        }
    }
    // down: group a, this CTA's half of the row tiles
    const int nrt = c.hv.rt1 - c.hv.rt0;
    const char* dgrp = dn ? dn + (long long)it.a * n_rtd * kQ4Unit + (long long)h * (n_rtd / 2) * kQ4Unit : nullptr;
    switch (it.kind) {
        case IT_ROUTER: return Ly.router + (half0(p.E / kRowTile) + it.b) * kF16Unit;
        case IT_GU: return gu + (half0(I / kHalfRow) + it.b) * kQ4Unit;
        case IT_LA: return Ly.lora_Ag + (half0(1) + it.b) * kF16Unit;
        case IT_LU: return Ly.lora_Au + (half0(1) + it.b) * kF16Unit;
        case IT_BG: return reinterpret_cast<const char*>(Ly.lora_Bg + (long long)it.a * r);
        case IT_BU: return reinterpret_cast<const char*>(Ly.lora_Bu + (long long)it.a * r);
        case IT_DQ:
        case IT_DQS: return dgrp + (long long)it.b * nrt * kQ4Quarter;
        case IT_DSC: return dgrp + 4LL * nrt * kQ4Quarter;
        case IT_ADT: return reinterpret_cast<const char*>(Ly.lora_AdT + (long long)it.a * r);
        case IT_BD: return reinterpret_cast<const char*>(Ly.lora_Bd + (long long)it.a * r);
        // head flush: both halves of d (seg = half)
        case IT_FC1: return Ly.fc1 + ((long long)it.seg * (p.H / kRowTile) * hn0 + it.b) * kF16Unit;
        case IT_FC2: return Ly.fc2 + ((long long)it.a * (p.E / kRowTile) + it.b) * kF16Step;
        default: return Ly.linit + ((long long)it.seg * (p.E / kRowTile) * hn0 + it.b) * kF16Unit;
    }
}

// The producer warp (all 32 lanes call this; it uses warp-wide shuffles): lane 0
// builds each layer's item table and decides how many of the next items can go
// (routing known, ring bytes and barrier slots free); the lanes then issue those
// copies in parallel.
__device__ void producer() {
    Ctx& c = ctx();
    const Prog& p = prg();
    Ctl* ctl = c.ctl;
    const int lane = threadIdx.x & 31;
    volatile int* ready = SM<volatile int>(c.pl.ready);
    int* lstart = SM<int>(c.pl.lin);   // linear start of the item in each slot
    const uint64_t pol = policy_evict_first();
    char* ring = g_smem + c.pl.ring;
    int lin = 0;      // linear ring position of the next item (lane 0)
    int k = 0;        // global index of the next item
    int front = 0;    // oldest item not known to be released (lane 0)
    if (__shfl_sync(0xffffffffu, lane == 0 ? (int)aborted() : 0, 0)) return;
    // the layers' tables, then this CTA's tables of the head flush.  Lane 0
    // builds tables in order, one ahead of the table being issued whenever that
    // table's slot is already free (a build never waits behind the ring).
    const int nl = n_layer_tabs(p);
    int nb = 0, kb = 0;   // lane 0: next table to build, global index of its first item
    auto build_next = [&](bool wait, int* fail) -> bool {
        int hl = -1, t0 = 0, t1 = 0;
        if (nb >= nl && !flush_table(p, c.nct, c.cta, nb - nl, &hl, &t0, &t1)) return false;
        // the table slot is free once the consumers finished table nb - kTables
        if (!wait && *(volatile int*)&ctl->cdone < nb - kTables + 1) return false;
        if (wait && !wait_flag(&ctl->cdone, nb - kTables + 1)) { *fail = 1; return false; }
        LayerTab* T = tab_of(nb);
        stamp_producer((nb << 8) | 0x80);
        T->k0 = kb;
        const bool built = nb < nl ? build_items(layer_shape(p, nb, has_router_phase(p, nb, c.step)), c.P,
                                                 c.pair, c.rank, p.ring_bytes, T, lin)
                                   : build_flush_items(p, hl, t0, t1, p.ring_bytes, T, lin);
        if (!built) {
            raise_error(EDGE0_EUNSUPPORTED);
            *fail = 1;
            return false;
        }
        __threadfence_block();
        *(volatile int*)&T->seq = nb + 1;
        stamp_producer((nb << 8) | 0x81);
        kb += T->n;
        ++nb;
        return true;
    };
    for (int l = 0;; ++l) {
        int fail = 0, have = 1;
        if (lane == 0) {
            if (nb <= l && !build_next(true, &fail)) have = 0;   // table l
            if (have && !fail && nb == l + 1) build_next(false, &fail);
        }
        if (__shfl_sync(0xffffffffu, fail, 0)) return;
        if (!__shfl_sync(0xffffffffu, have, 0)) break;
        LayerTab* T = tab_of(l);
        __syncwarp();
        const int n = T->n;
        bool have_routing = false;
        for (int i = 0; i < n;) {
            int m = 0;
            if (lane == 0) {
                // items i .. i + m - 1 can go now; wait only for the first one
                for (; m < 32 && i + m < n; ++m) {
                    const Item& it = T->it[i + m];
                    const int kk = k + m;
                    const bool routed = (it.kind == IT_GU || it.kind == IT_DSC || it.kind == IT_DQ ||
                                         it.kind == IT_DQS) && T->pl.seg[it.seg].slot >= 0;
                    if (routed && !have_routing) {
                        if (m > 0 && ready[l] != 1) break;
                        if (!wait_flag(&ready[l], 1)) { fail = 1; break; }
                        __threadfence_block();
                        have_routing = true;
                        stamp_producer((l << 8) | 0x82);
                    }
                    // slot kk and the item's ring bytes must be free: move `front` past the
                    // released items (waiting only for the batch's first item)
                    while (front < kk && (front <= kk - kSlots || it.lin + it.bytes - lstart[front % kSlots] > p.ring_bytes)) {
                        if (m > 0) {
                            if (!mbar_try_wait(empty_bar(front), item_parity(front))) break;
                        } else {
                            if (l >= nl && !mbar_try_wait(empty_bar(front), item_parity(front)))
                                stamp_producer((l << 8) | 0xE0 | ((front - T->k0 + 1024) << 20));
                            if (!mbar_wait(empty_bar(front), item_parity(front))) {
                                fail = 1;
                                break;
                            }
                        }
                        ++front;
                    }
                    if (fail) break;
                    if (front < kk && (front <= kk - kSlots || it.lin + it.bytes - lstart[front % kSlots] > p.ring_bytes)) break;
                    lstart[kk % kSlots] = it.lin;
                }
            }
            fail = __shfl_sync(0xffffffffu, fail, 0);
            m = __shfl_sync(0xffffffffu, m, 0);
            if (fail) return;
            __syncwarp();
            if (lane < m) {
                const Item& it = T->it[i + lane];
                const char* src = item_src(l < nl ? l : T->hl, T, it);
                uint64_t* fb = full_bar(k + lane);
                if (src == reinterpret_cast<const char*>(1)) {
                    raise_error(EDGE0_EINVAL);
                    mbar_arrive(fb);
                } else if (src) {
                    mbar_arrive_expect_tx(fb, (uint32_t)it.bytes);
                    bulk_g2s(ring + it.off, src, (uint32_t)it.bytes, fb, pol);
                } else {
                    mbar_arrive(fb);
                }
            }
            __syncwarp();
            if (lane == 0 && l >= nl && i < 64)   // flush: batch issued, with the front item
                stamp_producer((l << 8) | (0x90 + i) | ((front - T->k0 + 1024) << 20));
            i += m;
            k += m;
            if (lane == 0) *(volatile int*)&ctl->issued = k;
        }
        if (lane == 0) stamp_producer((l << 8) | 0x83);
    }
}

// ------------------------------------------------------------ consumers ----
__device__ __forceinline__ bool wait_item(const LayerTab* T, int i) {
    const Ctx& c = ctx();
    return mbar_wait(full_bar(T->k0 + i), item_parity(T->k0 + i));
}
__device__ __forceinline__ void release_item(const LayerTab* T, int i) {
    const Ctx& c = ctx();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(empty_bar(T->k0 + i));
}

// grid barrier: arrive (after the caller's cbar) and wait
// The arrival is an atomic that returns the count: the CTA whose arrival
// completes a barrier learns it at once instead of polling for its own update
// (the last to arrive is the one the whole grid waits for).
__device__ void bar_arrive() {
    const Ctx& c = ctx();
    if (threadIdx.x == 0) {
        __threadfence();
        c.ctl->bar_seen = atom_acq_rel_add_u64(&c.hdr->barrier, 1ull) + 1ull;
    }
}
__device__ __noinline__ bool bar_wait(unsigned long long& target) {
    const Ctx& c = ctx();
    if (threadIdx.x == 0) {
        target += (unsigned long long)c.nct;
        if (c.ctl->bar_seen < target && ld_acquire_u64(&c.hdr->barrier) < target) {
            const unsigned long long t0 = now_ns();
            for (unsigned it = 0; ld_acquire_u64(&c.hdr->barrier) < target; ++it) {
                if ((it & 15) == 15) {
                    if (should_abort()) { *(volatile int*)&c.ctl->abort = 1; break; }
                    if (now_ns() - t0 > ctx().ctl->tmo) { raise_error(EDGE0_ETIMEOUT); break; }
                }
            }
        }
    }
    return !cbar_or(aborted());
}

// send nfloats (multiple of 4) from this CTA's `src` into the peer's copy of
// `dst`, and wait for the peer's data in this CTA's `dst` (exchange barrier `which`)
__device__ __noinline__ bool exchange(int which, const float* src, float* dst, int nfloats,
                         uint32_t& phase) {
    const Ctx& c = ctx();
    uint64_t* bar = SM<uint64_t>(c.pl.xch) + which;
    const uint32_t peer = c.rank ^ 1u;
    if (threadIdx.x == 0) mbar_arrive_expect_tx(bar, (uint32_t)(nfloats * 4));
    const uint32_t rbar = mapa_shared(smem_u32(bar), peer);
    const uint32_t rdst = mapa_shared(smem_u32(dst), peer);
    for (int i = threadIdx.x; i < nfloats / 4; i += kConsumerThreads)
        st_async_v4(rdst + 16u * i, reinterpret_cast<const uint4*>(src)[i], rbar);
    const bool ok = mbar_wait(bar, phase & 1u);
    ++phase;
    return ok;
}

// B fragment of the x source for lane (g, t): token g / 2 in the even columns
struct XFrag {
    const uint2* base;
    int stride;   // uint2 per 16-input step
    bool live;
};
__device__ __forceinline__ XFrag xfrag() {
    const Ctx& c = ctx();
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3, tok = g >> 1;
    XFrag f;
    f.live = !(g & 1) && tok < prg().B;
    f.base = SM<uint2>(c.pl.xf) + (f.live ? tok : 0) * 4 + t;
    f.stride = prg().B * 4;
    return f;
}

// fp16 units [a, b) (x source) accumulated into acc (rows g, g + 8; column 2t = token t)
__device__ __forceinline__ void f16_run(const char* base, int a, int b, int gl0, float acc[4]) {
    const Ctx& c = ctx();
    const int lane = threadIdx.x & 31;
    const XFrag xf = xfrag();
    // one accumulator per 16-input step: consecutive MMAs do not wait on each other
    float as[4][4];
#pragma unroll
    for (int s = 0; s < 4; ++s) as[s][0] = as[s][1] = as[s][2] = as[s][3] = 0.f;
    for (int j = a; j < b; ++j) {
        const char* unit = base + (long long)j * kF16Unit;
        const int gl = gl0 + j;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const uint4 av = *reinterpret_cast<const uint4*>(unit + s * kF16Step + 16 * lane);
            uint2 bb = make_uint2(0u, 0u);
            if (xf.live) bb = xf.base[(gl * 4 + s) * xf.stride];
            const uint32_t A[4] = {av.x, av.y, av.z, av.w};
            mma_16816(as[s], A, bb.x, bb.y);
        }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] += (as[0][e] + as[1][e]) + (as[2][e] + as[3][e]);
}

// ------------------------------------------------------------ prologue ----
// RMSNorm gain of decode layer l into shared memory with cp.async (no registers
// held; it lands while the CTA still works on the layer before); build_x waits
// for its own copies, and its consumer barriers publish them.
__device__ __forceinline__ void prefetch_gamma(int l) {
    const Prog& p = prg();
    if (p.mode != MODE_DECODE || l >= p.L || !p.layers[l].gamma) return;
    __half* g = SM<__half>(ctx().pl.gam);
    const __half* src = p.layers[l].gamma;
    for (int i = threadIdx.x; i < p.d / 4; i += kConsumerThreads)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_u32(g + 4 * i)), "l"(src + 4 * i)
                     : "memory");
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
// x = fp16(RMSNorm(h) * gamma) for all tokens (decode; h updated by the previous
// layer's y first) or x = x_in; B fragments and group sums for this CTA's half
// of d.  The residual h stays in shared memory.  All global loads of a thread
// are issued before any is used (one round trip after the barrier).
__device__ __noinline__ void build_x(int l) {
    Ctx& c = ctx();
    const Prog& p = prg();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int B = p.B, d = p.d, n4 = B * d / 4;
    const bool decode = p.mode == MODE_DECODE;
    const LayerP& Ly = p.layers[l];
    __half* hs = SM<__half>(c.pl.hs);
    const float* y = (decode && l > 0) ? y_buf(c.par, p.layers[l - 1].sidx) : nullptr;
    const __half* hsrc = decode ? (l == 0 ? p.h_io : hs) : p.x_in;
    asm volatile("cp.async.wait_all;\n" ::: "memory");   // this thread's part of the gain
    uint2 hv[kMaxChunks];
    float4 yv[kMaxChunks];
#pragma unroll
    for (int j = 0; j < kMaxChunks; ++j) {
        const int i = tid + j * kConsumerThreads;
        if (i < n4) {
            hv[j] = *reinterpret_cast<const uint2*>(hsrc + 4 * i);
            if (y) yv[j] = __ldcg(reinterpret_cast<const float4*>(y + 4 * i));
        }
    }
    // h = fp16(h + y) into shared memory, sums of squares per token
    float ss[EDGE0_MAX_BATCH] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < kMaxChunks; ++j) {
        const int i = tid + j * kConsumerThreads;
        if (i < n4) {
            __half2 h01 = *reinterpret_cast<const __half2*>(&hv[j].x);
            __half2 h23 = *reinterpret_cast<const __half2*>(&hv[j].y);
            if (y) {
                h01 = __floats2half2_rn(__low2float(h01) + yv[j].x, __high2float(h01) + yv[j].y);
                h23 = __floats2half2_rn(__low2float(h23) + yv[j].z, __high2float(h23) + yv[j].w);
            }
            uint2 o;
            o.x = *reinterpret_cast<uint32_t*>(&h01);
            o.y = *reinterpret_cast<uint32_t*>(&h23);
            *reinterpret_cast<uint2*>(hs + 4 * i) = o;
            const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
            const float q = f01.x * f01.x + f01.y * f01.y + f23.x * f23.x + f23.y * f23.y;
            const int b = (4 * i) / d;
#pragma unroll
            for (int bb = 0; bb < EDGE0_MAX_BATCH; ++bb) if (bb == b) ss[bb] += q;
        }
    }
    float* red = SM<float>(c.pl.red);
    float* rs = red + B * kConsumerWarps;
    if (decode) {
        for (int b = 0; b < B; ++b) {
            const float sum = warp_sum(ss[b]);
            if (lane == 0) red[b * kConsumerWarps + wid] = sum;
        }
    }
    cbar();
    if (decode && tid < B) {
        float sum = 0.f;
        for (int w = 0; w < kConsumerWarps; ++w) sum += red[tid * kConsumerWarps + w];
        rs[tid] = rsqrtf(sum / (float)d + Ly.eps);
    }
    cbar();
    // x fragments and group sums of this CTA's half (the 16 threads of a group
    // are the 16 lanes of a half-warp)
    uint32_t* xf = SM<uint32_t>(c.pl.xf);
    float* xsum = SM<float>(c.pl.xsum);
    const __half* gam = (decode && Ly.gamma) ? SM<__half>(c.pl.gam) : nullptr;
    // one CTA keeps x of a head layer for the head flush
    __half* xs_out = (decode && c.cta == 0 && is_head_layer(p, l)) ? xs_buf(Ly.sidx) : nullptr;
#pragma unroll 1
    for (int j = 0; j * kConsumerThreads < n4; ++j) {
        const int i = tid + j * kConsumerThreads;
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        int b = 0, k = 0;
        if (i < n4) {
            b = (4 * i) / d;
            k = (4 * i) % d;
            const uint2 hh = *reinterpret_cast<const uint2*>(hs + 4 * i);
            const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&hh.x));
            const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&hh.y));
            x[0] = f01.x; x[1] = f01.y; x[2] = f23.x; x[3] = f23.y;
            if (decode) {
                float g4[4] = {1.f, 1.f, 1.f, 1.f};
                if (gam) {
                    const uint2 gg = *reinterpret_cast<const uint2*>(gam + k);
                    const float2 g01 = __half22float2(*reinterpret_cast<const __half2*>(&gg.x));
                    const float2 g23 = __half22float2(*reinterpret_cast<const __half2*>(&gg.y));
                    g4[0] = g01.x; g4[1] = g01.y; g4[2] = g23.x; g4[3] = g23.y;
                }
                const float r = rs[b];
                for (int e = 0; e < 4; ++e) x[e] = __half2float(__float2half_rn(x[e] * r * g4[e]));
            }
        }
        if (xs_out && i < n4) {
            const __half2 x01 = __floats2half2_rn(x[0], x[1]), x23 = __floats2half2_rn(x[2], x[3]);
            uint2 o;
            o.x = *reinterpret_cast<const uint32_t*>(&x01);
            o.y = *reinterpret_cast<const uint32_t*>(&x23);
            *reinterpret_cast<uint2*>(xs_out + 4 * i) = o;
        }
        float s4 = x[0] + x[1] + x[2] + x[3];
        for (int m = 8; m; m >>= 1) s4 += __shfl_xor_sync(0xffffffffu, s4, m);
        const int grp = k / kGroup;
        if (i < n4 && grp >= c.hv.gh0 && grp < c.hv.gh1) {
            const int kk = k % kGroup;
            const int sl = (grp - c.hv.gh0) * 4 + kk / 16;
            const int k1 = kk % 16, t1 = (k1 & 7) >> 1, w = k1 >> 3;
            const __half2 x01 = __floats2half2_rn(x[0], x[1]), x23 = __floats2half2_rn(x[2], x[3]);
            xf[((sl * B + b) * 4 + t1) * 2 + w] = *reinterpret_cast<const uint32_t*>(&x01);
            xf[((sl * B + b) * 4 + t1 + 1) * 2 + w] = *reinterpret_cast<const uint32_t*>(&x23);
            if ((lane & 15) == 0) xsum[(grp - c.hv.gh0) * B + b] = s4;
        }
    }
    cbar();
}

// ------------------------------------------------------------- phases -----
// g(tile, j0, j1, gl0) for each run of the units [a, b) of a unit item that lies
// in one row tile: units j0..j1-1 of the item, unit j is local group gl0 + j
template <class G>
__device__ __forceinline__ void tile_runs(const Item& it, int a, int b, G&& g) {
    const Ctx& c = ctx();
    const int ngh = c.hv.gh1 - c.hv.gh0;
    int j = a;
    while (j < b) {
        const int u = it.b + j, tile = u / ngh, grp = u - tile * ngh;
        const int e = b < j + (ngh - grp) ? b : j + (ngh - grp);
        g(tile, j, e, grp - j);
        j = e;
    }
}

// units of the unit items in [ia, ib) split over the warps; f(item, local unit
// range) runs on items the warp has units in; every item is released by every warp
template <class F>
__device__ bool warp_units(const LayerTab* T, int ia, int ib, F&& f, int wait_tag = -1) {
    const Ctx& c = ctx();
    const int wid = threadIdx.x >> 5;
    int tot = 0;
    for (int i = ia; i < ib; ++i)
        if (unit_kind(T->it[i].kind)) tot += T->it[i].n;
    int ua, ub;
    split_range(tot, kConsumerWarps, wid, &ua, &ub);
    int u = 0;
    bool ok = true;
    for (int i = ia; i < ib; ++i) {
        const Item& it = T->it[i];
        if (!unit_kind(it.kind)) continue;
        const int a = ua - u > 0 ? ua - u : 0, b = ub - u < it.n ? ub - u : it.n;
        u += it.n;
        if (a < b && ok) {
            if (!wait_item(T, i)) ok = false;
            else {
                if (wait_tag >= 0) { stamp(wait_tag); wait_tag = -1; }
                f(it, a, b);
            }
        }
        release_item(T, i);
    }
    return ok;
}

__device__ __forceinline__ bool seg_live(int l, const Seg& s) {
    const Ctx& c = ctx();
    return s.slot < 0 || s.slot < SM<int>(c.pl.ndist)[l];
}

// own router: partial logits of this CTA's units, into the layer's logits
__device__ bool phase_router(int l, const LayerTab* T) {
    Ctx& c = ctx();
    const Prog& p = prg();
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    float* lg = logr_buf(c.par, p.layers[l].sidx);
    return warp_units(T, 0, T->p1, [&](const Item& it, int a, int b) {
        tile_runs(it, a, b, [&](int tile, int j0, int j1, int gl0) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            f16_run(ring_at(it), j0, j1, gl0, acc);
            const int row = tile * kRowTile + g;
            if (t < p.B) {
                if (row < p.E) red_add_f32(lg + t * p.E + row, acc[0]);
                if (row + 8 < p.E) red_add_f32(lg + t * p.E + row + 8, acc[2]);
            }
        });
    });
}

// routing of an own-routed layer from its complete router logits
__device__ __noinline__ void route_layer(int l) {
    Ctx& c = ctx();
    const Prog& p = prg();
    const LayerP& Ly = p.layers[l];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    float* scr = SM<float>(c.pl.rscr);
    const float* lg = logr_buf(c.par, Ly.sidx);
    for (int i = tid; i < p.B * p.E; i += kConsumerThreads) {
        const int b = i / p.E, e = i - b * p.E;
        scr[b * 3 * p.E + e] = __ldcg(lg + i);
    }
    cbar();
    for (int b = wid; b < p.B; b += kConsumerWarps) {
        __shared__ int rid[EDGE0_MAX_BATCH][EDGE0_MAX_K];
        __shared__ float rw[EDGE0_MAX_BATCH][EDGE0_MAX_K];
        warp_route(scr + b * 3 * p.E, p.E, p.K, Ly.route_kind, Ly.n_groups, Ly.topk_groups,
                   Ly.route_scale, Ly.bias, scr + b * 3 * p.E + p.E, rid[b], rw[b], lane);
        if (lane < p.K) {
            ids_of(l)[b * p.K + lane] = rid[b][lane];
            w_of(l)[b * p.K + lane] = rw[b][lane];
        }
    }
    cbar();
    if (tid < 32) {
        const bool ok = make_dist_warp(l, lane);
        if (lane == 0) {
            if (!ok) raise_error(EDGE0_EINVAL);
            __threadfence_block();
            SM<volatile int>(c.pl.ready)[l] = 1;
        }
    }
    cbar();
}

// bounded wait (one thread) until a layer counter reaches `want`; false on
// abort or timeout
__device__ __noinline__ bool wait_count(const unsigned* cnt, unsigned want) {
    if (ld_acquire_u32(cnt) >= want) return true;
    const unsigned long long t0 = now_ns();
    for (unsigned it = 0; ld_acquire_u32(cnt) < want; ++it) {
        if ((it & 15) == 15) {
            if (should_abort()) return false;
            if (now_ns() - t0 > ctx().ctl->tmo) { raise_error(EDGE0_ETIMEOUT); return false; }
        }
    }
    return true;
}

// P1: partial gate/up sums of the pair's rows over this CTA's half of d; LoRA A
// units go straight into the layer's global sums, each warp counting the units it
// finished.  The warps take contiguous shares of the units; addresses come from
// registers (the table's constants loaded once, each item's fields once).  With
// LoRA on a shared pair, the last warp then waits for every LoRA A unit of the
// layer and loads the sums (A_gate x, A_up x) for the act.
__device__ bool phase1(int l, const LayerTab* T, bool lora_wait) {
    Ctx& c = ctx();
    const Prog& p = prg();
    const LayerP& Ly = p.layers[l];
    const int B = p.B;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
    float* part = SM<float>(c.pl.part);
    const char* ringb = g_smem + c.pl.ring;
    const int tok = g >> 1;
    const bool live = !(g & 1) && tok < B;
    const uint2* xfb = SM<uint2>(c.pl.xf) + (live ? tok : 0) * 4 + t;
    const int xstride = B * 4;
    const float* xs = SM<float>(c.pl.xsum);
    const int ngh = c.hv.gh1 - c.hv.gh0;
    const int k0 = T->k0, ia = T->p1, ib = T->p2;
    const int ndist = SM<int>(c.pl.ndist)[l];
    float* lora_g = lora_buf(c.par, Ly.sidx);
    int tot = 0;
    for (int i = ia; i < ib; ++i)
        if (unit_kind(T->it[i].kind)) tot += T->it[i].n;
    int ua, ub;
    split_range(tot, kConsumerWarps, wid, &ua, &ub);
    int u = 0;
    bool ok = true, first = true;
    for (int i = ia; i < ib; ++i) {
        const int kind = T->it[i].kind;
        if (!unit_kind(kind)) continue;
        const int in = T->it[i].n;
        const int a = ua - u > 0 ? ua - u : 0, b = ub - u < in ? ub - u : in;
        u += in;
        if (a < b && ok) {
            if (!mbar_wait(full_bar(k0 + i), item_parity(k0 + i))) {
                ok = false;
            } else {
                if (first) { stamp((l << 8) | 8); first = false; }
                const int ibase = T->it[i].b, seg = T->it[i].seg;
                const char* base = ringb + T->it[i].off;
                if (kind == IT_LA || kind == IT_LU) {
                    // one row tile (r <= 16 rows): units are groups ibase + j of this half
                    float as[4][4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) as[q][0] = as[q][1] = as[q][2] = as[q][3] = 0.f;
                    for (int j = a; j < b; ++j) {
                        const char* unit = base + j * kF16Unit;
                        const int gl = ibase + j;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint4 av = *reinterpret_cast<const uint4*>(unit + q * kF16Step + 16 * lane);
                            uint2 bb = make_uint2(0u, 0u);
                            if (live) bb = xfb[(gl * 4 + q) * xstride];
                            const uint32_t A[4] = {av.x, av.y, av.z, av.w};
                            mma_16816(as[q], A, bb.x, bb.y);
                        }
                    }
                    float* la = lora_g + (kind == IT_LA ? 0 : 16 * B);
                    if (t < B) {
                        red_add_f32(la + g * B + t, (as[0][0] + as[1][0]) + (as[2][0] + as[3][0]));
                        red_add_f32(la + (g + 8) * B + t, (as[0][2] + as[1][2]) + (as[2][2] + as[3][2]));
                    }
                    __threadfence();
                    __syncwarp();
                    if (lane == 0) red_release_add_u32(cnt_buf(c.par, Ly.sidx, CNT_LORA_A), (unsigned)(b - a));
                } else {
                    const int slot = T->pl.seg[seg].slot, hr0 = T->pl.seg[seg].hr0, hoff = T->pl.seg[seg].hoff;
                    if (slot < 0 || slot < ndist) {
                        // runs of units that lie in one row tile
                        int j = a;
                        while (j < b) {
                            const int uu = ibase + j, tile = uu / ngh, grp = uu - tile * ngh;
                            const int e = b < j + (ngh - grp) ? b : j + (ngh - grp);
                            const int gl0 = grp - j;
                            float r0 = 0.f, r1 = 0.f;
#pragma unroll 2
                            for (int jj = j; jj < e; ++jj) {
                                const char* unit = base + jj * kQ4Unit;
                                const uint4 wv = *reinterpret_cast<const uint4*>(unit + 16 * lane);
                                const uint2 sc = *reinterpret_cast<const uint2*>(unit + 512 + 8 * g);
                                const int gl = gl0 + jj;
                                const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
                                float as[4][4];
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    uint2 bb = make_uint2(0u, 0u);
                                    if (live) bb = xfb[(gl * 4 + q) * xstride];
                                    uint32_t A[4];
                                    q4_masks(w[q], A);
                                    as[q][0] = as[q][1] = as[q][2] = as[q][3] = 0.f;
                                    mma_16816(as[q], A, bb.x, bb.y);
                                }
                                const float a0 = (as[0][0] + as[1][0]) + (as[2][0] + as[3][0]);
                                const float a2 = (as[0][2] + as[1][2]) + (as[2][2] + as[3][2]);
                                const __half2 s0 = *reinterpret_cast<const __half2*>(&sc.x);
                                const __half2 s1 = *reinterpret_cast<const __half2*>(&sc.y);
                                const float xv = t < B ? xs[gl * B + t] : 0.f;
                                r0 += __low2float(s0) * kTwo24 * a0 + __high2float(s0) * xv;
                                r1 += __low2float(s1) * (kTwo24 / 16.0f) * a2 + __high2float(s1) * xv;
                            }
                            const int hl = hoff + tile - hr0;
                            if (t < B) {
                                atomicAdd(&part[(hl * 16 + g) * B + t], r0);
                                atomicAdd(&part[(hl * 16 + 8 + g) * B + t], r1);
                            }
                            j = e;
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(k0 + i));
    }
    if (lora_wait && wid == kConsumerWarps - 1) {
        // every LoRA A unit of the layer is in the global sums: load them
        bool w = true;
        if (lane == 0 && ok) w = wait_count(cnt_buf(c.par, Ly.sidx, CNT_LORA_A), 2u * (unsigned)(p.d / kGroup));
        w = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
        float* lsum = SM<float>(c.pl.vlo);
        if (ok && w)
            for (int q = lane; q < 32 * B; q += 32) lsum[q] = __ldcg(lora_g + q);
        ok = ok && w;
    }
    return ok;
}

// act = silu(gate) * up of all the pair's rows (partials of both CTAs, LoRA B
// terms for shared rows) -> hi/lo B fragments per 16-row quarter and their sums;
// for shared rows with LoRA, this CTA's half of the r entries of A_down act is
// added to the layer's v.  Every consumer thread runs every barrier here; the
// result is CTA-uniform.
__device__ bool compute_act(int l, const LayerTab* T, bool lora) {
    Ctx& c = ctx();
    const Prog& p = prg();
    const LayerP& Ly = p.layers[l];
    const int B = p.B, r = p.r, tid = threadIdx.x;
    const PairPlan& pl = T->pl;
    const float* part = SM<float>(c.pl.part);
    const float* recv = SM<float>(c.pl.recv);
    float* act32 = SM<float>(c.pl.act32);
    __half* af = SM<__half>(c.pl.af);
    float* qsum = SM<float>(c.pl.qsum);
    float* lsum = SM<float>(c.pl.vlo);   // A_gate x, A_up x of the layer (2 x 16 x B)
    float* lora_g = lora_buf(c.par, Ly.sidx);
    // LoRA items of the shared segment (segment 0 of a pair that owns shared rows)
    int ibg = -1, ibu = -1, iadt = -1, ssh = -1;
    bool ok = true;
    if (lora && pl.has_sh) {
        ssh = 0;
        ibg = T->ibg;
        ibu = T->ibu;
        iadt = T->iadt;
        ok = ibg >= 0 && ibu >= 0 && iadt >= 0;
        if (!ok && tid == 0) raise_error(EDGE0_EINVAL);
        // (the LoRA A sums were loaded into lsum at the end of P1)
        ok = ok && wait_item(T, ibg) && wait_item(T, ibu) && wait_item(T, iadt);
    }
    // af and qsum were cleared at the start of the layer
    ok = !cbar_or(!ok);
    stamp((l << 8) | 10);
    for (int i = tid; ok && i < pl.n_hr * 8 * B; i += kConsumerThreads) {
        const int hl = i / (8 * B), g = (i / B) % 8, b = i % B;
        int s = 0;
        while (s + 1 < pl.nseg && hl >= pl.seg[s + 1].hoff) ++s;
        const Seg& sg = pl.seg[s];
        float a = 0.f;
        if (seg_live(l, sg)) {
            const int row = (sg.hr0 + hl - sg.hoff) * kHalfRow + g;   // act row of the expert
            float gate = part[(hl * 16 + g) * B + b] + recv[(hl * 16 + g) * B + b];
            float up = part[(hl * 16 + 8 + g) * B + b] + recv[(hl * 16 + 8 + g) * B + b];
            if (s == ssh) {
                const int rl = row - sg.hr0 * kHalfRow;
                const __half* bg = reinterpret_cast<const __half*>(ring_at(T->it[ibg])) + rl * r;
                const __half* bu = reinterpret_cast<const __half*>(ring_at(T->it[ibu])) + rl * r;
                float dg = 0.f, du = 0.f;
                for (int q = 0; q < r; ++q) {
                    dg += __half2float(bg[q]) * lsum[q * B + b];
                    du += __half2float(bu[q]) * lsum[(16 + q) * B + b];
                }
                gate += Ly.lora_scale * dg;
                up += Ly.lora_scale * du;
            }
            a = silu_f(gate) * up;
            const int Ql = sg.qoff + row / 16 - sg.q0;
            const int k1 = row % 16, t1 = (k1 & 7) >> 1, w = k1 >> 3, sub = k1 & 1;
            const __half hi = __float2half_rn(a);
            const __half lo = __float2half_rn((a - __half2float(hi)) * kLoScale);
            af[(((Ql * B + b) * 2 + 0) * 4 + t1) * 4 + w * 2 + sub] = hi;
            af[(((Ql * B + b) * 2 + 1) * 4 + t1) * 4 + w * 2 + sub] = lo;
            atomicAdd(&qsum[Ql * B + b], a);
        }
        act32[(hl * 8 + g) * B + b] = a;
    }
    cbar();
    stamp((l << 8) | 11);
    // the non-unit P1 items (LoRA B rows of gate/up) are no longer needed; the
    // v warp keeps A_down^T until it has formed v (phase2)
    const bool vw = ssh >= 0 && (tid >> 5) == kVWarp;
    for (int i = T->p1; i < T->p2; ++i)
        if (!unit_kind(T->it[i].kind) && !(vw && i == iadt)) release_item(T, i);
    return !cbar_or(!ok);
}

// v[q][b] += sum over the pair's shared act rows of A_down[q][row] act[row][b]
// for q in this CTA's half of [0, r), by one warp (kVWarp) of a CTA that owns
// shared rows, while the other warps start the down rows; then the warp counts
// this CTA's shared rows and releases A_down^T.  Lane = (row phase js, output
// qi): each lane sums every fourth row of one q, two shuffles join the phases.
__device__ void lora_v_warp(int l, const LayerTab* T) {
    Ctx& c = ctx();
    const Prog& p = prg();
    const LayerP& Ly = p.layers[l];
    const int B = p.B, r = p.r, lane = threadIdx.x & 31;
    const PairPlan& pl = T->pl;
    const Seg& sg = pl.seg[0];
    const __half* adt = reinterpret_cast<const __half*>(ring_at(T->it[T->iadt]));
    const float* a32 = SM<float>(c.pl.act32) + sg.hoff * 8 * B;
    float* vg = lora_buf(c.par, Ly.sidx) + 32 * B;
    const int rows = (sg.hr1 - sg.hr0) * kHalfRow;
    const int q0 = c.rank ? r / 2 : 0, q1 = c.rank ? r : r / 2;
    const int qi = lane & 7, js = lane >> 3, q = q0 + qi;
    float acc[EDGE0_MAX_BATCH] = {0.f, 0.f, 0.f, 0.f};
    if (q < q1)
        for (int j = js; j < rows; j += 4) {
            const float a = __half2float(adt[j * r + q]);
#pragma unroll
            for (int b = 0; b < EDGE0_MAX_BATCH; ++b)
                if (b < B) acc[b] += a * a32[j * B + b];
        }
#pragma unroll
    for (int b = 0; b < EDGE0_MAX_BATCH; ++b) {
        acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], 8);
        acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], 16);
    }
    if (js == 0 && q < q1)
#pragma unroll
        for (int b = 0; b < EDGE0_MAX_BATCH; ++b)
            if (b < B) red_add_f32(vg + q * B + b, acc[b]);
    __syncwarp();
    if (lane == 0) {
        __threadfence();
        red_release_add_u32(cnt_buf(c.par, Ly.sidx, CNT_LORA_V), (unsigned)(sg.hr1 - sg.hr0));
    }
    release_item(T, T->iadt);
}

// P2: down rows of this CTA's half of d over the pair's act quarters -> y.  Each
// warp owns up to kMaxRtw consecutive row tiles and walks the layer's down groups
// once: the group's act fragments are loaded once, then every row tile of the
// warp runs its own accumulator chain.
constexpr int kMaxRtw = 4;   // row tiles of one warp (d <= kMaxD = 2048)
__device__ bool phase2(int l, const LayerTab* T, bool lora) {
    Ctx& c = ctx();
    const Prog& p = prg();
    const LayerP& Ly = p.layers[l];
    const int B = p.B, K = p.K, r = p.r, d = p.d;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
    const PairPlan& pl = T->pl;
    bool ok = true;
    if (lora && pl.has_sh && wid == kVWarp) lora_v_warp(l, T);
    for (int i = T->p2; i < T->p3 && ok; ++i) ok = wait_item(T, i);
    stamp((l << 8) | 9);
    if (ok && pl.n_hr > 0) {
        const uint2* afr = SM<uint2>(c.pl.af);
        const float* qsum = SM<float>(c.pl.qsum);
        const char* ring = g_smem + c.pl.ring;
        const int tok = g >> 1, part = g & 1;
        const bool blive = tok < B;
        const int nrt = c.hv.rt1 - c.hv.rt0;
        const int per = (nrt + kConsumerWarps - 1) / kConsumerWarps;
        const int i0 = wid * per;
        float y0[kMaxRtw], y1[kMaxRtw];
#pragma unroll
        for (int q = 0; q < kMaxRtw; ++q) y0[q] = y1[q] = 0.f;
        for (int di = 0; di < T->ndg; ++di) {
            const DGroup D = T->dg[di];
            const Seg& sg = pl.seg[D.seg];
            if (!seg_live(l, sg)) continue;
            // weight of the lane's token t for this segment's expert
            float w = 0.f;
            if (t < B) {
                if (sg.slot < 0) {
                    w = 1.f;
                } else {
                    const int e = dist_of(l)[sg.slot];
                    for (int k = 0; k < K; ++k)
                        if (ids_of(l)[t * K + k] == e) w += w_of(l)[t * K + k];
                }
            }
            uint2 bb[4];
            float qs = 0.f;
#pragma unroll
            for (int qi = 0; qi < 4; ++qi) {
                bb[qi] = make_uint2(0u, 0u);
                if (qi < D.nq) {
                    if (blive) bb[qi] = afr[(((D.ql0 + qi) * B + tok) * 2 + part) * 4 + t];
                    if (t < B) qs += qsum[(D.ql0 + qi) * B + t];
                }
            }
#pragma unroll
            for (int rr = 0; rr < kMaxRtw; ++rr) {
                const int i = i0 + rr;
                if (rr < per && i < nrt) {
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int qi = 0; qi < 4; ++qi) {
                        if (qi < D.nq) {
                            const uint32_t wq = *reinterpret_cast<const uint32_t*>(
                                ring + D.qoff[qi] + i * kQ4Quarter + 4 * lane);
                            uint32_t A[4];
                            q4_masks(wq, A);
                            mma_16816(acc, A, bb[qi].x, bb[qi].y);
                        }
                    }
                    const uint2 sc = *reinterpret_cast<const uint2*>(ring + D.soff + i * kQ4Scales + 8 * g);
                    const __half2 s0 = *reinterpret_cast<const __half2*>(&sc.x);
                    const __half2 s1 = *reinterpret_cast<const __half2*>(&sc.y);
                    y0[rr] += w * (__low2float(s0) * kTwo24 * (acc[0] + acc[1] * kLoInv) + __high2float(s0) * qs);
                    y1[rr] += w * (__low2float(s1) * (kTwo24 / 16.0f) * (acc[2] + acc[3] * kLoInv) +
                                   __high2float(s1) * qs);
                }
            }
        }
        // one vector reduction per 4 rows
        float* y = y_buf(c.par, Ly.sidx);
#pragma unroll
        for (int rr = 0; rr < kMaxRtw; ++rr) {
            const int i = i0 + rr;
            if (rr < per && i < nrt) {
                const int row = (c.hv.rt0 + i) * kRowTile + g;
                const float a0 = y0[rr], a1v = y1[rr];
                // rows g..g+3 of lanes with g % 4 == 0 as one vector reduction
                const float u1 = __shfl_down_sync(0xffffffffu, a0, 4), u2 = __shfl_down_sync(0xffffffffu, a0, 8),
                            u3 = __shfl_down_sync(0xffffffffu, a0, 12);
                const float v1 = __shfl_down_sync(0xffffffffu, a1v, 4), v2 = __shfl_down_sync(0xffffffffu, a1v, 8),
                            v3 = __shfl_down_sync(0xffffffffu, a1v, 12);
                if (t < B && (g & 3) == 0) {
                    red_add_v4_f32(y + (long long)t * d + row, a0, u1, u2, u3);
                    red_add_v4_f32(y + (long long)t * d + row + 8, a1v, v1, v2, v3);
                }
            }
        }
    }
    stamp((l << 8) | 12);
    // LoRA B_down rows of this CTA, once v is complete:
    // y[row] += scale * sum_q B_down[row][q] v[q]
    const int ibd = lora ? T->ibd : -1;
    if (ibd >= 0) {
        float* vs = SM<float>(c.pl.vlo);
        const int tid = threadIdx.x;
        const int n_sh = p.Is / kHalfRow;
        if (tid == 0 && ok) ok = wait_count(cnt_buf(c.par, Ly.sidx, CNT_LORA_V), 2u * (unsigned)n_sh);
        ok = !cbar_or(!ok);
        const float* vg = lora_buf(c.par, Ly.sidx) + 32 * B;
        for (int i = tid; ok && i < r * B; i += kConsumerThreads) vs[i] = __ldcg(vg + i);
        cbar();
        float* y = y_buf(c.par, Ly.sidx);
        for (int ii = ibd; ok && ii < T->p3; ++ii) {
            const Item& it = T->it[ii];
            if (it.kind != IT_BD) continue;
            const __half* bd = reinterpret_cast<const __half*>(ring_at(it));
            for (int i = tid; i < it.n * B; i += kConsumerThreads) {
                const int j = i / B, b = i % B;
                float s = 0.f;
                for (int q = 0; q < r; ++q) s += __half2float(bd[j * r + q]) * vs[q * B + b];
                red_add_f32(y + (long long)b * d + it.a + j, Ly.lora_scale * s);
            }
        }
    }
    for (int i = T->p2; i < T->p3; ++i) release_item(T, i);
    return ok;
}

// top-K of a head whose logits are complete (the last CTA to finish its head work)
__device__ __noinline__ void head_topk(int l) {
    Ctx& c = ctx();
    const Prog& p = prg();
    const LayerP& Ly = p.layers[l];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    float* scr = SM<float>(c.pl.rscr);
    const float* lg = logh_buf(c.par, Ly.sidx);
    for (int i = tid; i < p.B * p.E; i += kConsumerThreads) {
        const int b = i / p.E, e = i - b * p.E;
        const float v = __ldcg(lg + i);
        scr[b * 3 * p.E + e] = v;
        if (p.mode == MODE_HEAD && p.out_logits) p.out_logits[i] = v;
    }
    cbar();
    for (int b = wid; b < p.B; b += kConsumerWarps) {
        __shared__ int tid_[EDGE0_MAX_BATCH][EDGE0_MAX_K];
        __shared__ float tw_[EDGE0_MAX_BATCH][EDGE0_MAX_K];
        warp_route(scr + b * 3 * p.E, p.E, p.K, Ly.head_route_kind, Ly.head_n_groups, Ly.head_topk_groups,
                   Ly.head_route_scale, Ly.head_bias, scr + b * 3 * p.E + p.E, tid_[b], tw_[b], lane);
        if (lane < p.K) {
            if (p.mode == MODE_HEAD) {
                p.out_ids[b * p.K + lane] = tid_[b][lane];
                p.out_w[b * p.K + lane] = tw_[b][lane];
            } else {
                const long long o = (((long long)c.par * p.Ls + Ly.head_target) * p.B + b) * p.K + lane;
                p.pred_ids[o] = tid_[b][lane];
                p.pred_w[o] = tw_[b][lane];
            }
        }
    }
    cbar();
}

// x of head layer l over all of d as B fragments (the kept copy, or the input of
// a head-only call)
__device__ __noinline__ void load_x_full(int l) {
    Ctx& c = ctx();
    const Prog& p = prg();
    const int B = p.B, d = p.d, n4 = B * d / 4;
    const __half* src = p.mode == MODE_HEAD ? p.x_in : xs_buf(p.layers[l].sidx);
    uint32_t* xf = SM<uint32_t>(c.pl.xf);
    for (int i = threadIdx.x; i < n4; i += kConsumerThreads) {
        const int b = (4 * i) / d, k = (4 * i) % d;
        const uint2 v = __ldcg(reinterpret_cast<const uint2*>(src + 4 * i));
        const int sl = (k / kGroup) * 4 + (k % kGroup) / 16;
        const int k1 = k % 16, t1 = (k1 & 7) >> 1, w = k1 >> 3;
        xf[((sl * B + b) * 4 + t1) * 2 + w] = v.x;
        xf[((sl * B + b) * 4 + t1 + 1) * 2 + w] = v.y;
    }
    cbar();
}

// One table of the head flush: tasks [t0, t1) of head layer T->hl over all of d.
//   z = fc1 x + sum over executed e of fc1[:, d + e] + sum over previous e of
//       fc1[:, d + E + e]                       (16 rows per fc1 task)
//   logits += fc2[:, tile] GELU(z[tile])        (all E rows, per fc1 task)
//   logits += linear_init x + its one-hot columns  (16 rows per linear_init task)
// then the task count of the head; the CTA that completes it does the top-K.
// Every consumer thread runs every barrier; the result is CTA-uniform.
__device__ bool run_flush(int tl, const LayerTab* T, int& xl) {
    Ctx& c = ctx();
    const Prog& p = prg();
    const int l = T->hl;
    const LayerP& Ly = p.layers[l];
    const int B = p.B, K = p.K, E = p.E, H = p.H;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, g = lane >> 2, t = lane & 3;
    const int nH = H / kRowTile, hn0 = p.d / kGroup / 2;
    const int t0 = T->pl.hd0, t1 = T->pl.hd1;
    float* lg = logh_buf(c.par, Ly.sidx);
    float* zp = SM<float>(c.pl.zpart);   // [task][16][B]: z rows (fc1), logit rows (linear_init)
    if (xl != l) {
        load_x_full(l);
        xl = l;
    }
    stamp((tl << 8) | 20);
    for (int q = tid; q < (t1 - t0) * 16 * B; q += kConsumerThreads) zp[q] = 0.f;
    // one-hot columns of (task, row, token) = thread: loads issued before the units
    const int ti = tid / (16 * B), rr = (tid / B) % 16, bb = tid % B;
    const int task = t0 + ti;
    const bool mine = task < t1;
    float oh = 0.f;
    if (mine) {
        const int nprev = SM<int>(c.pl.nprv)[l];
        const int* ids = ids_of(l);
        const int* prv = prev_of(l);
        const __half* col = task < nH ? Ly.fc1_oh : Ly.linit_oh;
        const int stride = task < nH ? H : E;
        const int row = (task < nH ? task : task - nH) * kRowTile + rr;
        float v[2 * EDGE0_MAX_K];
#pragma unroll
        for (int k = 0; k < EDGE0_MAX_K; ++k) {
            v[k] = k < K ? __half2float(col[(long long)ids[bb * K + k] * stride + row]) : 0.f;
            v[EDGE0_MAX_K + k] = k < nprev ? __half2float(col[(long long)(E + prv[bb * K + k]) * stride + row]) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 2 * EDGE0_MAX_K; ++k) oh += v[k];
    }
    cbar();
    // fc1 and linear_init units of both halves of d.  Whole items are dealt to
    // the warps in turn (item i to warp i mod 16): the warps work on 16
    // consecutive items at once, so a table longer than the ring streams through
    // it, and each item's units (one row tile of one task) share one running sum.
    // The warp that processed an item releases it for all warps.
    bool ok = true;
    {
        const char* ringb = g_smem + c.pl.ring;
        const int tok = g >> 1;
        const bool live = !(g & 1) && tok < B;
        const uint2* xfb = SM<uint2>(c.pl.xf) + (live ? tok : 0) * 4 + t;
        const int xstride = B * 4;
        const int k0 = T->k0, n_units_items = T->p2;
        long long waited = 0, t_begin = clock64();   // trace: warp 0's waits and total
        for (int i = wid; i < n_units_items && ok; i += kConsumerWarps) {
            const int kind = T->it[i].kind, seg = T->it[i].seg, off = T->it[i].off, ib = T->it[i].b, in = T->it[i].n;
            const long long w0 = clock64();
            ok = mbar_wait(full_bar(k0 + i), item_parity(k0 + i));
            waited += clock64() - w0;
            if (ok) {
                // an item lies within one row tile of one half of d
                const int tile = ib / hn0, gl0 = ib - tile * hn0 + seg * hn0;
                const int tk = (kind == IT_FC1 ? tile : tile + nH) - t0;
                float as[4][4];
#pragma unroll
                for (int s = 0; s < 4; ++s) as[s][0] = as[s][1] = as[s][2] = as[s][3] = 0.f;
                const char* unit = ringb + off;
                for (int j = 0; j < in; ++j, unit += kF16Unit) {
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        const uint4 av = *reinterpret_cast<const uint4*>(unit + s * kF16Step + 16 * lane);
                        uint2 bb = make_uint2(0u, 0u);
                        if (live) bb = xfb[((gl0 + j) * 4 + s) * xstride];
                        const uint32_t A[4] = {av.x, av.y, av.z, av.w};
                        mma_16816(as[s], A, bb.x, bb.y);
                    }
                }
                if (t < B) {
                    atomicAdd(&zp[(tk * 16 + g) * B + t], (as[0][0] + as[1][0]) + (as[2][0] + as[3][0]));
                    atomicAdd(&zp[(tk * 16 + 8 + g) * B + t], (as[0][2] + as[1][2]) + (as[2][2] + as[3][2]));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_n(empty_bar(k0 + i), kConsumerWarps);
        }
        stamp_value((tl << 8) | 0x3E, (unsigned long long)(clock64() - t_begin));
        stamp_value((tl << 8) | 0x3F, (unsigned long long)waited);
    }
    ok = !cbar_or(!ok || aborted());
    stamp((tl << 8) | 21);
    // GELU (erf form) of the fc1 rows -> hi/lo B fragments per fc1 task; the
    // linear_init rows (with their one-hot columns) go into the logits
    __half* gf = SM<__half>(c.pl.gf);
    if (ok && mine) {
        if (task < nH) {
            const float z = zp[(ti * 16 + rr) * B + bb] + oh;
            const float gl = 0.5f * z * (1.0f + erff(z * 0.70710678118654752f));
            const int t1f = (rr & 7) >> 1, w = rr >> 3, sub = rr & 1;
            const __half hi = __float2half_rn(gl);
            const __half lo = __float2half_rn((gl - __half2float(hi)) * kLoScale);
            gf[(((ti * B + bb) * 2 + 0) * 4 + t1f) * 4 + w * 2 + sub] = hi;
            gf[(((ti * B + bb) * 2 + 1) * 4 + t1f) * 4 + w * 2 + sub] = lo;
        } else {
            red_add_f32(lg + bb * E + (task - nH) * kRowTile + rr, zp[(ti * 16 + rr) * B + bb] + oh);
        }
    }
    cbar();
    // fc2: the column block of each fc1 task over all E rows, from global memory
    // (K-major: block `task`, row tile e at (task E/16 + e) 512 B); one (task, row
    // tile) per warp in turn, the sum over tasks kept per row tile
    {
        const int nE = E / kRowTile, nf = (t1 < nH ? t1 : nH) - t0;
        const int tok = g >> 1, prt = g & 1;
        for (int e = wid; ok && nf > 0 && e < nE; e += kConsumerWarps) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int f = 0; f < nf; ++f) {
                const uint4 av = __ldg(reinterpret_cast<const uint4*>(
                    Ly.fc2 + ((long long)(t0 + f) * nE + e) * kF16Step + 16 * lane));
                uint2 bq = make_uint2(0u, 0u);
                if (tok < B) bq = SM<uint2>(c.pl.gf)[(f * B + tok) * 8 + prt * 4 + t];
                const uint32_t A[4] = {av.x, av.y, av.z, av.w};
                mma_16816(acc, A, bq.x, bq.y);
            }
            const int row = e * kRowTile + g;
            if (t < B) {
                red_add_f32(lg + t * E + row, acc[0] + acc[1] * kLoInv);
                red_add_f32(lg + t * E + row + 8, acc[2] + acc[3] * kLoInv);
            }
        }
    }
    ok = !cbar_or(!ok);
    stamp((tl << 8) | 22);
    // count this table's tasks; the CTA that completes the head does its top-K
    __threadfence();
    cbar();
    if (tid == 0) {
        const unsigned n = (unsigned)(t1 - t0);
        const unsigned old = atom_acq_rel_add_u32(cnt_buf(c.par, Ly.sidx, CNT_HEAD), n);
        c.ctl->last = ok && old + n == (unsigned)head_tasks(p);
    }
    cbar();
    if (c.ctl->last) head_topk(l);
    stamp((tl << 8) | 23);
    return !cbar_or(!ok);
}

// ------------------------------------------------------------ the kernel ---
__device__ void consumer() {
    Ctx& c = ctx();
    const Prog& p = prg();
    const int tid = threadIdx.x;
    const int B = p.B, d = p.d;
    unsigned long long bar_target = 0;
    if (tid == 0) {
        const unsigned long long v = ld_acquire_u64(&c.hdr->barrier);
        bar_target = v - v % (unsigned long long)c.nct;
    }
    uint32_t xph1 = 0;
    volatile int* ready = SM<volatile int>(c.pl.ready);
    {
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        stamp_value(0xFFF00, smid);   // trace: the SM this CTA runs on
    }
    float* part = SM<float>(c.pl.part);
    prefetch_gamma(0);
    // every decision to leave the loop is taken from a barrier reduction, so all
    // consumer threads leave together
    const int nl = n_layer_tabs(p);
    for (int l = 0; l < nl; ++l) {
        const LayerP& Ly = p.layers[l];
        LayerTab* T = tab_of(l);
        stamp((l << 8) | 0);
        if (tid == 0) wait_flag(&T->seq, l + 1);
        if (cbar_or(aborted())) break;
        const bool router = has_router_phase(p, l, c.step);
        const Shape Sh = layer_shape(p, l, router);
        for (int q = tid; q < T->pl.n_hr * 16 * B; q += kConsumerThreads) part[q] = 0.f;
        {
            // act fragments and quarter sums of this layer start at zero (partial quarters)
            uint32_t* af = SM<uint32_t>(c.pl.af);
            float* qsum = SM<float>(c.pl.qsum);
            for (int q = tid; q < T->pl.n_q * B * 2 * 4 * 2; q += kConsumerThreads) af[q] = 0u;
            for (int q = tid; q < T->pl.n_q * B; q += kConsumerThreads) qsum[q] = 0.f;
        }
        // ---------------- input x
        if (p.mode == MODE_DECODE && l > 0)
            if (!bar_wait(bar_target)) break;
        stamp((l << 8) | 24);   // the previous layer's grid barrier seen
        if (p.mode == MODE_DECODE || l == 0) build_x(l);
        prefetch_gamma(l + 1);   // build_x(l) is done with the gain of layer l
        stamp((l << 8) | 1);
        // ---------------- own routing
        if (router) {
            const bool ok = phase_router(l, T);
            if (cbar_or(!ok || aborted())) break;
            stamp((l << 8) | 40);   // router units done
            bar_arrive();
            if (!bar_wait(bar_target)) break;
            stamp((l << 8) | 42);   // the router barrier seen
            route_layer(l);
        }
        if (p.mode == MODE_DECODE && c.cta == 0) {
            for (int i = tid; i < B * p.K; i += kConsumerThreads)
                p.exec_ids[(((long long)c.par * p.Ls + Ly.sidx) * B) * p.K + i] = ids_of(l)[i];
        }
        if (ready[l] != 1) {
            if (tid == 0) raise_error(EDGE0_EINVAL);
            cbar();
            break;
        }
        stamp((l << 8) | 2);
        // ---------------- P1: gate/up partials, swap with the peer, act
        bool ok = phase1(l, T, Sh.lora && T->pl.has_sh);
        if (cbar_or(!ok || aborted())) break;
        stamp((l << 8) | 3);
        if (T->pl.n_hr > 0) {
            const int nmsg = T->pl.n_hr * 16 * B;
            ok = exchange(0, part, SM<float>(c.pl.recv), nmsg, xph1);
            if (cbar_or(!ok)) break;
        }
        stamp((l << 8) | 4);
        if (!compute_act(l, T, Sh.lora != 0)) break;
        stamp((l << 8) | 5);
        // ---------------- P2: down -> y, then this layer's barrier
        ok = phase2(l, T, Sh.lora != 0);
        if (cbar_or(!ok || aborted())) break;
        bar_arrive();
        stamp((l << 8) | 6);
        if (cbar_or(aborted())) break;
        if (tid == 0) *(volatile int*)&c.ctl->cdone = l + 1;
    }
    if (cbar_or(aborted())) return;
    if (nl > 0) {
        // ---------------- tail: the last layer's y is complete after its barrier
        if (!bar_wait(bar_target)) return;
        stamp((nl << 8) | 7);
        const float* Y = y_buf(c.par, p.layers[p.L - 1].sidx);
        const long long n = (long long)B * d;
        const long long a = n * c.cta / c.nct, b = n * (c.cta + 1) / c.nct;
        if (p.mode == MODE_DECODE) {
            const __half* hs = SM<__half>(c.pl.hs);
            for (long long i = a + tid; i < b; i += kConsumerThreads)
                p.h_io[i] = __float2half_rn(__half2float(hs[i]) + __ldcg(Y + i));
        } else if (p.mode == MODE_MOE) {
            for (long long i = a + tid; i < b; i += kConsumerThreads) p.y_out[i] = __float2half_rn(__ldcg(Y + i));
        }
    }
    // ---------------- head flush: every head layer's x and routing are final here
    int xl = -1;
    for (int j = 0;; ++j) {
        int hl, t0, t1;
        if (!flush_table(p, c.nct, c.cta, j, &hl, &t0, &t1)) break;
        const int tl = nl + j;
        LayerTab* T = tab_of(tl);
        if (tid == 0) wait_flag(&T->seq, tl + 1);
        if (cbar_or(aborted())) return;
        if (!run_flush(tl, T, xl)) return;
        if (tid == 0) *(volatile int*)&c.ctl->cdone = tl + 1;
    }
    if (c.cta == 0 && tid == 0 && p.step < 0) c.hdr->step = c.step + 1;
}

// The pair shape is part of the kernel (compile-time cluster dimensions): every
// launch of it, a profiler's replay included, runs in CTA pairs.
__global__ void __cluster_dims__(kClusterCtas, 1, 1) __launch_bounds__(kThreads, 1)
    engine_kernel(const __grid_constant__ Prog prog) {
    const int tid = threadIdx.x;
    // parameters and context into shared memory
    {
        const uint4* src = reinterpret_cast<const uint4*>(&prog);
        uint4* dst = reinterpret_cast<uint4*>(g_smem + kProgOff);
        for (int i = tid; i < (int)(sizeof(Prog) / 16); i += kThreads) dst[i] = src[i];
        if (tid == 0) {
            const char* s8 = reinterpret_cast<const char*>(&prog);
            for (int i = (int)(sizeof(Prog) / 16) * 16; i < (int)sizeof(Prog); ++i) g_smem[kProgOff + i] = s8[i];
            Ctx& cc = ctx();
            cc.pl = make_plan(prog, kCtxOff + kCtxBytes);
            cc.hdr = reinterpret_cast<WsHeader*>(prog.ws);
            cc.ctl = reinterpret_cast<Ctl*>(g_smem + cc.pl.ctl);
            cc.ws = ws_layout(prog.Ls, prog.B, prog.d, prog.E);
            cc.nct = gridDim.x;
            cc.cta = blockIdx.x;
            cc.rank = (int)cluster_ctarank();
            cc.pair = cc.cta / kClusterCtas;
            cc.P = cc.nct / kClusterCtas;
            cc.hv = halves(prog.d, prog.E, cc.rank);
        }
        __syncthreads();
    }
    Ctx& c = ctx();
    const Prog& p = prg();

    // the pair exchange addresses the other CTA of a two-CTA cluster: a launch
    // without that cluster shape records an error and touches no other CTA
    uint32_t ncl;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(ncl));
    if (ncl != (uint32_t)kClusterCtas || gridDim.x % kClusterCtas) {
        if (tid == 0) {
            atomicCAS(&c.hdr->error, 0, EDGE0_EUNSUPPORTED);
            atomicExch(&c.hdr->abort, 1);
        }
        return;
    }

    if (tid == 0) {
        Ctl* ctl = c.ctl;
        ctl->abort = 0;
        ctl->cdone = 0;
        ctl->issued = 0;
        ctl->last = 0;
        ctl->bar_seen = 0;
        ctl->step = p.step >= 0 ? p.step : ld_volatile_s32(&c.hdr->step);
        ctl->trace = c.cta < kTraceCtas ? ld_volatile_s32(&c.hdr->trace) : 0;
        const unsigned long long wn = ld_relaxed_u64(&c.hdr->wait_ns);
        ctl->tmo = wn ? wn : kDefaultWaitNs;
        ctl->tslot = 0;
        ctl->ptslot = kTraceProducer;
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(SM<uint64_t>(c.pl.full) + s, 1);
            mbar_init(SM<uint64_t>(c.pl.empty) + s, kConsumerWarps);
        }
        mbar_init(SM<uint64_t>(c.pl.xch) + 0, 1);
        mbar_init(SM<uint64_t>(c.pl.xch) + 1, 1);
        fence_mbar_init();
    }
    for (int i = tid; i < kTables; i += kThreads) tab_of(i)->seq = 0;
    __syncthreads();
    c.step = c.ctl->step;
    c.par = c.step & 1;
    // clear the other step parity of this launch's layers for the next step
    {
        const int op = c.par ^ 1;
        const long long per_y = (long long)p.B * p.d, per_l = (long long)p.B * p.E,
                        per_a = (long long)p.B * kLoraAcc, per = per_y + 2 * per_l + per_a;
        const long long tot = (long long)p.L * per;
        const long long a = tot * c.cta / c.nct, b = tot * (c.cta + 1) / c.nct;
        for (long long i = a + tid; i < b; i += kThreads) {
            const long long l = i / per, o = i % per;
            const int sidx = p.layers[l].sidx;
            if (o < per_y) y_buf(op, sidx)[o] = 0.f;
            else if (o < per_y + per_l) logr_buf(op, sidx)[o - per_y] = 0.f;
            else if (o < per_y + 2 * per_l) logh_buf(op, sidx)[o - per_y - per_l] = 0.f;
            else lora_buf(op, sidx)[o - per_y - 2 * per_l] = 0.f;
        }
        if (c.cta == 0)
            for (int i = tid; i < p.L * kLayerCounters; i += kThreads)
                cnt_buf(op, p.layers[i / kLayerCounters].sidx, 0)[i % kLayerCounters] = 0u;
    }
    // routing known at launch: predictions (prerouted layers, step > 0) or inputs;
    // previous-token ids of head layers
    for (int l = tid; l < p.L; l += kThreads) {
        const LayerP& Ly = p.layers[l];
        const int BK = p.B * p.K;
        const int32_t* src_i = nullptr;
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
        int flag = 0;
        if (src_i) {
            for (int i = 0; i < BK; ++i) {
                ids_of(l)[i] = src_i[i];
                w_of(l)[i] = src_w ? src_w[i] : 0.f;
            }
            if (!make_dist(l)) raise_error(EDGE0_EINVAL);
            flag = 1;
        }
        const int32_t* pv = nullptr;
        if (p.mode == MODE_HEAD) pv = p.prev_in;
        else if (p.mode == MODE_DECODE && (Ly.flags & LF_HEAD) && c.step > 0)
            pv = p.exec_ids + (((long long)((c.step - 1) & 1) * p.Ls + Ly.sidx) * p.B) * p.K;
        if (pv) {
            for (int i = 0; i < BK; ++i) {
                const int e = pv[i];
                if (e < 0 || e >= p.E) raise_error(EDGE0_EINVAL);
                prev_of(l)[i] = e < 0 || e >= p.E ? 0 : e;
            }
        }
        SM<int>(c.pl.nprv)[l] = pv ? p.K : 0;
        SM<volatile int>(c.pl.ready)[l] = flag;
    }
    __syncthreads();
    // the peer's barriers exist before any exchange
    cluster_sync_all();

    if (tid >= kConsumerThreads) {
        producer();   // the whole producer warp
        __syncwarp();
    } else {
        consumer();
        asm volatile("cp.async.wait_all;\n" ::: "memory");   // no gain copy outlives the CTA
    }
    __syncthreads();
    if (tid == 0 && aborted()) {
        // let copies still in flight into this CTA's ring land before it exits (bounded)
        const int issued = *(volatile int*)&c.ctl->issued;
        const unsigned long long t0 = now_ns();
        for (int k = issued > kSlots ? issued - kSlots : 0; k < issued; ++k)
            while (!mbar_try_wait(full_bar(k), item_parity(k)))
                if (now_ns() - t0 > 100000000ull) break;
        while (now_ns() - t0 < 20000ull) {}   // stores from the peer still in flight
    }
    __syncthreads();
    // neither CTA of a pair leaves while the other may still write into it
    cluster_sync_all();
}

// ------------------------------------------------------------------ host ---
namespace {
std::mutex g_grid_mutex;
int g_grid[64] = {};
int g_smem_max[64] = {};
}  // namespace

int engine_grid(int* nct) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return EDGE0_ECUDA;
    std::lock_guard<std::mutex> lock(g_grid_mutex);
    if (!g_grid[dev]) {
        int maxsm = 0;
        if (cudaDeviceGetAttribute(&maxsm, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return EDGE0_ECUDA;
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, engine_kernel) != cudaSuccess) return EDGE0_ECUDA;
        const int dyn = maxsm - (int)fa.sharedSizeBytes;
        if (cudaFuncSetAttribute(engine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn) != cudaSuccess)
            return EDGE0_ECUDA;
        // (the cluster shape comes from the kernel's compile-time dimensions)
        cudaLaunchConfig_t cfg;
        memset(&cfg, 0, sizeof(cfg));
        cfg.gridDim = dim3(kClusterCtas);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = dyn;
        int ncl = 0;
        if (cudaOccupancyMaxActiveClusters(&ncl, (void*)engine_kernel, &cfg) != cudaSuccess || ncl < 2)
            return EDGE0_ECUDA;
        g_grid[dev] = ncl * kClusterCtas;
        g_smem_max[dev] = dyn;
    }
    *nct = g_grid[dev];
    return EDGE0_OK;
}

int engine_smem_max() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(g_grid_mutex);
    return g_smem_max[dev];
}

// Derived launch fields for one set of shapes and grid: the pair-plan maxima over
// every kind of layer (shared expert, LoRA, own router: all 8 combinations), the
// ring that fits next to the fixed buffers, and the head flush's table size.
struct Derived {
    int mode, B, K, d, E, I, Is, H, r, nct, smem_max;
    int rc, slots_max, ps[2], hr_max, q_max, ring_bytes, ft, smem;
};

static int derive(Derived& D) {
    Prog p;
    memset(&p, 0, sizeof(p));
    p.mode = D.mode; p.L = 1; p.B = D.B; p.K = D.K; p.d = D.d; p.E = D.E; p.I = D.I; p.Is = D.Is;
    p.H = D.H; p.r = D.r;
    if (D.nct < 2 * kClusterCtas || D.nct % kClusterCtas) return EDGE0_EUNSUPPORTED;
    if (p.B <= 0 || p.B > EDGE0_MAX_BATCH) return EDGE0_EINVAL;
    if (p.d % 128 || p.d > kMaxD || p.E % kRowTile || p.H % 64 || p.I % 64 || p.Is % 64)
        return EDGE0_EUNSUPPORTED;
    if ((long long)p.B * p.d / 4 > (long long)kMaxChunks * kConsumerThreads) return EDGE0_EUNSUPPORTED;
    if (p.r <= 0 || p.r > 16) return EDGE0_EUNSUPPORTED;
    p.slots_max = p.mode == MODE_HEAD ? 0 : (p.B * p.K < p.E ? p.B * p.K : p.E);
    const int P = D.nct / kClusterCtas;
    // the plan's 32-bit splits: n * parts stays below 2^31
    if ((long long)(p.slots_max * (p.I / kHalfRow) + p.Is) * P >= (1LL << 31)) return EDGE0_EUNSUPPORTED;
    for (int f = 0; f < 2; ++f) p.ps[f] = shared_pairs(P, p.Is / kHalfRow, p.slots_max * (p.I / kHalfRow), f);
    p.ft = flush_tasks_max(p.B);
    if ((long long)EDGE0_MAX_LAYERS * head_tasks(p) * D.nct >= (1LL << 31)) return EDGE0_EUNSUPPORTED;
    p.hr_max = 1;
    p.q_max = 1;
    LayerTab T;   // scratch on the stack: the allocation-free entry point comes here too
    // one layer per combination of parts, in both passes (maxima, then ring capacity)
    for (int pass = 0; pass < 2; ++pass) {
        for (int combo = 0; combo < 8; ++combo) {
            p.layers[0].flags = ((combo & 1) ? LF_SHARED : 0) | ((combo & 2) ? LF_LORA : 0);
            const bool router = (combo & 4) && p.mode == MODE_DECODE;
            const Shape S = layer_shape(p, 0, router);
            for (int pair = 0; pair < P; ++pair)
                for (int rank = 0; rank < kClusterCtas; ++rank) {
                    int lin = 0;
                    if (!build_items(S, P, pair, rank, 1 << 30, &T, lin)) return EDGE0_EUNSUPPORTED;
                    if (pass == 0) {
                        if (T.pl.n_hr > p.hr_max) p.hr_max = T.pl.n_hr;
                        if (T.pl.n_q > p.q_max) p.q_max = T.pl.n_q;
                    } else {
                        // the consumers hold all down items of a layer (and the LoRA B
                        // rows) at once: they must fit in the ring next to one item of
                        // slack for the wrap-around
                        long long held = 0;
                        for (int i = T.p1; i < T.p3; ++i)
                            if (!unit_kind(T.it[i].kind)) held += T.it[i].bytes;
                        if (held + kItemMax > p.ring_bytes) return EDGE0_EUNSUPPORTED;
                    }
                }
        }
        if (pass == 0) {
            p.L = EDGE0_MAX_LAYERS;   // the fixed buffers of the largest call
            p.ring_bytes = 0;
            const int fixed = make_plan(p, kCtxOff + kCtxBytes).total;
            p.ring_bytes = ((D.smem_max - fixed) / 16) * 16;
            if (p.ring_bytes < kMinRing) return EDGE0_EUNSUPPORTED;
        }
    }
    // head flush tables: the fc2 items of a table are held until its fc2 step, next
    // to one item of slack; fewer tasks per table where the ring is short
    if (p.mode != MODE_MOE) {
        const int fc2b = (p.E / kRowTile) * kF16Step;
        if (fc2b > kItemMax) return EDGE0_EUNSUPPORTED;
        const int fit = (p.ring_bytes - kItemMax) / fc2b;
        if (fit < 1) return EDGE0_EUNSUPPORTED;
        if (p.ft > fit) p.ft = fit;
        const int nt = head_tasks(p);
        for (int t0 = 0; t0 < nt; t0 += p.ft) {
            const int t1 = t0 + p.ft < nt ? t0 + p.ft : nt;
            int lin = 0;
            if (!build_flush_items(p, 0, t0, t1, 1 << 30, &T, lin)) return EDGE0_EUNSUPPORTED;
            long long held = 0;
            for (int i = T.p2; i < T.n; ++i) held += T.it[i].bytes;
            if (held + kItemMax > p.ring_bytes) return EDGE0_EUNSUPPORTED;
        }
    }
    D.slots_max = p.slots_max;
    for (int f = 0; f < 2; ++f) D.ps[f] = p.ps[f];
    D.ft = p.ft;
    D.hr_max = p.hr_max;
    D.q_max = p.q_max;
    D.ring_bytes = p.ring_bytes;
    D.smem = make_plan(p, kCtxOff + kCtxBytes).total;
    return EDGE0_OK;
}

namespace {
constexpr int kDerivedCache = 16;
Derived g_derived[kDerivedCache];
int g_derived_n = 0, g_derived_next = 0;
}  // namespace

// Fills the derived fields of p for a grid of nct CTAs and checks the shapes
// against the engine's limits (cached per shape set; allocates nothing).
int engine_check(Prog& p, int nct, int smem_max, int* smem_bytes) {
    if (p.L <= 0 || p.L > EDGE0_MAX_LAYERS) return EDGE0_EINVAL;
    Derived key;
    memset(&key, 0, sizeof(key));
    key.mode = p.mode; key.B = p.B; key.K = p.K; key.d = p.d; key.E = p.E; key.I = p.I;
    key.Is = p.Is; key.H = p.H; key.r = p.r; key.nct = nct; key.smem_max = smem_max;
    std::lock_guard<std::mutex> lock(g_grid_mutex);
    int hit = -1;
    for (int i = 0; i < g_derived_n; ++i) {
        const Derived& d = g_derived[i];
        if (d.mode == key.mode && d.B == key.B && d.K == key.K && d.d == key.d && d.E == key.E &&
            d.I == key.I && d.Is == key.Is && d.H == key.H && d.r == key.r && d.nct == key.nct &&
            d.smem_max == key.smem_max) { hit = i; break; }
    }
    if (hit < 0) {
        key.rc = derive(key);
        hit = g_derived_next;
        g_derived[hit] = key;
        g_derived_next = (g_derived_next + 1) % kDerivedCache;
        if (g_derived_n < kDerivedCache) ++g_derived_n;
    }
    const Derived& d = g_derived[hit];
    if (d.rc) return d.rc;
    p.slots_max = d.slots_max;
    for (int f = 0; f < 2; ++f) p.ps[f] = d.ps[f];
    p.ft = d.ft;
    p.hr_max = d.hr_max;
    p.q_max = d.q_max;
    p.ring_bytes = d.ring_bytes;
    // the fixed buffers of this call's L are no larger than those the ring was sized with
    *smem_bytes = make_plan(p, kCtxOff + kCtxBytes).total;
    return EDGE0_OK;
}

int engine_launch(Prog& p, cudaStream_t stream) {
    int nct = 0;
    int rc = engine_grid(&nct);
    if (rc) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    int smem = 0;
    rc = engine_check(p, nct, g_smem_max[dev], &smem);
    if (rc) return rc;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(nct);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];   // the cluster shape is compiled into the kernel
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, engine_kernel, p) != cudaSuccess) return EDGE0_ECUDA;
    return EDGE0_OK;
}

}  // namespace edge0
