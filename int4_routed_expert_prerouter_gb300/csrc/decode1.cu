// Batch-1 decode kernel: one persistent launch runs every layer of a decode
// step for one sequence, and every prerouter head of the step.
//
// What one layer computes ("The Other Half of the Memory Wall": S3.1 "Math
// contract", S3.2 "Head", "Motivation", "Prediction-as-routing", S3.3):
//   x = fp16(RMSNorm(h) * gamma)
//   routing = the upstream head's prediction made one token earlier, or the
//             layer's own router + its routing rule (App. A)
//   y = sum_k w_k expert_{id_k}(x) + shared(x), expert = down(silu(gate) * up)
//       with int4 affine group-64 weights, the shared expert's gate, up and
//       down carrying unmerged LoRA deltas (alpha / r) B A v
//   h = fp16(h + y)
//
// Data flow.  Every value that crosses CTAs is a single-writer word: an fp32
// value (or an id) and the launch's 32-bit tag stored together as one 64-bit
// word, which is single-copy atomic; readers poll a word until it carries
// their tag.  No counters, fences or grid barriers stand between the layers:
// a CTA waits for exactly the words it reads.
//   * Gate/up: CTA pairs (clusters of two) own runs of half-row tiles ("hr": 8
//     act rows; the packed tile interleaves 8 gate and 8 up rows).  The two CTAs
//     split d in halves and swap partial sums through distributed shared
//     memory.  Routed pairs take the K routed slots' hr, shared pairs the shared
//     expert's (with its LoRA B_gate / B_up terms), one LoRA pair forms A_gate x
//     and A_up x and publishes them.  Each CTA of a pair publishes the act rows
//     of its parity (w_k act for routed rows).
//   * Down: CTA c < d/16 owns output row tile c.  It reads every act value of
//     the layer, applies that tile of every expert's down (and of the shared
//     expert's, with (alpha / r) B_down A_down act) and publishes the tile's y.
//   * Every CTA reads all of y to form the next layer's x; on a layer that
//     routes itself the last E/16 CTAs publish one router row tile each.
// Weights move by a producer warp: cp.async.bulk copies into a byte ring of
// shared memory, one block per (layer, phase) with its own mbarrier; blocks
// that depend only on predictions known at launch stream ahead of the compute
// by as many layers as the ring holds.  int4 nibbles enter m16n8k16
// tensor-core steps as fp16 subnormals (q 2^-24) through single masks; fp32
// activations travel as hi + lo fp16 columns.
//
// Every wait is bounded by the workspace's wait limit; on expiry the kernel
// records EDGE0_ETIMEOUT, sets the abort flag and leaves.
#include <stddef.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "internal.cuh"

namespace edge0 {
namespace d1 {

constexpr int kCW = 16;                  // consumer warps
constexpr int kCT = kCW * 32;            // consumer threads
constexpr int kT1 = kCT + 32;            // + the producer warp
constexpr int kMaxHr1 = 8;               // hr of one pair
constexpr int kMaxSeg1 = 3;              // expert runs of one pair
constexpr int kMaxPc = 24;               // copies of one block
constexpr int kBlocks = 16;              // block barriers
constexpr int kPieceMax = 32768;         // bytes of one bulk copy
constexpr int kMaxD1 = 2048;
constexpr int kMaxG1 = kMaxD1 / kGroup;  // groups of d
constexpr int kMaxNA = 4608;             // act values of a layer: K I + Is
constexpr int kMaxNS = kMaxNA / 16;      // their 16-row steps
constexpr int kMaxNG = kMaxNA / kGroup;  // their groups
constexpr int kPP = (kMaxNA / 2 + kCT - 1) / kCT;   // act word pairs of one thread
constexpr int kMsg = kMaxHr1 * 16;       // partial sums a pair exchanges
constexpr int kMaxK1 = EDGE0_MAX_K;
constexpr unsigned kTagMask = 0x3FFFFFFFu;   // launch tags: 1 .. kTagMask
constexpr unsigned kHoldBit = 0x40000000u;   // never in a written tag

__host__ __device__ inline void split1(int n, int parts, int i, int* a, int* b) {
    *a = (int)((long long)n * i / parts);
    *b = (int)((long long)n * (i + 1) / parts);
}
__host__ __device__ inline int ngh1(int d, int rank) {
    const int ng = d / kGroup;
    return rank ? ng - ng / 2 : ng / 2;
}

// ------------------------------------------------------------------ plan ----
struct Shape1 {
    int d, I, Is, E, K, H, r;
    int shared, lora;          // every layer of the launch has a shared expert / LoRA
    int P, Pr, Ps, Pl;         // pairs: all, routed, shared, LoRA
    int nct;                   // CTAs (2 P)
    int n_heads;
};
__host__ __device__ inline int n_act1(const Shape1& S) { return S.K * S.I + (S.shared ? S.Is : 0); }

enum Role1 : int { R1_ROUTED = 0, R1_SHARED = 1, R1_LORA = 2 };
struct Seg1 {
    int slot;                  // routed slot (index into the layer's K ids) or -1: shared
    int hr0, hr1;              // hr [hr0, hr1) of the expert
};
struct Plan1 {
    int role, nseg, n_hr;
    Seg1 seg[kMaxSeg1];
    int dt;                    // output row tile of the down phase (-1: none)
    int rt;                    // router row tile on layers that route themselves (-1: none)
    int t0, t1;                // head-flush tasks
};

__host__ __device__ inline bool plan1(const Shape1& S, int pair, int rank, Plan1& p) {
    p.role = R1_ROUTED;
    p.nseg = p.n_hr = 0;
    const int hpe = S.I / kHalfRow, n_rt = S.K * hpe, n_sh = S.shared ? S.Is / kHalfRow : 0;
    int a, b;
    if (pair < S.Pr) {
        split1(n_rt, S.Pr, pair, &a, &b);
        while (a < b) {
            if (p.nseg >= kMaxSeg1) return false;
            const int slot = a / hpe;
            const int end = (slot + 1) * hpe < b ? (slot + 1) * hpe : b;
            Seg1& s = p.seg[p.nseg++];
            s.slot = slot;
            s.hr0 = a - slot * hpe;
            s.hr1 = end - slot * hpe;
            p.n_hr += end - a;
            a = end;
        }
    } else if (pair < S.Pr + S.Ps) {
        p.role = R1_SHARED;
        split1(n_sh, S.Ps, pair - S.Pr, &a, &b);
        if (a < b) {
            p.seg[0].slot = -1;
            p.seg[0].hr0 = a;
            p.seg[0].hr1 = b;
            p.nseg = 1;
            p.n_hr = b - a;
        }
    } else {
        p.role = R1_LORA;
    }
    if (p.n_hr > kMaxHr1) return false;
    const int cta = 2 * pair + rank;
    p.dt = cta < S.d / kRowTile ? cta : -1;
    p.rt = S.nct - 1 - cta < S.E / kRowTile ? S.nct - 1 - cta : -1;
    split1(S.n_heads * (S.H / kRowTile + S.E / kRowTile), S.nct, cta, &p.t0, &p.t1);
    return true;
}

// Pairs: as many as the grid has, but no more than there are hr (+ the LoRA
// pair), so that every pair publishes act; then the LoRA pair (with LoRA) and
// the split of the rest that minimises the largest per-pair load in hr (a
// shared pair's LoRA B terms count as one more hr).  false if no split fits.
__host__ inline bool choose_pairs(Shape1& S, int grid_pairs) {
    const int hpe = S.I / kHalfRow, n_rt = S.K * hpe, n_sh = S.shared ? S.Is / kHalfRow : 0;
    S.Pl = S.lora ? 1 : 0;
    S.P = grid_pairs;
    if (S.P > S.Pl + n_rt + n_sh) S.P = S.Pl + n_rt + n_sh;
    S.nct = 2 * S.P;
    const int avail = S.P - S.Pl;
    if (!S.shared) {
        S.Ps = 0;
        S.Pr = avail;
        return S.Pr >= 1 && ceil_div(n_rt, S.Pr) <= kMaxHr1;
    }
    int best = 1 << 30, pick = -1;
    for (int ps = 1; ps < avail; ++ps) {
        const int pr = avail - ps;
        if (ps > n_sh || pr > n_rt) continue;
        const int cr = ceil_div(n_rt, pr), cs = ceil_div(n_sh, ps);
        if (cr > kMaxHr1 || cs > kMaxHr1) continue;
        const int cost = cr > cs + S.lora ? cr : cs + S.lora;
        if (cost <= best) { best = cost; pick = ps; }   // ties: more shared pairs
    }
    if (pick < 0) return false;
    S.Ps = pick;
    S.Pr = avail - pick;
    return true;
}

// ---------------------------------------------------------------- blocks ----
// A block is one (layer, phase) share of a CTA's weights, copied contiguously
// into the ring, in this order per layer:
//   b0 its router row tile over all of d (router CTAs, layers that route
//      themselves);
//   b1 gate/up units of the pair's hr over this CTA's half of d (the LoRA pair:
//      A_gate (rank 0) or A_up (rank 1) over all of d);
//   b3 the LoRA B_gate, B_up rows of the pair's act rows (shared pairs, LoRA);
//   b2 its output row tile of every routed expert's down, then of the shared
//      expert's, then (LoRA) A_down and the tile's rows of B_down;
// then two blocks per head-flush task.
enum PieceKind1 : int {
    K1_ROUTER = 0, K1_GU, K1_DOWN, K1_LA, K1_LU, K1_BG, K1_BU, K1_AD, K1_BD, K1_FC1, K1_FC2, K1_LINIT,
    K1_OHF, K1_OHL
};
struct Piece1 {
    int kind, seg;             // seg: the run (K1_GU) or the routed slot (K1_DOWN; -1: shared)
    long long src;             // byte offset in the source matrix (of the expert, for K1_GU/K1_DOWN)
    int bytes, dst;            // size and offset in the block
};
struct Block1 {
    int n, bytes;
    Piece1 pc[kMaxPc];
};
struct Lay1 {
    Block1 b0, b1, b3, b2;
    int bu;                    // b3 offset of the B_up rows (B_gate rows at 0)
    int ad, bd;                // b2 offsets of A_down and of the B_down rows
    int seg_base[kMaxSeg1];    // pair-local act row of each run's first row
};

__host__ __device__ inline bool add_piece(Block1& B, int kind, int seg, long long src, long long bytes) {
    while (bytes > 0) {
        if (B.n >= kMaxPc) return false;
        const int n = bytes > kPieceMax ? kPieceMax : (int)bytes;
        Piece1& pc = B.pc[B.n++];
        pc.kind = kind;
        pc.seg = seg;
        pc.src = src;
        pc.bytes = n;
        pc.dst = B.bytes;
        B.bytes += n;
        src += n;
        bytes -= n;
    }
    return true;
}

__host__ __device__ inline bool layout1(const Shape1& S, const Plan1& p, int rank, Lay1& L) {
    L.b0.n = L.b0.bytes = L.b1.n = L.b1.bytes = L.b3.n = L.b3.bytes = L.b2.n = L.b2.bytes = 0;
    L.bu = L.ad = L.bd = 0;
    const int ng = S.d / kGroup, ng0 = ng / 2, ng1 = ng - ng0, ngh = ngh1(S.d, rank);
    bool ok = true;
    // b0: router row tile rt over all of d (packed fp16 [E x d]: the first half of
    // d for every row tile, then the second half)
    if (p.rt >= 0) {
        const long long nE = S.E / kRowTile;
        ok &= add_piece(L.b0, K1_ROUTER, 0, (long long)p.rt * ng0 * kF16Unit, (long long)ng0 * kF16Unit);
        ok &= add_piece(L.b0, K1_ROUTER, 0, nE * ng0 * kF16Unit + (long long)p.rt * ng1 * kF16Unit,
                        (long long)ng1 * kF16Unit);
    }
    if (p.role == R1_LORA) {
        // LoRA A (packed fp16 [r x d], one row tile: its two halves back to back
        // are the row tile's groups in order)
        ok &= add_piece(L.b1, rank ? K1_LU : K1_LA, 0, 0, (long long)ng * kF16Unit);
    } else {
        // b1: gate/up units [hr][group of the half] of each run, back to back
        int base = 0;
        for (int s = 0; s < p.nseg; ++s) {
            const Seg1& sg = p.seg[s];
            const long long tiles = (sg.slot < 0 ? S.Is : S.I) / kHalfRow;
            const long long half0 = tiles * ng0 * kQ4Unit;
            ok &= add_piece(L.b1, K1_GU, s, rank * half0 + (long long)sg.hr0 * ngh * kQ4Unit,
                            (long long)(sg.hr1 - sg.hr0) * ngh * kQ4Unit);
            L.seg_base[s] = base;
            base += 8 * (sg.hr1 - sg.hr0);
        }
        // b3: LoRA B_gate, B_up rows (row-major [Is, r] fp16) of the pair's act rows
        if (p.role == R1_SHARED && S.lora && p.nseg > 0) {
            const long long rb = 2LL * S.r, row0 = 8LL * p.seg[0].hr0, rows = 8LL * p.n_hr;
            ok &= add_piece(L.b3, K1_BG, 0, row0 * rb, rows * rb);
            L.bu = L.b3.bytes;
            ok &= add_piece(L.b3, K1_BU, 0, row0 * rb, rows * rb);
        }
    }
    // b2: output row tile dt of every expert's down (row-tile major units)
    if (p.dt >= 0) {
        const long long ui = (long long)(S.I / kGroup) * kQ4Unit, us = (long long)(S.Is / kGroup) * kQ4Unit;
        for (int k = 0; k < S.K; ++k) ok &= add_piece(L.b2, K1_DOWN, k, p.dt * ui, ui);
        if (S.shared) ok &= add_piece(L.b2, K1_DOWN, -1, p.dt * us, us);
        if (S.shared && S.lora) {
            // A_down (packed fp16 [r x Is]: one row tile, its groups in order) and
            // the tile's rows of B_down (row-major [d, r])
            L.ad = L.b2.bytes;
            ok &= add_piece(L.b2, K1_AD, 0, 0, (long long)(S.Is / kGroup) * kF16Unit);
            L.bd = L.b2.bytes;
            ok &= add_piece(L.b2, K1_BD, 0, 16LL * p.dt * 2 * S.r, 16LL * 2 * S.r);
        }
    }
    return ok;
}

// Head-flush task j of a head: fc1 row tile j (j < H/16) with its fc2 column
// block, else linear_init row tile j - H/16, dense parts over all of d; and the
// 16 entries of the row tile in each of the n2 one-hot columns the head's
// features select (rows of the transposed columns, 32 bytes each: ids[k2] is
// column e for executed expert e, E + e for previous expert e).  Two blocks:
//   half 0: the row tile's groups of the first half of d;
//   half 1: the groups of the second half, then (fc1) the fc2 block, then the
//           one-hot rows.
// flush_piece(., half, i, ...) is copy i of a block; false past its last.
__host__ __device__ inline bool flush_piece(const Shape1& S, int j, int half, int i, const int* ids, int n2,
                                            Piece1& pc) {
    const int ng = S.d / kGroup, ng0 = ng / 2, ng1 = ng - ng0, nH = S.H / kRowTile, nE = S.E / kRowTile;
    const bool fc1 = j < nH;
    const int jr = fc1 ? j : j - nH;
    const int rows = fc1 ? nH : nE;   // row tiles of the dense matrix
    pc.seg = 0;
    if (half == 0) {
        if (i != 0) return false;
        pc.kind = fc1 ? K1_FC1 : K1_LINIT;
        pc.src = (long long)jr * ng0 * kF16Unit;
        pc.bytes = ng0 * kF16Unit;
        pc.dst = 0;
        return true;
    }
    if (i == 0) {
        pc.kind = fc1 ? K1_FC1 : K1_LINIT;
        pc.src = (long long)rows * ng0 * kF16Unit + (long long)jr * ng1 * kF16Unit;
        pc.bytes = ng1 * kF16Unit;
        pc.dst = 0;
        return true;
    }
    int dst = ng1 * kF16Unit;
    if (fc1) {
        if (i == 1) {
            pc.kind = K1_FC2;
            pc.src = (long long)jr * nE * kF16Step;
            pc.bytes = nE * kF16Step;
            pc.dst = dst;
            return true;
        }
        dst += nE * kF16Step;
        --i;
    }
    const int k2 = i - 1;
    if (k2 >= n2) return false;
    pc.kind = fc1 ? K1_OHF : K1_OHL;
    pc.src = ((long long)(ids ? ids[k2] : 0) * (fc1 ? S.H : S.E) + 16LL * jr) * 2;
    pc.bytes = 32;
    pc.dst = dst + 32 * k2;
    return true;
}
// the block as a copy list
__host__ __device__ inline bool flush_block(const Shape1& S, int j, int half, Block1& B, const int* ids = nullptr,
                                            int n2 = 0) {
    B.n = B.bytes = 0;
    Piece1 pc;
    for (int i = 0; flush_piece(S, j, half, i, ids, n2, pc); ++i) {
        if (B.n >= kMaxPc || pc.bytes > kPieceMax) return false;
        B.pc[B.n++] = pc;
        B.bytes = pc.dst + pc.bytes;
    }
    return true;
}
// bytes of flush_block(S, j, half, ., ., n2), without building it
__host__ __device__ inline int flush_bytes(const Shape1& S, int j, int half, int n2) {
    const int ng = S.d / kGroup, ng0 = ng / 2;
    if (half == 0) return ng0 * kF16Unit;
    return (ng - ng0) * kF16Unit + (j < S.H / kRowTile ? (S.E / kRowTile) * kF16Step : 0) + n2 * 32;
}

// ring placement shared by the producer and the consumers: a block starts at the
// ring offset `off` unless it would cross the ring's end, then at offset 0 of
// the next lap; `pos` counts ring bytes passed (skipped tails included)
struct Ring1 {
    int pos, off;
};
__host__ __device__ inline int place1(Ring1& r, int bytes, int ring) {
    if (r.off + bytes > ring) {
        r.pos += ring - r.off;
        r.off = 0;
    }
    const int at = r.off;
    r.pos += bytes;
    r.off += bytes;
    if (r.off == ring) r.off = 0;
    return at;
}

// --------------------------------------------------------------- workspace ----
// After the header, per step parity p and state row s (tagged: the value's
// 32 bits in the low half of a 64-bit word, the launch's tag in the high half):
//   y     [2][Ls][d]    tagged  layer output (writer: the row tile's CTA)
//   act   [2][Ls][NA]   tagged  act of the layer, NA = K I + Is: routed slot k at
//                               k I (times w_k), the shared expert at K I
//   logr  [2][Ls][E]    tagged  own-router logits (writer: the row tile's CTA)
//   lax   [2][Ls][32]   tagged  A_gate x (0-15), A_up x (16-31)
//   ex    [2][Ls][K]    tagged  executed ids (writer: CTA 0)
//   xs    [Ls][d/2]     tagged  x as fp16 pairs (writer: CTA 0, head layers)
//   logh  [2][Ls][E]    fp32    head logits (vector reductions; the other
//                               parity's are cleared for the next step)
//   cnt   [2][Ls]       u32     head tasks done (cleared likewise)
// and the trace area at the end of the workspace.
struct Ws1 {
    long long y, act, logr, lax, ex, xs, logh, cnt, end;
};
__host__ __device__ inline Ws1 ws1(int Ls, int d, int E, int K, int NA) {
    Ws1 w;
    long long o = kWsHeaderBytes;
    w.y = o;    o += 2LL * Ls * d * 8;
    w.act = o;  o += 2LL * Ls * NA * 8;
    w.logr = o; o += 2LL * Ls * E * 8;
    w.lax = o;  o += 2LL * Ls * 32 * 8;
    w.ex = o;   o += (2LL * Ls * K * 8 + 255) / 256 * 256;
    w.xs = o;   o += (long long)Ls * d / 2 * 8;
    w.logh = o; o += 2LL * Ls * E * 4;
    w.cnt = o;  o += (2LL * Ls * 4 + 255) / 256 * 256;
    w.end = o;
    return w;
}
constexpr long long kTraceBytes = (long long)kTraceCtas * kTraceSlots * 8;

// ------------------------------------------------------ shared memory ----
struct Sm1 {
    uint64_t full[kBlocks];
    uint64_t xbar;
    int abort;                            // CTA abort flag (read after consumer barriers)
    int topk;                             // flush: this CTA completed the current head
    int issued;                           // blocks issued by the producer
    int released_blocks;                  // blocks the consumers are done with
    int released;                         // ring position up to which blocks are free
    unsigned long long wait_ns;
    int trace, tslot, ptslot;
    int flush_after;                      // the head flush follows this layer (-1: no heads)
    // arrays: each 16-byte aligned (some are read and written as vectors)
    __align__(16) int route_ready[EDGE0_MAX_LAYERS];
    __align__(16) int ids[EDGE0_MAX_LAYERS][kMaxK1];
    __align__(16) float w[EDGE0_MAX_LAYERS][kMaxK1];
    __align__(16) int heads[EDGE0_MAX_LAYERS];
    __align__(16) int fids[2 * kMaxK1];   // flush: one-hot columns of the current head
    __align__(16) Shape1 S;
    __align__(16) Plan1 plan;
    __align__(16) Lay1 lay;
    __align__(16) float red[kCW];
    __align__(16) float lax[32];
    __align__(16) float xsum[kMaxG1];
    __align__(16) float gsum[kMaxNG];
    __align__(16) float mine[kMsg];
    __align__(16) float recv[kMsg];
    __align__(16) float part[kCW][kMsg];
    __align__(16) float logits[EDGE0_MAX_E];
    __align__(16) float rscr[2 * EDGE0_MAX_E];
    __align__(16) __half h[kMaxD1];
    __align__(16) uint2 xf[kMaxG1 * 16];  // [group][t][step]: x as B fragments
    __align__(16) uint2 af[kMaxNS * 8];   // [act step][lane < 8]: act hi (lanes 0-3), lo (4-7)
    __align__(16) uint2 gf[8];            // GELU(z) of a flush task, same form
};
static_assert(offsetof(Sm1, h) % 16 == 0 && offsetof(Sm1, xf) % 16 == 0 && offsetof(Sm1, af) % 16 == 0 &&
                  offsetof(Sm1, part) % 16 == 0 && offsetof(Sm1, mine) % 16 == 0,
              "vector-accessed shared arrays are 16-byte aligned");
constexpr int kSm1Bytes = (int)((sizeof(Sm1) + 127) / 128 * 128);

extern __shared__ __align__(128) char d1_smem[];
__device__ __forceinline__ Sm1& sm() { return *reinterpret_cast<Sm1*>(d1_smem); }
__device__ __forceinline__ char* ring() { return d1_smem + kSm1Bytes; }

// ---------------------------------------------------------------- helpers ----
__device__ __forceinline__ unsigned long long now1() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void cbar1() { named_bar_sync(1, kCT); }
// consumer barrier returning the OR of `v` over the consumer threads: every
// decision to leave is taken from one, so all consumer threads take it together
__device__ __forceinline__ bool cbar_or1(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n"
        " selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(kCT)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ int vload(const int* p) { return *(const volatile int*)p; }

__device__ __noinline__ void fail1(WsHeader* hdr, int code) {
    atomicCAS(&hdr->error, 0, code);
    atomicExch(&hdr->abort, 1);
    *(volatile int*)&sm().abort = 1;
}
// another CTA's abort is adopted locally: the exit path then drains this CTA's
// copies in flight
__device__ __forceinline__ bool gone1(WsHeader* hdr) {
    if (vload(&sm().abort)) return true;
    if (ld_volatile_s32(&hdr->abort)) {
        *(volatile int*)&sm().abort = 1;
        return true;
    }
    return false;
}
// every 16th turn of a wait loop: false once the launch gave up or the wait ran
// past its limit (then EDGE0_ETIMEOUT is recorded)
__device__ __forceinline__ bool keep_waiting(WsHeader* hdr, unsigned it, unsigned long long t0) {
    if ((it & 15) != 15) return true;
    if (gone1(hdr)) return false;
    if (now1() - t0 > sm().wait_ns) {
        fail1(hdr, EDGE0_ETIMEOUT);
        return false;
    }
    return true;
}

// tagged words
__device__ __forceinline__ unsigned long long tagged(unsigned tag, float v) {
    return ((unsigned long long)tag << 32) | __float_as_uint(v);
}
__device__ __forceinline__ float tval(unsigned long long w) { return __uint_as_float((unsigned)(w & 0xFFFFFFFFu)); }
__device__ __forceinline__ bool tok(unsigned long long w, unsigned tag) { return (unsigned)(w >> 32) == tag; }
// one word once it carries `tag` (bounded; false on give-up)
__device__ __forceinline__ bool poll1(WsHeader* hdr, const unsigned long long* p, unsigned tag, float* v) {
    unsigned long long w = ld_relaxed_u64(p);
    if (!tok(w, tag)) {
        const unsigned long long t0 = now1();
        for (unsigned it = 0; !tok(w, tag); ++it) {
            if (!keep_waiting(hdr, it, t0)) return false;
            w = ld_relaxed_u64(p);
        }
    }
    *v = tval(w);
    return true;
}
// a pair of words loaded already as w: re-polled until both carry `tag`
__device__ __forceinline__ bool settle2(WsHeader* hdr, const unsigned long long* p, unsigned tag, ulonglong2& w) {
    if (tok(w.x, tag) && tok(w.y, tag)) return true;
    const unsigned long long t0 = now1();
    for (unsigned it = 0;; ++it) {
        if (!keep_waiting(hdr, it, t0)) return false;
        w = ld_relaxed_u64x2(p);
        if (tok(w.x, tag) && tok(w.y, tag)) return true;
    }
}

// trace stamps (thread 0 of the consumers, lane 0 of the producer)
__device__ __noinline__ void stamp_slow1(const Prog& p, int tag, bool producer) {
    Sm1& s = sm();
    int* slot = producer ? &s.ptslot : &s.tslot;
    const int lim = producer ? kTraceSlots : 3072;
    if (*slot + 3 > lim) return;
    unsigned long long* tr =
        reinterpret_cast<unsigned long long*>(p.ws + p.ws_bytes - kTraceBytes) + (long long)blockIdx.x * kTraceSlots;
    long long c;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(c));
    tr[*slot] = (unsigned long long)tag;
    tr[*slot + 1] = now1();
    tr[*slot + 2] = (unsigned long long)c;
    *slot += 3;
}
__device__ __forceinline__ void stamp1(const Prog& p, int tag) {
    if (sm().trace && threadIdx.x == 0) stamp_slow1(p, tag, false);
}

// parity wait with CTA-scope acquire (the bulk copies into this CTA's ring)
__device__ __forceinline__ bool mbar_try_wait_cta(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// bounded wait on a block or exchange barrier phase; false on abort/timeout
__device__ __noinline__ bool mbar_wait1(WsHeader* hdr, uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = now1();
    for (unsigned it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (!keep_waiting(hdr, it, t0)) return false;
    }
}

__device__ __forceinline__ float h2f(uint16_t v) { return __half2float(__ushort_as_half(v)); }
// scales of rows g and g + 8 of a row tile: (s_g, b_g, s_g8, b_g8)
__device__ __forceinline__ float4 scales4(const char* p) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    return make_float4(h2f((uint16_t)(v.x & 0xFFFF)), h2f((uint16_t)(v.x >> 16)), h2f((uint16_t)(v.y & 0xFFFF)),
                       h2f((uint16_t)(v.y >> 16)));
}
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}
// an fp32 value as element k (0..15) of a 16-row B step held as 8 uint2 lane
// slots: its fp16 hi part in the column of lanes 0-3, the fp16 of the rest
// times kLoScale in the column of lanes 4-7
__device__ __forceinline__ void put_hilo(uint2* step, int k, float v) {
    const __half hi = __float2half_rn(v);
    const __half lo = __float2half_rn((v - __half2float(hi)) * kLoScale);
    __half* hh = reinterpret_cast<__half*>(step);
    const int kk = k & 7, t = kk >> 1, wv = k >> 3, e = kk & 1;
    hh[(t * 2 + wv) * 2 + e] = hi;
    hh[((4 + t) * 2 + wv) * 2 + e] = lo;
}
// the 16 row sums of a tile once every consumer warp wrote part[w][0..15]
__device__ __forceinline__ float tile_sum(const Sm1& s, int i) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kCW; ++w) v += s.part[w][i];
    return v;
}
// partial sums of rows g, g + 8 (lanes 4g) into part[warp]
__device__ __forceinline__ void put_part(Sm1& s, float a0, float a1) {
    const int lane = threadIdx.x & 31;
    if ((lane & 3) == 0) {
        s.part[threadIdx.x >> 5][lane >> 2] = a0;
        s.part[threadIdx.x >> 5][(lane >> 2) + 8] = a1;
    }
}

// ---------------------------------------------------------------- producer ----
__device__ __forceinline__ bool own_routed1(const Prog& p, int l, int step) {
    return step == 0 || !(p.layers[l].flags & LF_PREROUTED);
}

__device__ const char* piece_src1(const Prog& p, const Piece1& pc, int l) {
    const Sm1& s = sm();
    const LayerP& Ly = p.layers[l];
    switch (pc.kind) {
        case K1_ROUTER: return Ly.router + pc.src;
        case K1_GU: {
            const Seg1& sg = s.plan.seg[pc.seg];
            if (sg.slot < 0) return Ly.sh_gu + pc.src;
            return Ly.gu + (long long)s.ids[l][sg.slot] * q4_bytes(2 * p.I, p.d) + pc.src;
        }
        case K1_DOWN:
            if (pc.seg < 0) return Ly.sh_down_rows + pc.src;
            return Ly.down_rows + (long long)s.ids[l][pc.seg] * q4_bytes(p.d, p.I) + pc.src;
        case K1_LA: return Ly.lora_Ag + pc.src;
        case K1_LU: return Ly.lora_Au + pc.src;
        case K1_BG: return reinterpret_cast<const char*>(Ly.lora_Bg) + pc.src;
        case K1_BU: return reinterpret_cast<const char*>(Ly.lora_Bu) + pc.src;
        case K1_AD: return Ly.lora_Ad + pc.src;
        case K1_BD: return reinterpret_cast<const char*>(Ly.lora_Bd) + pc.src;
        case K1_FC1: return Ly.fc1 + pc.src;
        case K1_FC2: return Ly.fc2 + pc.src;
        case K1_OHF: return reinterpret_cast<const char*>(Ly.fc1_oh) + pc.src;
        case K1_OHL: return reinterpret_cast<const char*>(Ly.linit_oh) + pc.src;
        default: return Ly.linit + pc.src;
    }
}

struct Stream1 {
    Ring1 r;
    int nb;
};

// the whole producer warp: place a block of `bytes`, wait for its room, arm its
// barrier; its ring offset, or -1 on give-up
__device__ int open_block1(const Prog& p, WsHeader* hdr, Stream1& q, int bytes) {
    Sm1& s = sm();
    const int off = place1(q.r, bytes, p.ring1);
    const int end = q.r.pos;
    int ok = 1;
    if ((threadIdx.x & 31) == 0) {
        const unsigned long long t0 = now1();
        for (unsigned it = 0;; ++it) {
            if (end - vload(&s.released) <= p.ring1 && q.nb - vload(&s.released_blocks) < kBlocks) break;
            if (!keep_waiting(hdr, it, t0)) { ok = 0; break; }
        }
        if (ok) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&s.full[q.nb % kBlocks], (uint32_t)bytes);
        }
    }
    return __shfl_sync(0xffffffffu, ok, 0) ? off : -1;
}
__device__ __forceinline__ void close_block1(const Prog& p, Stream1& q, int tag) {
    Sm1& s = sm();
    ++q.nb;
    if ((threadIdx.x & 31) == 0) {
        *(volatile int*)&s.issued = q.nb;
        if (s.trace) stamp_slow1(p, tag, true);
    }
    __syncwarp();
}

// a layer block: copy i by lane i, i + 32, ...
__device__ bool issue1(const Prog& p, WsHeader* hdr, Stream1& q, const Block1& B, int l, uint64_t pol, int tag) {
    if (B.bytes == 0) return true;
    const int off = open_block1(p, hdr, q, B.bytes);
    if (off < 0) return false;
    Sm1& s = sm();
    for (int i = threadIdx.x & 31; i < B.n; i += 32) {
        const Piece1& pc = B.pc[i];
        bulk_g2s(ring() + off + pc.dst, piece_src1(p, pc, l), (uint32_t)pc.bytes, &s.full[q.nb % kBlocks], pol);
    }
    close_block1(p, q, tag);
    return true;
}

// a flush block (task j of head layer l, half h): copy i by lane i
__device__ bool issue_flush1(const Prog& p, WsHeader* hdr, Stream1& q, int j, int h, int n2, int l, uint64_t pol,
                             int tag) {
    Sm1& s = sm();
    const int off = open_block1(p, hdr, q, flush_bytes(s.S, j, h, n2));
    if (off < 0) return false;
    Piece1 pc;
    if (flush_piece(s.S, j, h, threadIdx.x & 31, s.fids, n2, pc))
        bulk_g2s(ring() + off + pc.dst, piece_src1(p, pc, l), (uint32_t)pc.bytes, &s.full[q.nb % kBlocks], pol);
    close_block1(p, q, tag);
    return true;
}

// the head flush's blocks: a task's one-hot rows are gathered by the head
// layer's executed ids (this launch's tagged words) and previous ids (what the
// previous launch left in exec_ids)
__device__ bool produce_flush1(const Prog& p, WsHeader* hdr, const Ws1& W, Stream1& q, int step, int par,
                               unsigned tag, uint64_t pol) {
    Sm1& s = sm();
    const int lane = threadIdx.x & 31;
    const int tph = p.H / kRowTile + p.E / kRowTile;
    const int n2 = p.K + (step > 0 ? p.K : 0);
    int cur = -1;
    for (int t = s.plan.t0; t < s.plan.t1; ++t) {
        const int l = s.heads[t / tph];
        if (l != cur) {
            const int sidx = p.layers[l].sidx;
            int ok = 1;
            if (lane < n2) {
                int e;
                if (lane < p.K) {
                    float v = 0.f;
                    const unsigned long long* ex =
                        reinterpret_cast<const unsigned long long*>(p.ws + W.ex) + ((long long)par * p.Ls + sidx) * p.K;
                    ok = poll1(hdr, ex + lane, tag, &v);
                    e = (int)__float_as_uint(v);
                } else {
                    e = ld_volatile_s32(p.exec_ids + ((long long)(par ^ 1) * p.Ls + sidx) * p.K + (lane - p.K));
                }
                e = e < 0 || e >= p.E ? 0 : e;
                s.fids[lane] = lane < p.K ? e : p.E + e;
            }
            __syncwarp();
            if (!__all_sync(0xffffffffu, ok)) return false;
            cur = l;
        }
        const int j = t % tph, tg = 0xF000 | (t - s.plan.t0);
        if (!issue_flush1(p, hdr, q, j, 0, n2, l, pol, tg)) return false;
        if (!issue_flush1(p, hdr, q, j, 1, n2, l, pol, tg)) return false;
    }
    return true;
}

__device__ void producer1(const Prog& p, WsHeader* hdr, const Ws1& W, int step, int par, unsigned tag) {
    Sm1& s = sm();
    const int lane = threadIdx.x & 31;
    const uint64_t pol = policy_evict_first();
    const Plan1& pl = s.plan;
    const Lay1& L = s.lay;
    Stream1 q{{0, 0}, 0};
    auto route_wait = [&](int l) -> bool {   // the layer's own routing is done (lane 0 polls)
        int ok = 1;
        if (lane == 0) {
            const unsigned long long t0 = now1();
            for (unsigned it = 0; !vload(&s.route_ready[l]); ++it)
                if (!keep_waiting(hdr, it, t0)) { ok = 0; break; }
        }
        return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    for (int l = 0; l < p.L; ++l) {
        const bool own = own_routed1(p, l, step);
        if (own && !issue1(p, hdr, q, L.b0, l, pol, (l << 8) | 0x80)) return;
        // blocks that read routed experts follow the layer's routing
        bool known = !own;
        if (pl.role == R1_ROUTED && pl.nseg > 0 && !known) {
            if (!route_wait(l)) return;
            known = true;
        }
        if (!issue1(p, hdr, q, L.b1, l, pol, (l << 8) | 0x81)) return;
        if (!issue1(p, hdr, q, L.b3, l, pol, (l << 8) | 0x83)) return;
        if (L.b2.bytes && !known && !route_wait(l)) return;
        if (!issue1(p, hdr, q, L.b2, l, pol, (l << 8) | 0x82)) return;
        // the head flush runs right after the last layer that owns a head
        if (l == s.flush_after && !produce_flush1(p, hdr, W, q, step, par, tag, pol)) return;
    }
}

// ---------------------------------------------------------------- consumers ----
struct Cons1 {
    Ring1 r;                   // ring placement (same sequence as the producer's)
    int nb;                    // blocks taken
    int off;                   // ring offset of the current block
    int end;                   // ring position after it
};
// next block: its ring offset; waits for its data (every consumer thread)
__device__ __forceinline__ bool take1(const Prog& p, WsHeader* hdr, Cons1& c, int bytes) {
    c.off = place1(c.r, bytes, p.ring1);
    c.end = c.r.pos;
    Sm1& s = sm();
    uint64_t* bar = &s.full[c.nb % kBlocks];
    const uint32_t par = (uint32_t)((c.nb / kBlocks) & 1);
    const bool ok = mbar_try_wait_cta(bar, par) || mbar_wait1(hdr, bar, par);
    ++c.nb;
    return ok;
}
// after a consumer barrier that follows the last read of every block taken so far
__device__ __forceinline__ void give1(const Cons1& c) {
    if (threadIdx.x == 0) {
        Sm1& s = sm();
        *(volatile int*)&s.released = c.end;
        *(volatile int*)&s.released_blocks = c.nb;
    }
}

// B fragments of x for group g: lanes 0-3 hold (k 2t, 2t+1 | 2t+8, 2t+9) of steps 0-3
__device__ __forceinline__ void xfrag(const Sm1& s, int g, int lane, uint4& xa, uint4& xb) {
    xa = xb = make_uint4(0u, 0u, 0u, 0u);
    if (lane < 4) {
        const uint4* src = reinterpret_cast<const uint4*>(&s.xf[(g * 4 + lane) * 4]);
        xa = src[0];
        xb = src[1];
    }
}
// x elements 4i .. 4i+3 (as two fp16 pairs) into the B fragments
__device__ __forceinline__ void put_x4(Sm1& s, int i, uint32_t x01, uint32_t x23) {
    const int k = 4 * i, g = k / kGroup, kk = k % kGroup, st = kk / 16, k16 = kk % 16;
    const int wv = k16 >> 3, t = (k16 & 7) >> 1;
    uint32_t* xw = reinterpret_cast<uint32_t*>(s.xf);
    xw[((g * 4 + t) * 4 + st) * 2 + wv] = x01;
    xw[((g * 4 + t + 1) * 4 + st) * 2 + wv] = x23;
}

// h = fp16(h + y) (y: the previous layer's tagged words; y == null: h from
// h_in), x = fp16(h * rsqrt(mean(h^2) + eps) * gamma) over all of d as B
// fragments and group sums.  Thread i owns elements 4i .. 4i+3.  false: a poll
// gave up (uniform).
__device__ bool build_x1(const Prog& p, WsHeader* hdr, int l, const __half* h_in, const unsigned long long* y,
                         unsigned want, uint2 gam, unsigned long long* xs_out, unsigned tag, __half* dbg_prev) {
    Sm1& s = sm();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, n4 = p.d / 4;
    float hf[4] = {0.f, 0.f, 0.f, 0.f};
    float q = 0.f;
    bool ok = true;
    if (tid < n4) {
        const uint2 hv = h_in ? *reinterpret_cast<const uint2*>(h_in + 4 * tid)
                              : *reinterpret_cast<const uint2*>(&s.h[4 * tid]);
        __half2 h01 = *reinterpret_cast<const __half2*>(&hv.x), h23 = *reinterpret_cast<const __half2*>(&hv.y);
        if (y) {
            ulonglong2 a = ld_relaxed_u64x2(y + 4 * tid), b = ld_relaxed_u64x2(y + 4 * tid + 2);
            ok = settle2(hdr, y + 4 * tid, want, a) && settle2(hdr, y + 4 * tid + 2, want, b);
            h01 = __floats2half2_rn(__low2float(h01) + tval(a.x), __high2float(h01) + tval(a.y));
            h23 = __floats2half2_rn(__low2float(h23) + tval(b.x), __high2float(h23) + tval(b.y));
        }
        uint2 o;
        o.x = *reinterpret_cast<const uint32_t*>(&h01);
        o.y = *reinterpret_cast<const uint32_t*>(&h23);
        *reinterpret_cast<uint2*>(&s.h[4 * tid]) = o;
        if (dbg_prev) *reinterpret_cast<uint2*>(dbg_prev + 4 * tid) = o;
        hf[0] = __low2float(h01); hf[1] = __high2float(h01); hf[2] = __low2float(h23); hf[3] = __high2float(h23);
        q = hf[0] * hf[0] + hf[1] * hf[1] + hf[2] * hf[2] + hf[3] * hf[3];
    }
    q = warp_sum(q);
    if (lane == 0) s.red[wid] = q;
    if (cbar_or1(!ok)) return false;
    float ss = 0.f;
#pragma unroll
    for (int w = 0; w < kCW; ++w) ss += s.red[w];
    const float rs = rsqrtf(ss / (float)p.d + p.layers[l].eps);
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (tid < n4) {
        const float2 g01 = __half22float2(*reinterpret_cast<const __half2*>(&gam.x));
        const float2 g23 = __half22float2(*reinterpret_cast<const __half2*>(&gam.y));
        x[0] = __half2float(__float2half_rn(hf[0] * rs * g01.x));
        x[1] = __half2float(__float2half_rn(hf[1] * rs * g01.y));
        x[2] = __half2float(__float2half_rn(hf[2] * rs * g23.x));
        x[3] = __half2float(__float2half_rn(hf[3] * rs * g23.y));
    }
    float sum = x[0] + x[1] + x[2] + x[3];
#pragma unroll
    for (int m = 8; m; m >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, m);
    if (tid < n4) {
        const uint32_t x01 = pack2(x[0], x[1]), x23 = pack2(x[2], x[3]);
        put_x4(s, tid, x01, x23);
        if ((lane & 15) == 0) s.xsum[4 * tid / kGroup] = sum;
        if (xs_out) {
            xs_out[2 * tid] = ((unsigned long long)tag << 32) | x01;
            xs_out[2 * tid + 1] = ((unsigned long long)tag << 32) | x23;
        }
    }
    cbar1();
    return true;
}

// fp16 units u0, u0 + ustride, ... < u1 of a packed row tile against x groups
// xg0 + u: partial sums of rows g, g + 8 (lanes 4g) added into a0 / a1
__device__ __forceinline__ void f16_units(const Sm1& s, const char* base, int u0, int u1, int ustride, int xg0,
                                          int lane, float& a0, float& a1) {
    for (int u = u0; u < u1; u += ustride) {
        const char* unit = base + (long long)u * kF16Unit;
        uint4 xa, xb;
        xfrag(s, xg0 + u, lane, xa, xb);
        const uint32_t xbv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
        float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int st = 0; st < 4; ++st) {
            const uint4 a = *reinterpret_cast<const uint4*>(unit + st * kF16Step + 16 * lane);
            const uint32_t A[4] = {a.x, a.y, a.z, a.w};
            mma_16816(c, A, xbv[2 * st], xbv[2 * st + 1]);
        }
        a0 += c[0];
        a1 += c[2];
    }
}

// gate/up partial sums of the pair's hr over this CTA's half of d (groups g0 +
// [0, ngh)): warp w takes groups [ngh w / 16, ngh (w + 1) / 16) of every hr
__device__ void gateup1(const char* blk, int ngh, int g0, int n_hr) {
    Sm1& s = sm();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int ga, gb;
    split1(ngh, kCW, wid, &ga, &gb);
    float acc[kMaxHr1][2];
#pragma unroll
    for (int j = 0; j < kMaxHr1; ++j) acc[j][0] = acc[j][1] = 0.f;
    for (int g = ga; g < gb; ++g) {
        uint4 xa, xb;
        xfrag(s, g0 + g, lane, xa, xb);
        const float xsm = s.xsum[g0 + g];
#pragma unroll
        for (int j = 0; j < kMaxHr1; ++j) {
            if (j < n_hr) {
                const char* unit = blk + (long long)(j * ngh + g) * kQ4Unit;
                const uint4 wv = *reinterpret_cast<const uint4*>(unit + 16 * lane);
                float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t A[4];
                q4_masks(wv.x, A);
                mma_16816(c0, A, xa.x, xa.y);
                q4_masks(wv.y, A);
                mma_16816(c1, A, xa.z, xa.w);
                q4_masks(wv.z, A);
                mma_16816(c0, A, xb.x, xb.y);
                q4_masks(wv.w, A);
                mma_16816(c1, A, xb.z, xb.w);
                const float4 sc = scales4(unit + 512 + (lane >> 2) * 8);
                acc[j][0] += sc.x * kTwo24 * (c0[0] + c1[0]) + sc.y * xsm;
                acc[j][1] += sc.z * (kTwo24 / 16.f) * (c0[2] + c1[2]) + sc.w * xsm;
            }
        }
    }
    if ((lane & 3) == 0) {   // every warp writes its rows (zero without groups)
        const int g8 = lane >> 2;
#pragma unroll
        for (int j = 0; j < kMaxHr1; ++j)
            if (j < n_hr) {
                s.part[wid][j * 16 + g8] = acc[j][0];
                s.part[wid][j * 16 + g8 + 8] = acc[j][1];
            }
    }
}

// act of the pair's act rows of this CTA's parity (pair-local row i = thread
// i, i % 2 == rank), w_k act for routed rows, the shared expert's rows with
// their LoRA B terms, published as tagged words.  m0 / m1: the partial gate/up
// sums of rank 0 / rank 1.
__device__ void act1(const Prog& p, int l, int rank, const float* m0, const float* m1, const char* blk3, bool lora,
                     unsigned long long* act_out, unsigned tag) {
    Sm1& s = sm();
    const int i = threadIdx.x;
    const Plan1& pl = s.plan;
    if (i >= 8 * pl.n_hr || (i & 1) != rank) return;
    int sg = 0;
    while (sg + 1 < pl.nseg && i >= s.lay.seg_base[sg + 1]) ++sg;
    const Seg1& seg = pl.seg[sg];
    const int row = 8 * seg.hr0 + i - s.lay.seg_base[sg];   // expert-local act row
    const int hl = i >> 3, r8 = i & 7;
    float gt = m0[hl * 16 + r8] + m1[hl * 16 + r8];
    float up = m0[hl * 16 + 8 + r8] + m1[hl * 16 + 8 + r8];
    float wt = 1.f;
    if (seg.slot >= 0) {
        wt = s.w[l][seg.slot];
    } else if (lora) {
        // unmerged LoRA on the shared gate and up [S3.3]: + (alpha / r) B (A x)
        const int r = p.r;
        const __half* bg = reinterpret_cast<const __half*>(blk3) + (long long)i * r;
        const __half* bu = reinterpret_cast<const __half*>(blk3 + s.lay.bu) + (long long)i * r;
        float dg = 0.f, du = 0.f;
        if ((r & 7) == 0) {
            for (int j = 0; j < r; j += 8) {
                const uint4 gv = *reinterpret_cast<const uint4*>(bg + j);
                const uint4 uv = *reinterpret_cast<const uint4*>(bu + j);
                const __half2* g2 = reinterpret_cast<const __half2*>(&gv);
                const __half2* u2 = reinterpret_cast<const __half2*>(&uv);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float2 gf = __half22float2(g2[c]), uf = __half22float2(u2[c]);
                    dg += gf.x * s.lax[j + 2 * c] + gf.y * s.lax[j + 2 * c + 1];
                    du += uf.x * s.lax[16 + j + 2 * c] + uf.y * s.lax[16 + j + 2 * c + 1];
                }
            }
        } else {
            for (int j = 0; j < r; ++j) {
                dg += __half2float(bg[j]) * s.lax[j];
                du += __half2float(bu[j]) * s.lax[16 + j];
            }
        }
        const float ls = p.layers[l].lora_scale;
        gt += ls * dg;
        up += ls * du;
    }
    const long long gi = (seg.slot >= 0 ? (long long)seg.slot * p.I : (long long)p.K * p.I) + row;
    st_relaxed_u64(act_out + gi, tagged(tag, silu_f(gt) * up * wt));
}

// The down phase of output row tile dt.  Every act value of the layer (tagged
// words, two per load) becomes hi/lo B fragments with exact group sums; then
// the tile's units of every expert (unit u = act group u), and with LoRA
// (alpha / r) B_down (A_down act_shared): warp w < Is/64 forms v_w = A_down
// [:, group w] act_shared[group w] and adds B_down[tile] v_w (B_down is linear,
// so the sum over w is B_down v).  The tile's 16 y values go out as tagged
// words.  false: a poll gave up (uniform).
__device__ bool down_tile1(const Prog& p, WsHeader* hdr, int l, const char* blk2, const unsigned long long* act_in,
                           unsigned want, bool lora, unsigned long long* y_out, int dt, unsigned tag) {
    Sm1& s = sm();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int NA = n_act1(s.S), NG = NA / kGroup, NP = NA / 2;
    ulonglong2 wd[kPP];
#pragma unroll
    for (int i = 0; i < kPP; ++i) {
        const int q = tid + kCT * i;
        wd[i] = make_ulonglong2(0ull, 0ull);
        if (q < NP) wd[i] = ld_relaxed_u64x2(act_in + 2 * q);
    }
    bool ok = true;
#pragma unroll
    for (int i = 0; i < kPP; ++i) {
        const int q = tid + kCT * i;   // q < NP is uniform over a warp (NP is a multiple of 32)
        float v0 = 0.f, v1 = 0.f;
        if (q < NP) {
            if (ok) ok = settle2(hdr, act_in + 2 * q, want, wd[i]);
            v0 = tval(wd[i].x);
            v1 = tval(wd[i].y);
            put_hilo(&s.af[(q >> 3) * 8], (2 * q) & 15, v0);
            put_hilo(&s.af[(q >> 3) * 8], (2 * q + 1) & 15, v1);
        }
        const float gs = warp_sum(v0 + v1);   // a warp holds one group of 64
        if (lane == 0 && q < NP) s.gsum[q >> 5] = gs;
    }
    if (cbar_or1(!ok)) return false;
    float a0 = 0.f, a1 = 0.f;
    for (int u = wid; u < NG; u += kCW) {
        const char* unit = blk2 + (long long)u * kQ4Unit;
        const uint4 wv = *reinterpret_cast<const uint4*>(unit + 16 * lane);
        uint2 b[4];
#pragma unroll
        for (int st = 0; st < 4; ++st) b[st] = lane < 8 ? s.af[(4 * u + st) * 8 + lane] : make_uint2(0u, 0u);
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t A[4];
        q4_masks(wv.x, A);
        mma_16816(c0, A, b[0].x, b[0].y);
        q4_masks(wv.y, A);
        mma_16816(c1, A, b[1].x, b[1].y);
        q4_masks(wv.z, A);
        mma_16816(c0, A, b[2].x, b[2].y);
        q4_masks(wv.w, A);
        mma_16816(c1, A, b[3].x, b[3].y);
        const float4 sc = scales4(unit + 512 + (lane >> 2) * 8);
        const float gs = s.gsum[u];
        a0 += sc.x * kTwo24 * ((c0[0] + c1[0]) + (c0[1] + c1[1]) * kLoInv) + sc.y * gs;
        a1 += sc.z * (kTwo24 / 16.f) * ((c0[2] + c1[2]) + (c0[3] + c1[3]) * kLoInv) + sc.w * gs;
    }
    if (lora && wid < p.Is / kGroup) {
        const int r = p.r, g8 = lane >> 2, t = lane & 3;
        const int ush = (p.K * p.I) / kGroup + wid;   // act group of the shared unit
        const char* unit = blk2 + s.lay.ad + (long long)wid * kF16Unit;
        float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int st = 0; st < 4; ++st) {
            const uint4 a = *reinterpret_cast<const uint4*>(unit + st * kF16Step + 16 * lane);
            const uint32_t A[4] = {a.x, a.y, a.z, a.w};
            const uint2 b = lane < 8 ? s.af[(4 * ush + st) * 8 + lane] : make_uint2(0u, 0u);
            mma_16816(c, A, b.x, b.y);
        }
        // v_w[g8], v_w[g8 + 8] sit in lanes 4 g8; as the B operand (k = the rank
        // index) lane t < 4 takes the hi, lane 4 + t the lo parts of
        // v[2t], v[2t+1] | v[2t+8], v[2t+9]
        const float vr = c[0] + c[1] * kLoInv, vr8 = c[2] + c[3] * kLoInv;
        const float v0 = __shfl_sync(0xffffffffu, vr, 8 * t), v1 = __shfl_sync(0xffffffffu, vr, 8 * t + 4);
        const float v8 = __shfl_sync(0xffffffffu, vr8, 8 * t), v9 = __shfl_sync(0xffffffffu, vr8, 8 * t + 4);
        uint32_t b0 = 0u, b1 = 0u;
        if (lane < 8) {
            auto part16 = [&](float v) {
                const float hi = __half2float(__float2half_rn(v));
                return lane < 4 ? hi : (v - hi) * kLoScale;
            };
            b0 = pack2(part16(v0), part16(v1));
            b1 = pack2(part16(v8), part16(v9));
        }
        // A: the tile's B_down rows g8 and g8 + 8, k = the rank index (zero past r)
        const __half* bd = reinterpret_cast<const __half*>(blk2 + s.lay.bd);
        const __half zero = __float2half_rn(0.f);
        auto at = [&](int rw, int kk) { return kk < r ? bd[rw * r + kk] : zero; };
        __half2 q0 = __halves2half2(at(g8, 2 * t), at(g8, 2 * t + 1));
        __half2 q1 = __halves2half2(at(g8 + 8, 2 * t), at(g8 + 8, 2 * t + 1));
        __half2 q2 = __halves2half2(at(g8, 2 * t + 8), at(g8, 2 * t + 9));
        __half2 q3 = __halves2half2(at(g8 + 8, 2 * t + 8), at(g8 + 8, 2 * t + 9));
        const uint32_t A[4] = {*reinterpret_cast<uint32_t*>(&q0), *reinterpret_cast<uint32_t*>(&q1),
                               *reinterpret_cast<uint32_t*>(&q2), *reinterpret_cast<uint32_t*>(&q3)};
        float e[4] = {0.f, 0.f, 0.f, 0.f};
        mma_16816(e, A, b0, b1);
        const float ls = p.layers[l].lora_scale;
        a0 += ls * (e[0] + e[1] * kLoInv);
        a1 += ls * (e[2] + e[3] * kLoInv);
    }
    put_part(s, a0, a1);
    cbar1();
    if (tid < 16) st_relaxed_u64(y_out + 16 * dt + tid, tagged(tag, tile_sum(s, tid)));
    return true;
}

// ------------------------------------------------------------ head flush ----
// x of a head layer over all of d as B fragments (tagged fp16 pairs)
__device__ bool flush_head1(const Prog& p, WsHeader* hdr, const unsigned long long* xs, unsigned want) {
    Sm1& s = sm();
    const int tid = threadIdx.x;
    bool ok = true;
    if (tid < p.d / 4) {
        ulonglong2 w = ld_relaxed_u64x2(xs + 2 * tid);
        ok = settle2(hdr, xs + 2 * tid, want, w);
        put_x4(s, tid, (uint32_t)w.x, (uint32_t)w.y);
    }
    return !cbar_or1(!ok);
}

// one task of head layer l (see flush_piece); its logits summed into lg
__device__ void flush_task1(const Prog& p, int j, int n2, const char* blkA, const char* blkB, float* lg) {
    Sm1& s = sm();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, g8 = lane >> 2;
    const int nH = p.H / kRowTile, nE = p.E / kRowTile, ng = p.d / kGroup, ng0 = ng / 2;
    const bool fc1 = j < nH;
    const int row0 = 16 * (fc1 ? j : j - nH);
    // dense part: warp w takes groups w, w + 16, ... (the first half of d from
    // block A, the second from block B)
    float a0 = 0.f, a1 = 0.f;
    f16_units(s, blkA, wid, ng0, kCW, 0, lane, a0, a1);
    int u1 = wid;
    while (u1 < ng0) u1 += kCW;
    f16_units(s, blkB, u1 - ng0, ng - ng0, kCW, ng0, lane, a0, a1);
    put_part(s, a0, a1);
    cbar1();
    if (tid < 16) {
        float z = tile_sum(s, tid);
        // one-hot columns of the executed and previous masks [S3.2 "Head"]: the
        // rows of the transposed columns that the producer gathered into block B
        // (the concatenated features are never materialised)
        const __half* oh = reinterpret_cast<const __half*>(blkB + (long long)(ng - ng0) * kF16Unit +
                                                           (fc1 ? (long long)nE * kF16Step : 0LL));
        for (int k2 = 0; k2 < n2; ++k2) z += __half2float(oh[k2 * 16 + tid]);
        if (fc1) {
            // erf-GELU [S3.2 "Head"], then fc2 columns row0 .. row0+15 below
            put_hilo(s.gf, tid, 0.5f * z * (1.f + erff(z * 0.70710678118654752f)));
        } else {
            red_add_f32(lg + row0 + tid, z);
        }
    }
    if (fc1) {
        cbar1();
        const uint2 b = lane < 8 ? s.gf[lane] : make_uint2(0u, 0u);
        const char* fc2 = blkB + (long long)(ng - ng0) * kF16Unit;
        for (int rt = wid; rt < nE; rt += kCW) {
            const uint4 a = *reinterpret_cast<const uint4*>(fc2 + (long long)rt * kF16Step + 16 * lane);
            const uint32_t A[4] = {a.x, a.y, a.z, a.w};
            float c[4] = {0.f, 0.f, 0.f, 0.f};
            mma_16816(c, A, b.x, b.y);
            if ((lane & 3) == 0) {
                red_add_f32(lg + rt * 16 + g8, c[0] + c[1] * kLoInv);
                red_add_f32(lg + rt * 16 + g8 + 8, c[2] + c[3] * kLoInv);
            }
        }
    }
}

// ---------------------------------------------------------------- consumers ----
__device__ void consumer1(const Prog& p, WsHeader* hdr, const Ws1& W, int step, int par, unsigned tag) {
    Sm1& s = sm();
    const int tid = threadIdx.x, lane = tid & 31;
    const int rank = (int)cluster_ctarank();
    const int cta = blockIdx.x, nct = gridDim.x;
    const Plan1& pl = s.plan;
    const Lay1& L = s.lay;
    const int ng = p.d / kGroup, ngh = ngh1(p.d, rank), g0 = rank ? ng / 2 : 0;
    const bool lora = s.S.lora && pl.role == R1_SHARED && pl.nseg > 0;
    const bool lora_dn = s.S.lora && s.S.shared;
    // with the workspace's hold hook set, the first poll of the launch waits for
    // a tag that is never written (a bounded wait that runs out, for tests)
    const bool hold = ld_volatile_s32(&hdr->hold) > 0;
    bool first = true;
    auto want = [&]() -> unsigned {
        const unsigned w = (first && hold) ? (tag | kHoldBit) : tag;
        first = false;
        return w;
    };
    auto row = [&](long long base, int sidx, long long n) {   // tagged row (par, sidx) of n words
        return reinterpret_cast<unsigned long long*>(p.ws + base) + ((long long)par * p.Ls + sidx) * n;
    };
    const int NA = n_act1(s.S);
    Cons1 c{{0, 0}, 0, 0, 0};
    int nx = 0;   // pair exchanges so far
    const uint32_t peer = (uint32_t)rank ^ 1u;
    const uint32_t rbar = mapa_shared(smem_u32(&s.xbar), peer);
    const uint32_t rrecv = mapa_shared(smem_u32(s.recv), peer);
    const bool xch = pl.n_hr > 0;
    const int msg = pl.n_hr * 16;
    // RMSNorm gain of layer 0 (then of the next layer, loaded a layer ahead)
    const int n4 = p.d / 4;
    auto gain = [&](int l) {
        uint2 g = make_uint2(0x3C003C00u, 0x3C003C00u);   // 1.0 in fp16
        if (l < p.L && p.layers[l].gamma && tid < n4)
            g = __ldg(reinterpret_cast<const uint2*>(p.layers[l].gamma + 4 * tid));
        return g;
    };
    uint2 gam = gain(0);
    // ---- head flush (after the last layer that owns a head).  A CTA adds its
    // finished tasks of a head to the head's count once; the one that completes
    // the count routes.  false: the launch gave up (uniform).
    auto flush = [&]() -> bool {
        const int tph = p.H / kRowTile + p.E / kRowTile;
        const int n2 = p.K + (step > 0 ? p.K : 0);
        int xl = -1, ndone = 0;
        for (int t = pl.t0; t < pl.t1; ++t) {
            const int hi = t / tph, j = t % tph, l = s.heads[hi];
            const LayerP& Ly = p.layers[l];
            const int sidx = Ly.sidx;
            if (l != xl) {
                const unsigned long long* xs =
                    reinterpret_cast<const unsigned long long*>(p.ws + W.xs) + (long long)sidx * (p.d / 2);
                if (!flush_head1(p, hdr, xs, want())) return false;
                xl = l;
            }
            float* lg = reinterpret_cast<float*>(p.ws + W.logh) + ((long long)par * p.Ls + sidx) * p.E;
            stamp1(p, 0xF100 | (t - pl.t0));
            bool ok = take1(p, hdr, c, flush_bytes(s.S, j, 0, n2));
            const char* blkA = ring() + c.off;
            ok = take1(p, hdr, c, flush_bytes(s.S, j, 1, n2)) && ok;
            const char* blkB = ring() + c.off;
            stamp1(p, 0xF200 | (t - pl.t0));
            if (ok) flush_task1(p, j, n2, blkA, blkB, lg);
            if (cbar_or1(!ok || vload(&s.abort))) return false;
            give1(c);
            stamp1(p, 0xF300 | (t - pl.t0));
            ++ndone;
            const bool head_end = t + 1 == pl.t1 || (t + 1) / tph != hi;
            if (!head_end) continue;
            if (tid == 0) {
                __threadfence();
                unsigned* cnt = reinterpret_cast<unsigned*>(p.ws + W.cnt) + ((long long)par * p.Ls + sidx);
                s.topk = atom_acq_rel_add_u32(cnt, (unsigned)ndone) + (unsigned)ndone == (unsigned)tph;
            }
            ndone = 0;
            cbar1();
            if (s.topk && tid < 32) {
                // the head's prediction for its target layer at the next token [S3.2]
                for (int e = lane; e < p.E; e += 32) s.logits[e] = __ldcg(lg + e);
                __syncwarp();
                const long long o = ((long long)par * p.Ls + Ly.head_target) * p.K;
                warp_route(s.logits, p.E, p.K, Ly.head_route_kind, Ly.head_n_groups, Ly.head_topk_groups,
                           Ly.head_route_scale, Ly.head_bias, s.rscr, p.pred_ids + o, p.pred_w + o, lane);
                if (p.dbg_logits)
                    for (int e = lane; e < p.E; e += 32) p.dbg_logits[(long long)l * p.E + e] = s.logits[e];
            }
            cbar1();
        }
        return true;
    };
    bool broke = true;   // left the layer loop early (set false when it completes)
    for (int l = 0;; ++l) {
        if (l == p.L) {
            broke = false;
            break;
        }
        const LayerP& Ly = p.layers[l];
        const bool own = own_routed1(p, l, step);
        const int sidx = Ly.sidx;
        stamp1(p, (l << 8) | 0);
        // the exchange barrier of this layer is armed before the peer can send:
        // layer 0's here, the next layer's right after this layer's exchange
        if (l == 0 && xch && tid == 0) mbar_arrive_expect_tx(&s.xbar, (uint32_t)(msg * 4));
        // ---- x, from the previous layer's y
        const unsigned long long* yprev = l > 0 ? row(W.y, p.layers[l - 1].sidx, p.d) : nullptr;
        unsigned long long* xs_out =
            (cta == 0 && (Ly.flags & LF_HEAD))
                ? reinterpret_cast<unsigned long long*>(p.ws + W.xs) + (long long)sidx * (p.d / 2)
                : nullptr;
        __half* dbg = (p.dbg_h && cta == 0 && l > 0) ? p.dbg_h + (long long)(l - 1) * p.d : nullptr;
        if (!build_x1(p, hdr, l, l == 0 ? p.h_io : nullptr, yprev, l > 0 ? want() : tag, gam, xs_out, tag, dbg))
            break;
        gam = gain(l + 1);
        stamp1(p, (l << 8) | 2);
        // ---- routing of a layer that routes itself
        if (own) {
            unsigned long long* logr = row(W.logr, sidx, p.E);
            bool ok = true;
            if (L.b0.bytes) {
                // this CTA's router row tile, published as tagged logits
                ok = take1(p, hdr, c, L.b0.bytes);
                float a0 = 0.f, a1 = 0.f;
                if (ok) f16_units(s, ring() + c.off, tid >> 5, ng, kCW, 0, lane, a0, a1);
                put_part(s, a0, a1);
                if (cbar_or1(!ok)) break;
                give1(c);
                if (tid < 16) st_relaxed_u64(logr + 16 * pl.rt + tid, tagged(tag, tile_sum(s, tid)));
            }
            // CTAs whose weights or act depend on the routing route (CTA 0 records it)
            const bool routes = (pl.role == R1_ROUTED && pl.nseg > 0) || pl.dt >= 0 || cta == 0;
            if (routes) {
                const unsigned wt = want();
                if (tid < p.E) ok = poll1(hdr, logr + tid, wt, &s.logits[tid]);
            }
            if (cbar_or1(!ok)) break;
            if (routes) {
                if (tid < 32)
                    warp_route(s.logits, p.E, p.K, Ly.route_kind, Ly.n_groups, Ly.topk_groups, Ly.route_scale,
                               Ly.bias, s.rscr, s.ids[l], s.w[l], lane);
                cbar1();
                if (tid == 0) *(volatile int*)&s.route_ready[l] = 1;
            }
        }
        if (cta == 0 && tid < p.K) {
            p.exec_ids[((long long)par * p.Ls + sidx) * p.K + tid] = s.ids[l][tid];
            st_relaxed_u64(row(W.ex, sidx, p.K) + tid, ((unsigned long long)tag << 32) | (unsigned)s.ids[l][tid]);
        }
        stamp1(p, (l << 8) | 4);
        // ---- gate/up (or LoRA A) partial sums
        if (L.b1.bytes) {
            const bool ok = take1(p, hdr, c, L.b1.bytes);
            stamp1(p, (l << 8) | 9);
            const char* blk1 = ring() + c.off;
            if (pl.role == R1_LORA) {
                float a0 = 0.f, a1 = 0.f;
                if (ok) f16_units(s, blk1, tid >> 5, ng, kCW, 0, lane, a0, a1);
                put_part(s, a0, a1);
            } else if (ok) {
                gateup1(blk1, ngh, g0, pl.n_hr);
            }
            if (cbar_or1(!ok || vload(&s.abort))) break;
            give1(c);
        }
        stamp1(p, (l << 8) | 5);
        if (pl.role == R1_LORA) {
            // rank 0: A_gate x (words 0-15), rank 1: A_up x (16-31)
            if (tid < 16) st_relaxed_u64(row(W.lax, sidx, 32) + 16 * rank + tid, tagged(tag, tile_sum(s, tid)));
        } else if (xch) {
            // ---- swap the partial sums with the peer, then act
            if (tid < msg) {
                const float v = tile_sum(s, tid);
                s.mine[tid] = v;
                st_async_b32(rrecv + 4u * tid, v, rbar);
            }
            bool ok = true;
            if (lora && tid >= kCT - 32) ok = poll1(hdr, row(W.lax, sidx, 32) + lane, want(), &s.lax[lane]);
            if (tid == 0) {
                if (!mbar_wait1(hdr, &s.xbar, (uint32_t)(nx & 1))) ok = false;
                else if (l + 1 < p.L) mbar_arrive_expect_tx(&s.xbar, (uint32_t)(msg * 4));
            }
            ++nx;
            bool ok3 = true;
            if (L.b3.bytes) ok3 = take1(p, hdr, c, L.b3.bytes);
            if (cbar_or1(!ok || !ok3 || vload(&s.abort))) break;
            stamp1(p, (l << 8) | 6);
            act1(p, l, rank, rank ? s.recv : s.mine, rank ? s.mine : s.recv, ring() + c.off, lora,
                 row(W.act, sidx, NA), tag);
            if (L.b3.bytes) {
                cbar1();
                give1(c);
            }
        }
        stamp1(p, (l << 8) | 7);
        // ---- down: this CTA's output row tile
        if (pl.dt >= 0) {
            const bool ok = take1(p, hdr, c, L.b2.bytes);
            stamp1(p, (l << 8) | 10);
            if (cbar_or1(!ok)) break;
            if (!down_tile1(p, hdr, l, ring() + c.off, row(W.act, sidx, NA), want(), lora_dn, row(W.y, sidx, p.d),
                            pl.dt, tag))
                break;
            cbar1();
            give1(c);
        }
        stamp1(p, (l << 8) | 8);
        if (l == s.flush_after && !flush()) break;
    }
    if (broke) {
        if (tid == 0) *(volatile int*)&s.abort = 1;
        return;
    }
    stamp1(p, 0xFF00);
    // ---- the last layer's output into h_io, a slice per CTA (every CTA read
    // h_io at layer 0 before it published anything the last y depends on)
    const unsigned long long* ylast = row(W.y, p.layers[p.L - 1].sidx, p.d);
    const unsigned wt = want();
    const int a = p.d * cta / nct, b = p.d * (cta + 1) / nct;
    bool ok = true;
    for (int i = a + tid; i < b && ok; i += kCT) {
        float yv = 0.f;
        ok = poll1(hdr, ylast + i, wt, &yv);
        const __half h = __float2half_rn(__half2float(s.h[i]) + yv);
        p.h_io[i] = h;
        if (p.dbg_h) p.dbg_h[(long long)(p.L - 1) * p.d + i] = h;
    }
    if (cbar_or1(!ok)) return;
    if (cta == 0 && tid == 0) {
        if (p.step < 0) hdr->step = step + 1;
        hdr->serial = tag;   // the next launch tags with serial + 1
    }
}

// ------------------------------------------------------------------ kernel ----
__global__ void __cluster_dims__(kClusterCtas, 1, 1) __launch_bounds__(kT1, 1)
    decode1_kernel(const __grid_constant__ Prog p) {
    Sm1& s = sm();
    const int tid = threadIdx.x;
    WsHeader* hdr = reinterpret_cast<WsHeader*>(p.ws);
    uint32_t ncl;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(ncl));
    if (ncl != (uint32_t)kClusterCtas || (int)gridDim.x != 2 * p.pairs1[0]) {
        if (tid == 0) {
            atomicCAS(&hdr->error, 0, EDGE0_EUNSUPPORTED);
            atomicExch(&hdr->abort, 1);
        }
        return;
    }
    const int rank = (int)cluster_ctarank(), pair = blockIdx.x / 2;
    const int shared = (p.layers[0].flags & LF_SHARED) != 0;
    const Ws1 W = ws1(p.Ls, p.d, p.E, p.K, p.K * p.I + (shared ? p.Is : 0));
    __shared__ int s_step;
    __shared__ unsigned s_tag;
    if (tid == 0) {
        s.abort = 0;
        s.topk = 0;
        s.issued = 0;
        s.released_blocks = 0;
        s.released = 0;
        const unsigned long long wn = ld_relaxed_u64(&hdr->wait_ns);
        s.wait_ns = wn ? wn : kDefaultWaitNs;
        s.trace = blockIdx.x < kTraceCtas ? ld_volatile_s32(&hdr->trace) : 0;
        s.tslot = 0;
        s.ptslot = 3072;
        for (int i = 0; i < kBlocks; ++i) mbar_init(&s.full[i], 1);
        mbar_init(&s.xbar, 1);
        fence_mbar_init();
        s_step = p.step >= 0 ? p.step : ld_volatile_s32(&hdr->step);
        s_tag = ((unsigned)ld_volatile_s32(reinterpret_cast<const int*>(&hdr->serial)) % kTagMask) + 1u;
        // the plan of this CTA and the layout of its blocks
        Shape1 S;
        S.d = p.d; S.I = p.I; S.Is = p.Is; S.E = p.E; S.K = p.K; S.H = p.H; S.r = p.r;
        S.shared = shared;
        S.lora = (p.layers[0].flags & LF_LORA) != 0;
        S.P = p.pairs1[0]; S.Pr = p.pairs1[1]; S.Ps = p.pairs1[2]; S.Pl = p.pairs1[3];
        S.nct = gridDim.x;
        int nh = 0;
        s.flush_after = -1;
        for (int l = 0; l < p.L; ++l)
            if (p.layers[l].flags & LF_HEAD) {
                s.heads[nh++] = l;
                s.flush_after = l;
            }
        S.n_heads = nh;
        s.S = S;
        if (!plan1(S, pair, rank, s.plan) || !layout1(S, s.plan, rank, s.lay)) fail1(hdr, EDGE0_EUNSUPPORTED);
    }
    __syncthreads();
    const int step = s_step, par = step & 1;
    // clear the other step parity's head logits and task counts for the next step
    {
        const int op = par ^ 1;
        const long long tot = (long long)p.L * p.E;
        const long long a = tot * blockIdx.x / gridDim.x, b = tot * (blockIdx.x + 1) / gridDim.x;
        for (long long i = a + tid; i < b; i += kT1) {
            const long long l = i / p.E, o = i % p.E;
            reinterpret_cast<float*>(p.ws + W.logh)[((long long)op * p.Ls + p.layers[l].sidx) * p.E + o] = 0.f;
        }
        if (blockIdx.x == 0)
            for (int l = tid; l < p.L; l += kT1)
                reinterpret_cast<unsigned*>(p.ws + W.cnt)[(long long)op * p.Ls + p.layers[l].sidx] = 0u;
    }
    // routing known at launch: the predictions of prerouted layers (step > 0)
    for (int l = tid; l < p.L; l += kT1) s.route_ready[l] = 0;
    for (int i = tid; i < p.L * p.K; i += kT1) {
        const int l = i / p.K, k = i % p.K;
        if (step > 0 && (p.layers[l].flags & LF_PREROUTED)) {
            const long long o = ((long long)((step - 1) & 1) * p.Ls + p.layers[l].sidx) * p.K + k;
            int e = p.pred_ids[o];
            if (e < 0 || e >= p.E) {
                fail1(hdr, EDGE0_EINVAL);
                e = 0;
            }
            s.ids[l][k] = e;
            s.w[l][k] = p.pred_w[o];
        }
    }
    __syncthreads();
    // the peer's barriers exist before any exchange
    cluster_sync_all();
    if (!vload(&s.abort)) {
        if (tid >= kCT) producer1(p, hdr, W, step, par, s_tag);
        else consumer1(p, hdr, W, step, par, s_tag);
    }
    __syncthreads();
    if (tid == 0 && vload(&s.abort)) {
        // let copies still in flight into this CTA's ring land before it exits (bounded)
        const int issued = vload(&s.issued);
        const unsigned long long t0 = now1();
        for (int k = issued > kBlocks ? issued - kBlocks : 0; k < issued; ++k)
            while (!mbar_try_wait(&s.full[k % kBlocks], (uint32_t)((k / kBlocks) & 1)))
                if (now1() - t0 > 100000000ull) break;
        while (now1() - t0 < 20000ull) {}   // stores from the peer still in flight
    }
    __syncthreads();
    // neither CTA of a pair leaves while the other may still write into it
    cluster_sync_all();
}

}  // namespace d1

// ------------------------------------------------------------------- host ----
using namespace d1;

long long decode1_ws_bytes(int Ls, int d, int E, int K, int I, int Is) {
    if (Ls <= 0 || d <= 0 || E <= 0 || K <= 0 || I <= 0 || Is < 0) return 0;
    return ws1(Ls, d, E, K, K * I + Is).end + kTraceBytes;
}

namespace {
std::mutex g_d1_mutex;
int g_d1_grid[64] = {};
int g_d1_smem[64] = {};

struct Key1 {
    int d, I, Is, E, K, H, r, shared, lora, n_heads, nct, smem;
    int rc, P, Pr, Ps, Pl, ring;
};
constexpr int kKeys = 16;
Key1 g_keys[kKeys];
int g_nkeys = 0, g_next_key = 0;

int grid1(int* nct, int* smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return EDGE0_ECUDA;
    if (!g_d1_grid[dev]) {
        int maxsm = 0;
        if (cudaDeviceGetAttribute(&maxsm, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return EDGE0_ECUDA;
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, decode1_kernel) != cudaSuccess) return EDGE0_ECUDA;
        const int dyn = maxsm - (int)fa.sharedSizeBytes;
        if (cudaFuncSetAttribute(decode1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn) != cudaSuccess)
            return EDGE0_ECUDA;
        cudaLaunchConfig_t cfg;
        memset(&cfg, 0, sizeof(cfg));
        cfg.gridDim = dim3(kClusterCtas);
        cfg.blockDim = dim3(kT1);
        cfg.dynamicSmemBytes = dyn;
        int ncl = 0;
        if (cudaOccupancyMaxActiveClusters(&ncl, (void*)decode1_kernel, &cfg) != cudaSuccess || ncl < 4)
            return EDGE0_ECUDA;
        g_d1_grid[dev] = ncl * kClusterCtas;
        g_d1_smem[dev] = dyn;
    }
    *nct = g_d1_grid[dev];
    *smem = g_d1_smem[dev];
    return EDGE0_OK;
}

// the pairs, every CTA's plan and blocks for the shapes on a grid of at most
// k.nct CTAs: every output and router row tile has its CTA, the ring holds the
// largest block
int derive1(Key1& k) {
    Shape1 S;
    S.d = k.d; S.I = k.I; S.Is = k.Is; S.E = k.E; S.K = k.K; S.H = k.H; S.r = k.r;
    S.shared = k.shared; S.lora = k.lora; S.n_heads = k.n_heads;
    if (k.nct % kClusterCtas || k.nct < 8) return EDGE0_EUNSUPPORTED;
    if (n_act1(S) > kMaxNA || n_act1(S) % kGroup) return EDGE0_EUNSUPPORTED;
    if (S.lora && (!S.shared || S.Is / kGroup > kCW || S.r > 16)) return EDGE0_EUNSUPPORTED;
    if (!choose_pairs(S, k.nct / kClusterCtas)) return EDGE0_EUNSUPPORTED;
    if (S.d / kRowTile > S.nct || S.E / kRowTile > S.nct) return EDGE0_EUNSUPPORTED;
    const int ring = ((k.smem - kSm1Bytes) / 128) * 128;
    if (ring < 2 * kPieceMax) return EDGE0_EUNSUPPORTED;
    int biggest = 0;
    for (int pair = 0; pair < S.P; ++pair)
        for (int rank = 0; rank < kClusterCtas; ++rank) {
            Plan1 pl;
            Lay1 L;
            if (!plan1(S, pair, rank, pl) || !layout1(S, pl, rank, L)) return EDGE0_EUNSUPPORTED;
            if (pl.role != R1_LORA && pl.n_hr < 1) return EDGE0_EUNSUPPORTED;   // every pair publishes
            const Block1* bl[4] = {&L.b0, &L.b1, &L.b3, &L.b2};
            for (const Block1* b : bl) biggest = b->bytes > biggest ? b->bytes : biggest;
        }
    const int tph = S.H / kRowTile + S.E / kRowTile;
    for (int j = 0; j < tph && S.n_heads > 0; ++j)
        for (int h = 0; h < 2; ++h) {
            Block1 B;
            if (!flush_block(S, j, h, B, nullptr, 2 * S.K) || B.n > 32) return EDGE0_EUNSUPPORTED;
            biggest = B.bytes > biggest ? B.bytes : biggest;
        }
    // a task's two blocks are held together (with a ring tail skipped between)
    if (S.n_heads > 0 && flush_bytes(S, 0, 0, 2 * S.K) + 2 * flush_bytes(S, 0, 1, 2 * S.K) > ring)
        return EDGE0_EUNSUPPORTED;
    if (biggest > ring) return EDGE0_EUNSUPPORTED;
    k.P = S.P; k.Pr = S.Pr; k.Ps = S.Ps; k.Pl = S.Pl;
    k.ring = ring;
    return EDGE0_OK;
}
}  // namespace

int decode1_check(Prog& p) {
    if (p.mode != MODE_DECODE || p.B != 1) return EDGE0_EUNSUPPORTED;
    if (p.d % 128 || p.d > kMaxD1 || p.E % kRowTile || p.E > EDGE0_MAX_E || p.H % kRowTile) return EDGE0_EUNSUPPORTED;
    if (p.I % kGroup || p.Is % kGroup || p.r <= 0 || p.r > 16 || p.K > kMaxK1) return EDGE0_EUNSUPPORTED;
    const int f0 = p.layers[0].flags & (LF_SHARED | LF_LORA);
    if (p.ws_bytes < decode1_ws_bytes(p.Ls, p.d, p.E, p.K, p.I, (f0 & LF_SHARED) ? p.Is : 0))
        return EDGE0_EUNSUPPORTED;
    int n_heads = 0;
    for (int l = 0; l < p.L; ++l) {
        const LayerP& Ly = p.layers[l];
        if ((Ly.flags & (LF_SHARED | LF_LORA)) != f0) return EDGE0_EUNSUPPORTED;
        if (Ly.slot_table || Ly.gu_host || !Ly.down_rows) return EDGE0_EUNSUPPORTED;
        if ((Ly.flags & LF_SHARED) && !Ly.sh_down_rows) return EDGE0_EUNSUPPORTED;
        if ((Ly.flags & LF_LORA) && !Ly.lora_Ad) return EDGE0_EUNSUPPORTED;
        if (Ly.flags & LF_HEAD) ++n_heads;
        // every tagged word of a launch has one writer: one layer per state row
        for (int m = 0; m < l; ++m)
            if (p.layers[m].sidx == Ly.sidx) return EDGE0_EUNSUPPORTED;
        // bulk copies read whole 16-byte lines of every source
        if (((uintptr_t)Ly.gu | (uintptr_t)Ly.down_rows | (uintptr_t)Ly.router | (uintptr_t)Ly.sh_down_rows) & 15)
            return EDGE0_EUNSUPPORTED;
        if (Ly.gamma && ((uintptr_t)Ly.gamma & 7)) return EDGE0_EUNSUPPORTED;
    }
    Key1 k;
    memset(&k, 0, sizeof(k));
    int rc = grid1(&k.nct, &k.smem);
    if (rc) return rc;
    k.d = p.d; k.I = p.I; k.Is = p.Is; k.E = p.E; k.K = p.K; k.H = p.H; k.r = p.r;
    k.shared = (f0 & LF_SHARED) != 0;
    k.lora = (f0 & LF_LORA) != 0;
    k.n_heads = n_heads;
    std::lock_guard<std::mutex> lock(g_d1_mutex);
    int hit = -1;
    for (int i = 0; i < g_nkeys; ++i) {
        const Key1& q = g_keys[i];
        if (q.d == k.d && q.I == k.I && q.Is == k.Is && q.E == k.E && q.K == k.K && q.H == k.H && q.r == k.r &&
            q.shared == k.shared && q.lora == k.lora && q.n_heads == k.n_heads && q.nct == k.nct && q.smem == k.smem) {
            hit = i;
            break;
        }
    }
    if (hit < 0) {
        k.rc = derive1(k);
        hit = g_next_key;
        g_keys[hit] = k;
        g_next_key = (g_next_key + 1) % kKeys;
        if (g_nkeys < kKeys) ++g_nkeys;
    }
    const Key1& q = g_keys[hit];
    if (q.rc) return q.rc;
    p.pairs1[0] = q.P;
    p.pairs1[1] = q.Pr;
    p.pairs1[2] = q.Ps;
    p.pairs1[3] = q.Pl;
    p.ring1 = q.ring;
    return EDGE0_OK;
}

int decode1_launch(Prog& p, cudaStream_t stream) {
    int rc = decode1_check(p);
    if (rc) return rc;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(2 * p.pairs1[0]);
    cfg.blockDim = dim3(kT1);
    cfg.dynamicSmemBytes = kSm1Bytes + p.ring1;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];   // the cluster shape is compiled into the kernel
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode1_kernel, p) != cudaSuccess) return EDGE0_ECUDA;
    return EDGE0_OK;
}

}  // namespace edge0
