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
// Data flow.  One CTA per SM.  Every value that crosses CTAs is a
// single-writer word: an fp32 value (or an id) and the launch's 32-bit tag
// stored together as one 64-bit word, which is single-copy atomic; readers poll
// a word until it carries their tag.  No counters, fences or grid barriers
// stand between the layers: a CTA waits for exactly the words it reads.
//   * Every CTA forms x from all of the previous layer's y.  Consumer warp w
//     owns a fixed slice of d (whole groups of 64): it keeps h for that slice in
//     registers and builds x there straight into tensor-core B fragments.
//   * Gate/up: each expert CTA owns a run of half-row tiles ("hr": 8 act rows;
//     the packed tile interleaves 8 gate and 8 up rows) of the routed slots or
//     the shared expert, over all of d; it publishes those act rows (w_k act for
//     routed rows, the shared expert's with its LoRA B_gate / B_up terms).  The
//     last CTAs form the LoRA A_gate x, A_up x partial sums instead.
//   * Down: CTA c < d/16 owns output row tile c.  Each of its warps reads the
//     act values of its act groups straight into B fragments and applies that
//     tile of every expert's down (and the shared expert's, with (alpha / r)
//     B_down A_down act); the tile's y goes out after one reduction.
//   * On a layer that routes itself, E/16 CTAs publish one router row tile each
//     and every CTA that needs the routing runs the routing rule.
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
#include <vector>

#include "common.cuh"
#include "internal.cuh"

namespace edge0 {
namespace d1 {

constexpr int kCW = 16;                  // consumer warps
constexpr int kCT = kCW * 32;            // consumer threads
constexpr int kT1 = kCT + 32;            // + the producer warp
constexpr int kMaxHr1 = 5;               // hr of one CTA
constexpr int kMaxSeg1 = 3;              // expert runs of one CTA
constexpr int kMaxPc = 24;               // copies of one block
constexpr int kBlocks = 16;              // block barriers
constexpr int kPieceMax = 32768;         // bytes of one bulk copy
constexpr int kMaxD1 = 2048;
constexpr int kMaxGW = kMaxD1 / kGroup / kCW;   // groups of d a warp owns
constexpr int kMaxNA = 4608;             // act values of a layer: K I + Is
constexpr int kMaxUW = (kMaxNA / kGroup + kCW - 1) / kCW;   // act groups a warp owns
constexpr int kMaxNQ = 4;                // LoRA-A CTAs per matrix
constexpr int kMaxK1 = EDGE0_MAX_K;
constexpr unsigned kTagMask = 0x3FFFFFFFu;   // launch tags: 1 .. kTagMask
constexpr unsigned kHoldBit = 0x40000000u;   // never in a written tag
static_assert(kMaxGW == 2, "a warp's slice of d is at most two groups (128 values, 4 per lane)");

__host__ __device__ inline void split1(int n, int parts, int i, int* a, int* b) {
    *a = (int)((long long)n * i / parts);
    *b = (int)((long long)n * (i + 1) / parts);
}

// ------------------------------------------------------------------ plan ----
struct Shape1 {
    int d, I, Is, E, K, H, r;
    int shared, lora;          // every layer of the launch has a shared expert / LoRA
    int nct;                   // CTAs
    int NQ;                    // LoRA-A CTAs per matrix (0 without LoRA)
    int n_heads;
};
__host__ __device__ inline int n_act1(const Shape1& S) { return S.K * S.I + (S.shared ? S.Is : 0); }
__host__ __device__ inline int n_hr_all(const Shape1& S) { return n_act1(S) / kHalfRow; }
__host__ __device__ inline int n_lora_ctas(const Shape1& S) { return S.lora ? 2 * S.NQ : 0; }

enum Role1 : int { R1_EXPERT = 0, R1_LORA = 1 };
struct Seg1 {
    int slot;                  // routed slot (index into the layer's K ids) or -1: shared
    int hr0, hr1;              // hr [hr0, hr1) of the expert
};
struct Plan1 {
    int role, nseg, n_hr;
    Seg1 seg[kMaxSeg1];
    int shr;                   // the run of the shared expert (-1: none)
    int lm, la0, la1;          // LoRA CTA: matrix (0 A_gate, 1 A_up), its groups of d
    int dt;                    // output row tile of the down phase (-1: none)
    int rt;                    // router row tile on layers that route themselves (-1: none)
    int t0, t1;                // head-flush tasks
};

// The hr of all experts in order (routed slot 0, 1, ..., then the shared
// expert) are split evenly over the expert CTAs [0, nct - 2 NQ); the last 2 NQ
// CTAs form LoRA A partial sums (NQ per matrix, each over a range of groups).
__host__ __device__ inline bool plan1(const Shape1& S, int c, Plan1& p) {
    p.role = R1_EXPERT;
    p.nseg = p.n_hr = 0;
    p.shr = -1;
    p.lm = p.la0 = p.la1 = 0;
    const int hpe = S.I / kHalfRow, n_rt = S.K * hpe, nG = S.nct - n_lora_ctas(S);
    if (c < nG) {
        int a, b;
        split1(n_hr_all(S), nG, c, &a, &b);
        while (a < b) {
            if (p.nseg >= kMaxSeg1) return false;
            Seg1& s = p.seg[p.nseg];
            if (a < n_rt) {
                const int slot = a / hpe, end = (slot + 1) * hpe < b ? (slot + 1) * hpe : b;
                s.slot = slot;
                s.hr0 = a - slot * hpe;
                s.hr1 = end - slot * hpe;
                a = end;
            } else {
                s.slot = -1;
                s.hr0 = a - n_rt;
                s.hr1 = b - n_rt;
                p.shr = p.nseg;
                a = b;
            }
            p.n_hr += s.hr1 - s.hr0;
            ++p.nseg;
        }
    } else {
        p.role = R1_LORA;
        const int j = c - nG;
        p.lm = j / S.NQ;
        split1(S.d / kGroup, S.NQ, j % S.NQ, &p.la0, &p.la1);
    }
    if (p.n_hr > kMaxHr1) return false;
    p.dt = c < S.d / kRowTile ? c : -1;
    const int rt = (2 * S.nct - 1 - n_lora_ctas(S) - c) % S.nct;
    p.rt = rt < S.E / kRowTile ? rt : -1;
    split1(S.n_heads * (S.H / kRowTile + S.E / kRowTile), S.nct, c, &p.t0, &p.t1);
    return true;
}

// ---------------------------------------------------------------- blocks ----
// A block is one (layer, phase) share of a CTA's weights, copied contiguously
// into the ring, in this order per layer:
//   b0 its router row tile over all of d (router CTAs, layers that route
//      themselves): the row tile's groups in order;
//   b1 its gate/up units over all of d: the first half of d for every hr of
//      every run, then the second half (a LoRA CTA: its groups of A_gate or A_up);
//   b3 the LoRA B_gate, B_up rows of its shared act rows;
//   b2 its output row tile of every routed expert's down, then of the shared
//      expert's (one unit per act group, in act order), then (LoRA) A_down and
//      the tile's rows of B_down;
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
    int seg_base[kMaxSeg1];    // CTA-local act row of each run's first row
};

// one CTA's entry of the plan table: its Plan1, then its Lay1
constexpr int kTab1Stride = (int)((sizeof(Plan1) + sizeof(Lay1) + 255) / 256 * 256);

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

__host__ __device__ inline bool layout1(const Shape1& S, const Plan1& p, Lay1& L) {
    L.b0.n = L.b0.bytes = L.b1.n = L.b1.bytes = L.b3.n = L.b3.bytes = L.b2.n = L.b2.bytes = 0;
    L.bu = L.ad = L.bd = 0;
    const int ng = S.d / kGroup, ng0 = ng / 2, ng1 = ng - ng0;
    bool ok = true;
    // b0: router row tile rt (packed fp16 [E x d]: the first half of d for every
    // row tile, then the second half)
    if (p.rt >= 0) {
        const long long nE = S.E / kRowTile;
        ok &= add_piece(L.b0, K1_ROUTER, 0, (long long)p.rt * ng0 * kF16Unit, (long long)ng0 * kF16Unit);
        ok &= add_piece(L.b0, K1_ROUTER, 0, nE * ng0 * kF16Unit + (long long)p.rt * ng1 * kF16Unit,
                        (long long)ng1 * kF16Unit);
    }
    if (p.role == R1_LORA) {
        // LoRA A (packed fp16 [r x d], one row tile: its two halves back to back
        // are the row tile's groups in order)
        ok &= add_piece(L.b1, p.lm ? K1_LU : K1_LA, 0, (long long)p.la0 * kF16Unit,
                        (long long)(p.la1 - p.la0) * kF16Unit);
    } else {
        // b1: gate/up units (packed [half][tile][group of the half]) of each run
        int base = 0;
        for (int h = 0; h < 2; ++h)
            for (int s = 0; s < p.nseg; ++s) {
                const Seg1& sg = p.seg[s];
                const long long tiles = (sg.slot < 0 ? S.Is : S.I) / kHalfRow;
                const int ngh = h ? ng1 : ng0;
                ok &= add_piece(L.b1, K1_GU, s, (h ? tiles * ng0 * kQ4Unit : 0) + (long long)sg.hr0 * ngh * kQ4Unit,
                                (long long)(sg.hr1 - sg.hr0) * ngh * kQ4Unit);
                if (h == 0) {
                    L.seg_base[s] = base;
                    base += 8 * (sg.hr1 - sg.hr0);
                }
            }
        // b3: LoRA B_gate, B_up rows (row-major [Is, r] fp16) of the shared run
        if (S.lora && p.shr >= 0) {
            const Seg1& sg = p.seg[p.shr];
            const long long rb = 2LL * S.r, row0 = 8LL * sg.hr0, rows = 8LL * (sg.hr1 - sg.hr0);
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
//   y     [2][Ls][d]        tagged  layer output (writer: the row tile's CTA)
//   act   [2][Ls][NA]       tagged  act of the layer, NA = K I + Is: routed slot k
//                                   at k I (times w_k), the shared expert at K I
//   logr  [2][Ls][E]        tagged  own-router logits (writer: the row tile's CTA)
//   lax   [2][Ls][8][16]    tagged  partial A_gate x (rows 0 .. NQ-1), A_up x
//                                   (rows NQ .. 2 NQ-1)
//   ex    [2][Ls][K]        tagged  executed ids (writer: CTA 0)
//   xs    [Ls][d/2]         tagged  x as fp16 pairs (writer: CTA 0, head layers)
//   logh  [2][Ls][E]        fp32    head logits (vector reductions; the other
//                                   parity's are cleared for the next step)
//   cnt   [2][Ls]           u32     head tasks done (cleared likewise)
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
    w.lax = o;  o += 2LL * Ls * 2 * kMaxNQ * 16 * 8;
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
    int abort;                            // CTA abort flag (read after consumer barriers)
    int topk;                             // flush: this CTA completed the current head
    int issued;                           // blocks issued by the producer
    int released_blocks;                  // blocks the consumers are done with
    int released;                         // ring position up to which blocks are free
    unsigned long long wait_ns;
    int trace, tslot, ptslot;
    int flush_after;                      // the head flush follows this layer (-1: no heads)
    // the launch's layer descriptors: read from shared memory, not the kernel
    // parameter block
    __align__(16) LayerP ly[EDGE0_MAX_LAYERS];
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
    __align__(16) float partg[kCW][kMaxHr1 * 16];   // gate/up (LoRA A) partial sums per warp
    __align__(16) float partd[kCW][16];             // down / router / flush partial sums per warp
    __align__(16) float logits[EDGE0_MAX_E];
    __align__(16) float rscr[2 * EDGE0_MAX_E];
    __align__(16) uint2 gf[8];            // GELU(z) of a flush task as a hi/lo B step
    // per-warp B fragments: x of the warp's groups [group][t][step] (lanes 0-3
    // read them), and one act group [step][lane < 8] as hi (lanes 0-3) / lo (4-7)
    __align__(16) uint2 xw[kCW][kMaxGW * 16];
    __align__(16) uint2 aw[kCW][32];
};
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
// past its limit (then EDGE0_ETIMEOUT is recorded); out of line, so that the
// many wait loops stay small in the instruction cache
__device__ __noinline__ bool wait_check(WsHeader* hdr, unsigned long long t0) {
    if (gone1(hdr)) return false;
    if (now1() - t0 > sm().wait_ns) {
        fail1(hdr, EDGE0_ETIMEOUT);
        return false;
    }
    return true;
}
__device__ __forceinline__ bool keep_waiting(WsHeader* hdr, unsigned it, unsigned long long t0) {
    return (it & 15) != 15 || wait_check(hdr, t0);
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

// two pairs loaded already as a, b: both re-polled together until all four
// words carry `tag` (each re-poll costs one round trip to L2, so the loads that
// are still pending go out together)
__device__ __forceinline__ bool settle22(WsHeader* hdr, const unsigned long long* pa, const unsigned long long* pb,
                                         unsigned tag, ulonglong2& a, ulonglong2& b) {
    if (tok(a.x, tag) && tok(a.y, tag) && tok(b.x, tag) && tok(b.y, tag)) return true;
    const unsigned long long t0 = now1();
    for (unsigned it = 0;; ++it) {
        if (!keep_waiting(hdr, it, t0)) return false;
        a = ld_relaxed_u64x2(pa);
        b = ld_relaxed_u64x2(pb);
        if (tok(a.x, tag) && tok(a.y, tag) && tok(b.x, tag) && tok(b.y, tag)) return true;
    }
}

// trace stamps (thread 0 of the consumers, lane 0 of the producer): tag, global
// timer, SM cycle counter (inline: a call would wait for the caller's loads)
__device__ __forceinline__ void stamp_slow1(const Prog& p, int tag, bool producer) {
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
// per-warp stamp k (< 3) of the middle layer: lane 0 of each consumer warp, at
// trace slots 2800 + 9 warp + 3 k
__device__ __forceinline__ void wstamp1(const Prog& p, int l, int k) {
    if (sm().trace && l == p.L / 2 && (threadIdx.x & 31) == 0) {
        unsigned long long* tr = reinterpret_cast<unsigned long long*>(p.ws + p.ws_bytes - kTraceBytes) +
                                 (long long)blockIdx.x * kTraceSlots + 2800 + 9 * (threadIdx.x >> 5) + 3 * k;
        long long c;
        asm volatile("mov.u64 %0, %%clock64;" : "=l"(c));
        tr[0] = 0xA000u | (unsigned)(k << 8) | (threadIdx.x >> 5);
        tr[1] = now1();
        tr[2] = (unsigned long long)c;
    }
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
// bounded wait on a block barrier phase; false on abort/timeout
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
__device__ __forceinline__ float2 unpack2(uint32_t v) {
    return __half22float2(*reinterpret_cast<const __half2*>(&v));
}
// an fp32 pair as its fp16 hi parts and as the fp16 of the rests times kLoScale
__device__ __forceinline__ void hilo2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __half ha = __float2half_rn(a), hb = __float2half_rn(b);
    hi = (uint32_t)__half_as_ushort(ha) | ((uint32_t)__half_as_ushort(hb) << 16);
    lo = pack2((a - __half2float(ha)) * kLoScale, (b - __half2float(hb)) * kLoScale);
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
// per-warp partial sums of rows g, g + 8 (lanes 4g) of a row tile
__device__ __forceinline__ void put_partd(Sm1& s, float a0, float a1) {
    const int lane = threadIdx.x & 31;
    if ((lane & 3) == 0) {
        s.partd[threadIdx.x >> 5][lane >> 2] = a0;
        s.partd[threadIdx.x >> 5][(lane >> 2) + 8] = a1;
    }
}
__device__ __forceinline__ float sum_partd(const Sm1& s, int i) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kCW; ++w) v += s.partd[w][i];
    return v;
}

// A 16-row fp16 unit (4 steps of 512 bytes) against one group of x held as B
// fragments: partial sums of rows g, g + 8 (lanes 4g, column 0)
__device__ __forceinline__ void f16_unit(const char* unit, const uint32_t (&xb)[4][2], int lane, float& a0,
                                         float& a1) {
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int st = 0; st < 4; ++st) {
        const uint4 a = *reinterpret_cast<const uint4*>(unit + st * kF16Step + 16 * lane);
        const uint32_t A[4] = {a.x, a.y, a.z, a.w};
        mma_16816(c, A, xb[st][0], xb[st][1]);
    }
    a0 += c[0];
    a1 += c[2];
}
// A 16-row int4 unit against one group given as B fragments (b[st] = (b0, b1)),
// with its scales: s 2^24 C + b * (the group's sum); with `lo` the B columns
// carry a hi / lo pair (C = column 0 + column 1 / kLoScale)
__device__ __forceinline__ void q4_unit(const char* unit, const uint32_t (&b)[4][2], float gsum, bool lo, int lane,
                                        float& a0, float& a1) {
    const uint4 wv = *reinterpret_cast<const uint4*>(unit + 16 * lane);
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t A[4];
    q4_masks(wv.x, A);
    mma_16816(c0, A, b[0][0], b[0][1]);
    q4_masks(wv.y, A);
    mma_16816(c1, A, b[1][0], b[1][1]);
    q4_masks(wv.z, A);
    mma_16816(c0, A, b[2][0], b[2][1]);
    q4_masks(wv.w, A);
    mma_16816(c1, A, b[3][0], b[3][1]);
    const float4 sc = scales4(unit + 512 + (lane >> 2) * 8);
    const float r0 = (c0[0] + c1[0]) + (lo ? (c0[1] + c1[1]) * kLoInv : 0.f);
    const float r1 = (c0[2] + c1[2]) + (lo ? (c0[3] + c1[3]) * kLoInv : 0.f);
    a0 += sc.x * kTwo24 * r0 + sc.y * gsum;
    a1 += sc.z * (kTwo24 / 16.f) * r1 + sc.w * gsum;
}

// ---------------------------------------------------------------- producer ----
__device__ __forceinline__ bool own_routed1(int l, int step) {
    return step == 0 || !(sm().ly[l].flags & LF_PREROUTED);
}

__device__ const char* piece_src1(const Prog& p, const Piece1& pc, int l) {
    const Sm1& s = sm();
    const LayerP& Ly = s.ly[l];
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
            __nanosleep(64);   // leave the issue slots of its SM sub-partition to the consumers
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
            const int sidx = s.ly[l].sidx;
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
            for (unsigned it = 0; !vload(&s.route_ready[l]); ++it) {
                if (!keep_waiting(hdr, it, t0)) { ok = 0; break; }
            }
        }
        return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    bool routed_rows = false;   // b1 reads routed experts
    for (int sg = 0; sg < pl.nseg; ++sg) routed_rows |= pl.seg[sg].slot >= 0;
    for (int l = 0; l < p.L; ++l) {
        const bool own = own_routed1(l, step);
        if (own && !issue1(p, hdr, q, L.b0, l, pol, (l << 8) | 0x80)) return;
        // blocks that read routed experts follow the layer's routing
        bool known = !own;
        if (routed_rows && !known) {
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
// ring release up to a block's end: after a consumer barrier that follows the
// last read of every block up to it
struct Mark1 {
    int end, nb;
};
__device__ __forceinline__ Mark1 mark1(const Cons1& c) { return Mark1{c.end, c.nb}; }
__device__ __forceinline__ void give1(const Mark1& m) {
    if (threadIdx.x == 0) {
        Sm1& s = sm();
        *(volatile int*)&s.released = m.end;
        *(volatile int*)&s.released_blocks = m.nb;
    }
}

// A warp's slice of d: groups [gw0, gw0 + ngw), 4 values per lane (lane l: 4l ..
// 4l + 3 of the slice).  x of a slice as B fragments: lanes 0-3 of the warp hold,
// for local group gl and step st, (x[k 2t, 2t+1], x[k 2t+8, 2t+9]) with k =
// 64 gl + 16 st; each lane stores its two fp16 pairs (x01 = values 0, 1, x23 =
// values 2, 3) where they belong, then lanes 0-3 read theirs.
__device__ __forceinline__ void x_frags(uint32_t x01, uint32_t x23, int ngw, uint32_t (&xb)[kMaxGW][4][2]) {
    const int lane = threadIdx.x & 31;
    uint32_t* xw = reinterpret_cast<uint32_t*>(sm().xw[threadIdx.x >> 5]);
    {
        const int k = 4 * lane, gl = k / kGroup, kk = k % kGroup, st = kk / 16, k16 = kk % 16;
        const int wv = k16 >> 3, t = (k16 & 7) >> 1;
        if (gl < kMaxGW) {
            xw[((gl * 4 + t) * 4 + st) * 2 + wv] = x01;
            xw[((gl * 4 + t + 1) * 4 + st) * 2 + wv] = x23;
        }
    }
    __syncwarp();
#pragma unroll
    for (int gl = 0; gl < kMaxGW; ++gl) {
        uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
        if (lane < 4 && gl < ngw) {
            const uint4* src = reinterpret_cast<const uint4*>(xw + (gl * 4 + lane) * 8);
            a = src[0];
            b = src[1];
        }
        xb[gl][0][0] = a.x; xb[gl][0][1] = a.y; xb[gl][1][0] = a.z; xb[gl][1][1] = a.w;
        xb[gl][2][0] = b.x; xb[gl][2][1] = b.y; xb[gl][3][0] = b.z; xb[gl][3][1] = b.w;
    }
    __syncwarp();
}

__device__ void consumer1(const Prog& p, WsHeader* hdr, const Ws1& W, int step, int par, unsigned tag) {
    Sm1& s = sm();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int cta = blockIdx.x, nct = gridDim.x;
    const Plan1& pl = s.plan;
    const Lay1& L = s.lay;
    const int ng = p.d / kGroup, ng0 = ng / 2, ng1 = ng - ng0;
    const bool lora_up = s.S.lora && pl.shr >= 0;   // this CTA's shared rows carry LoRA B terms
    const bool lora_dn = s.S.lora && s.S.shared;
    const int NQ = s.S.NQ;
    // this warp's slice of d
    int gw0, gw1;
    split1(ng, kCW, wid, &gw0, &gw1);
    const int ngw = gw1 - gw0;
    const int e0 = kGroup * gw0 + 4 * lane;           // first of this lane's 4 values
    const bool mine = 4 * lane < kGroup * ngw;        // the lane holds values
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
    const int NA = n_act1(s.S), NG = NA / kGroup, KIg = p.K * p.I / kGroup;
    Cons1 c{{0, 0}, 0, 0, 0};
    // h of this lane's 4 values (fp16 pairs), the RMSNorm gain of the next layer
    uint32_t h01 = 0u, h23 = 0u;
    auto gain = [&](int l) {
        uint2 g = make_uint2(0x3C003C00u, 0x3C003C00u);   // 1.0 in fp16
        if (l < p.L && s.ly[l].gamma && mine) g = __ldg(reinterpret_cast<const uint2*>(s.ly[l].gamma + e0));
        return g;
    };
    if (mine) {
        const uint2 hv = *reinterpret_cast<const uint2*>(p.h_io + e0);
        h01 = hv.x;
        h23 = hv.y;
    }
    uint2 gam = gain(0);
    uint32_t xb[kMaxGW][4][2];
    float xsum[kMaxGW];
    // x of a head layer from its tagged fp16 pairs (the head flush)
    auto load_x = [&](const unsigned long long* xs, unsigned wt) -> bool {
        bool ok = true;
        ulonglong2 w = make_ulonglong2(0ull, 0ull);
        if (mine) {
            w = ld_relaxed_u64x2(xs + e0 / 2);
            ok = settle2(hdr, xs + e0 / 2, wt, w);
        }
        x_frags((uint32_t)w.x, (uint32_t)w.y, ngw, xb);
        return !cbar_or1(!ok);
    };
    // ---- head flush (after the last layer that owns a head).  A CTA adds its
    // finished tasks of a head to the head's count once; the one that completes
    // the count routes.  false: the launch gave up (uniform).
    auto flush = [&]() -> bool {
        const int tph = p.H / kRowTile + p.E / kRowTile, nH = p.H / kRowTile, nE = p.E / kRowTile;
        const int n2 = p.K + (step > 0 ? p.K : 0);
        int xl = -1, ndone = 0;
        for (int t = pl.t0; t < pl.t1; ++t) {
            const int hi = t / tph, j = t % tph, l = s.heads[hi];
            const LayerP& Ly = s.ly[l];
            const int sidx = Ly.sidx;
            if (l != xl) {
                const unsigned long long* xs =
                    reinterpret_cast<const unsigned long long*>(p.ws + W.xs) + (long long)sidx * (p.d / 2);
                if (!load_x(xs, want())) return false;
                xl = l;
            }
            float* lg = reinterpret_cast<float*>(p.ws + W.logh) + ((long long)par * p.Ls + sidx) * p.E;
            stamp1(p, 0xF100 | (t - pl.t0));
            bool ok = take1(p, hdr, c, flush_bytes(s.S, j, 0, n2));
            const char* blkA = ring() + c.off;
            ok = take1(p, hdr, c, flush_bytes(s.S, j, 1, n2)) && ok;
            const char* blkB = ring() + c.off;
            const Mark1 mk = mark1(c);
            stamp1(p, 0xF200 | (t - pl.t0));
            const bool fc1 = j < nH;
            const int row0 = 16 * (fc1 ? j : j - nH);
            float a0 = 0.f, a1 = 0.f;
            if (ok)
                for (int gl = 0; gl < ngw; ++gl) {
                    const int g = gw0 + gl;
                    f16_unit(g < ng0 ? blkA + (long long)g * kF16Unit : blkB + (long long)(g - ng0) * kF16Unit, xb[gl],
                             lane, a0, a1);
                }
            put_partd(s, a0, a1);
            if (cbar_or1(!ok)) return false;
            if (tid < 16) {
                float z = sum_partd(s, tid);
                // one-hot columns of the executed and previous masks [S3.2 "Head"]:
                // the rows of the transposed columns gathered into block B (the
                // concatenated features are never materialised)
                const __half* oh = reinterpret_cast<const __half*>(blkB + (long long)ng1 * kF16Unit +
                                                                   (fc1 ? (long long)nE * kF16Step : 0LL));
                for (int k2 = 0; k2 < n2; ++k2) z += __half2float(oh[k2 * 16 + tid]);
                if (fc1) put_hilo(s.gf, tid, 0.5f * z * (1.f + erff(z * 0.70710678118654752f)));   // erf-GELU
                else red_add_f32(lg + row0 + tid, z);
            }
            if (fc1) {
                // fc2 columns row0 .. row0 + 15 against GELU(z)
                cbar1();
                const uint2 b = lane < 8 ? s.gf[lane] : make_uint2(0u, 0u);
                const char* fc2 = blkB + (long long)ng1 * kF16Unit;
                for (int rt = wid; rt < nE; rt += kCW) {
                    const uint4 a = *reinterpret_cast<const uint4*>(fc2 + (long long)rt * kF16Step + 16 * lane);
                    const uint32_t A[4] = {a.x, a.y, a.z, a.w};
                    float cc[4] = {0.f, 0.f, 0.f, 0.f};
                    mma_16816(cc, A, b.x, b.y);
                    if ((lane & 3) == 0) {
                        red_add_f32(lg + rt * 16 + (lane >> 2), cc[0] + cc[1] * kLoInv);
                        red_add_f32(lg + rt * 16 + (lane >> 2) + 8, cc[2] + cc[3] * kLoInv);
                    }
                }
            }
            if (cbar_or1(vload(&s.abort))) return false;
            give1(mk);
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
    Mark1 pend{0, 0};            // blocks read before the next consumer barrier
    bool broke = true;           // left the layer loop early (set false when it completes)
    for (int l = 0;; ++l) {
        if (l == p.L) {
            broke = false;
            break;
        }
        const LayerP& Ly = s.ly[l];
        const bool own = own_routed1(l, step);
        const int sidx = Ly.sidx;
        stamp1(p, (l << 8) | 0);
        // ---- h = fp16(h + y_prev), x = fp16(RMSNorm(h) gamma) over this warp's slice
        {
            bool ok = true;
            if (l > 0 && mine) {
                const unsigned long long* yp = row(W.y, s.ly[l - 1].sidx, p.d) + e0;
                const unsigned wt = want();
                ulonglong2 a = ld_relaxed_u64x2(yp), b = ld_relaxed_u64x2(yp + 2);
                ok = settle22(hdr, yp, yp + 2, wt, a, b);
                wstamp1(p, l, 0);
                const float2 f01 = unpack2(h01), f23 = unpack2(h23);
                h01 = pack2(f01.x + tval(a.x), f01.y + tval(a.y));
                h23 = pack2(f23.x + tval(b.x), f23.y + tval(b.y));
            }
            if (mine && p.dbg_h && cta == 0 && l > 0)
                *reinterpret_cast<uint2*>(p.dbg_h + (long long)(l - 1) * p.d + e0) = make_uint2(h01, h23);
            const float2 f01 = unpack2(h01), f23 = unpack2(h23);
            float q = mine ? f01.x * f01.x + f01.y * f01.y + f23.x * f23.x + f23.y * f23.y : 0.f;
            q = warp_sum(q);
            if (lane == 0) s.red[wid] = q;
            stamp1(p, (l << 8) | 0x21);
            if (cbar_or1(!ok)) break;
            give1(pend);
            float ss = 0.f;
#pragma unroll
            for (int w = 0; w < kCW; ++w) ss += s.red[w];
            const float rs = rsqrtf(ss / (float)p.d + Ly.eps);
            const float2 g01 = unpack2(gam.x), g23 = unpack2(gam.y);
            const float x0 = __half2float(__float2half_rn(f01.x * rs * g01.x));
            const float x1 = __half2float(__float2half_rn(f01.y * rs * g01.y));
            const float x2 = __half2float(__float2half_rn(f23.x * rs * g23.x));
            const float x3 = __half2float(__float2half_rn(f23.y * rs * g23.y));
            const uint32_t x01 = mine ? pack2(x0, x1) : 0u, x23 = mine ? pack2(x2, x3) : 0u;
            float gs = mine ? x0 + x1 + x2 + x3 : 0.f;
#pragma unroll
            for (int m = 8; m; m >>= 1) gs += __shfl_xor_sync(0xffffffffu, gs, m);
            xsum[0] = __shfl_sync(0xffffffffu, gs, 0);
            xsum[1] = __shfl_sync(0xffffffffu, gs, 16);
            x_frags(x01, x23, ngw, xb);
            if (cta == 0 && (Ly.flags & LF_HEAD) && mine) {
                unsigned long long* xs = reinterpret_cast<unsigned long long*>(p.ws + W.xs) + (long long)sidx * (p.d / 2);
                xs[e0 / 2] = ((unsigned long long)tag << 32) | x01;
                xs[e0 / 2 + 1] = ((unsigned long long)tag << 32) | x23;
            }
        }
        gam = gain(l + 1);
        stamp1(p, (l << 8) | 2);
        // ---- routing of a layer that routes itself
        if (own) {
            unsigned long long* logr = row(W.logr, sidx, p.E);
            bool ok = true;
            if (L.b0.bytes) {
                // this CTA's router row tile, published as tagged logits
                ok = take1(p, hdr, c, L.b0.bytes);
                const char* blk0 = ring() + c.off;
                pend = mark1(c);
                float a0 = 0.f, a1 = 0.f;
                if (ok)
                    for (int gl = 0; gl < ngw; ++gl)
                        f16_unit(blk0 + (long long)(gw0 + gl) * kF16Unit, xb[gl], lane, a0, a1);
                put_partd(s, a0, a1);
                if (cbar_or1(!ok)) break;
                give1(pend);
                if (tid < 16) st_relaxed_u64(logr + 16 * pl.rt + tid, tagged(tag, sum_partd(s, tid)));
            }
            // CTAs whose weights or act depend on the routing route (CTA 0 records it)
            const bool routes = pl.role == R1_EXPERT || pl.dt >= 0 || cta == 0;
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
        // ---- gate/up (LoRA A) partial sums of this warp's slice of d
        if (L.b1.bytes) {
            bool ok = take1(p, hdr, c, L.b1.bytes);
            const char* blk1 = ring() + c.off;
            pend = mark1(c);
            stamp1(p, (l << 8) | 9);
            if (pl.role == R1_LORA) {
                float a0 = 0.f, a1 = 0.f;
                if (ok)
                    for (int gl = 0; gl < ngw; ++gl) {
                        const int g = gw0 + gl;
                        if (g >= pl.la0 && g < pl.la1)
                            f16_unit(blk1 + (long long)(g - pl.la0) * kF16Unit, xb[gl], lane, a0, a1);
                    }
                if ((lane & 3) == 0) {
                    s.partg[wid][lane >> 2] = a0;
                    s.partg[wid][(lane >> 2) + 8] = a1;
                }
            } else {
                // unit (hr j, group g): the first half of d for every hr, then the second
                const char* base[kMaxGW];
                long long jstride[kMaxGW];
#pragma unroll
                for (int gl = 0; gl < kMaxGW; ++gl) {
                    const int g = gw0 + gl;
                    base[gl] = g < ng0 ? blk1 + (long long)g * kQ4Unit
                                       : blk1 + ((long long)pl.n_hr * ng0 + (g - ng0)) * kQ4Unit;
                    jstride[gl] = (long long)(g < ng0 ? ng0 : ng1) * kQ4Unit;
                }
#pragma unroll 2
                for (int j = 0; j < pl.n_hr; ++j) {
                    float a0 = 0.f, a1 = 0.f;
#pragma unroll
                    for (int gl = 0; gl < kMaxGW; ++gl)
                        if (ok && gl < ngw) q4_unit(base[gl] + j * jstride[gl], xb[gl], xsum[gl], false, lane, a0, a1);
                    if ((lane & 3) == 0) {
                        s.partg[wid][j * 16 + (lane >> 2)] = a0;
                        s.partg[wid][j * 16 + (lane >> 2) + 8] = a1;
                    }
                }
            }
            stamp1(p, (l << 8) | 0x27);
            if (cbar_or1(!ok || vload(&s.abort))) break;
            give1(pend);
        }
        stamp1(p, (l << 8) | 5);
        if (pl.role == R1_LORA) {
            if (tid < 16) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < kCW; ++w) v += s.partg[w][tid];
                unsigned long long* lax = row(W.lax, sidx, 2 * kMaxNQ * 16);
                st_relaxed_u64(lax + (cta - (nct - 2 * NQ)) * 16 + tid, tagged(tag, v));
            }
        } else {
            // ---- act of this CTA's rows: the routed rows right away; the shared
            // expert's rows with LoRA once warp 15 has the A_gate x, A_up x sums
            // (a barrier of the act warps and warp 15 only)
            bool ok3 = true;
            const char* blk3 = nullptr;
            if (L.b3.bytes) {
                ok3 = take1(p, hdr, c, L.b3.bytes);
                blk3 = ring() + c.off;
                pend = mark1(c);
            }
            const int nrow = 8 * pl.n_hr, nwa = (nrow + 31) / 32;
            auto act_row = [&](int i, bool shared_rows) {
                int sg = 0;
                while (sg + 1 < pl.nseg && i >= L.seg_base[sg + 1]) ++sg;
                const Seg1& seg = pl.seg[sg];
                if ((seg.slot < 0) != shared_rows) return;
                const int rw = 8 * seg.hr0 + i - L.seg_base[sg];   // expert-local act row
                const int j = i >> 3, r8 = i & 7;
                float gt = 0.f, up = 0.f;
#pragma unroll
                for (int w = 0; w < kCW; ++w) {
                    gt += s.partg[w][j * 16 + r8];
                    up += s.partg[w][j * 16 + 8 + r8];
                }
                float wt = 1.f;
                if (seg.slot >= 0) {
                    wt = s.w[l][seg.slot];
                } else if (lora_up) {
                    // unmerged LoRA on the shared gate and up [S3.3]: + (alpha / r) B (A x)
                    const int r = p.r, lr = i - L.seg_base[sg];
                    const __half* bg = reinterpret_cast<const __half*>(blk3) + (long long)lr * r;
                    const __half* bu = reinterpret_cast<const __half*>(blk3 + L.bu) + (long long)lr * r;
                    float dg = 0.f, du = 0.f;
                    for (int q = 0; q < r; ++q) {
                        dg += __half2float(bg[q]) * s.lax[q];
                        du += __half2float(bu[q]) * s.lax[16 + q];
                    }
                    gt += Ly.lora_scale * dg;
                    up += Ly.lora_scale * du;
                }
                const long long gi = (seg.slot >= 0 ? (long long)seg.slot * p.I : (long long)p.K * p.I) + rw;
                st_relaxed_u64(row(W.act, sidx, NA) + gi, tagged(tag, silu_f(gt) * up * wt));
            };
            if (tid < nrow && ok3) act_row(tid, false);
            if (lora_up) {
                if (wid == kCW - 1) {
                    // A_gate x (lanes 0-15), A_up x (16-31): the LoRA CTAs' partial sums
                    bool okl = true;
                    const unsigned long long* lax = row(W.lax, sidx, 2 * kMaxNQ * 16);
                    const unsigned wt = want();
                    const int m = lane >> 4, r = lane & 15;
                    // the NQ partial sums, re-polled together while any is pending
                    unsigned long long pw[kMaxNQ];
                    unsigned pend_q = 0;
#pragma unroll
                    for (int qq = 0; qq < kMaxNQ; ++qq) {
                        pw[qq] = qq < NQ ? ld_relaxed_u64(lax + (m * NQ + qq) * 16 + r) : 0ull;
                        if (qq < NQ && !tok(pw[qq], wt)) pend_q |= 1u << qq;
                    }
                    if (pend_q) {
                        const unsigned long long t0 = now1();
                        for (unsigned it = 0; pend_q; ++it) {
                            if (!keep_waiting(hdr, it, t0)) {
                                okl = false;
                                break;
                            }
#pragma unroll
                            for (int qq = 0; qq < kMaxNQ; ++qq)
                                if ((pend_q >> qq) & 1u) pw[qq] = ld_relaxed_u64(lax + (m * NQ + qq) * 16 + r);
#pragma unroll
                            for (int qq = 0; qq < kMaxNQ; ++qq)
                                if (((pend_q >> qq) & 1u) && tok(pw[qq], wt)) pend_q &= ~(1u << qq);
                        }
                    }
                    float v = 0.f;
#pragma unroll
                    for (int qq = 0; qq < kMaxNQ; ++qq)
                        if (qq < NQ) v += tval(pw[qq]);
                    s.lax[lane] = okl ? v : 0.f;
                }
                if (wid < nwa || wid == kCW - 1) named_bar_sync(2, 32 * (nwa + 1));
            }
            if (tid < nrow && ok3) act_row(tid, true);
        }
        stamp1(p, (l << 8) | 7);
        // ---- down: this CTA's output row tile; warp w takes act groups w, w + 16, ...
        if (pl.dt >= 0) {
            bool ok = take1(p, hdr, c, L.b2.bytes);
            const char* blk2 = ring() + c.off;
            pend = mark1(c);
            stamp1(p, (l << 8) | 10);
            const unsigned long long* act = row(W.act, sidx, NA);
            const unsigned wt = want();
            // this lane's pair of every act group of the warp: all loads go out
            // first; a group is taken as soon as it is complete (groups of the
            // shared expert, which come last, wait for the LoRA terms), and the
            // groups still pending are re-polled together
            ulonglong2 wd[kMaxUW];
            unsigned pend_u = 0;
#pragma unroll
            for (int i = 0; i < kMaxUW; ++i) {
                const int u = wid + kCW * i;
                wd[i] = make_ulonglong2(0ull, 0ull);
                if (u < NG) {
                    wd[i] = ld_relaxed_u64x2(act + (long long)u * kGroup + 2 * lane);
                    if (!(tok(wd[i].x, wt) && tok(wd[i].y, wt))) pend_u |= 1u << i;
                }
            }
            wstamp1(p, l, 1);
            float a0 = 0.f, a1 = 0.f;
            const int t = lane & 3;
#pragma unroll 1
            for (int i = 0; i < kMaxUW; ++i) {
                const int u = wid + kCW * i;
                if (u < NG) {
                    if (ok && ((pend_u >> i) & 1u)) {
                        const unsigned long long t0 = now1();
                        for (unsigned it = 0; (pend_u >> i) & 1u; ++it) {
                            if (!keep_waiting(hdr, it, t0)) {
                                ok = false;
                                break;
                            }
#pragma unroll
                            for (int q = 0; q < kMaxUW; ++q)
                                if ((pend_u >> q) & 1u)
                                    wd[q] = ld_relaxed_u64x2(act + (long long)(wid + kCW * q) * kGroup + 2 * lane);
#pragma unroll
                            for (int q = 0; q < kMaxUW; ++q)
                                if (((pend_u >> q) & 1u) && tok(wd[q].x, wt) && tok(wd[q].y, wt)) pend_u &= ~(1u << q);
                        }
                    }
                    const float v0 = tval(wd[i].x), v1 = tval(wd[i].y);
                    uint32_t hi, lo;
                    hilo2(v0, v1, hi, lo);
                    const float gsum = warp_sum(v0 + v1);
                    // B fragments of the act group: lane t < 4 the hi parts, lane
                    // 4 + t the lo parts of act k 2t, 2t+1 | 2t+8, 2t+9 of each step;
                    // this lane's pair is act k = 2 lane, 2 lane + 1
                    uint32_t* aw = reinterpret_cast<uint32_t*>(s.aw[wid]);
                    {
                        const int st = lane >> 3, pt = lane & 3, wv = (lane >> 2) & 1;
                        aw[(st * 8 + pt) * 2 + wv] = hi;
                        aw[(st * 8 + 4 + pt) * 2 + wv] = lo;
                    }
                    __syncwarp();
                    uint32_t b[4][2];
#pragma unroll
                    for (int st = 0; st < 4; ++st) {
                        const uint2 v = lane < 8 ? s.aw[wid][st * 8 + lane] : make_uint2(0u, 0u);
                        b[st][0] = v.x;
                        b[st][1] = v.y;
                    }
                    __syncwarp();
                    q4_unit(blk2 + (long long)u * kQ4Unit, b, gsum, true, lane, a0, a1);
                    if (lora_dn && u >= KIg) {
                        // (alpha / r) B_down[tile] (A_down[:, group] act_shared[group]):
                        // B_down is linear, so the groups' products sum to B_down v
                        const int wi = u - KIg, r = p.r, g8 = lane >> 2;
                        float cc[4] = {0.f, 0.f, 0.f, 0.f};
                        const char* unit = blk2 + L.ad + (long long)wi * kF16Unit;
#pragma unroll
                        for (int st = 0; st < 4; ++st) {
                            const uint4 a = *reinterpret_cast<const uint4*>(unit + st * kF16Step + 16 * lane);
                            const uint32_t A[4] = {a.x, a.y, a.z, a.w};
                            mma_16816(cc, A, b[st][0], b[st][1]);
                        }
                        // v[g8], v[g8 + 8] sit in lanes 4 g8; as the B operand (k =
                        // the rank index) lane t < 4 takes the hi, lane 4 + t the lo
                        // parts of v[2t], v[2t+1] | v[2t+8], v[2t+9]
                        const float vr = cc[0] + cc[1] * kLoInv, vr8 = cc[2] + cc[3] * kLoInv;
                        const float v0s = __shfl_sync(0xffffffffu, vr, 8 * t);
                        const float v1s = __shfl_sync(0xffffffffu, vr, 8 * t + 4);
                        const float v8s = __shfl_sync(0xffffffffu, vr8, 8 * t);
                        const float v9s = __shfl_sync(0xffffffffu, vr8, 8 * t + 4);
                        uint32_t h0, l0, h1, l1;
                        hilo2(v0s, v1s, h0, l0);
                        hilo2(v8s, v9s, h1, l1);
                        const uint32_t bb0 = lane < 4 ? h0 : (lane < 8 ? l0 : 0u);
                        const uint32_t bb1 = lane < 4 ? h1 : (lane < 8 ? l1 : 0u);
                        // A: the tile's B_down rows g8 and g8 + 8, k = the rank index (zero past r)
                        const __half* bd = reinterpret_cast<const __half*>(blk2 + L.bd);
                        const __half zero = __float2half_rn(0.f);
                        auto at = [&](int rw, int kk) { return kk < r ? bd[rw * r + kk] : zero; };
                        __half2 q0 = __halves2half2(at(g8, 2 * t), at(g8, 2 * t + 1));
                        __half2 q1 = __halves2half2(at(g8 + 8, 2 * t), at(g8 + 8, 2 * t + 1));
                        __half2 q2 = __halves2half2(at(g8, 2 * t + 8), at(g8, 2 * t + 9));
                        __half2 q3 = __halves2half2(at(g8 + 8, 2 * t + 8), at(g8 + 8, 2 * t + 9));
                        const uint32_t A[4] = {*reinterpret_cast<uint32_t*>(&q0), *reinterpret_cast<uint32_t*>(&q1),
                                               *reinterpret_cast<uint32_t*>(&q2), *reinterpret_cast<uint32_t*>(&q3)};
                        float e[4] = {0.f, 0.f, 0.f, 0.f};
                        mma_16816(e, A, bb0, bb1);
                        a0 += Ly.lora_scale * (e[0] + e[1] * kLoInv);
                        a1 += Ly.lora_scale * (e[2] + e[3] * kLoInv);
                    }
                }
            }
            put_partd(s, a0, a1);
            wstamp1(p, l, 2);
            stamp1(p, (l << 8) | 0x25);
            if (cbar_or1(!ok || vload(&s.abort))) break;
            give1(pend);
            if (tid < 16) st_relaxed_u64(row(W.y, sidx, p.d) + 16 * pl.dt + tid, tagged(tag, sum_partd(s, tid)));
        }
        stamp1(p, (l << 8) | 8);
        if (l == s.flush_after) {
            if (!flush()) break;
            pend = mark1(c);
        }
    }
    if (broke) {
        if (tid == 0) *(volatile int*)&s.abort = 1;
        return;
    }
    stamp1(p, 0xFF00);
    // ---- the last layer's output into h_io, a slice per CTA (every CTA read
    // h_io at layer 0 before it published anything the last y depends on)
    const unsigned long long* ylast = row(W.y, s.ly[p.L - 1].sidx, p.d);
    const unsigned wt = want();
    const int a = p.d * cta / nct, b = p.d * (cta + 1) / nct;
    bool ok = true;
    if (mine && e0 + 4 > a && e0 < b) {
        const float2 f01 = unpack2(h01), f23 = unpack2(h23);
        const float hv[4] = {f01.x, f01.y, f23.x, f23.y};
        ulonglong2 ya = ld_relaxed_u64x2(ylast + e0), yb = ld_relaxed_u64x2(ylast + e0 + 2);
        ok = settle22(hdr, ylast + e0, ylast + e0 + 2, wt, ya, yb);
        const float yv[4] = {tval(ya.x), tval(ya.y), tval(yb.x), tval(yb.y)};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int e = e0 + k;
            if (e < a || e >= b) continue;
            const __half h = __float2half_rn(hv[k] + yv[k]);
            p.h_io[e] = h;
            if (p.dbg_h) p.dbg_h[(long long)(p.L - 1) * p.d + e] = h;
        }
    }
    if (cbar_or1(!ok)) return;
    if (cta == 0 && tid == 0) {
        if (p.step < 0) hdr->step = step + 1;
        hdr->serial = tag;   // the next launch tags with serial + 1
    }
}

// ------------------------------------------------------------------ kernel ----
__global__ void __launch_bounds__(kT1, 1) decode1_kernel(const __grid_constant__ Prog p) {
    Sm1& s = sm();
    const int tid = threadIdx.x;
    long long c_entry;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(c_entry));
    const unsigned long long g_entry = now1();
    WsHeader* hdr = reinterpret_cast<WsHeader*>(p.ws);
    if ((int)gridDim.x != p.grid1[0]) {
        if (tid == 0) {
            atomicCAS(&hdr->error, 0, EDGE0_EUNSUPPORTED);
            atomicExch(&hdr->abort, 1);
        }
        return;
    }
    // header words this launch reads (all loads in flight before the first use)
    const unsigned long long hdr_wait = ld_relaxed_u64(&hdr->wait_ns);
    const int hdr_trace = ld_volatile_s32(&hdr->trace), hdr_step = ld_volatile_s32(&hdr->step);
    const int hdr_serial = ld_volatile_s32(reinterpret_cast<const int*>(&hdr->serial));
    {
        // the layer descriptors from their device copy (a read of the kernel
        // parameter block at a different address per lane is serialised)
        static_assert(sizeof(LayerP) % 8 == 0, "layer descriptors copy as 8-byte words");
        const unsigned long long* src = reinterpret_cast<const unsigned long long*>(p.ly1);
        unsigned long long* dst = reinterpret_cast<unsigned long long*>(s.ly);
        const int n = p.L * (int)(sizeof(LayerP) / 8);
        for (int i = tid; i < n; i += kT1) dst[i] = __ldg(src + i);
    }
    __syncthreads();
    const unsigned long long g_ly = now1();
    const int shared = (s.ly[0].flags & LF_SHARED) != 0;
    const Ws1 W = ws1(p.Ls, p.d, p.E, p.K, p.K * p.I + (shared ? p.Is : 0));
    __shared__ int s_step;
    __shared__ unsigned s_tag;
    if (tid == 0) {
        s.abort = 0;
        s.topk = 0;
        s.issued = 0;
        s.released_blocks = 0;
        s.released = 0;
        s.wait_ns = hdr_wait ? hdr_wait : kDefaultWaitNs;
        s.trace = blockIdx.x < kTraceCtas ? hdr_trace : 0;
        s.tslot = 0;
        s.ptslot = 3072;
        for (int i = 0; i < kBlocks; ++i) mbar_init(&s.full[i], 1);
        fence_mbar_init();
        s_step = p.step >= 0 ? p.step : hdr_step;
        s_tag = ((unsigned)hdr_serial % kTagMask) + 1u;
        // the plan of this CTA and the layout of its blocks
        Shape1 S;
        S.d = p.d; S.I = p.I; S.Is = p.Is; S.E = p.E; S.K = p.K; S.H = p.H; S.r = p.r;
        S.shared = shared;
        S.lora = (s.ly[0].flags & LF_LORA) != 0;
        S.nct = gridDim.x;
        S.NQ = S.lora ? p.grid1[1] : 0;
        S.n_heads = p.n_heads1;
        s.flush_after = p.n_heads1 > 0 ? p.heads1[p.n_heads1 - 1] : -1;
        s.S = S;
    }
    for (int i = tid; i < p.n_heads1; i += kT1) s.heads[i] = p.heads1[i];
    const unsigned long long g_t0 = now1();
    {
        // this CTA's plan and block layout, built on the host
        static_assert(sizeof(Plan1) % 8 == 0 && sizeof(Lay1) % 8 == 0, "plans copy as 8-byte words");
        const unsigned long long* src =
            reinterpret_cast<const unsigned long long*>(p.tab1 + (long long)blockIdx.x * kTab1Stride);
        unsigned long long* dp = reinterpret_cast<unsigned long long*>(&s.plan);
        unsigned long long* dl = reinterpret_cast<unsigned long long*>(&s.lay);
        constexpr int np = (int)(sizeof(Plan1) / 8), nl = (int)(sizeof(Lay1) / 8);
        for (int i = tid; i < np + nl; i += kT1) {
            if (i < np) dp[i] = src[i];
            else dl[i - np] = src[i];
        }
    }
    __syncthreads();
    if (s.trace && tid == 0) {   // the kernel's entry, and the CTA's plan built
        unsigned long long* tr = reinterpret_cast<unsigned long long*>(p.ws + p.ws_bytes - kTraceBytes) +
                                 (long long)blockIdx.x * kTraceSlots;
        tr[0] = 0xFFF0u;
        tr[1] = g_entry;
        tr[2] = (unsigned long long)c_entry;
        tr[3] = 0xFFF2u;
        tr[4] = g_ly;
        tr[5] = 0;
        tr[6] = 0xFFF3u;
        tr[7] = g_t0;
        tr[8] = 0;
        s.tslot = 9;
        stamp_slow1(p, 0xFFF1, false);
    }
    const int step = s_step, par = step & 1;
    // clear the other step parity's head logits and task counts for the next step
    {
        const int op = par ^ 1;
        const long long tot = (long long)p.L * p.E;
        const long long a = tot * blockIdx.x / gridDim.x, b = tot * (blockIdx.x + 1) / gridDim.x;
        for (long long i = a + tid; i < b; i += kT1) {
            const long long l = i / p.E, o = i % p.E;
            reinterpret_cast<float*>(p.ws + W.logh)[((long long)op * p.Ls + s.ly[l].sidx) * p.E + o] = 0.f;
        }
        if (blockIdx.x == 0)
            for (int l = tid; l < p.L; l += kT1)
                reinterpret_cast<unsigned*>(p.ws + W.cnt)[(long long)op * p.Ls + s.ly[l].sidx] = 0u;
    }
    // routing known at launch: the predictions of prerouted layers (step > 0)
    for (int l = tid; l < p.L; l += kT1) s.route_ready[l] = 0;
    for (int i = tid; i < p.L * p.K; i += kT1) {
        const int l = i / p.K, k = i % p.K;
        if (step > 0 && (s.ly[l].flags & LF_PREROUTED)) {
            const long long o = ((long long)((step - 1) & 1) * p.Ls + s.ly[l].sidx) * p.K + k;
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
    }
    __syncthreads();
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
    int d, I, Is, E, K, H, r, shared, lora, n_heads, nct, smem, dev;
    int rc, grid, NQ, ring;
    char* tab;                // device table: every CTA's Plan1 + Lay1 (kTab1Stride bytes each)
};
constexpr int kKeys = 16;
Key1 g_keys[kKeys];
int g_nkeys = 0, g_next_key = 0;

int grid1(int* nct, int* smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return EDGE0_ECUDA;
    if (!g_d1_grid[dev]) {
        int maxsm = 0, nsm = 0;
        if (cudaDeviceGetAttribute(&maxsm, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return EDGE0_ECUDA;
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, decode1_kernel) != cudaSuccess) return EDGE0_ECUDA;
        const int dyn = maxsm - (int)fa.sharedSizeBytes;
        if (cudaFuncSetAttribute(decode1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn) != cudaSuccess)
            return EDGE0_ECUDA;
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode1_kernel, kT1, dyn) != cudaSuccess ||
            per_sm < 1)
            return EDGE0_ECUDA;
        g_d1_grid[dev] = nsm;   // one CTA per SM, all resident at once (cooperative launch)
        g_d1_smem[dev] = dyn;
    }
    *nct = g_d1_grid[dev];
    *smem = g_d1_smem[dev];
    return EDGE0_OK;
}

// the grid, every CTA's plan and blocks for the shapes on at most k.nct CTAs:
// every expert CTA owns hr (so every CTA publishes something that each layer's
// y depends on), every output and router row tile has its CTA, the ring holds
// the largest block
int derive1(Key1& k, std::vector<char>* table = nullptr) {
    Shape1 S;
    S.d = k.d; S.I = k.I; S.Is = k.Is; S.E = k.E; S.K = k.K; S.H = k.H; S.r = k.r;
    S.shared = k.shared; S.lora = k.lora; S.n_heads = k.n_heads;
    const int ng = S.d / kGroup;
    if (ng < 2 || ng > kCW * kMaxGW) return EDGE0_EUNSUPPORTED;
    if (n_act1(S) > kMaxNA || n_act1(S) % kGroup) return EDGE0_EUNSUPPORTED;
    if (S.lora && (!S.shared || S.Is / kGroup > kCW || S.r > 16)) return EDGE0_EUNSUPPORTED;
    S.NQ = S.lora ? (ng < kMaxNQ ? ng : kMaxNQ) : 0;
    const int nla = n_lora_ctas(S);
    int nct = k.nct;
    if (nct - nla > n_hr_all(S)) nct = n_hr_all(S) + nla;
    S.nct = nct;
    if (nct - nla < 1 || S.d / kRowTile > nct || S.E / kRowTile > nct) return EDGE0_EUNSUPPORTED;
    if (ceil_div(n_hr_all(S), nct - nla) > kMaxHr1) return EDGE0_EUNSUPPORTED;
    const int ring = ((k.smem - kSm1Bytes) / 128) * 128;
    if (ring < 2 * kPieceMax) return EDGE0_EUNSUPPORTED;
    int biggest = 0;
    std::vector<char> local;
    std::vector<char>& tab = table ? *table : local;
    tab.assign((size_t)nct * kTab1Stride, 0);
    for (int c = 0; c < nct; ++c) {
        Plan1 pl;
        Lay1 L;
        memset(&pl, 0, sizeof(pl));
        memset(&L, 0, sizeof(L));
        if (!plan1(S, c, pl) || !layout1(S, pl, L)) return EDGE0_EUNSUPPORTED;
        if (pl.role == R1_EXPERT && pl.n_hr < 1) return EDGE0_EUNSUPPORTED;
        const Block1* bl[4] = {&L.b0, &L.b1, &L.b3, &L.b2};
        for (const Block1* b : bl) biggest = b->bytes > biggest ? b->bytes : biggest;
        memcpy(tab.data() + (size_t)c * kTab1Stride, &pl, sizeof(pl));
        memcpy(tab.data() + (size_t)c * kTab1Stride + sizeof(pl), &L, sizeof(L));
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
    k.grid = nct;
    k.NQ = S.NQ;
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
        if (Ly.flags & LF_HEAD) p.heads1[n_heads] = l;
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
    if (cudaGetDevice(&k.dev) != cudaSuccess) return EDGE0_ECUDA;
    k.d = p.d; k.I = p.I; k.Is = p.Is; k.E = p.E; k.K = p.K; k.H = p.H; k.r = p.r;
    k.shared = (f0 & LF_SHARED) != 0;
    k.lora = (f0 & LF_LORA) != 0;
    k.n_heads = n_heads;
    p.n_heads1 = n_heads;
    std::lock_guard<std::mutex> lock(g_d1_mutex);
    int hit = -1;
    for (int i = 0; i < g_nkeys; ++i) {
        const Key1& q = g_keys[i];
        if (q.d == k.d && q.I == k.I && q.Is == k.Is && q.E == k.E && q.K == k.K && q.H == k.H && q.r == k.r &&
            q.shared == k.shared && q.lora == k.lora && q.n_heads == k.n_heads && q.nct == k.nct && q.smem == k.smem &&
            q.dev == k.dev) {
            hit = i;
            break;
        }
    }
    if (hit < 0) {
        std::vector<char> tab;
        k.rc = derive1(k, &tab);
        if (k.rc == EDGE0_OK) {
            // the plan table on the device, once per shape and device (kept while
            // the key stays cached)
            if (cudaMalloc(&k.tab, tab.size()) != cudaSuccess) {
                k.tab = nullptr;
                k.rc = EDGE0_ECUDA;
            } else if (cudaMemcpy(k.tab, tab.data(), tab.size(), cudaMemcpyHostToDevice) != cudaSuccess) {
                cudaFree(k.tab);
                k.tab = nullptr;
                k.rc = EDGE0_ECUDA;
            }
        }
        hit = g_next_key;
        if (g_keys[hit].tab) {
            // a launch may still read the table of the key it replaces: cudaFree
            // waits for the device to finish its work first
            int cur = 0;
            cudaGetDevice(&cur);
            cudaSetDevice(g_keys[hit].dev);
            cudaFree(g_keys[hit].tab);
            cudaSetDevice(cur);
        }
        g_keys[hit] = k;
        g_next_key = (g_next_key + 1) % kKeys;
        if (g_nkeys < kKeys) ++g_nkeys;
    }
    const Key1& q = g_keys[hit];
    if (q.rc) return q.rc;
    p.grid1[0] = q.grid;
    p.grid1[1] = q.NQ;
    p.ring1 = q.ring;
    p.tab1 = q.tab;
    return EDGE0_OK;
}

namespace {
// device copies of the layer descriptor arrays of recent launches: a model's
// decode steps pass the same descriptors every step, so after the first step
// the launch finds its copy here (a copy is freed only when evicted; cudaFree
// waits for the device's work first)
struct DescCopy {
    int dev = -1;
    std::vector<char> host;
    LayerP* dptr = nullptr;
};
constexpr int kDescCopies = 8;
DescCopy g_desc[kDescCopies];
int g_desc_next = 0;

int layer_copy(Prog& p) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EDGE0_ECUDA;
    const size_t n = sizeof(LayerP) * (size_t)p.L;
    const char* src = reinterpret_cast<const char*>(p.layers);
    std::lock_guard<std::mutex> lock(g_d1_mutex);
    for (DescCopy& e : g_desc)
        if (e.dptr && e.dev == dev && e.host.size() == n && memcmp(e.host.data(), src, n) == 0) {
            p.ly1 = e.dptr;
            return EDGE0_OK;
        }
    DescCopy& e = g_desc[g_desc_next];
    g_desc_next = (g_desc_next + 1) % kDescCopies;
    if (e.dptr) {
        int cur = 0;
        cudaGetDevice(&cur);
        cudaSetDevice(e.dev);
        cudaFree(e.dptr);
        cudaSetDevice(cur);
        e.dptr = nullptr;
    }
    void* d = nullptr;
    if (cudaMalloc(&d, n) != cudaSuccess) return EDGE0_ECUDA;
    if (cudaMemcpy(d, src, n, cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaFree(d);
        return EDGE0_ECUDA;
    }
    e.dev = dev;
    e.host.assign(src, src + n);
    e.dptr = reinterpret_cast<LayerP*>(d);
    p.ly1 = e.dptr;
    return EDGE0_OK;
}
}  // namespace

int decode1_launch(Prog& p, cudaStream_t stream) {
    int rc = decode1_check(p);
    if (rc) return rc;
    rc = layer_copy(p);
    if (rc) return rc;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(p.grid1[0]);
    cfg.blockDim = dim3(kT1);
    cfg.dynamicSmemBytes = kSm1Bytes + p.ring1;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];   // every CTA resident at once: the CTAs wait on one another
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode1_kernel, p) != cudaSuccess) return EDGE0_ECUDA;
    return EDGE0_OK;
}

}  // namespace edge0
