// Batch-1 decode kernel: one persistent launch runs every layer of a decode
// step for one sequence, then every prerouter head of the step.
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
// Work split.  The grid is one CTA per SM in clusters of two ("pairs"); every
// expert is cut into half-row tiles ("hr": 8 act rows, whose packed gate/up tile
// interleaves its 8 gate and 8 up rows).  Pairs take one of three roles, fixed
// for the launch:
//   routed pairs  a contiguous run of the K routed slots' hr;
//   shared pairs  a contiguous run of the shared expert's hr, with its LoRA B
//                 terms: B_gate/B_up on their act rows, and B_down applied to
//                 the partial v = A_down act of their own rows (B_down is
//                 linear, so the partial products sum to B_down v);
//   a LoRA pair   A_gate x and A_up x, published as (value, tag) words that the
//                 shared pairs poll.
// The two CTAs of a pair split d in halves for gate/up, swap their partial
// sums through distributed shared memory, form act for all of the pair's rows
// and apply the matching columns of down to their half of the output rows.
// Layer outputs are summed into global memory with vector reductions; one grid
// barrier per layer (two on a layer that routes itself) publishes them.
//
// Weights move by a producer warp: cp.async.bulk copies into a byte ring of
// shared memory, one block per (layer, phase) with its own mbarrier.  The
// blocks of prerouted layers depend only on predictions known at launch, so
// the stream runs ahead of the compute by as many layers as the ring holds.
// int4 nibbles enter m16n8k16 tensor-core steps as fp16 subnormals (q 2^-24)
// through single masks; fp32 activations travel as hi + lo fp16 columns.
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
constexpr int kMaxSig = 9;               // 16-row act steps of one pair (+ the last slot: LoRA v)
constexpr int kMaxPc = 24;               // copies of one block
constexpr int kMaxParts = 8;             // (expert run, group) parts of a pair's down block
constexpr int kBlocks = 16;              // block barriers
constexpr int kPieceMax = 32768;         // bytes of one bulk copy
constexpr int kMaxD1 = 2048;
constexpr int kMaxG1 = kMaxD1 / kGroup;  // groups of d
constexpr int kMaxTw = kMaxD1 / 2 / kRowTile / kCW;   // down row tiles of one warp
constexpr int kMsg = kMaxHr1 * 16;       // partial sums a pair exchanges
constexpr int kMaxK1 = EDGE0_MAX_K;
constexpr int kNY = 1;                   // copies of each layer's y: pair p adds into copy p % kNY

__host__ __device__ inline void split1(int n, int parts, int i, int* a, int* b) {
    *a = (int)((long long)n * i / parts);
    *b = (int)((long long)n * (i + 1) / parts);
}
__host__ __device__ inline int ngh1(int d, int rank) {
    const int ng = d / kGroup;
    return rank ? ng - ng / 2 : ng / 2;
}
__host__ __device__ inline int nrth1(int d, int rank) {
    const int n = d / kRowTile;
    return rank ? n - n / 2 : n / 2;
}

// ------------------------------------------------------------------ plan ----
struct Shape1 {
    int d, I, Is, E, K, H, r;
    int shared, lora;          // every layer of the launch has a shared expert / LoRA
    int P, Pr, Ps, Pl;         // pairs: all, routed, shared, LoRA
    int n_heads;
};
enum Role1 : int { R1_ROUTED = 0, R1_SHARED = 1, R1_LORA = 2 };
struct Seg1 {
    int slot;                  // routed slot (index into the layer's K ids) or -1: shared
    int hr0, hr1;              // hr [hr0, hr1) of the expert
};
struct Plan1 {
    int role, nseg, n_hr;
    Seg1 seg[kMaxSeg1];
    int ru0, ru1;              // router units (row tile x group of this CTA's half)
    int t0, t1;                // head-flush tasks
};

__host__ __device__ inline bool plan1(const Shape1& S, int pair, int rank, Plan1& p) {
    p.role = R1_ROUTED;
    p.nseg = p.n_hr = 0;
    p.ru0 = p.ru1 = p.t0 = p.t1 = 0;
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
    split1((S.E / kRowTile) * ngh1(S.d, rank), S.P, pair, &p.ru0, &p.ru1);
    split1(S.n_heads * (S.H / kRowTile + S.E / kRowTile), 2 * S.P, 2 * pair + rank, &p.t0, &p.t1);
    return true;
}

// Pairs per role: the LoRA pair (with LoRA), then the split of the rest that
// minimises the largest per-pair load in hr (a shared pair's LoRA B terms count
// as one more hr).  0 if no split fits the kernel's limits.
__host__ inline int choose_pairs(Shape1& S) {
    const int hpe = S.I / kHalfRow, n_rt = S.K * hpe, n_sh = S.shared ? S.Is / kHalfRow : 0;
    S.Pl = S.lora ? 1 : 0;
    const int avail = S.P - S.Pl;
    if (!S.shared) {
        S.Ps = 0;
        S.Pr = avail;
        return ceil_div(n_rt, S.Pr) <= kMaxHr1;
    }
    int best = 1 << 30, pick = -1;
    for (int ps = 1; ps < avail; ++ps) {
        const int cr = ceil_div(n_rt, avail - ps), cs = ceil_div(n_sh, ps);
        if (cr > kMaxHr1 || cs > kMaxHr1) continue;
        const int cost = cr > cs + S.lora ? cr : cs + S.lora;
        if (cost <= best) { best = cost; pick = ps; }   // ties: more shared pairs
    }
    if (pick < 0) return 0;
    S.Ps = pick;
    S.Pr = avail - pick;
    return 1;
}

// ---------------------------------------------------------------- blocks ----
// A block is one (layer, phase) share of a CTA's weights, copied contiguously
// into the ring: P0 router units (layers that route themselves), P1 gate/up
// (LoRA A_gate / A_up on the LoRA pair), P2 down (+ on shared pairs the LoRA
// rows B_gate, B_up, A_down^T of the pair's act rows and B_down of this CTA's
// output half); one block per head-flush task.
enum PieceKind1 : int {
    K1_ROUTER = 0, K1_GU, K1_DOWN, K1_LA, K1_LU, K1_BG, K1_BU, K1_ADT, K1_BD, K1_FC1, K1_FC2, K1_LINIT,
    K1_OHF, K1_OHL
};
struct Piece1 {
    int kind, seg;
    long long src;             // byte offset in the source matrix (of the expert, for K1_GU/K1_DOWN)
    int bytes, dst;            // size and offset in the block
};
struct Block1 {
    int n, bytes;
    Piece1 pc[kMaxPc];
};
struct Part1 {                 // one (expert run, group of I) of the down block
    int seg, sa, sb;           // expert-local 16-row steps [sa, sb]
    int sig0;                  // act step index of sa
    int words, scales;         // block offsets: step sa's words, the group's scales
};
struct Lay1 {
    Block1 b0, b1, b2;
    int la, lu, bg, bu, adt, bd;        // block offsets of the LoRA parts
    int nparts;
    Part1 part[kMaxParts];
    int nsig;
    int sig_seg[kMaxSig], sig_step[kMaxSig];
    int seg_base[kMaxSeg1];             // pair-local act row of each run's first row
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
    L.b0.n = L.b0.bytes = L.b1.n = L.b1.bytes = L.b2.n = L.b2.bytes = 0;
    L.la = L.lu = L.bg = L.bu = L.adt = L.bd = 0;
    L.nparts = L.nsig = 0;
    const int ng = S.d / kGroup, ng0 = ng / 2, ngh = ngh1(S.d, rank);
    bool ok = true;
    // P0: router units of this CTA's half of d (packed fp16 [E x d], by halves)
    if (p.ru1 > p.ru0)
        ok &= add_piece(L.b0, K1_ROUTER, 0,
                        (long long)rank * (S.E / kRowTile) * ng0 * kF16Unit + (long long)p.ru0 * kF16Unit,
                        (long long)(p.ru1 - p.ru0) * kF16Unit);
    if (p.role == R1_LORA) {
        // LoRA A (packed fp16 [r x d], one row tile: its two halves back to back
        // are the row tile's groups in order): rank 0 A_gate, rank 1 A_up, all of d
        L.la = 0;
        ok &= add_piece(L.b1, rank ? K1_LU : K1_LA, 0, 0, (long long)ng * kF16Unit);
        return ok;
    }
    // P1: gate/up units [hr][group of the half] of each run, back to back
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
    const bool lora_rows = p.role == R1_SHARED && S.lora && p.nseg > 0;
    // P2: per run and group of I, the 16-row steps the run touches over this
    // CTA's half of the output row tiles, then the group's scales (down packed
    // K-major: per group [half 0 words, half 0 scales, half 1 words, half 1 scales])
    const int nrt = S.d / kRowTile, nh = nrth1(S.d, rank), nh0 = nrt / 2;
    const long long gstride = (long long)kQ4Unit * nrt;
    const long long hoff = rank ? (long long)kQ4Unit * nh0 : 0;
    for (int s = 0; s < p.nseg; ++s) {
        const Seg1& sg = p.seg[s];
        const int sa = sg.hr0 / 2, sb = (sg.hr1 - 1) / 2;
        const int sig0 = L.nsig;
        for (int st = sa; st <= sb; ++st) {
            if (L.nsig >= kMaxSig - 1) return false;
            L.sig_seg[L.nsig] = s;
            L.sig_step[L.nsig] = st;
            ++L.nsig;
        }
        for (int gi = sa / 4; gi <= sb / 4; ++gi) {
            if (L.nparts >= kMaxParts) return false;
            const int a = (sa > 4 * gi ? sa : 4 * gi) - 4 * gi;
            const int b = (sb < 4 * gi + 3 ? sb : 4 * gi + 3) - 4 * gi;
            const long long gb = gi * gstride + hoff;
            Part1& P = L.part[L.nparts++];
            P.seg = s;
            P.sa = 4 * gi + a;
            P.sb = 4 * gi + b;
            P.sig0 = sig0 + (P.sa - sa);
            P.words = L.b2.bytes;
            if (b == 3) {   // the run's last words are followed by the scales
                ok &= add_piece(L.b2, K1_DOWN, s, gb + (long long)a * nh * kQ4Quarter,
                                (long long)(4 - a) * nh * kQ4Quarter + (long long)nh * kQ4Scales);
                P.scales = P.words + (4 - a) * nh * kQ4Quarter;
            } else {
                ok &= add_piece(L.b2, K1_DOWN, s, gb + (long long)a * nh * kQ4Quarter,
                                (long long)(b - a + 1) * nh * kQ4Quarter);
                P.scales = L.b2.bytes;
                ok &= add_piece(L.b2, K1_DOWN, s, gb + 4LL * nh * kQ4Quarter, (long long)nh * kQ4Scales);
            }
        }
    }
    if (lora_rows) {
        // LoRA rows (row-major [rows, r] fp16): B_gate, B_up and A_down^T of the
        // pair's act rows, B_down of this CTA's output half
        const long long rb = 2LL * S.r, row0 = 8LL * p.seg[0].hr0, rows = 8LL * p.n_hr;
        L.bg = L.b2.bytes;
        ok &= add_piece(L.b2, K1_BG, 0, row0 * rb, rows * rb);
        L.bu = L.b2.bytes;
        ok &= add_piece(L.b2, K1_BU, 0, row0 * rb, rows * rb);
        L.adt = L.b2.bytes;
        ok &= add_piece(L.b2, K1_ADT, 0, row0 * rb, rows * rb);
        L.bd = L.b2.bytes;
        ok &= add_piece(L.b2, K1_BD, 0, (rank ? 16LL * nh0 : 0LL) * rb, 16LL * nh * rb);
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
    int dst = 0;
    if (i == 0) {
        pc.kind = fc1 ? K1_FC1 : K1_LINIT;
        pc.src = (long long)rows * ng0 * kF16Unit + (long long)jr * ng1 * kF16Unit;
        pc.bytes = ng1 * kF16Unit;
        pc.dst = 0;
        return true;
    }
    dst = ng1 * kF16Unit;
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
// After the header, per step parity p and state row s:
//   y      [2][Ls][kNY][d] fp32  layer output (vector reductions; kNY copies spread
//                                the reductions, their sum is the output)
//   logr   [2][Ls][E]   fp32  own-router logits
//   logh   [2][Ls][E]   fp32  head logits (row of the head's owner)
//   lax    [2][Ls][32]  u64   A_gate x, A_up x as (fp32 bits, launch tag)
//   cnt    [2][Ls]      u32   head tasks done
//   xs     [Ls][d]      fp16  x of each layer, for the head flush
// and the trace area at the end of the workspace.
struct Ws1 {
    long long y, logr, logh, lax, cnt, xs, end;
};
__host__ __device__ inline Ws1 ws1(int Ls, int d, int E) {
    Ws1 w;
    long long o = kWsHeaderBytes;
    w.y = o;    o += 2LL * Ls * kNY * d * 4;
    w.logr = o; o += 2LL * Ls * E * 4;
    w.logh = o; o += 2LL * Ls * E * 4;
    w.lax = o;  o += 2LL * Ls * 32 * 8;
    w.cnt = o;  o += (2LL * Ls * 4 + 255) / 256 * 256;
    w.xs = o;   o += ((long long)Ls * d * 2 + 255) / 256 * 256;
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
    unsigned gu_warps;                    // consumer warps with gate/up (or LoRA A) partials
    unsigned fl_warps;                    // consumer warps with head-flush dense partials
    // arrays: each 16-byte aligned (some are read and written as vectors)
    __align__(16) int route_ready[EDGE0_MAX_LAYERS];
    __align__(16) int ids[EDGE0_MAX_LAYERS][kMaxK1];
    __align__(16) float w[EDGE0_MAX_LAYERS][kMaxK1];
    __align__(16) int heads[EDGE0_MAX_LAYERS];
    __align__(16) Shape1 S;
    __align__(16) Plan1 plan;
    __align__(16) Lay1 lay;
    __align__(16) float red[kCW];
    __align__(16) float lax[32];
    __align__(16) float v[16];
    __align__(16) float xsum[kMaxG1];
    __align__(16) float stepsum[kMaxSig];
    __align__(16) float mine[kMsg];
    __align__(16) float recv[kMsg];
    __align__(16) float actw[kMaxHr1 * 8];
    __align__(16) float part[kCW][kMsg];
    __align__(16) float logits[EDGE0_MAX_E];
    __align__(16) float rscr[2 * EDGE0_MAX_E];
    __align__(16) __half h[kMaxD1];
    __align__(16) uint2 xf[kMaxG1 * 16];  // [group][t][step]: x as B fragments
    __align__(16) uint2 af[kMaxSig * 8];  // [act step][lane < 8]: act hi (lanes 0-3), lo (4-7)
    __align__(16) uint2 gf[8];            // GELU(z) of a flush task, same form
};
static_assert(offsetof(Sm1, h) % 16 == 0 && offsetof(Sm1, xf) % 16 == 0 &&
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
    Sm1& s = sm();
    if (s.trace && threadIdx.x == 0 && s.tslot + 3 <= 3072) {
        unsigned long long* tr = reinterpret_cast<unsigned long long*>(p.ws + p.ws_bytes - kTraceBytes) +
                                 (long long)blockIdx.x * kTraceSlots + s.tslot;
        long long c;
        asm volatile("mov.u64 %0, %%clock64;" : "=l"(c));
        tr[0] = (unsigned long long)tag;
        tr[1] = now1();
        tr[2] = (unsigned long long)c;
        s.tslot += 3;
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

// bounded wait on a block or exchange barrier phase; false on abort/timeout
__device__ __noinline__ bool mbar_wait1(WsHeader* hdr, uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = now1();
    for (unsigned it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31) == 31) {
            if (gone1(hdr)) return false;
            if (now1() - t0 > sm().wait_ns) {
                fail1(hdr, EDGE0_ETIMEOUT);
                return false;
            }
        }
    }
}

// Grid barriers.  Two counters: `barrier` counts layer-end arrivals (one per CTA
// and layer), `barrier_r` router arrivals (one per CTA and layer that routes
// itself).  Every CTA arrives at a layer's router barrier before its end
// barrier and waits for the end barrier before the next layer, so neither
// counter can reach a barrier's count while a CTA has yet to arrive at it (CTAs
// that do not wait for the router barrier arrive at the end one right away; on
// a shared counter their arrivals could complete the router barrier early).
// thread 0 arrives after the caller's consumer barrier (all of the CTA's global
// writes before it are ordered by the fence)
__device__ __forceinline__ void grid_arrive1(unsigned long long* ctr) {
    if (threadIdx.x == 0) {
        __threadfence();
        red_release_add_u64(ctr, 1ull);
    }
}
// thread 0 polls, then a consumer barrier; false on abort/timeout (uniform)
__device__ __noinline__ bool grid_wait1(WsHeader* hdr, const unsigned long long* ctr, unsigned long long target) {
    if (threadIdx.x == 0 && ld_acquire_u64(ctr) < target) {
        const unsigned long long t0 = now1();
        for (unsigned it = 0; ld_acquire_u64(ctr) < target; ++it) {
            if ((it & 15) == 15) {
                if (gone1(hdr)) {
                    *(volatile int*)&sm().abort = 1;
                    break;
                }
                if (now1() - t0 > sm().wait_ns) {
                    fail1(hdr, EDGE0_ETIMEOUT);
                    break;
                }
            }
        }
    }
    return !cbar_or1(vload(&sm().abort) != 0);
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

// ---------------------------------------------------------------- producer ----
__device__ __forceinline__ bool own_routed1(const Prog& p, int l, int step) {
    return step == 0 || !(p.layers[l].flags & LF_PREROUTED);
}

__device__ const char* piece_src1(const Prog& p, const Piece1& pc, int l) {
    const Sm1& s = sm();
    const LayerP& Ly = p.layers[l];
    switch (pc.kind) {
        case K1_ROUTER: return Ly.router + pc.src;
        case K1_GU:
        case K1_DOWN: {
            const Seg1& sg = s.plan.seg[pc.seg];
            const bool gu = pc.kind == K1_GU;
            if (sg.slot < 0) return (gu ? Ly.sh_gu : Ly.sh_down) + pc.src;
            const long long stride = gu ? q4_bytes(2 * p.I, p.d) : q4_bytes(p.d, p.I);
            return (gu ? Ly.gu : Ly.down) + (long long)s.ids[l][sg.slot] * stride + pc.src;
        }
        case K1_LA: return Ly.lora_Ag + pc.src;
        case K1_LU: return Ly.lora_Au + pc.src;
        case K1_BG: return reinterpret_cast<const char*>(Ly.lora_Bg) + pc.src;
        case K1_BU: return reinterpret_cast<const char*>(Ly.lora_Bu) + pc.src;
        case K1_ADT: return reinterpret_cast<const char*>(Ly.lora_AdT) + pc.src;
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
// one flush block (task j of head layer l, half h): as issue1, with copy i made
// by lane i straight from flush_piece
__device__ bool issue_flush1(const Prog& p, WsHeader* hdr, Stream1& q, int j, int h, const int* ids, int n2, int l,
                             uint64_t pol, int tag);

// the whole producer warp: place a block, wait for its room, arm its barrier,
// issue its copies (one lane per copy)
__device__ bool issue1(const Prog& p, WsHeader* hdr, Stream1& q, const Block1& B, int l, uint64_t pol, int tag) {
    Sm1& s = sm();
    const int lane = threadIdx.x & 31;
    if (B.bytes == 0) return true;
    const int off = place1(q.r, B.bytes, p.ring1);
    const int end = q.r.pos;
    int ok = 1;
    if (lane == 0) {
        const unsigned long long t0 = now1();
        for (unsigned it = 0;; ++it) {
            if (end - vload(&s.released) <= p.ring1 && q.nb - vload(&s.released_blocks) < kBlocks) break;
            if ((it & 63) == 63) {
                if (gone1(hdr)) { ok = 0; break; }
                if (now1() - t0 > s.wait_ns) { fail1(hdr, EDGE0_ETIMEOUT); ok = 0; break; }
            }
        }
        if (ok) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&s.full[q.nb % kBlocks], (uint32_t)B.bytes);
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) return false;
    for (int i = lane; i < B.n; i += 32) {
        const Piece1& pc = B.pc[i];
        bulk_g2s(ring() + off + pc.dst, piece_src1(p, pc, l), (uint32_t)pc.bytes, &s.full[q.nb % kBlocks], pol);
    }
    ++q.nb;
    if (lane == 0) {
        *(volatile int*)&s.issued = q.nb;
        if (s.trace) stamp_slow1(p, tag, true);
    }
    __syncwarp();
    return true;
}

__device__ bool issue_flush1(const Prog& p, WsHeader* hdr, Stream1& q, int j, int h, const int* ids, int n2, int l,
                             uint64_t pol, int tag) {
    Sm1& s = sm();
    const int lane = threadIdx.x & 31;
    const int bytes = flush_bytes(s.S, j, h, n2);
    const int off = place1(q.r, bytes, p.ring1);
    const int end = q.r.pos;
    int ok = 1;
    if (lane == 0) {
        const unsigned long long t0 = now1();
        for (unsigned it = 0;; ++it) {
            if (end - vload(&s.released) <= p.ring1 && q.nb - vload(&s.released_blocks) < kBlocks) break;
            if ((it & 63) == 63) {
                if (gone1(hdr)) { ok = 0; break; }
                if (now1() - t0 > s.wait_ns) { fail1(hdr, EDGE0_ETIMEOUT); ok = 0; break; }
            }
        }
        if (ok) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&s.full[q.nb % kBlocks], (uint32_t)bytes);
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) return false;
    Piece1 pc;
    if (flush_piece(s.S, j, h, lane, ids, n2, pc))
        bulk_g2s(ring() + off + pc.dst, piece_src1(p, pc, l), (uint32_t)pc.bytes, &s.full[q.nb % kBlocks], pol);
    ++q.nb;
    if (lane == 0) {
        *(volatile int*)&s.issued = q.nb;
        if (s.trace) stamp_slow1(p, tag, true);
    }
    __syncwarp();
    return true;
}

// the head flush's blocks: a task's one-hot rows are gathered by the head layer's
// executed (this step) and previous (last step) ids, read once the barrier that
// ends that layer has passed
__device__ bool produce_flush1(const Prog& p, WsHeader* hdr, Stream1& q, int step, int par, unsigned long long base,
                               uint64_t pol) {
    Sm1& s = sm();
    const int lane = threadIdx.x & 31;
    const int tph = p.H / kRowTile + p.E / kRowTile;
    const int n2 = p.K + (step > 0 ? p.K : 0);
    int cur = -1;
    __shared__ int fids[2 * kMaxK1];
    for (int t = s.plan.t0; t < s.plan.t1; ++t) {
        const int l = s.heads[t / tph];
        if (l != cur) {
            const unsigned long long need = base + (unsigned long long)gridDim.x * ((unsigned long long)l + 1);
            int ok = 1;
            if (lane == 0 && ld_acquire_u64(&hdr->barrier) < need) {
                const unsigned long long t0 = now1();
                for (unsigned it = 0; ld_acquire_u64(&hdr->barrier) < need; ++it) {
                    if ((it & 15) == 15) {
                        if (gone1(hdr)) { ok = 0; break; }
                        if (now1() - t0 > s.wait_ns) { fail1(hdr, EDGE0_ETIMEOUT); ok = 0; break; }
                    }
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
            const int sidx = p.layers[l].sidx;
            if (lane < n2) {
                const int k = lane < p.K ? lane : lane - p.K;
                const int32_t* src = p.exec_ids + ((long long)((lane < p.K ? par : par ^ 1)) * p.Ls + sidx) * p.K;
                int e = ld_volatile_s32(src + k);
                e = e < 0 || e >= p.E ? 0 : e;
                fids[lane] = lane < p.K ? e : p.E + e;
            }
            __syncwarp();
            cur = l;
        }
        const int j = t % tph, tg = 0xF000 | (t - s.plan.t0);
        if (!issue_flush1(p, hdr, q, j, 0, fids, n2, l, pol, tg)) return false;
        if (!issue_flush1(p, hdr, q, j, 1, fids, n2, l, pol, tg)) return false;
    }
    return true;
}

__device__ void producer1(const Prog& p, WsHeader* hdr, int step, int par, unsigned long long base) {
    Sm1& s = sm();
    const int lane = threadIdx.x & 31;
    const uint64_t pol = policy_evict_first();
    Stream1 q{{0, 0}, 0};
    for (int l = 0; l < p.L; ++l) {
        const bool own = own_routed1(p, l, step);
        if (own && !issue1(p, hdr, q, s.lay.b0, l, pol, (l << 8) | 0x80)) return;
        if (own && s.plan.role == R1_ROUTED && s.plan.nseg > 0) {
            // the routed weights of a layer that routes itself follow its routing
            int ok = 1;
            if (lane == 0) {
                const unsigned long long t0 = now1();
                for (unsigned it = 0; !vload(&s.route_ready[l]); ++it) {
                    if ((it & 63) == 63) {
                        if (gone1(hdr)) { ok = 0; break; }
                        if (now1() - t0 > s.wait_ns) { fail1(hdr, EDGE0_ETIMEOUT); ok = 0; break; }
                    }
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) return;
        }
        if (!issue1(p, hdr, q, s.lay.b1, l, pol, (l << 8) | 0x81)) return;
        if (!issue1(p, hdr, q, s.lay.b2, l, pol, (l << 8) | 0x82)) return;
        // the head flush runs right after the last layer that owns a head
        if (l == s.flush_after && !produce_flush1(p, hdr, q, step, par, base, pol)) return;
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
// after a consumer barrier that follows the last read of the current block
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

// x = fp16(h * rsqrt(mean(h^2) + eps) * gamma) after h = fp16(h + y) (y == null:
// h from h_in); B fragments and group sums of x over groups [g0, g1) of d.
// Thread i owns elements 4i .. 4i+3.
__device__ void build_x1(const Prog& p, int l, const __half* h_in, const float* y, uint2 gam, int g0, int g1,
                         __half* xs_out, __half* dbg_prev) {
    Sm1& s = sm();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, n4 = p.d / 4;
    float hf[4] = {0.f, 0.f, 0.f, 0.f};
    float q = 0.f;
    if (tid < n4) {
        const uint2 hv = h_in ? *reinterpret_cast<const uint2*>(h_in + 4 * tid)
                              : *reinterpret_cast<const uint2*>(&s.h[4 * tid]);
        __half2 h01 = *reinterpret_cast<const __half2*>(&hv.x), h23 = *reinterpret_cast<const __half2*>(&hv.y);
        if (y) {
            float4 yv = __ldcg(reinterpret_cast<const float4*>(y + 4 * tid));
#pragma unroll
            for (int q = 1; q < kNY; ++q) {
                const float4 u = __ldcg(reinterpret_cast<const float4*>(y + (long long)q * p.d + 4 * tid));
                yv.x += u.x; yv.y += u.y; yv.z += u.z; yv.w += u.w;
            }
            h01 = __floats2half2_rn(__low2float(h01) + yv.x, __high2float(h01) + yv.y);
            h23 = __floats2half2_rn(__low2float(h23) + yv.z, __high2float(h23) + yv.w);
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
    cbar1();
    float ss = 0.f;
#pragma unroll
    for (int w = 0; w < kCW; ++w) ss += s.red[w];
    const float rs = rsqrtf(ss / (float)p.d + p.layers[l].eps);
    const int k = 4 * tid, g = k / kGroup;
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
    if (tid < n4 && g >= g0 && g < g1) {
        const int kk = k % kGroup, st = kk / 16, k16 = kk % 16, wv = k16 >> 3, t = (k16 & 7) >> 1;
        const int gl = g - g0;
        uint32_t* xw = reinterpret_cast<uint32_t*>(s.xf);
        xw[((gl * 4 + t) * 4 + st) * 2 + wv] = pack2(x[0], x[1]);
        xw[((gl * 4 + t + 1) * 4 + st) * 2 + wv] = pack2(x[2], x[3]);
        if ((lane & 15) == 0) s.xsum[gl] = sum;
        if (xs_out) {
            uint2 o;
            o.x = pack2(x[0], x[1]);
            o.y = pack2(x[2], x[3]);
            *reinterpret_cast<uint2*>(xs_out + k) = o;
        }
    }
    cbar1();
}

// own-router units of this CTA: partial logits summed into logr
__device__ void router_units1(const Prog& p, const char* blk, float* logr, int xg0) {
    const Sm1& s = sm();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, g8 = lane >> 2;
    const int ngh = ngh1(p.d, cluster_ctarank());
    for (int u = s.plan.ru0 + wid; u < s.plan.ru1; u += kCW) {
        const int rt = u / ngh, g = u - rt * ngh;
        const char* unit = blk + (long long)(u - s.plan.ru0) * kF16Unit;
        uint4 xa, xb;
        xfrag(s, xg0 + g, lane, xa, xb);
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t xbv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
        for (int st = 0; st < 4; ++st) {
            const uint4 a = *reinterpret_cast<const uint4*>(unit + st * kF16Step + 16 * lane);
            const uint32_t A[4] = {a.x, a.y, a.z, a.w};
            mma_16816(c, A, xbv[2 * st], xbv[2 * st + 1]);
        }
        if ((lane & 3) == 0) {
            red_add_f32(logr + rt * 16 + g8, c[0]);
            red_add_f32(logr + rt * 16 + g8 + 8, c[2]);
        }
    }
}

// gate/up partial sums of the pair's hr over this CTA's half of d: warp w takes
// groups [ngh w / 16, ngh (w + 1) / 16) of every hr
__device__ void gateup1(const Prog& p, const char* blk, int ngh, int n_hr) {
    Sm1& s = sm();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int ga, gb;
    split1(ngh, kCW, wid, &ga, &gb);
    if (ga >= gb) return;
    float acc[kMaxHr1][2];
#pragma unroll
    for (int j = 0; j < kMaxHr1; ++j) acc[j][0] = acc[j][1] = 0.f;
    for (int g = ga; g < gb; ++g) {
        uint4 xa, xb;
        xfrag(s, g, lane, xa, xb);
        const float xsm = s.xsum[g];
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
    stamp1(p, 0xE010);
    if ((lane & 3) == 0) {
        const int g8 = lane >> 2;
#pragma unroll
        for (int j = 0; j < kMaxHr1; ++j)
            if (j < n_hr) {
                s.part[wid][j * 16 + g8] = acc[j][0];
                s.part[wid][j * 16 + g8 + 8] = acc[j][1];
            }
    }
}

// LoRA A x of one matrix over all of d (the LoRA pair: rank 0 A_gate, rank 1
// A_up): partial sums of its 16 rows into part (warp w takes groups w, w + 16, ...)
__device__ void lora_a1(const char* blk, int ng) {
    Sm1& s = sm();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    float a0 = 0.f, a1 = 0.f;
    for (int g = wid; g < ng; g += kCW) {
        const char* unit = blk + (long long)g * kF16Unit;
        uint4 xa, xb;
        xfrag(s, g, lane, xa, xb);
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
    if ((lane & 3) == 0) {
        const int g8 = lane >> 2;
        s.part[wid][g8] = a0;
        s.part[wid][g8 + 8] = a1;
    }
}

// act of every act row of the pair, weighted by its routing weight, as hi/lo B
// fragments per 16-row step, with per-step sums; thread (sigma, k) owns row k of
// act step sigma.  m0 / m1: the partial gate/up sums of rank 0 / rank 1; blk2:
// the down block (the LoRA rows of a shared pair).
__device__ void act1(const Prog& p, int l, const float* m0, const float* m1, const char* blk2, bool lora) {
    Sm1& s = sm();
    const int tid = threadIdx.x;
    const Lay1& L = s.lay;
    if ((tid & ~31) >= L.nsig * 16) return;   // whole warps only: full-mask shuffles below
    const bool live = tid < L.nsig * 16;
    const int sig = live ? tid >> 4 : 0, k = tid & 15;
    const int sg = L.sig_seg[sig];
    const Seg1& seg = s.plan.seg[sg];
    const int row = 16 * L.sig_step[sig] + k;   // expert-local act row
    float aw = 0.f;
    if (live && row >= 8 * seg.hr0 && row < 8 * seg.hr1) {
        const int i = L.seg_base[sg] + row - 8 * seg.hr0;   // pair-local act row
        const int hl = i >> 3, r8 = i & 7;
        float gt = m0[hl * 16 + r8] + m1[hl * 16 + r8];
        float up = m0[hl * 16 + 8 + r8] + m1[hl * 16 + 8 + r8];
        float wt = 1.f;
        if (seg.slot >= 0) {
            wt = s.w[l][seg.slot];
        } else if (lora) {
            // unmerged LoRA on the shared gate and up [S3.3]: + (alpha / r) B (A x)
            const int r = p.r;
            const __half* bg = reinterpret_cast<const __half*>(blk2 + L.bg) + (long long)i * r;
            const __half* bu = reinterpret_cast<const __half*>(blk2 + L.bu) + (long long)i * r;
            float dg = 0.f, du = 0.f;
            if ((r & 7) == 0) {
                for (int j = 0; j < r; j += 8) {
                    const uint4 gv = *reinterpret_cast<const uint4*>(bg + j);
                    const uint4 uv = *reinterpret_cast<const uint4*>(bu + j);
                    const __half2* g2 = reinterpret_cast<const __half2*>(&gv);
                    const __half2* u2 = reinterpret_cast<const __half2*>(&uv);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 gf = __half22float2(g2[q]), uf = __half22float2(u2[q]);
                        dg += gf.x * s.lax[j + 2 * q] + gf.y * s.lax[j + 2 * q + 1];
                        du += uf.x * s.lax[16 + j + 2 * q] + uf.y * s.lax[16 + j + 2 * q + 1];
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
        aw = silu_f(gt) * up * wt;
        s.actw[i] = aw;
    }
    const __half hi = __float2half_rn(aw);
    const __half lo = __float2half_rn((aw - __half2float(hi)) * kLoScale);
    __half* af = reinterpret_cast<__half*>(s.af);
    const int kk = k & 7, t = kk >> 1, wv = k >> 3, hh = kk & 1;
    if (live) {
        af[((sig * 8 + t) * 2 + wv) * 2 + hh] = hi;        // lanes 0-3: hi column
        af[((sig * 8 + 4 + t) * 2 + wv) * 2 + hh] = lo;    // lanes 4-7: lo column
    }
    float sum = aw;
#pragma unroll
    for (int m = 8; m; m >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, m);
    if (live && k == 0) s.stepsum[sig] = sum;
}

// down of the pair's act over this CTA's half of the output row tiles: warp w
// takes row tiles [nh w / 16, nh (w + 1) / 16); results into yacc
// With `lora` (a shared pair): + (alpha / r) B_down v_pair on the same rows, one
// MMA per row tile with B_down's rows as the A operand (k = the rank, zero
// beyond r) and v_pair as hi/lo columns.
__device__ void down1(const Prog& p, int l, const char* blk2, int nh, bool lora, float* yout) {
    Sm1& s = sm();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const Lay1& L = s.lay;
    int ta, tb;
    split1(nh, kCW, wid, &ta, &tb);
    float y[kMaxTw][2];
#pragma unroll
    for (int j = 0; j < kMaxTw; ++j) y[j][0] = y[j][1] = 0.f;
    if (lora) {
        const int r = p.r, g8 = lane >> 2, t = lane & 3;
        const float ls = p.layers[l].lora_scale;
        uint2 bv = make_uint2(0u, 0u);
        if (lane < 8) bv = s.af[kMaxSig * 8 - 8 + lane];   // v_pair hi/lo (written by lora_v1)
        const __half* bd = reinterpret_cast<const __half*>(blk2 + L.bd);
        const __half zero = __float2half_rn(0.f);
#pragma unroll
        for (int j = 0; j < kMaxTw; ++j) {
            const int rt = ta + j;
            if (rt < tb) {
                // A fragment: rows rt*16 + g8 (+ 8), k = 2t, 2t+1 (+ 8)
                const __half* r0 = bd + (long long)(rt * 16 + g8) * r;
                const __half* r1 = r0 + 8LL * r;
                auto at = [&](const __half* row, int k) { return k < r ? row[k] : zero; };
                __half2 a0 = __halves2half2(at(r0, 2 * t), at(r0, 2 * t + 1));
                __half2 a1 = __halves2half2(at(r1, 2 * t), at(r1, 2 * t + 1));
                __half2 a2 = __halves2half2(at(r0, 2 * t + 8), at(r0, 2 * t + 9));
                __half2 a3 = __halves2half2(at(r1, 2 * t + 8), at(r1, 2 * t + 9));
                const uint32_t A[4] = {*reinterpret_cast<uint32_t*>(&a0), *reinterpret_cast<uint32_t*>(&a1),
                                       *reinterpret_cast<uint32_t*>(&a2), *reinterpret_cast<uint32_t*>(&a3)};
                float c[4] = {0.f, 0.f, 0.f, 0.f};
                mma_16816(c, A, bv.x, bv.y);
                y[j][0] += ls * (c[0] + c[1] * kLoInv);
                y[j][1] += ls * (c[2] + c[3] * kLoInv);
            }
        }
    }
    for (int pi = 0; pi < L.nparts; ++pi) {
        const Part1& P = L.part[pi];
        const int nst = P.sb - P.sa + 1;
        uint2 a[4];
        float psum = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            a[j] = make_uint2(0u, 0u);
            if (j < nst) {
                if (lane < 8) a[j] = s.af[(P.sig0 + j) * 8 + lane];
                psum += s.stepsum[P.sig0 + j];
            }
        }
        const char* wb = blk2 + P.words + 4 * lane;
        const long long sstride = (long long)nh * kQ4Quarter;
#pragma unroll
        for (int j = 0; j < kMaxTw; ++j) {
            const int rt = ta + j;
            if (rt < tb) {
                float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (q < nst) {
                        const uint32_t wv = *reinterpret_cast<const uint32_t*>(wb + q * sstride + rt * kQ4Quarter);
                        uint32_t A[4];
                        q4_masks(wv, A);
                        if (q & 1) mma_16816(c1, A, a[q].x, a[q].y);
                        else mma_16816(c0, A, a[q].x, a[q].y);
                    }
                }
                const float4 sc = scales4(blk2 + P.scales + rt * kQ4Scales + (lane >> 2) * 8);
                y[j][0] += sc.x * kTwo24 * ((c0[0] + c1[0]) + (c0[1] + c1[1]) * kLoInv) + sc.y * psum;
                y[j][1] += sc.z * (kTwo24 / 16.f) * ((c0[2] + c1[2]) + (c0[3] + c1[3]) * kLoInv) + sc.w * psum;
            }
        }
    }
    stamp1(p, 0xE020);
    // rows g (y[j][0]) and g + 8 (y[j][1]) sit in lanes 4g: lane q < 4 gathers rows
    // 4q .. 4q+3 of the tile and adds them into the layer's y with one vector reduction
#pragma unroll
    for (int j = 0; j < kMaxTw; ++j) {
        if (ta + j < tb) {
            float v[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int src = (lane & 1) * 16 + 4 * m;
                const float a = __shfl_sync(0xffffffffu, y[j][0], src);
                const float b = __shfl_sync(0xffffffffu, y[j][1], src);
                v[m] = (lane & 2) ? b : a;
            }
            if (lane < 4) red_add_v4_f32(yout + (ta + j) * 16 + 4 * lane, v[0], v[1], v[2], v[3]);
        }
    }
    stamp1(p, 0xE021);
}

// the shared pair's partial v = A_down^T-rows . act of its own rows (64 threads:
// thread 4 r + c sums rows c, c + 4, ...)
__device__ void lora_v1(const char* blk2, int r, int rows) {
    Sm1& s = sm();
    const int tid = threadIdx.x;
    if (tid >= 64) return;
    const int rr = tid >> 2, c = tid & 3;
    float v = 0.f;
    if (rr < r) {
        const __half* adt = reinterpret_cast<const __half*>(blk2 + s.lay.adt);
        for (int i = c; i < rows; i += 4) v += __half2float(adt[(long long)i * r + rr]) * s.actw[i];
    }
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    if (c == 0 && rr < 16) {
        s.v[rr] = v;
        // as the B operand of down1's LoRA MMA (k = rr): lanes 0-3 hi, 4-7 lo
        const __half hi = __float2half_rn(v);
        const __half lo = __float2half_rn((v - __half2float(hi)) * kLoScale);
        __half* bf = reinterpret_cast<__half*>(&s.af[kMaxSig * 8 - 8]);
        const int kk = rr & 7, t = kk >> 1, wv = rr >> 3, hh = kk & 1;
        bf[(t * 2 + wv) * 2 + hh] = hi;
        bf[((4 + t) * 2 + wv) * 2 + hh] = lo;
    }
}

// ------------------------------------------------------------ head flush ----
// x of head layer l over all of d as B fragments
__device__ void flush_head1(const Prog& p, const __half* xs) {
    Sm1& s = sm();
    const int tid = threadIdx.x, n4 = p.d / 4;
    if (tid < n4) {
        const uint2 v = __ldcg(reinterpret_cast<const uint2*>(xs + 4 * tid));
        const int k = 4 * tid, g = k / kGroup, kk = k % kGroup, st = kk / 16, k16 = kk % 16;
        const int wv = k16 >> 3, t = (k16 & 7) >> 1;
        uint32_t* xw = reinterpret_cast<uint32_t*>(s.xf);
        xw[((g * 4 + t) * 4 + st) * 2 + wv] = v.x;
        xw[((g * 4 + t + 1) * 4 + st) * 2 + wv] = v.y;
    }
    cbar1();
}

// one task of head layer l (see flush_block); its logits summed into lg
__device__ void flush_task1(const Prog& p, int l, int j, int n2, const char* blkA, const char* blkB, float* lg) {
    Sm1& s = sm();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, g8 = lane >> 2;
    const LayerP& Ly = p.layers[l];
    const int nH = p.H / kRowTile, nE = p.E / kRowTile, ng = p.d / kGroup;
    const bool fc1 = j < nH;
    const int row0 = 16 * (fc1 ? j : j - nH);
    (void)Ly;
    // dense part: warp w takes groups [ng w / 16, ng (w + 1) / 16) of the row tile
    int ga, gb;
    split1(ng, kCW, wid, &ga, &gb);
    float acc0 = 0.f, acc1 = 0.f;
    for (int g = ga; g < gb; ++g) {
        uint4 xa, xb;
        xfrag(s, g, lane, xa, xb);
        const uint32_t xbv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
        const char* unit = g < ng / 2 ? blkA + (long long)g * kF16Unit : blkB + (long long)(g - ng / 2) * kF16Unit;
        float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int st = 0; st < 4; ++st) {
            const uint4 a = *reinterpret_cast<const uint4*>(unit + st * kF16Step + 16 * lane);
            const uint32_t A[4] = {a.x, a.y, a.z, a.w};
            mma_16816(c, A, xbv[2 * st], xbv[2 * st + 1]);
        }
        acc0 += c[0];
        acc1 += c[2];
    }
    if ((lane & 3) == 0) {
        s.part[wid][g8] = acc0;
        s.part[wid][g8 + 8] = acc1;
    }
    cbar1();
    if (tid < 16) {
        float z = 0.f;
        for (int w = 0; w < kCW; ++w)
            if ((s.fl_warps >> w) & 1u) z += s.part[w][tid];
        // one-hot columns of the executed and previous masks [S3.2 "Head"]: the
        // rows of the transposed columns that the producer gathered into the block
        // (the concatenated features are never materialised)
        const __half* oh = reinterpret_cast<const __half*>(blkB + (long long)(ng - ng / 2) * kF16Unit +
                                                           (fc1 ? (long long)nE * kF16Step : 0LL));
        for (int k2 = 0; k2 < n2; ++k2) z += __half2float(oh[k2 * 16 + tid]);
        if (fc1) {
            // erf-GELU [S3.2 "Head"], then fc2 columns row0 .. row0+15 below
            const float gl = 0.5f * z * (1.f + erff(z * 0.70710678118654752f));
            const __half hi = __float2half_rn(gl);
            const __half lo = __float2half_rn((gl - __half2float(hi)) * kLoScale);
            __half* gf = reinterpret_cast<__half*>(s.gf);
            const int kk = tid & 7, t = kk >> 1, wv = tid >> 3, hh = kk & 1;
            gf[(t * 2 + wv) * 2 + hh] = hi;
            gf[((4 + t) * 2 + wv) * 2 + hh] = lo;
        } else {
            red_add_f32(lg + row0 + tid, z);
        }
    }
    if (fc1) {
        cbar1();
        const uint2 b = lane < 8 ? s.gf[lane] : make_uint2(0u, 0u);
        const char* fc2 = blkB + (long long)(ng - ng / 2) * kF16Unit;
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

// routing of a complete logit row by warp 0 (logits read from global memory)
__device__ void route_row1(const float* lg, int E, int K, int kind, int ng, int G, float scale, const float* bias,
                           int* ids, float* w) {
    Sm1& s = sm();
    const int lane = threadIdx.x & 31;
    for (int e = lane; e < E; e += 32) s.logits[e] = __ldcg(lg + e);
    __syncwarp();
    warp_route(s.logits, E, K, kind, ng, G, scale, bias, s.rscr, ids, w, lane);
}

// ---------------------------------------------------------------- consumers ----
__device__ void consumer1(const Prog& p, WsHeader* hdr, const Ws1& W, int step, int par, unsigned tag,
                          unsigned long long base, unsigned long long base_r) {
    Sm1& s = sm();
    const int tid = threadIdx.x;
    const int rank = (int)cluster_ctarank();
    const int cta = blockIdx.x, nct = gridDim.x;
    const Plan1& pl = s.plan;
    const Lay1& L = s.lay;
    const int ng = p.d / kGroup, ngh = ngh1(p.d, rank), g0 = rank ? ng / 2 : 0;
    const int nh = nrth1(p.d, rank), row0 = rank ? 16 * (p.d / kRowTile / 2) : 0;
    const bool lora = s.S.lora && pl.role == R1_SHARED && pl.nseg > 0;
    const int hold = ld_volatile_s32(&hdr->hold);
    unsigned long long nend = 0, nrt = 0;   // layer-end and router barriers arrived at
    bool first_wait = true;
    // counter value once `n` barriers of a counter with launch base `b` completed
    auto target = [&](unsigned long long b, unsigned long long n) {
        unsigned long long t = b + (unsigned long long)nct * n;
        if (first_wait) t += (unsigned long long)(hold > 0 ? hold : 0);
        return t;
    };
    Cons1 c{{0, 0}, 0, 0, 0};
    int nx = 0;   // pair exchanges so far
    const uint32_t peer = (uint32_t)rank ^ 1u;
    const uint32_t rbar = mapa_shared(smem_u32(&s.xbar), peer);
    const uint32_t rrecv = mapa_shared(smem_u32(s.recv), peer);
    const bool xch = pl.n_hr > 0;
    const int msg = pl.n_hr * 16;
    // x fragments held: this CTA's half of d, or all of d on the LoRA pair
    const int xa0 = pl.role == R1_LORA ? 0 : g0, xa1 = pl.role == R1_LORA ? ng : g0 + ngh;
    // RMSNorm gain of layer 0 (then of the next layer, loaded a layer ahead)
    const int n4 = p.d / 4;
    auto gain = [&](int l) {
        uint2 g = make_uint2(0x3C003C00u, 0x3C003C00u);   // 1.0 in fp16
        if (l < p.L && p.layers[l].gamma && tid < n4)
            g = __ldg(reinterpret_cast<const uint2*>(p.layers[l].gamma + 4 * tid));
        return g;
    };
    uint2 gam = gain(0);
    // ---- head flush (after the last layer that owns a head): x of a head layer
    // is final once the barrier that ends the layer has passed.  A CTA adds its
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
                if (!grid_wait1(hdr, &hdr->barrier, target(base, (unsigned long long)l + 1))) return false;
                first_wait = false;
                flush_head1(p, reinterpret_cast<const __half*>(p.ws + W.xs) + (long long)sidx * p.d);
                xl = l;
            }
            float* lg = reinterpret_cast<float*>(p.ws + W.logh) + ((long long)par * p.Ls + sidx) * p.E;
            stamp1(p, 0xF100 | (t - pl.t0));
            bool ok = take1(p, hdr, c, flush_bytes(s.S, j, 0, n2));
            const char* blkA = ring() + c.off;
            ok = take1(p, hdr, c, flush_bytes(s.S, j, 1, n2)) && ok;
            const char* blkB = ring() + c.off;
            stamp1(p, 0xF200 | (t - pl.t0));
            if (ok) flush_task1(p, l, j, n2, blkA, blkB, lg);
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
                const long long o = ((long long)par * p.Ls + Ly.head_target) * p.K;
                route_row1(lg, p.E, p.K, Ly.head_route_kind, Ly.head_n_groups, Ly.head_topk_groups,
                           Ly.head_route_scale, Ly.head_bias, p.pred_ids + o, p.pred_w + o);
                if (p.dbg_logits)
                    for (int e = tid; e < p.E; e += 32) p.dbg_logits[(long long)l * p.E + e] = s.logits[e];
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
        float* y = reinterpret_cast<float*>(p.ws + W.y) + (((long long)par * p.Ls + sidx) * kNY + (cta >> 1) % kNY) * p.d;
        stamp1(p, (l << 8) | 0);
        // the exchange barrier of this layer is armed before the peer can send:
        // layer 0's here, the next layer's before this layer's grid arrival
        if (l == 0 && xch && tid == 0) mbar_arrive_expect_tx(&s.xbar, (uint32_t)(msg * 4));
        // ---- x: the previous layer's y is complete after its barrier
        const float* yprev = nullptr;
        if (l > 0) {
            if (!grid_wait1(hdr, &hdr->barrier, target(base, nend))) break;
            first_wait = false;
            yprev = reinterpret_cast<const float*>(p.ws + W.y) + ((long long)par * p.Ls + p.layers[l - 1].sidx) * kNY * p.d;
        }
        stamp1(p, (l << 8) | 1);
        __half* xs_out = cta < 2 ? reinterpret_cast<__half*>(p.ws + W.xs) + (long long)sidx * p.d : nullptr;
        __half* dbg = (p.dbg_h && cta == 0 && l > 0) ? p.dbg_h + (long long)(l - 1) * p.d : nullptr;
        build_x1(p, l, l == 0 ? p.h_io : nullptr, yprev, gam, xa0, xa1, xs_out, dbg);
        gam = gain(l + 1);
        stamp1(p, (l << 8) | 2);
        // ---- routing
        if (own) {
            float* logr = reinterpret_cast<float*>(p.ws + W.logr) + ((long long)par * p.Ls + sidx) * p.E;
            bool ok = true;
            if (L.b0.bytes) {
                ok = take1(p, hdr, c, L.b0.bytes);
                if (ok) router_units1(p, ring() + c.off, logr, g0 - xa0);
            }
            if (cbar_or1(!ok || vload(&s.abort))) break;
            if (L.b0.bytes) give1(c);
            stamp1(p, (l << 8) | 11);
            grid_arrive1(&hdr->barrier_r);
            ++nrt;
            if (pl.role == R1_ROUTED && (pl.nseg > 0 || cta == 0)) {
                if (!grid_wait1(hdr, &hdr->barrier_r, target(base_r, nrt))) break;
                first_wait = false;
                stamp1(p, (l << 8) | 3);
                if (tid < 32)
                    route_row1(logr, p.E, p.K, Ly.route_kind, Ly.n_groups, Ly.topk_groups, Ly.route_scale, Ly.bias,
                               s.ids[l], s.w[l]);
                cbar1();
                if (tid == 0) *(volatile int*)&s.route_ready[l] = 1;
            }
        }
        if (cta == 0 && tid < p.K) p.exec_ids[((long long)par * p.Ls + sidx) * p.K + tid] = s.ids[l][tid];
        stamp1(p, (l << 8) | 4);
        // ---- gate/up (or LoRA A) partial sums over this CTA's half, swapped with the peer
        if (L.b1.bytes) {
            const bool ok = take1(p, hdr, c, L.b1.bytes);
            stamp1(p, (l << 8) | 9);
            const char* blk1 = ring() + c.off;
            if (ok) {
                if (pl.role == R1_LORA) lora_a1(blk1, ng);
                else gateup1(p, blk1, ngh, pl.n_hr);
            }
            if (cbar_or1(!ok || vload(&s.abort))) break;
            give1(c);
        }
        stamp1(p, (l << 8) | 5);
        if (xch) {
            if (tid < msg) {
                float v = 0.f;
                for (int w = 0; w < kCW; ++w)
                    if ((s.gu_warps >> w) & 1u) v += s.part[w][tid];
                s.mine[tid] = v;
                st_async_b32(rrecv + 4u * tid, v, rbar);
            }
            if (lora && tid >= kCT - 32) {
                // A_gate x, A_up x from the LoRA pair: (value, tag) words of this launch
                const unsigned long long* src =
                    reinterpret_cast<const unsigned long long*>(p.ws + W.lax) + ((long long)par * p.Ls + sidx) * 32;
                const int ln = tid & 31;
                const unsigned long long t0 = now1();
                unsigned long long v = ld_relaxed_u64(src + ln);
                for (unsigned it = 0; !__all_sync(0xffffffffu, (unsigned)(v >> 32) == tag); ++it) {
                    if ((it & 15) == 15) {
                        int bad = 0;
                        if (ln == 0) {
                            if (gone1(hdr)) bad = 1;
                            else if (now1() - t0 > s.wait_ns) { fail1(hdr, EDGE0_ETIMEOUT); bad = 1; }
                        }
                        if (__shfl_sync(0xffffffffu, bad, 0)) break;
                    }
                    v = ld_relaxed_u64(src + ln);
                }
                s.lax[ln] = __uint_as_float((unsigned)(v & 0xFFFFFFFFu));
            }
            if (tid == 0) {
                if (!mbar_wait1(hdr, &s.xbar, (uint32_t)(nx & 1))) *(volatile int*)&s.abort = 1;
                else if (l + 1 < p.L) mbar_arrive_expect_tx(&s.xbar, (uint32_t)(msg * 4));
            }
            ++nx;
            if (cbar_or1(vload(&s.abort) != 0)) break;
        }
        const float* m0 = rank ? s.recv : s.mine;
        const float* m1 = rank ? s.mine : s.recv;
        stamp1(p, (l << 8) | 6);
        if (pl.role == R1_LORA) {
            // (value, tag) words: rank 0 A_gate x (words 0-15), rank 1 A_up x (16-31)
            if (tid < 16) {
                float v = 0.f;
                for (int w = 0; w < kCW; ++w)
                    if ((s.gu_warps >> w) & 1u) v += s.part[w][tid];
                unsigned long long* dst =
                    reinterpret_cast<unsigned long long*>(p.ws + W.lax) + ((long long)par * p.Ls + sidx) * 32;
                st_relaxed_u64(dst + 16 * rank + tid, ((unsigned long long)tag << 32) | __float_as_uint(v));
            }
            cbar1();
            grid_arrive1(&hdr->barrier);
            ++nend;
            if (l == s.flush_after && !flush()) break;
            continue;
        }
        // ---- act, down, y
        if (L.b2.bytes) {
            const bool ok = take1(p, hdr, c, L.b2.bytes);
            stamp1(p, (l << 8) | 10);
            const char* blk2 = ring() + c.off;
            if (ok) act1(p, l, m0, m1, blk2, lora);
            if (cbar_or1(!ok || vload(&s.abort))) break;
            stamp1(p, (l << 8) | 7);
            if (lora) {
                lora_v1(blk2, p.r, 8 * pl.n_hr);
                cbar1();
            }
            down1(p, l, blk2, nh, lora, y + row0);
            cbar1();
            stamp1(p, 0xE022);
            give1(c);
        } else {
            cbar1();
        }
        stamp1(p, (l << 8) | 8);
        grid_arrive1(&hdr->barrier);
        ++nend;
        if (l == s.flush_after && !flush()) break;
    }
    if (broke) {
        if (tid == 0) *(volatile int*)&s.abort = 1;
        return;
    }
    stamp1(p, 0xFF00);
    // ---- the last layer's output
    if (!grid_wait1(hdr, &hdr->barrier, target(base, nend))) return;
    const float* ylast = reinterpret_cast<const float*>(p.ws + W.y) + ((long long)par * p.Ls + p.layers[p.L - 1].sidx) * kNY * p.d;
    const int a = p.d * cta / nct, b = p.d * (cta + 1) / nct;
    for (int i = a + tid; i < b; i += kCT) {
        float yv = 0.f;
#pragma unroll
        for (int q = 0; q < kNY; ++q) yv += __ldcg(ylast + (long long)q * p.d + i);
        const __half h = __float2half_rn(__half2float(s.h[i]) + yv);
        p.h_io[i] = h;
        if (p.dbg_h) p.dbg_h[(long long)(p.L - 1) * p.d + i] = h;
    }
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
    const Ws1 W = ws1(p.Ls, p.d, p.E);
    __shared__ unsigned long long s_base, s_base_r;
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
        const unsigned long long v = ld_acquire_u64(&hdr->barrier);
        s_base = v - v % (unsigned long long)gridDim.x;
        const unsigned long long vr = ld_acquire_u64(&hdr->barrier_r);
        s_base_r = vr - vr % (unsigned long long)gridDim.x;
        s_step = p.step >= 0 ? p.step : ld_volatile_s32(&hdr->step);
        s_tag = (ld_volatile_s32(reinterpret_cast<const int*>(&hdr->serial)) & 0x3FFFFFFF) + 1;
        // the plan of this CTA and the layout of its blocks
        Shape1 S;
        S.d = p.d; S.I = p.I; S.Is = p.Is; S.E = p.E; S.K = p.K; S.H = p.H; S.r = p.r;
        S.shared = (p.layers[0].flags & LF_SHARED) != 0;
        S.lora = (p.layers[0].flags & LF_LORA) != 0;
        S.P = p.pairs1[0]; S.Pr = p.pairs1[1]; S.Ps = p.pairs1[2]; S.Pl = p.pairs1[3];
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
        // warps that write partial sums (the others' part rows are not read)
        const int ngh = ngh1(p.d, rank), ng = p.d / kGroup;
        unsigned gm = 0, fm = 0;
        for (int w = 0; w < kCW; ++w) {
            int a, b;
            split1(ngh, kCW, w, &a, &b);
            if (s.plan.role == R1_LORA ? w < ng : a < b) gm |= 1u << w;
            split1(ng, kCW, w, &a, &b);
            if (a < b) fm |= 1u << w;
        }
        s.gu_warps = gm;
        s.fl_warps = fm;
    }
    __syncthreads();
    const int step = s_step, par = step & 1;
    // clear the other step parity of this launch's layers for the next step
    {
        const int op = par ^ 1;
        const long long dy = (long long)kNY * p.d;
        const long long per = dy + 2LL * p.E + 64;   // floats: y copies, logr, logh, lax (32 u64)
        const long long tot = (long long)p.L * per;
        const long long a = tot * blockIdx.x / gridDim.x, b = tot * (blockIdx.x + 1) / gridDim.x;
        for (long long i = a + tid; i < b; i += kT1) {
            const long long l = i / per, o = i % per;
            const long long row = (long long)op * p.Ls + p.layers[l].sidx;
            float* dst;
            if (o < dy) dst = reinterpret_cast<float*>(p.ws + W.y) + row * dy + o;
            else if (o < dy + p.E) dst = reinterpret_cast<float*>(p.ws + W.logr) + row * p.E + (o - dy);
            else if (o < dy + 2LL * p.E) dst = reinterpret_cast<float*>(p.ws + W.logh) + row * p.E + (o - dy - p.E);
            else dst = reinterpret_cast<float*>(p.ws + W.lax) + row * 64 + (o - dy - 2LL * p.E);
            *dst = 0.f;
        }
        if (blockIdx.x == 0)
            for (int l = tid; l < p.L; l += kT1)
                reinterpret_cast<unsigned*>(p.ws + W.cnt)[(long long)op * p.Ls + p.layers[l].sidx] = 0u;
    }
    // routing known at launch: the predictions of prerouted layers (step > 0)
    for (int i = tid; i < p.L * p.K; i += kT1) {
        const int l = i / p.K, k = i % p.K;
        s.route_ready[l] = 0;
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
        if (tid >= kCT) producer1(p, hdr, step, par, s_base);
        else consumer1(p, hdr, W, step, par, s_tag, s_base, s_base_r);
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

long long decode1_ws_bytes(int Ls, int d, int E) {
    if (Ls <= 0 || d <= 0 || E <= 0) return 0;
    return ws1(Ls, d, E).end + kTraceBytes;
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

// every CTA's plan and blocks for the shapes: the ring must hold the largest block
int derive1(Key1& k) {
    Shape1 S;
    S.d = k.d; S.I = k.I; S.Is = k.Is; S.E = k.E; S.K = k.K; S.H = k.H; S.r = k.r;
    S.shared = k.shared; S.lora = k.lora; S.n_heads = k.n_heads;
    S.P = k.nct / kClusterCtas;
    if (S.P < 4 || k.nct % kClusterCtas) return EDGE0_EUNSUPPORTED;
    if (!choose_pairs(S)) return EDGE0_EUNSUPPORTED;
    if (S.Pr < 1) return EDGE0_EUNSUPPORTED;
    const int ring = ((k.smem - kSm1Bytes) / 128) * 128;
    if (ring < 2 * kPieceMax) return EDGE0_EUNSUPPORTED;
    int biggest = 0;
    for (int pair = 0; pair < S.P; ++pair)
        for (int rank = 0; rank < kClusterCtas; ++rank) {
            Plan1 pl;
            Lay1 L;
            if (!plan1(S, pair, rank, pl) || !layout1(S, pl, rank, L)) return EDGE0_EUNSUPPORTED;
            const int m = L.b0.bytes > L.b1.bytes ? L.b0.bytes : L.b1.bytes;
            biggest = m > biggest ? m : biggest;
            biggest = L.b2.bytes > biggest ? L.b2.bytes : biggest;
        }
    const int tph = S.H / kRowTile + S.E / kRowTile;
    for (int j = 0; j < tph && S.n_heads > 0; ++j)
        for (int h = 0; h < 2; ++h) {
            Block1 B;
            if (!flush_block(S, j, h, B, nullptr, 2 * S.K) || B.n > 32) return EDGE0_EUNSUPPORTED;
            biggest = B.bytes > biggest ? B.bytes : biggest;
        }
    // a task's two blocks are held together
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
    if (p.ws_bytes < decode1_ws_bytes(p.Ls, p.d, p.E)) return EDGE0_EUNSUPPORTED;
    const int f0 = p.layers[0].flags & (LF_SHARED | LF_LORA);
    int n_heads = 0;
    for (int l = 0; l < p.L; ++l) {
        const LayerP& Ly = p.layers[l];
        if ((Ly.flags & (LF_SHARED | LF_LORA)) != f0) return EDGE0_EUNSUPPORTED;
        if (Ly.slot_table || Ly.gu_host) return EDGE0_EUNSUPPORTED;
        if (Ly.flags & LF_HEAD) ++n_heads;
        // bulk copies read whole 16-byte lines of every source
        if (((uintptr_t)Ly.gu | (uintptr_t)Ly.down | (uintptr_t)Ly.router) & 15) return EDGE0_EUNSUPPORTED;
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
    int nct = 0, smem = 0;
    rc = grid1(&nct, &smem);
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
