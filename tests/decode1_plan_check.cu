// Host-side check of the batch-1 decode kernel's work split (no GPU needed): for
// several shapes and grids, every CTA's plan and block layouts as the kernel
// builds them.  Checked: every expert CTA owns half-row tiles, and every
// half-row tile of every routed slot and of the shared expert is owned by
// exactly one CTA; the act rows the CTAs publish cover the layer's act vector
// exactly once; every group of A_gate and A_up has one LoRA CTA; every output
// row tile and router row tile has exactly one CTA, every head-flush task
// exactly one; every gate/up unit sits where the consumers look for it and
// comes from the right source unit; every copy lies inside its source matrix,
// starts and ends on 16 bytes and stays inside its block; the down block holds
// one unit per act group, in act order; every block fits the ring.
// Compiled and run by tests/test_decode1_plan.py; exits non-zero on a failure.
#include "decode1.cu"

#include <cstdio>
#include <vector>

using namespace edge0;
using namespace edge0::d1;

static int fails = 0;
#define CHECK(c, ...)                                                    \
    do {                                                                 \
        if (!(c)) {                                                      \
            ++fails;                                                     \
            if (fails < 30) {                                            \
                printf("FAIL %s:%d ", __FILE__, __LINE__);               \
                printf(__VA_ARGS__);                                     \
                printf("\n");                                            \
            }                                                            \
        }                                                                \
    } while (0)

static long long src_size(const Shape1& S, const Plan1& pl, const Piece1& pc) {
    switch (pc.kind) {
        case K1_ROUTER: return f16_bytes(S.E, S.d);
        case K1_GU: return q4_bytes(2 * (pl.seg[pc.seg].slot < 0 ? S.Is : S.I), S.d);
        case K1_DOWN: return q4_bytes(S.d, pc.seg < 0 ? S.Is : S.I);
        case K1_LA: case K1_LU: return f16_bytes(S.r, S.d);
        case K1_BG: case K1_BU: return 2LL * S.Is * S.r;
        case K1_AD: return f16_bytes(S.r, S.Is);
        case K1_BD: return 2LL * S.d * S.r;
        case K1_FC1: return f16_bytes(S.H, S.d);
        case K1_FC2: return f16_bytes(S.E, S.H);
        case K1_LINIT: return f16_bytes(S.E, S.d);
        case K1_OHF: return 2LL * 2 * S.E * S.H;
        case K1_OHL: return 2LL * 2 * S.E * S.E;
    }
    return -1;
}

static void check_block(const Shape1& S, const Plan1& pl, const Block1& B, int ring, const char* what) {
    int at = 0;
    for (int i = 0; i < B.n; ++i) {
        const Piece1& pc = B.pc[i];
        CHECK(pc.dst == at, "%s piece %d dst %d != %d", what, i, pc.dst, at);
        CHECK(pc.bytes > 0 && pc.bytes <= kPieceMax && pc.bytes % 16 == 0, "%s piece %d bytes %d", what, i, pc.bytes);
        CHECK(pc.src >= 0 && pc.src % 16 == 0, "%s piece %d src %lld", what, i, pc.src);
        CHECK(pc.src + pc.bytes <= src_size(S, pl, pc), "%s piece %d kind %d outside its source (%lld + %d > %lld)",
              what, i, pc.kind, pc.src, pc.bytes, src_size(S, pl, pc));
        at += pc.bytes;
    }
    CHECK(at == B.bytes, "%s bytes %d != %d", what, at, B.bytes);
    CHECK(B.bytes <= ring, "%s block of %d bytes > ring %d", what, B.bytes, ring);
}

static void check_shape(const char* name, int d, int E, int K, int I, int Is, int H, int r, bool shared, bool lora,
                        int n_heads, int nct, bool must) {
    Key1 k;
    memset(&k, 0, sizeof(k));
    k.d = d; k.I = I; k.Is = Is; k.E = E; k.K = K; k.H = H; k.r = r;
    k.shared = shared; k.lora = lora; k.n_heads = n_heads; k.nct = nct;
    k.smem = 232448 - 1024;
    const int rc = derive1(k);
    printf("%-30s grid %3d rc=%d: %d CTAs, %d LoRA-A CTAs per matrix, ring %d\n", name, nct, rc, k.grid, k.NQ,
           k.ring);
    CHECK(rc == 0 || !must, "%s: the grid must take the shape (rc %d)", name, rc);
    if (rc) return;
    CHECK(k.grid <= nct, "%s: more CTAs than the grid", name);
    Shape1 S;
    S.d = d; S.I = I; S.Is = Is; S.E = E; S.K = K; S.H = H; S.r = r;
    S.shared = shared; S.lora = lora; S.n_heads = n_heads;
    S.nct = k.grid; S.NQ = k.NQ;
    const int hpe = I / 8, n_sh = shared ? Is / 8 : 0, NA = n_act1(S), ng = d / 64;
    std::vector<int> cov_rt(K * hpe, 0), cov_sh(n_sh, 0), cov_act(NA, 0), cov_dt(d / 16, 0), cov_r(E / 16, 0);
    std::vector<int> cov_la(2 * ng, 0);
    const int tph = H / 16 + E / 16;
    std::vector<int> cov_task(n_heads * tph, 0);
    for (int c = 0; c < S.nct; ++c) {
        Plan1 pl;
        Lay1 L;
        const bool ok = plan1(S, c, pl) && layout1(S, pl, L);
        CHECK(ok, "%s CTA %d: plan/layout refused", name, c);
        if (!ok) continue;
        if (pl.role == R1_LORA) {
            CHECK(c >= S.nct - 2 * S.NQ, "LoRA CTA %d", c);
            for (int g = pl.la0; g < pl.la1; ++g) ++cov_la[pl.lm * ng + g];
            CHECK(L.b1.bytes == (pl.la1 - pl.la0) * 2048 && L.b3.bytes == 0, "LoRA CTA blocks");
        } else {
            CHECK(pl.n_hr >= 1, "%s CTA %d owns no hr", name, c);
        }
        CHECK(pl.n_hr <= kMaxHr1, "n_hr %d", pl.n_hr);
        int nh = 0;
        for (int s = 0; s < pl.nseg; ++s) {
            const Seg1& sg = pl.seg[s];
            CHECK(sg.hr0 < sg.hr1, "empty run");
            CHECK(L.seg_base[s] == 8 * nh, "seg_base %d != %d", L.seg_base[s], 8 * nh);
            CHECK((sg.slot < 0) == (s == pl.shr), "shared run index");
            nh += sg.hr1 - sg.hr0;
            for (int h = sg.hr0; h < sg.hr1; ++h) {
                if (sg.slot < 0) { CHECK(h < n_sh, "shared hr %d", h); if (h < n_sh) ++cov_sh[h]; }
                else { CHECK(sg.slot < K && h < hpe, "slot %d hr %d", sg.slot, h); if (sg.slot < K && h < hpe) ++cov_rt[sg.slot * hpe + h]; }
            }
        }
        CHECK(nh == pl.n_hr, "n_hr");
        // the act rows this CTA publishes (as its act threads map them)
        for (int i = 0; i < 8 * pl.n_hr; ++i) {
            int sg = 0;
            while (sg + 1 < pl.nseg && i >= L.seg_base[sg + 1]) ++sg;
            const Seg1& seg = pl.seg[sg];
            const int row = 8 * seg.hr0 + i - L.seg_base[sg];
            const long long gi = (seg.slot >= 0 ? (long long)seg.slot * I : (long long)K * I) + row;
            CHECK(gi >= 0 && gi < NA, "act index %lld", gi);
            if (gi >= 0 && gi < NA) ++cov_act[gi];
        }
        if (pl.dt >= 0) { CHECK(pl.dt == c && pl.dt < d / 16, "dt %d", pl.dt); ++cov_dt[pl.dt]; }
        if (pl.rt >= 0) { CHECK(pl.rt < E / 16, "rt %d", pl.rt); ++cov_r[pl.rt]; }
        for (int t = pl.t0; t < pl.t1; ++t) ++cov_task[t];
        check_block(S, pl, L.b0, k.ring, "b0");
        check_block(S, pl, L.b1, k.ring, "b1");
        check_block(S, pl, L.b3, k.ring, "b3");
        check_block(S, pl, L.b2, k.ring, "b2");
        CHECK(L.b0.bytes == (pl.rt >= 0 ? ng * 2048 : 0), "b0 bytes");
        if (pl.role == R1_EXPERT) {
            CHECK(L.b1.bytes == pl.n_hr * ng * 576, "b1 bytes");
            // gate/up unit (hr j, group g) as the consumers address it: the first
            // half of d for every hr, then the second half
            int j = 0;
            for (int s = 0; s < pl.nseg; ++s)
                for (int h = pl.seg[s].hr0; h < pl.seg[s].hr1; ++h, ++j)
                    for (int g = 0; g < ng; ++g) {
                        const int ng0 = ng / 2, ng1 = ng - ng0;
                        const long long at = g < ng0 ? ((long long)j * ng0 + g) * 576
                                                     : ((long long)pl.n_hr * ng0 + (long long)j * ng1 + (g - ng0)) * 576;
                        // the piece that holds it, and the source unit it copies
                        const int half = g < ng0 ? 0 : 1, gh = g < ng0 ? g : g - ng0, ngh = half ? ng1 : ng0;
                        const long long tiles = (pl.seg[s].slot < 0 ? Is : I) / 8;
                        const long long src = (half ? tiles * ng0 * 576 : 0) + ((long long)h * ngh + gh) * 576;
                        bool found = false;
                        for (int q = 0; q < L.b1.n; ++q) {
                            const Piece1& pc = L.b1.pc[q];
                            if (pc.seg == s && at >= pc.dst && at < pc.dst + pc.bytes) {
                                found = true;
                                CHECK(pc.src + (at - pc.dst) == src, "gate/up unit (%d, %d) of CTA %d from the wrong source", j, g, c);
                            }
                        }
                        CHECK(found, "gate/up unit (%d, %d) of CTA %d outside b1", j, g, c);
                    }
            CHECK(L.b3.bytes == ((lora && pl.shr >= 0) ? 2 * 16 * r * (pl.seg[pl.shr].hr1 - pl.seg[pl.shr].hr0) : 0),
                  "b3 bytes");
        }
        if (pl.dt >= 0) {
            // one unit per act group, in act order, then (LoRA) A_down and B_down rows
            int u = 0;
            for (int i = 0; i < L.b2.n; ++i) {
                const Piece1& pc = L.b2.pc[i];
                if (pc.kind != K1_DOWN) continue;
                CHECK(pc.dst == u * 576, "down unit %d at %d", u, pc.dst);
                const int per = (pc.seg < 0 ? Is : I) / 64;
                CHECK(pc.src == (long long)pl.dt * per * 576, "down tile source");
                CHECK(pc.seg == (u < K * (I / 64) ? u / (I / 64) : -1), "down unit %d slot %d", u, pc.seg);
                u += pc.bytes / 576;
            }
            CHECK(u == NA / 64, "down units %d != %d", u, NA / 64);
            if (lora) CHECK(L.ad == u * 576 && L.bd == L.ad + (Is / 64) * 2048 && L.b2.bytes == L.bd + 32 * r,
                            "LoRA down parts");
            else CHECK(L.b2.bytes == u * 576, "b2 bytes");
        } else {
            CHECK(L.b2.bytes == 0, "b2 without a tile");
        }
    }
    for (size_t i = 0; i < cov_rt.size(); ++i) CHECK(cov_rt[i] == 1, "%s routed hr %zu covered %d", name, i, cov_rt[i]);
    for (size_t i = 0; i < cov_sh.size(); ++i) CHECK(cov_sh[i] == 1, "%s shared hr %zu covered %d", name, i, cov_sh[i]);
    for (size_t i = 0; i < cov_act.size(); ++i) CHECK(cov_act[i] == 1, "%s act %zu published %d times", name, i, cov_act[i]);
    for (size_t i = 0; i < cov_dt.size(); ++i) CHECK(cov_dt[i] == 1, "%s output tile %zu: %d", name, i, cov_dt[i]);
    for (size_t i = 0; i < cov_r.size(); ++i) CHECK(cov_r[i] == 1, "%s router tile %zu: %d", name, i, cov_r[i]);
    for (size_t i = 0; i < cov_task.size(); ++i) CHECK(cov_task[i] == 1, "task %zu: %d", i, cov_task[i]);
    for (size_t i = 0; i < cov_la.size(); ++i) CHECK(cov_la[i] == (lora ? 1 : 0), "%s LoRA A group %zu: %d", name, i, cov_la[i]);
    // flush blocks with the one-hot rows of the extreme columns (0 and 2E - 1)
    std::vector<int> ids(2 * K);
    for (int q = 0; q < 2; ++q) {
        for (int i = 0; i < 2 * K; ++i) ids[i] = q ? (i < K ? E - 1 - i : 2 * E - 1 - (i - K)) : (i < K ? i : E + i - K);
        for (int j = 0; j < tph && n_heads; ++j)
            for (int h = 0; h < 2; ++h) {
                Block1 B;
                CHECK(flush_block(S, j, h, B, ids.data(), 2 * K), "flush block %d/%d", j, h);
                CHECK(flush_bytes(S, j, h, 2 * K) == B.bytes, "flush_bytes %d != %d", flush_bytes(S, j, h, 2 * K), B.bytes);
                CHECK(h == 0 || flush_bytes(S, j, h, K) == B.bytes - 32 * K, "flush_bytes without previous ids");
                CHECK(B.n <= 32, "more copies than producer lanes");
                Plan1 pl;
                plan1(S, 0, pl);
                check_block(S, pl, B, k.ring, "flush");
            }
    }
    // the two blocks of an fc1 task read the whole row tile of fc1 once
    if (n_heads) {
        Block1 A, B;
        flush_block(S, 0, 0, A);
        flush_block(S, 0, 1, B);
        CHECK(A.pc[0].bytes + B.pc[0].bytes == 32 * d, "fc1 row tile bytes");
    }
}

int main() {
    printf("shared-memory state %d bytes\n", kSm1Bytes);
    const int grids[] = {152, 148, 76, 32};
    for (int nct : grids) {
        const bool big = nct >= 128;   // d = 2048 needs 128 output row tiles
        check_shape("35B stack (33 heads)", 2048, 256, 4, 512, 512, 512, 16, true, true, 33, nct, big);
        check_shape("35B layer ring", 2048, 256, 4, 512, 512, 512, 16, true, true, 1, nct, big);
        check_shape("toy", 256, 16, 2, 128, 128, 64, 4, true, true, 1, nct, true);
        check_shape("35B no LoRA", 2048, 256, 4, 512, 512, 512, 16, true, false, 2, nct, big);
        check_shape("35B no shared", 2048, 256, 4, 512, 512, 512, 16, false, false, 0, nct, big);
        check_shape("8B shapes E=32 K=8", 1536, 32, 8, 512, 512, 512, 16, true, true, 2, nct, nct >= 96);
        check_shape("d=1536 K=2", 1536, 64, 2, 512, 256, 256, 8, true, true, 3, nct, nct >= 96);
        check_shape("35B E=16 (small)", 2048, 16, 4, 512, 512, 512, 16, true, true, 1, nct, big);
        check_shape("35B E=32 L=1 (no heads)", 2048, 32, 4, 512, 512, 512, 16, true, true, 0, nct, big);
    }
    if (fails) {
        printf("%d FAILURES\n", fails);
        return 1;
    }
    printf("ALL OK\n");
    return 0;
}
