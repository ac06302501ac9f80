// Host-side check of the persistent engine's work split (no GPU needed): for
// layer shapes of every kind and several grids, the pair plans and copy items
// that the producer warps would build, and the head flush's task tables.
// Checked: every half-row tile, LoRA A unit, B_down row tile, router unit and
// head task is owned exactly once; every copy item stays inside its source
// matrix and its ring; LoRA work sits on the pairs that own shared rows.
// Compiled and run by tests/test_engine_plan.py; exits non-zero on a failure.
#include "engine.cu"
#include <cstdio>
#include <vector>
#include <set>

using namespace edge0;

static int fails = 0;
#define CHECK(c, ...) do { if (!(c)) { ++fails; if (fails < 20) { printf("FAIL %s:%d ", __FILE__, __LINE__); printf(__VA_ARGS__); printf("\n"); } } } while (0)

void check_shape(const char* name, int d, int E, int K, int I, int Is, int H, int r, int B, bool shared,
                 bool lora, bool head, bool router, int nct) {
    Prog p;
    memset(&p, 0, sizeof(p));
    p.mode = MODE_DECODE; p.L = 1; p.B = B; p.K = K; p.d = d; p.E = E; p.I = I; p.Is = Is; p.H = H; p.r = r;
    p.layers[0].flags = (shared ? LF_SHARED : 0) | (lora ? LF_LORA : 0) | (head ? LF_HEAD : 0) | (router ? 0 : LF_PREROUTED);
    p.step = router ? 0 : 1;
    int smem = 0;
    int rc = engine_check(p, nct, 232448 - 1024, &smem);
    printf("%-28s rc=%d smem=%d ring=%d hr_max=%d q_max=%d slots=%d\n", name, rc, smem, p.ring_bytes, p.hr_max, p.q_max, p.slots_max);
    // the full GB300 grid takes every shape; a smaller grid may refuse one
    // whose items do not fit the ring (a recorded EDGE0_EUNSUPPORTED, no launch)
    CHECK(rc == 0 || (rc == EDGE0_EUNSUPPORTED && nct < 148), "engine_check %d", rc);
    if (rc) return;
    CHECK(smem <= 232448 - 1024, "smem");
    const Shape S = layer_shape(p, 0, router);
    const int P = nct / 2;
    const int hpe = I / 8, n_sh = shared ? Is / 8 : 0;
    std::vector<int> cov_sh(n_sh, 0), cov_rt(p.slots_max * hpe, 0);
    std::vector<int> cov_head(H / 16 + E / 16, 0);
    const int n_gd = d / 64;
    int max_items = 0, max_bytes = 0, max_held = 0;
    for (int pair = 0; pair < P; ++pair) {
        PairPlan ref;
        for (int rank = 0; rank < 2; ++rank) {
            LayerTab T;
            int lin = 0;
            bool ok = build_items(S, P, pair, rank, p.ring_bytes, &T, lin);
            CHECK(ok, "build_items pair %d rank %d", pair, rank);
            const PairPlan& pl = T.pl;
            if (rank == 0) ref = pl;
            else {
                CHECK(ref.n_hr == pl.n_hr && ref.nseg == pl.nseg && ref.has_sh == pl.has_sh,
                      "pair plans differ between ranks");
            }
            CHECK(pl.n_hr <= p.hr_max && pl.n_q <= p.q_max, "maxima");
            if (rank == 0) {
                for (int s = 0; s < pl.nseg; ++s) {
                    const Seg& g = pl.seg[s];
                    for (int h = g.hr0; h < g.hr1; ++h) {
                        if (g.slot < 0) cov_sh[h]++;
                        else cov_rt[g.slot * hpe + h]++;
                    }
                    CHECK(g.q0 == g.hr0 / 2 && g.q1 == (g.hr1 + 1) / 2, "quarters");
                }
            }
            // items: ring placement and source bounds
            const Halves hv = halves(d, E, rank);
            long long held = 0;
            int tot_units_router = 0;
            for (int i = 0; i < T.n; ++i) {
                const Item& it = T.it[i];
                CHECK(it.bytes > 0 && it.bytes <= kItemMax && it.bytes % 16 == 0, "item bytes %d", it.bytes);
                CHECK(it.off % 16 == 0 && it.off + it.bytes <= p.ring_bytes, "item ring placement");
                if (it.bytes > max_bytes) max_bytes = it.bytes;
                long long lo = 0, hi = 0, lim = 0;   // source byte range and buffer size
                const int n_rtd = d / 16, ngh = hv.gh1 - hv.gh0, nrt = hv.rt1 - hv.rt0;
                auto half0 = [&](int tiles) { return (long long)rank * tiles * (n_gd / 2); };
                const int Iexp = (it.kind == IT_GU || it.kind == IT_DQ || it.kind == IT_DQS || it.kind == IT_DSC) &&
                                 T.pl.seg[it.seg].slot < 0 ? Is : I;
                const long long dgrp = (long long)it.a * n_rtd * kQ4Unit + (long long)rank * (n_rtd / 2) * kQ4Unit;
                switch (it.kind) {
                    case IT_ROUTER: lo = (half0(E / 16) + it.b) * kF16Unit; lim = f16_bytes(E, d);
                        CHECK(it.b + it.n <= (E / 16) * ngh, "router units"); break;
                    case IT_GU: lo = (half0(Iexp / 8) + it.b) * kQ4Unit; lim = q4_bytes(2 * Iexp, d);
                        CHECK(it.b + it.n <= (Iexp / 8) * ngh, "gu units"); break;
                    case IT_LA: case IT_LU: lo = (half0(1) + it.b) * kF16Unit; lim = f16_bytes(r, d);
                        CHECK(it.b + it.n <= ngh, "lora units"); break;
                    case IT_BG: case IT_BU: lo = (long long)it.a * r * 2; lim = (long long)Is * r * 2; break;
                    case IT_DQ: case IT_DQS: lo = dgrp + (long long)it.b * nrt * kQ4Quarter; lim = q4_bytes(d, Iexp);
                        CHECK(lo + it.bytes <= dgrp + (long long)nrt * kQ4Unit, "down run past the half");
                        CHECK(it.b + it.n <= 4, "steps"); break;
                    case IT_DSC: lo = dgrp + 4LL * nrt * kQ4Quarter; lim = q4_bytes(d, Iexp);
                        CHECK(lo + it.bytes == dgrp + (long long)nrt * kQ4Unit, "scales"); break;
                    case IT_ADT: lo = (long long)it.a * r * 2; lim = (long long)Is * r * 2; break;
                    case IT_BD: lo = (long long)it.a * r * 2; lim = (long long)d * r * 2; break;
                    case IT_FC1: lo = (half0(H / 16) + it.b) * kF16Unit; lim = f16_bytes(H, d);
                        CHECK(it.b + it.n <= (H / 16) * ngh, "fc1 units"); break;
                    case IT_FC2: lo = ((long long)it.a * (E / 16) + it.b) * kF16Step; lim = f16_bytes(E, H);
                        CHECK(it.b + it.n <= E / 16, "fc2 rows"); break;
                    default: lo = (half0(E / 16) + it.b) * kF16Unit; lim = f16_bytes(E, d);
                        CHECK(it.b + it.n <= (E / 16) * ngh, "linit units"); break;
                }
                hi = lo + it.bytes;
                CHECK(lo >= 0 && hi <= lim, "item kind %d source [%lld, %lld) outside %lld", it.kind, lo, hi, lim);
                if (i >= T.p1 && i < T.p3 && !unit_kind(it.kind)) held += it.bytes;
            }
            CHECK(held + kItemMax <= p.ring_bytes, "held bytes");
            // LA items come first in P1
            for (int i = T.p1; i < T.n; ++i)
                if (T.it[i].kind == IT_LA || T.it[i].kind == IT_LU)
                    for (int j = T.p1; j < i; ++j)
                        CHECK(T.it[j].kind == IT_LA || T.it[j].kind == IT_LU, "LA item after another kind");
            if (held > max_held) max_held = (int)held;
            if (T.n > max_items) max_items = T.n;
            (void)tot_units_router;
        }
    }
    for (int h = 0; h < n_sh; ++h) CHECK(cov_sh[h] == 1, "shared hr %d covered %d times", h, cov_sh[h]);
    for (size_t h = 0; h < cov_rt.size(); ++h) CHECK(cov_rt[h] == 1, "routed hr %zu covered %d times", h, cov_rt[h]);
    // LoRA A units and B_down row tiles per rank: each exactly once, on the
    // pairs that own shared rows
    if (lora && shared) for (int rank = 0; rank < 2; ++rank) {
        const Halves hv = halves(d, E, rank);
        const int ngh = hv.gh1 - hv.gh0, nrt = hv.rt1 - hv.rt0;
        std::vector<int> cla(2 * ngh, 0), cbd(nrt, 0);
        for (int pair = 0; pair < P; ++pair) {
            PairPlan pl; pair_plan(S, P, pair, rank, pl);
            if (pl.la1 > pl.la0) CHECK(pair < S.ps, "LoRA A units on routed pair %d", pair);
            if (pl.bd1 > pl.bd0) CHECK(pair < S.ps, "B_down rows on routed pair %d", pair);
            for (int u = pl.la0; u < pl.la1; ++u) cla[u]++;
            for (int u = pl.bd0; u < pl.bd1; ++u) cbd[u]++;
        }
        for (int u = 0; u < 2 * ngh; ++u) CHECK(cla[u] == 1, "LoRA A unit %d covered %d", u, cla[u]);
        for (int u = 0; u < nrt; ++u) CHECK(cbd[u] == 1, "B_down row tile %d covered %d", u, cbd[u]);
    }
    printf("    ps=%d (P=%d)\n", S.ps, P);
    // router coverage per rank
    if (router) for (int rank = 0; rank < 2; ++rank) {
        const Halves hv = halves(d, E, rank);
        std::vector<int> cov((E / 16) * (hv.gh1 - hv.gh0), 0);
        for (int pair = 0; pair < P; ++pair) {
            PairPlan pl; pair_plan(S, P, pair, rank, pl);
            for (int u = pl.ru0; u < pl.ru1; ++u) cov[u]++;
        }
        for (size_t u = 0; u < cov.size(); ++u) CHECK(cov[u] == 1, "router unit %zu rank %d covered %d", u, rank, cov[u]);
    }
    printf("    max items %d, max item bytes %d, max held %d\n", max_items, max_bytes, max_held);
}

void check_flush(const char* name, int mode, int L, int d, int E, int K, int H, int B, int nct) {
    Prog p;
    memset(&p, 0, sizeof(p));
    p.mode = mode; p.L = L; p.B = B; p.K = K; p.d = d; p.E = E; p.I = 512; p.Is = 512; p.H = H; p.r = 16;
    for (int l = 0; l < L; ++l) {
        p.layers[l].flags = LF_SHARED | LF_LORA | (l >= 6 && l <= 38 ? LF_HEAD : 0);
        p.layers[l].sidx = l;
    }
    int smem = 0;
    const int rc = engine_check(p, nct, 232448 - 1024, &smem);
    CHECK(rc == 0 || (rc == EDGE0_EUNSUPPORTED && nct < 148), "%s engine_check %d", name, rc);
    if (rc) {
        printf("%-28s grid %d: unsupported\n", name, nct);
        return;
    }
    const int nh = n_heads(p), nt = head_tasks(p), nH = H / 16, nE = E / 16, hn0 = d / 128;
    std::vector<int> cov(nh * nt, 0);
    int max_tabs = 0, max_items = 0;
    for (int cta = 0; cta < nct; ++cta) {
        int lin = 0, j = 0, hl, t0, t1;
        for (; flush_table(p, nct, cta, j, &hl, &t0, &t1); ++j) {
            CHECK(is_head_layer(p, hl) && t0 < t1 && t1 <= nt && t1 - t0 <= p.ft, "table");
            int hi = 0;
            for (int l = 0; l < hl; ++l) hi += is_head_layer(p, l);
            for (int t = t0; t < t1; ++t) cov[hi * nt + t]++;
            LayerTab T;
            CHECK(build_flush_items(p, hl, t0, t1, p.ring_bytes, &T, lin), "build_flush_items");
            if (T.n > max_items) max_items = T.n;
            long long held = 0;
            for (int i = 0; i < T.n; ++i) {
                const Item& it = T.it[i];
                CHECK(it.off % 16 == 0 && it.off + it.bytes <= p.ring_bytes && it.bytes <= kItemMax, "ring");
                long long lo, lim;
                if (it.kind == IT_FC1) { lo = ((long long)it.seg * nH * hn0 + it.b) * 2048; lim = (long long)H * d * 2;
                    CHECK(it.b + it.n <= nH * hn0 && (it.b / hn0) == it.a && (it.b + it.n - 1) / hn0 == it.a, "fc1 units"); }
                else if (it.kind == IT_LINIT) { lo = ((long long)it.seg * nE * hn0 + it.b) * 2048; lim = (long long)E * d * 2;
                    CHECK((it.b / hn0) == it.a && (it.b + it.n - 1) / hn0 == it.a, "linit units"); }
                else { CHECK(it.kind == IT_FC2 && i >= T.p2, "fc2 order"); lo = ((long long)it.a * nE + it.b) * 512; lim = (long long)E * H * 2; held += it.bytes; }
                CHECK(lo >= 0 && lo + it.bytes <= lim, "flush source");
                CHECK(it.seg == 0 || it.seg == 1, "half");
            }
            CHECK(held + kItemMax <= p.ring_bytes, "flush held");
        }
        if (j > max_tabs) max_tabs = j;
    }
    for (int i = 0; i < nh * nt; ++i) CHECK(cov[i] == 1, "%s flush task %d covered %d", name, i, cov[i]);
    printf("%-28s heads %d tasks/head %d ft %d max tables/CTA %d max items %d\n", name, nh, nt, p.ft, max_tabs, max_items);
}

int main() {
    for (int nct : {152, 148, 76, 32}) {
        check_flush("flush 35b stack", MODE_DECODE, 40, 2048, 256, 4, 512, 1, nct);
        check_flush("flush 35b stack B=4", MODE_DECODE, 40, 2048, 256, 4, 512, 4, nct);
        check_flush("flush 8b", MODE_DECODE, 24, 1536, 128, 8, 512, 2, nct);
        check_flush("flush head-only", MODE_HEAD, 1, 2048, 256, 4, 512, 1, nct);
        check_flush("flush toy", MODE_DECODE, 40, 256, 16, 2, 64, 3, nct);
    }
    for (int nct : {152, 148, 76, 32}) {
        printf("--- grid %d\n", nct);
        check_shape("35b prerouted head+lora", 2048, 256, 4, 512, 512, 512, 16, 1, true, true, true, false, nct);
        check_shape("35b own-routed", 2048, 256, 4, 512, 512, 512, 16, 1, true, true, false, true, nct);
        check_shape("35b B=4", 2048, 256, 4, 512, 512, 512, 16, 4, true, true, true, true, nct);
        check_shape("8b B=1", 1536, 128, 8, 512, 512, 512, 16, 1, true, true, true, true, nct);
        check_shape("8b B=2", 1536, 128, 8, 512, 512, 512, 16, 2, true, true, true, false, nct);
        check_shape("toy", 256, 16, 2, 128, 128, 64, 4, 1, true, true, true, true, nct);
        check_shape("toy B=3", 256, 16, 2, 128, 128, 64, 4, 3, true, true, true, true, nct);
        check_shape("moe no shared", 2048, 32, 4, 512, 512, 64, 16, 2, false, false, false, false, nct);
        check_shape("35b lora no head", 2048, 256, 4, 512, 512, 512, 16, 1, true, true, false, false, nct);
        check_shape("35b B=4 r=4", 2048, 256, 4, 512, 512, 512, 4, 4, true, true, true, false, nct);
        check_shape("r=1", 256, 16, 2, 128, 128, 64, 1, 2, true, true, true, false, nct);
    }
    printf("%s (%d failures)\n", fails ? "FAILED" : "ALL OK", fails);
    return fails != 0;
}
