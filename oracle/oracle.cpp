// Edge0 prerouted int4 MoE decode path -- CPU ORACLE (test infrastructure only).
//
// Plain single-threaded restatement, in fp64, of what the decode path computes.
// It is used by the tests, by the smoke check and by the bench's CPU-baseline leg;
// nothing in the product path links or calls it.  Each routine names the passage
// (page title + section) it follows; see oracle.h for the page list.
#include "oracle.h"

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <vector>

namespace {

// Affine group size of the int4 format [P1 S2 "Quantization": "int4 affine group-64"].
constexpr int kGroup = 64;

double h2d(uint16_t h) { return orc_half_to_double(h); }

}  // namespace

extern "C" {

// ---------------------------------------------------------------- fp16 -----
// IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
double orc_half_to_double(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1f;
    const int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = std::ldexp((double)f, -24);                      // subnormal: f * 2^-24
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = std::ldexp(1.0 + (double)f / 1024.0, e - 15);
    }
    return sign ? -v : v;
}

// Round to nearest, ties to even, directly from fp64 (no double rounding).
uint16_t orc_double_to_half(double v) {
    if (std::isnan(v)) return 0x7e00;
    const uint16_t sign = std::signbit(v) ? 0x8000 : 0;
    const double a = std::fabs(v);
    if (a >= 65520.0) return sign | 0x7c00;                  // rounds to infinity
    if (a < std::ldexp(1.0, -14)) {
        // subnormal range: spacing 2^-24; m == 1024 lands exactly on the smallest normal
        const double m = std::nearbyint(a * 16777216.0);
        return sign | (uint16_t)m;
    }
    int e2;
    const double fr = std::frexp(a, &e2);                    // a = fr * 2^e2, fr in [0.5, 1)
    int E = e2 - 1;                                          // a = (2 fr) * 2^E
    double m = std::nearbyint((2.0 * fr - 1.0) * 1024.0);    // exact product, RNE
    if (m >= 1024.0) { m = 0.0; E += 1; }
    if (E + 15 >= 31) return sign | 0x7c00;
    return sign | (uint16_t)(((E + 15) << 10) | (int)m);
}

// ---------------------------------------------------------------- int4 -----
// [P3 "Architectural Deep Dive": uint32 words holding eight 4-bit values,
//  layout [E, out, in/8]]; nibble order (low nibble = lowest input index) is
// the reading stated in the design notes.
void orc_int4_unpack(const uint32_t* packed, long n_words, uint8_t* nibbles) {
    for (long j = 0; j < n_words; ++j)
        for (int i = 0; i < 8; ++i) nibbles[8 * j + i] = (packed[j] >> (4 * i)) & 0xf;
}

void orc_int4_pack(const uint8_t* nibbles, long n_words, uint32_t* packed) {
    for (long j = 0; j < n_words; ++j) {
        uint32_t w = 0;
        for (int i = 0; i < 8; ++i) w |= (uint32_t)(nibbles[8 * j + i] & 0xf) << (4 * i);
        packed[j] = w;
    }
}

// w[o, i] = s[o, i/64] * q[o, i] + b[o, i/64]   [P1 S2; P3; P4 QuantSpec(mode="affine")]
void orc_int4_dequant(const orc_q4* m, double* w) {
    const int wpr = m->in / 8, gpr = m->in / kGroup;
    for (int o = 0; o < m->out; ++o)
        for (int i = 0; i < m->in; ++i) {
            const uint32_t word = m->q[(long)o * wpr + i / 8];
            const int q = (word >> (4 * (i % 8))) & 0xf;
            const double s = h2d(m->s[(long)o * gpr + i / kGroup]);
            const double b = h2d(m->b[(long)o * gpr + i / kGroup]);
            w[(long)o * m->in + i] = s * q + b;
        }
}

void orc_int4_matvec(const orc_q4* m, const double* v, double* y) {
    const int wpr = m->in / 8, gpr = m->in / kGroup;
    for (int o = 0; o < m->out; ++o) {
        double acc = 0.0;
        for (int i = 0; i < m->in; ++i) {
            const uint32_t word = m->q[(long)o * wpr + i / 8];
            const int q = (word >> (4 * (i % 8))) & 0xf;
            const double s = h2d(m->s[(long)o * gpr + i / kGroup]);
            const double b = h2d(m->b[(long)o * gpr + i / kGroup]);
            acc += (s * q + b) * v[i];
        }
        y[o] = acc;
    }
}

void orc_f16_matvec(const uint16_t* W, int out, int in, int ld, const double* v, double* y) {
    for (int o = 0; o < out; ++o) {
        double acc = 0.0;
        for (int i = 0; i < in; ++i) acc += h2d(W[(long)o * ld + i]) * v[i];
        y[o] = acc;
    }
}

// erf-GELU, the exact form 0.5 z (1 + erf(z / sqrt 2))  [P1 S3.2 "Head"; P4 gelu_erf]
double orc_gelu_erf(double z) { return 0.5 * z * (1.0 + std::erf(z / std::sqrt(2.0))); }

double orc_silu(double z) { return z / (1.0 + std::exp(-z)); }

// down(silu(gate(x)) * up(x))  [P1 S3.1 "Math contract"; P3 SwiGLU listing]
void orc_expert_swiglu(const orc_q4* gate, const orc_q4* up, const orc_q4* down,
                       const double* x, double* y) {
    const int I = gate->out;
    std::vector<double> g(I), u(I), a(I);
    orc_int4_matvec(gate, x, g.data());
    orc_int4_matvec(up, x, u.data());
    for (int i = 0; i < I; ++i) a[i] = orc_silu(g[i]) * u[i];
    orc_int4_matvec(down, a.data(), y);
}

// dy = (alpha / r) * B (A v)   [P1 S3.3 "Deployment keeps it unmerged"; P2 eq.]
void orc_lora_delta(const uint16_t* A, const uint16_t* B, int r, int in, int out,
                    double alpha, const double* v, double* dy) {
    std::vector<double> av(r);
    orc_f16_matvec(A, r, in, in, v, av.data());
    for (int o = 0; o < out; ++o) {
        double acc = 0.0;
        for (int j = 0; j < r; ++j) acc += h2d(B[(long)o * r + j]) * av[j];
        dy[o] = (alpha / r) * acc;
    }
}

// ------------------------------------------------------------- routing -----
// Plain selection: repeatedly take the largest remaining score, lower index first.
void orc_topk(const float* score, int n, int k, int32_t* idx) {
    std::vector<char> taken(n, 0);
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < n; ++e) {
            if (taken[e]) continue;
            if (best < 0 || score[e] > score[best]) best = e;
        }
        taken[best] = 1;
        idx[j] = best;
    }
}

// Softmax-topk with renormalisation  [P1 App. A "Softmax-topk"; P4 norm_topk_prob=True]
// g = softmax(l); inds = topk(g, K); w = g[inds] / sum_inds g.  softmax is monotone,
// so ranking g and ranking the fp32 logits pick the same experts.
void orc_route_softmax_topk(const float* logits, const float* bias, int E, int K,
                            int32_t* ids, float* w) {
    std::vector<float> l(E);
    for (int e = 0; e < E; ++e) l[e] = bias ? (float)(logits[e] + bias[e]) : logits[e];
    double mx = l[0];
    for (int e = 1; e < E; ++e) mx = std::fmax(mx, (double)l[e]);
    std::vector<double> g(E);
    double z = 0.0;
    for (int e = 0; e < E; ++e) { g[e] = std::exp((double)l[e] - mx); z += g[e]; }
    for (int e = 0; e < E; ++e) g[e] /= z;
    orc_topk(l.data(), E, K, ids);
    double sel = 0.0;
    for (int k = 0; k < K; ++k) sel += g[ids[k]];
    for (int k = 0; k < K; ++k) w[k] = (float)(g[ids[k]] / sel);
}

// Sigmoid-group  [P1 App. A "Sigmoid-group"; P1 S2 "MoE routing"]
void orc_route_sigmoid_group(const float* logits, const float* bias, int E, int K,
                             int n_groups, int G, float scale, int32_t* ids, float* w) {
    // sigma in fp32: the selection is decided in the precision the kernel uses
    std::vector<float> sig(E), sel(E);
    for (int e = 0; e < E; ++e) {
        sig[e] = (float)(1.0 / (1.0 + std::exp(-(double)logits[e])));
        sel[e] = bias ? (float)(sig[e] + bias[e]) : sig[e];
    }
    const int per = E / n_groups;
    std::vector<float> gscore(n_groups);
    for (int gi = 0; gi < n_groups; ++gi) {
        int32_t top2[2];
        orc_topk(sel.data() + gi * per, per, 2, top2);
        gscore[gi] = sel[gi * per + top2[0]] + sel[gi * per + top2[1]];
    }
    std::vector<int32_t> keep(G);
    orc_topk(gscore.data(), n_groups, G, keep.data());
    std::vector<float> masked(E, -INFINITY);
    for (int j = 0; j < G; ++j)
        for (int e = keep[j] * per; e < (keep[j] + 1) * per; ++e) masked[e] = sel[e];
    orc_topk(masked.data(), E, K, ids);
    double sum = 0.0;
    for (int k = 0; k < K; ++k) sum += sig[ids[k]];
    for (int k = 0; k < K; ++k) w[k] = (float)(scale * (double)sig[ids[k]] / (sum + 1e-20));
}

void orc_apply_route(const orc_route* r, const float* logits, int E, int K, int32_t* ids, float* w) {
    if (r->kind == ORC_ROUTE_SIGMOID_GROUP)
        orc_route_sigmoid_group(logits, r->bias, E, K, r->n_groups, r->topk_groups, r->scale,
                                ids, w);
    else
        orc_route_softmax_topk(logits, r->bias, E, K, ids, w);
}

// ---------------------------------------------------------------- head -----
// head(feats) = linear_init(feats) + fc2(gelu_erf(fc1(feats))),
// feats = concat[x, executed one-hot, previous one-hot], f_in = d + 2E
// [P1 S3.2 "Head"; P2 "Prerouter Head Architecture"; P4 PrerouterHead]
void orc_prerouter_logits(const uint16_t* fc1, const uint16_t* fc2, const uint16_t* linit,
                          int d, int E, int H, const uint16_t* x,
                          const int32_t* exec_ids, const int32_t* prev_ids, int K,
                          float* logits) {
    const int f_in = d + 2 * E;
    std::vector<double> feats(f_in, 0.0);
    for (int i = 0; i < d; ++i) feats[i] = h2d(x[i]);
    for (int k = 0; k < K; ++k) feats[d + exec_ids[k]] = 1.0;
    if (prev_ids)
        for (int k = 0; k < K; ++k) feats[d + E + prev_ids[k]] = 1.0;
    std::vector<double> z(H), g(H), o2(E), o1(E);
    orc_f16_matvec(fc1, H, f_in, f_in, feats.data(), z.data());
    for (int j = 0; j < H; ++j) g[j] = orc_gelu_erf(z[j]);
    orc_f16_matvec(fc2, E, H, H, g.data(), o2.data());
    orc_f16_matvec(linit, E, f_in, f_in, feats.data(), o1.data());
    for (int e = 0; e < E; ++e) logits[e] = (float)(o1[e] + o2[e]);
}

void orc_rmsnorm(const uint16_t* h, const uint16_t* gamma, int d, double eps, uint16_t* x) {
    double ss = 0.0;
    for (int i = 0; i < d; ++i) { const double v = h2d(h[i]); ss += v * v; }
    const double inv = 1.0 / std::sqrt(ss / d + eps);
    for (int i = 0; i < d; ++i)
        x[i] = orc_double_to_half(h2d(h[i]) * inv * (gamma ? h2d(gamma[i]) : 1.0));
}

// ----------------------------------------------------------------- MoE -----
namespace {

orc_q4 expert_mat(const uint32_t* q, const uint16_t* s, const uint16_t* b, int e, int out, int in) {
    orc_q4 m;
    m.q = q + (long)e * out * (in / 8);
    m.s = s + (long)e * out * (in / kGroup);
    m.b = b + (long)e * out * (in / kGroup);
    m.out = out;
    m.in = in;
    return m;
}

// routed part for one token: sum_k w_k expert_{ids_k}(x)
void routed_one(const orc_moe* m, const double* x, const int32_t* ids, const float* w, double* y) {
    std::vector<double> o(m->d);
    for (int i = 0; i < m->d; ++i) y[i] = 0.0;
    for (int k = 0; k < m->K; ++k) {
        const int e = ids[k];
        orc_q4 g = expert_mat(m->gate_q, m->gate_s, m->gate_b, e, m->I, m->d);
        orc_q4 u = expert_mat(m->up_q, m->up_s, m->up_b, e, m->I, m->d);
        orc_q4 dn = expert_mat(m->down_q, m->down_s, m->down_b, e, m->d, m->I);
        orc_expert_swiglu(&g, &u, &dn, x, o.data());
        for (int i = 0; i < m->d; ++i) y[i] += (double)w[k] * o[i];
    }
}

}  // namespace

void orc_moe_forward(const orc_moe* m, const uint16_t* x, const int32_t* ids, const float* w,
                     int B, uint16_t* y16, double* y) {
    std::vector<double> xv(m->d), yr(m->d), ys(m->d);
    for (int b = 0; b < B; ++b) {
        for (int i = 0; i < m->d; ++i) xv[i] = h2d(x[(long)b * m->d + i]);
        routed_one(m, xv.data(), ids + (long)b * m->K, w + (long)b * m->K, yr.data());
        if (m->sh_gate_q) {
            orc_q4 g = expert_mat(m->sh_gate_q, m->sh_gate_s, m->sh_gate_b, 0, m->Is, m->d);
            orc_q4 u = expert_mat(m->sh_up_q, m->sh_up_s, m->sh_up_b, 0, m->Is, m->d);
            orc_q4 dn = expert_mat(m->sh_down_q, m->sh_down_s, m->sh_down_b, 0, m->d, m->Is);
            orc_expert_swiglu(&g, &u, &dn, xv.data(), ys.data());
        } else {
            for (int i = 0; i < m->d; ++i) ys[i] = 0.0;
        }
        for (int i = 0; i < m->d; ++i) {
            const double v = yr[i] + ys[i];
            if (y) y[(long)b * m->d + i] = v;
            if (y16) y16[(long)b * m->d + i] = orc_double_to_half(v);
        }
    }
}

// -------------------------------------------------------------- layers -----
// One decode layer at step t (synthetic stack: attention is the identity):
//   x = RMSNorm(h); routing = upstream head's prediction made at t-1 (prerouted
//   layers, t > 0) or this layer's own router; h += routed experts + shared
//   expert with unmerged LoRA on its projections; the head owned by this layer
//   predicts its target layer's routing for t+1 from x and the executed and
//   previous one-hot masks.
// [P1 S3.2 "Motivation", "Head", "Prediction-as-routing", "Feature drift";
//  P1 S3.3; P1 Fig. 1 caption]
void orc_decode_layer(const orc_layer* layers, int l, orc_state* st, uint16_t* h, int t,
                      orc_record* rec) {
    const orc_layer* Ly = &layers[l];
    const orc_moe* m = &Ly->moe;
    const int d = m->d, E = m->E, K = m->K, B = st->B, L = st->L;
    const int cur = t & 1, prv = (t + 1) & 1;
    std::vector<uint16_t> x16(d);
    std::vector<double> x(d), yr(d), g, u, a, o(d), dl(d);
    std::vector<float> logits(E);
    for (int b = 0; b < B; ++b) {
        uint16_t* hb = h + (long)b * d;
        orc_rmsnorm(hb, Ly->gamma, d, Ly->eps, x16.data());
        for (int i = 0; i < d; ++i) x[i] = h2d(x16[i]);

        int32_t* ids = st->exec_ids + (((long)cur * L + l) * B + b) * K;
        std::vector<float> w(K);
        if (Ly->prerouted && t > 0) {
            const long p = (((long)prv * L + l) * B + b) * K;
            for (int k = 0; k < K; ++k) { ids[k] = st->pred_ids[p + k]; w[k] = st->pred_w[p + k]; }
        } else {
            std::vector<double> lg(E);
            orc_f16_matvec(Ly->router, E, d, d, x.data(), lg.data());
            for (int e = 0; e < E; ++e) logits[e] = (float)lg[e];
            orc_apply_route(&Ly->route, logits.data(), E, K, ids, w.data());
            if (rec && rec->router_logits)
                std::memcpy(rec->router_logits + ((long)l * B + b) * E, logits.data(), sizeof(float) * E);
        }

        routed_one(m, x.data(), ids, w.data(), yr.data());

        // shared expert with unmerged LoRA on gate, up and down
        const int Is = m->Is;
        g.assign(Is, 0.0); u.assign(Is, 0.0); a.assign(Is, 0.0);
        std::vector<double> ys(d, 0.0);
        if (m->sh_gate_q) {
            orc_q4 G = expert_mat(m->sh_gate_q, m->sh_gate_s, m->sh_gate_b, 0, Is, d);
            orc_q4 U = expert_mat(m->sh_up_q, m->sh_up_s, m->sh_up_b, 0, Is, d);
            orc_q4 D = expert_mat(m->sh_down_q, m->sh_down_s, m->sh_down_b, 0, d, Is);
            orc_int4_matvec(&G, x.data(), g.data());
            orc_int4_matvec(&U, x.data(), u.data());
            if (Ly->lora_Ag) {
                std::vector<double> dg(Is), du(Is);
                orc_lora_delta(Ly->lora_Ag, Ly->lora_Bg, Ly->r, d, Is, Ly->alpha, x.data(), dg.data());
                orc_lora_delta(Ly->lora_Au, Ly->lora_Bu, Ly->r, d, Is, Ly->alpha, x.data(), du.data());
                for (int i = 0; i < Is; ++i) { g[i] += dg[i]; u[i] += du[i]; }
            }
            for (int i = 0; i < Is; ++i) a[i] = orc_silu(g[i]) * u[i];
            orc_int4_matvec(&D, a.data(), ys.data());
            if (Ly->lora_Ad) {
                orc_lora_delta(Ly->lora_Ad, Ly->lora_Bd, Ly->r, Is, d, Ly->alpha, a.data(), dl.data());
                for (int i = 0; i < d; ++i) ys[i] += dl[i];
            }
        }
        for (int i = 0; i < d; ++i) hb[i] = orc_double_to_half(h2d(hb[i]) + yr[i] + ys[i]);

        if (Ly->fc1) {
            const int32_t* prev = t > 0 ? st->exec_ids + (((long)prv * L + l) * B + b) * K : nullptr;
            orc_prerouter_logits(Ly->fc1, Ly->fc2, Ly->linit, d, E, Ly->H, x16.data(), ids, prev,
                                 K, logits.data());
            const int tg = Ly->head_target;
            const long p = (((long)cur * L + tg) * B + b) * K;
            orc_apply_route(&layers[tg].route, logits.data(), E, K, st->pred_ids + p, st->pred_w + p);
            if (rec && rec->head_logits)
                std::memcpy(rec->head_logits + ((long)l * B + b) * E, logits.data(), sizeof(float) * E);
        }
        if (rec) {
            if (rec->x) std::memcpy(rec->x + ((long)l * B + b) * d, x16.data(), 2 * d);
            if (rec->ids) std::memcpy(rec->ids + ((long)l * B + b) * K, ids, 4 * K);
            if (rec->w) std::memcpy(rec->w + ((long)l * B + b) * K, w.data(), 4 * K);
            if (rec->hout) std::memcpy(rec->hout + ((long)l * B + b) * d, hb, 2 * d);
        }
    }
}

void orc_decode_step(const orc_layer* layers, orc_state* st, uint16_t* h, int t, orc_record* rec) {
    for (int l = 0; l < st->L; ++l) orc_decode_layer(layers, l, st, h, t, rec);
}

}  // extern "C"
