// C ABI entry points of libedge0: argument validation on the host, translation
// of the public descriptors into the engine's kernel parameter block, launch.
#include <stddef.h>
#include <string.h>

#include "internal.cuh"

using namespace edge0;

namespace {

bool al16(const void* p) { return ((uintptr_t)p & 15) == 0; }   // (null counts as aligned)

struct Dims {
    int d, E, K, I, Is, H, r;
};

int check_route(const edge0_route& r, int E, int K) {
    if (r.kind == EDGE0_ROUTE_SOFTMAX_TOPK) return EDGE0_OK;
    if (r.kind != EDGE0_ROUTE_SIGMOID_GROUP) return EDGE0_EINVAL;
    if (r.n_groups <= 0 || r.n_groups > 32 || E % r.n_groups) return EDGE0_EINVAL;
    if (E / r.n_groups < 2) return EDGE0_EINVAL;
    if (r.topk_groups <= 0 || r.topk_groups > r.n_groups) return EDGE0_EINVAL;
    if (K > r.topk_groups * (E / r.n_groups)) return EDGE0_EINVAL;
    return EDGE0_OK;
}

int check_dims(const Dims& D, int B, int max_b = EDGE0_MAX_BATCH) {
    if (B <= 0 || B > max_b) return EDGE0_EINVAL;
    if (D.d <= 0 || D.d % kGroup || D.I <= 0 || D.I % kGroup || D.Is <= 0 || D.Is % kGroup)
        return EDGE0_EINVAL;
    if (D.H <= 0 || D.H % kGroup) return EDGE0_EINVAL;
    if (D.E <= 0 || D.E > EDGE0_MAX_E || D.E % 16) return EDGE0_EINVAL;
    if (D.K <= 0 || D.K > EDGE0_MAX_K || D.K > D.E) return EDGE0_EINVAL;
    if (D.r <= 0 || D.r > 16) return EDGE0_EINVAL;
    return EDGE0_OK;
}

void route_into(const edge0_route& r, int* kind, int* ng, int* tg, float* sc, const float** bias) {
    *kind = r.kind;
    *ng = r.n_groups > 0 ? r.n_groups : 1;
    *tg = r.topk_groups > 0 ? r.topk_groups : 1;
    *sc = r.scale;
    *bias = r.bias;
}

// The kernel parameter block of a call (~32 KB): one per calling thread, reused
// by every call of that thread (no heap allocation per call; a call holds it
// only until it has enqueued its launches).
Prog* call_prog() {
    static thread_local Prog prog;
    return &prog;
}

int fill_layer(const edge0_layer_desc& Ld, const Dims& D, int Lstate, LayerP& P) {
    const edge0_moe_desc& m = Ld.moe;
    if (m.d != D.d || m.E != D.E || m.K != D.K || m.I != D.I || m.Is != D.Is) return EDGE0_EINVAL;
    if (!m.gate_up || !m.down || !Ld.router) return EDGE0_EINVAL;
    if (!al16(m.gate_up) || !al16(m.down) || !al16(Ld.router)) return EDGE0_EINVAL;
    if (m.slot_table && m.n_slots <= 0) return EDGE0_EINVAL;
    memset(&P, 0, sizeof(P));
    P.gu = (const char*)m.gate_up;
    P.down = (const char*)m.down;
    P.slot_table = m.slot_table;
    P.n_slots = m.slot_table ? m.n_slots : m.E;
    if ((m.host_gate_up != nullptr) != (m.host_down != nullptr)) return EDGE0_EINVAL;
    if (m.host_gate_up && (!m.slot_table || !al16(m.host_gate_up) || !al16(m.host_down))) return EDGE0_EINVAL;
    P.gu_host = (const char*)m.host_gate_up;
    P.down_host = (const char*)m.host_down;
    if (m.tier_counts && ((uintptr_t)m.tier_counts & 7)) return EDGE0_EINVAL;
    P.tier_counts = m.tier_counts;
    if (!al16(m.down_rows) || !al16(m.sh_down_rows)) return EDGE0_EINVAL;
    P.down_rows = (const char*)m.down_rows;
    P.sh_down_rows = (const char*)m.sh_down_rows;
    P.ready = (void*)Ld.ready;
    P.router = (const char*)Ld.router;
    P.gamma = (const __half*)Ld.gamma;
    if (Ld.gamma && ((uintptr_t)Ld.gamma & 7)) return EDGE0_EINVAL;
    P.eps = Ld.eps;
    int rc = check_route(Ld.route, D.E, D.K);
    if (rc) return rc;
    route_into(Ld.route, &P.route_kind, &P.n_groups, &P.topk_groups, &P.route_scale, &P.bias);
    int flags = 0;
    if (Ld.prerouted) flags |= LF_PREROUTED;
    if (m.sh_gate_up || m.sh_down) {
        if (!m.sh_gate_up || !m.sh_down) return EDGE0_EINVAL;
        if (!al16(m.sh_gate_up) || !al16(m.sh_down)) return EDGE0_EINVAL;
        P.sh_gu = (const char*)m.sh_gate_up;
        P.sh_down = (const char*)m.sh_down;
        flags |= LF_SHARED;
    }
    const edge0_lora_desc &lg = Ld.lora_gate, &lu = Ld.lora_up, &ld = Ld.lora_down;
    if (lg.A || lu.A || ld.A_T) {
        if (!(flags & LF_SHARED)) return EDGE0_EINVAL;
        if (!lg.A || !lu.A || !ld.A_T || !lg.B || !lu.B || !ld.B) return EDGE0_EINVAL;
        if (lg.r != D.r || lu.r != D.r || ld.r != D.r) return EDGE0_EINVAL;
        if (lg.in != D.d || lg.out != D.Is || lu.in != D.d || lu.out != D.Is || ld.in != D.Is ||
            ld.out != D.d)
            return EDGE0_EINVAL;
        if (lg.alpha != lu.alpha || lg.alpha != ld.alpha) return EDGE0_EINVAL;
        if (!al16(lg.A) || !al16(lu.A) || !al16(ld.A_T) || !al16(lg.B) || !al16(lu.B) || !al16(ld.B) ||
            !al16(ld.A))
            return EDGE0_EINVAL;
        P.lora_Ag = (const char*)lg.A;
        P.lora_Au = (const char*)lu.A;
        P.lora_AdT = (const __half*)ld.A_T;
        P.lora_Ad = (const char*)ld.A;   // optional: the batch-1 kernel needs it
        P.lora_Bg = (const __half*)lg.B;
        P.lora_Bu = (const __half*)lu.B;
        P.lora_Bd = (const __half*)ld.B;
        P.lora_scale = lg.alpha / (float)D.r;
        flags |= LF_LORA;
    }
    if (Ld.has_head) {
        const edge0_head_desc& h = Ld.head;
        if (h.d != D.d || h.E != D.E || h.H != D.H || h.K != D.K) return EDGE0_EINVAL;
        if (!h.fc1_dense || !h.fc1_oh_T || !h.fc2 || !h.linit_dense || !h.linit_oh_T)
            return EDGE0_EINVAL;
        if (!al16(h.fc1_dense) || !al16(h.fc1_oh_T) || !al16(h.fc2) || !al16(h.linit_dense) ||
            !al16(h.linit_oh_T))
            return EDGE0_EINVAL;
        if (Ld.head_target < 0 || Ld.head_target >= Lstate) return EDGE0_EINVAL;
        rc = check_route(h.route, D.E, D.K);
        if (rc) return rc;
        P.fc1 = (const char*)h.fc1_dense;
        P.fc1_oh = (const __half*)h.fc1_oh_T;
        P.fc2 = (const char*)h.fc2;
        P.linit = (const char*)h.linit_dense;
        P.linit_oh = (const __half*)h.linit_oh_T;
        route_into(h.route, &P.head_route_kind, &P.head_n_groups, &P.head_topk_groups,
                   &P.head_route_scale, &P.head_bias);
        P.head_target = Ld.head_target;
        flags |= LF_HEAD;
    }
    if (Ld.index < 0 || Ld.index >= Lstate) return EDGE0_EINVAL;
    P.sidx = Ld.index;
    P.flags = flags;
    return EDGE0_OK;
}

void set_dims(Prog& p, const Dims& D, int B) {
    p.B = B;
    p.d = D.d;
    p.E = D.E;
    p.K = D.K;
    p.I = D.I;
    p.Is = D.Is;
    p.H = D.H;
    p.r = D.r;
}

int check_ws(int Ls, const Dims& D, int B, const void* ws, size_t bytes) {
    if (!ws || !al16(ws)) return EDGE0_EINVAL;
    if ((long long)bytes < ws_layout(Ls, B, D.d, D.E).total) return EDGE0_EINVAL;
    return EDGE0_OK;
}

int decode_common(const edge0_layer_desc* layers, int L, uint16_t* h, edge0_route_state* st, int B,
                  int step, cudaStream_t stream) {
    if (!layers || !h || !st || L <= 0 || L > EDGE0_MAX_LAYERS) return EDGE0_EINVAL;
    if (!st->pred_ids || !st->pred_w || !st->exec_ids) return EDGE0_EINVAL;
    if (st->B != B || st->L <= 0 || st->K != layers[0].moe.K) return EDGE0_EINVAL;
    if (!al16(h)) return EDGE0_EINVAL;
    Dims D;
    D.d = layers[0].moe.d;
    D.E = layers[0].moe.E;
    D.K = layers[0].moe.K;
    D.I = layers[0].moe.I;
    D.Is = layers[0].moe.Is;
    // every head of one call has one width, every LoRA one rank
    D.H = 64;
    D.r = 16;
    for (int l = 0; l < L; ++l)
        if (layers[l].has_head) { D.H = layers[l].head.H; break; }
    for (int l = 0; l < L; ++l)
        if (layers[l].lora_gate.A) { D.r = layers[l].lora_gate.r; break; }
    const bool batched = B > EDGE0_MAX_BATCH;
    int rc = check_dims(D, B, batched ? EDGE0_MAX_BATCHED : EDGE0_MAX_BATCH);
    if (rc) return rc;
    if (batched) {
        // the batched path: explicit steps, d in halves of whole groups
        if (step < 0 || D.d % 128) return EDGE0_EINVAL;
        const int Imax = D.I > D.Is ? D.I : D.Is;
        if (!st->workspace || !al16(st->workspace) ||
            (long long)st->workspace_bytes < batch_ws_layout(st->L, B, D.d, D.E, D.K, Imax, D.H).total)
            return EDGE0_EINVAL;
    } else {
        rc = check_ws(st->L, D, B, st->workspace, st->workspace_bytes);
        if (rc) return rc;
    }
    static_assert(sizeof(Prog) <= 32000, "kernel parameter block too large");
    Prog* p = call_prog();
    memset(p, 0, sizeof(Prog));
    p->mode = MODE_DECODE;
    p->L = L;
    set_dims(*p, D, B);
    p->step = step;
    p->h_io = (__half*)h;
    p->pred_ids = st->pred_ids;
    p->pred_w = st->pred_w;
    p->exec_ids = st->exec_ids;
    p->Ls = st->L;
    p->ws = (char*)st->workspace;
    p->ws_bytes = (long long)st->workspace_bytes;
    if (B == 1) {
        p->dbg_h = (__half*)st->record_h;
        p->dbg_logits = st->record_logits;
    }
    for (int l = 0; l < L && rc == EDGE0_OK; ++l) rc = fill_layer(layers[l], D, st->L, p->layers[l]);
    if (rc == EDGE0_OK) {
        if (batched) rc = batch_decode(*p, stream);
        else if (B == 1 && decode1_check(*p) == EDGE0_OK) rc = decode1_launch(*p, stream);
        else rc = engine_launch(*p, stream);
    }
    return rc;
}

}  // namespace

extern "C" const char* edge0_status_string(int status) {
    switch (status) {
        case EDGE0_OK: return "ok";
        case EDGE0_EINVAL: return "invalid argument";
        case EDGE0_ECUDA: return "CUDA runtime error";
        case EDGE0_ETIMEOUT: return "a bounded device wait timed out";
        case EDGE0_EUNSUPPORTED: return "shape not supported by this build";
        default: return "unknown status";
    }
}

extern "C" size_t edge0_workspace_bytes(int L, int B, int d, int E) {
    if (L <= 0 || B <= 0 || d <= 0 || E <= 0) return 0;
    return (size_t)ws_layout(L, B, d, E).total;
}

extern "C" size_t edge0_decode_workspace_bytes(int L, int B, int d, int E, int K, int I, int Is, int H) {
    if (L <= 0 || B <= 0 || d <= 0 || E <= 0 || K <= 0 || I <= 0 || Is <= 0 || H <= 0) return 0;
    if (B == 1) {
        // one sequence: room for the batch-1 kernel's layout too
        const long long n = ws_layout(L, B, d, E).total, n1 = decode1_ws_bytes(L, d, E, K, I, Is);
        return (size_t)(n > n1 ? n : n1);
    }
    if (B <= EDGE0_MAX_BATCH) return (size_t)ws_layout(L, B, d, E).total;
    if (B > EDGE0_MAX_BATCHED) return 0;
    return (size_t)batch_ws_layout(L, B, d, E, K, I > Is ? I : Is, H).total;
}

extern "C" int edge0_state_init(edge0_route_state* st, cudaStream_t stream) {
    if (!st || !st->pred_ids || !st->pred_w || !st->exec_ids || !st->workspace) return EDGE0_EINVAL;
    if (st->L <= 0 || st->B <= 0 || st->K <= 0) return EDGE0_EINVAL;
    const size_t n = (size_t)2 * st->L * st->B * st->K;
    if (cudaMemsetAsync(st->pred_ids, 0, n * 4, stream) != cudaSuccess) return EDGE0_ECUDA;
    if (cudaMemsetAsync(st->pred_w, 0, n * 4, stream) != cudaSuccess) return EDGE0_ECUDA;
    if (cudaMemsetAsync(st->exec_ids, 0, n * 4, stream) != cudaSuccess) return EDGE0_ECUDA;
    if (cudaMemsetAsync(st->workspace, 0, st->workspace_bytes, stream) != cudaSuccess)
        return EDGE0_ECUDA;
    return EDGE0_OK;
}

extern "C" int edge0_state_error(const edge0_route_state* st, cudaStream_t stream, int* status) {
    if (!st || !st->workspace || !status) return EDGE0_EINVAL;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return EDGE0_ECUDA;
    WsHeader h;
    if (cudaMemcpy(&h, st->workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
        return EDGE0_ECUDA;
    *status = h.error;
    if (h.error || h.abort) {
        // a launch that gave up leaves its accumulators, counters and barrier
        // count part-way: the whole state starts again from zero
        edge0_route_state s2 = *st;
        if (edge0_state_init(&s2, stream) != EDGE0_OK) return EDGE0_ECUDA;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return EDGE0_ECUDA;
    }
    return EDGE0_OK;
}

extern "C" int edge0_state_set_wait_limit(edge0_route_state* st, unsigned long long wait_ns,
                                          cudaStream_t stream) {
    if (!st || !st->workspace || st->workspace_bytes < sizeof(WsHeader)) return EDGE0_EINVAL;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return EDGE0_ECUDA;
    char* dst = (char*)st->workspace + offsetof(WsHeader, wait_ns);
    if (cudaMemcpy(dst, &wait_ns, sizeof(wait_ns), cudaMemcpyHostToDevice) != cudaSuccess) return EDGE0_ECUDA;
    return EDGE0_OK;
}

extern "C" int edge0_decode_layer(const edge0_layer_desc* layer, uint16_t* h_inout,
                                  edge0_route_state* st, int B, int step, cudaStream_t stream) {
    return decode_common(layer, 1, h_inout, st, B, step, stream);
}

extern "C" int edge0_decode_step(const edge0_layer_desc* layers, int L, uint16_t* h_inout,
                                 edge0_route_state* st, int B, int step, cudaStream_t stream) {
    return decode_common(layers, L, h_inout, st, B, step, stream);
}

extern "C" size_t edge0_prefill_workspace_bytes(int T, int d, int E, int K, int I, int Is) {
    if (T <= 0 || T > kMaxPrefill || d <= 0 || E <= 0 || K <= 0 || I <= 0 || Is <= 0) return 0;
    return (size_t)batch_ws_layout(1, T, d, E, K, I > Is ? I : Is, 16).total;
}

extern "C" int edge0_prefill(const edge0_layer_desc* layers, int L, uint16_t* h, int T, int32_t* ids_out,
                             unsigned flags, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (flags & ~EDGE0_PREFILL_TCGEN05_GATE_UP) return EDGE0_EINVAL;
    if (!layers || !h || L <= 0 || L > EDGE0_MAX_LAYERS || T <= 0 || T > kMaxPrefill) return EDGE0_EINVAL;
    if (!al16(h) || !workspace || !al16(workspace) || ((uintptr_t)ids_out & 3)) return EDGE0_EINVAL;
    Dims D;
    D.d = layers[0].moe.d;
    D.E = layers[0].moe.E;
    D.K = layers[0].moe.K;
    D.I = layers[0].moe.I;
    D.Is = layers[0].moe.Is;
    D.H = 64;
    D.r = 16;
    for (int l = 0; l < L; ++l)
        if (layers[l].lora_gate.A) { D.r = layers[l].lora_gate.r; break; }
    int rc = check_dims(D, T, kMaxPrefill);
    if (rc) return rc;
    if (D.d % 128) return EDGE0_EINVAL;
    const size_t need = edge0_prefill_workspace_bytes(T, D.d, D.E, D.K, D.I, D.Is);
    if (need == 0 || workspace_bytes < need) return EDGE0_EINVAL;
    Prog* p = call_prog();
    memset(p, 0, sizeof(Prog));
    p->mode = MODE_PREFILL;
    p->L = L;
    set_dims(*p, D, T);
    p->h_io = (__half*)h;
    p->Ls = L;
    p->ws = (char*)workspace;
    p->ws_bytes = (long long)workspace_bytes;
    for (int l = 0; l < L && rc == EDGE0_OK; ++l) {
        // a prefill reads no route state: a layer's state row is not used
        edge0_layer_desc Ld = layers[l];
        Ld.index = 0;
        Ld.has_head = 0;     // nor a head: the prerouter is not used at prefill
        rc = fill_layer(Ld, D, 1, p->layers[l]);
        if (rc == EDGE0_OK && (p->layers[l].slot_table || p->layers[l].gu_host)) rc = EDGE0_EINVAL;
    }
    if (rc == EDGE0_OK) {
        // the header (error word) and the layer-output accumulators start at zero
        const BatchWs W = batch_ws_layout(1, T, D.d, D.E, D.K, D.I > D.Is ? D.I : D.Is, 16);
        if (cudaMemsetAsync(workspace, 0, kWsHeaderBytes, stream) != cudaSuccess ||
            cudaMemsetAsync((char*)workspace + W.y, 0, (size_t)T * D.d * 4, stream) != cudaSuccess)
            rc = EDGE0_ECUDA;
    }
    p->tc_gu = (flags & EDGE0_PREFILL_TCGEN05_GATE_UP) ? 1 : 0;
    if (rc == EDGE0_OK) rc = batch_prefill(*p, ids_out, stream);
    return rc;
}

extern "C" int edge0_moe_int4_forward(const edge0_moe_desc* moe, const uint16_t* x,
                                      const int32_t* ids, const float* w, int B, uint16_t* y,
                                      void* workspace, size_t workspace_bytes,
                                      cudaStream_t stream) {
    if (!moe || !x || !ids || !w || !y) return EDGE0_EINVAL;
    if (!moe->gate_up || !moe->down) return EDGE0_EINVAL;
    if (!al16(x) || !al16(y)) return EDGE0_EINVAL;
    Dims D{moe->d, moe->E, moe->K, moe->I, moe->Is > 0 ? moe->Is : 64, 64, 16};
    int rc = check_dims(D, B);
    if (rc) return rc;
    rc = check_ws(1, D, B, workspace, workspace_bytes);
    if (rc) return rc;
    edge0_layer_desc L;
    memset(&L, 0, sizeof(L));
    L.moe = *moe;
    L.moe.Is = D.Is;
    L.router = moe->gate_up;   // not used in this mode; satisfies the layer check
    L.route.kind = EDGE0_ROUTE_SOFTMAX_TOPK;
    Prog* p = call_prog();
    memset(p, 0, sizeof(Prog));
    p->mode = MODE_MOE;
    p->L = 1;
    set_dims(*p, D, B);
    p->step = -1;   // alternate the workspace's parities call by call
    p->x_in = (const __half*)x;
    p->ids_in = ids;
    p->w_in = w;
    p->y_out = (__half*)y;
    p->Ls = 1;
    p->ws = (char*)workspace;
    rc = fill_layer(L, D, 1, p->layers[0]);
    if (rc == EDGE0_OK) rc = engine_launch(*p, stream);
    return rc;
}

extern "C" int edge0_prerouter_topk(const edge0_head_desc* head, const uint16_t* x,
                                    const int32_t* exec_ids, const int32_t* prev_ids, int B,
                                    int32_t* out_ids, float* out_w, float* out_logits,
                                    void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!head || !x || !exec_ids || !out_ids || !out_w) return EDGE0_EINVAL;
    if (!al16(x)) return EDGE0_EINVAL;
    Dims D{head->d, head->E, head->K, 64, 64, head->H, 16};
    int rc = check_dims(D, B);
    if (rc) return rc;
    rc = check_ws(1, D, B, workspace, workspace_bytes);
    if (rc) return rc;
    edge0_layer_desc L;
    memset(&L, 0, sizeof(L));
    L.moe.d = D.d;
    L.moe.E = D.E;
    L.moe.K = D.K;
    L.moe.I = D.I;
    L.moe.Is = D.Is;
    L.moe.gate_up = L.moe.down = head->fc2;   // not used in this mode
    L.router = head->fc2;
    L.route.kind = EDGE0_ROUTE_SOFTMAX_TOPK;
    L.has_head = 1;
    L.head = *head;
    L.head_target = 0;
    Prog* p = call_prog();
    memset(p, 0, sizeof(Prog));
    p->mode = MODE_HEAD;
    p->L = 1;
    set_dims(*p, D, B);
    p->step = -1;
    p->x_in = (const __half*)x;
    p->exec_in = exec_ids;
    p->prev_in = prev_ids;
    p->out_ids = out_ids;
    p->out_w = out_w;
    p->out_logits = out_logits;
    p->Ls = 1;
    p->ws = (char*)workspace;
    rc = fill_layer(L, D, 1, p->layers[0]);
    if (rc == EDGE0_OK) rc = engine_launch(*p, stream);
    return rc;
}
