/*
 * Edge0 prerouted int4 MoE decode path -- CPU ORACLE (test infrastructure only).
 *
 * A plain, single-threaded, slow and obviously correct restatement of what the
 * decode hot path computes, in fp64.  It shares no code, header, table or helper
 * with the CUDA library; only tests, the smoke check and the bench's CPU-baseline
 * leg may load it.
 *
 * Sources (page title + section):
 *   [P1] "The Other Half of the Memory Wall: Serving 35B MoEs from SSD with Trained
 *        Routing Prediction" (arXiv HTML): S2 "MoE routing", S3.1 "Math contract",
 *        S3.2 "Head" / "Prediction-as-routing" / "Feature drift", S3.3, App. A.
 *   [P2] the reading guide of the same paper: "Prerouter Head Architecture" and
 *        "Unmerged Adapter Execution" equations.
 *   [P3] "Inside Edge0-35B": "Architectural Deep Dive: MoE Tensor Math and Packing".
 *   [P4] "Edge0 streams a 35B MoE off SSD. I counted the bytes it can't stream.":
 *        the PrerouterHead class and "Counting the bytes".
 *
 * Conventions
 *   fp16 values are passed as their IEEE binary16 bit patterns (uint16_t).
 *   int4 matrices use the pages' MLX affine layout: packed uint32 [out, in/8]
 *   (nibble i of word j = input element 8j+i, low nibble first), scales and
 *   biases [out, in/64]; w = s*q + b.
 *   Every routine runs on one thread and allocates only with malloc/free.
 */
#ifndef EDGE0_ORACLE_H
#define EDGE0_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- fp16 <-> fp64, IEEE 754 binary16, round to nearest even ---- */
double orc_half_to_double(uint16_t h);
uint16_t orc_double_to_half(double v);

/* ---- int4 affine group-64 format [P1 S2 "Quantization"; P3; P4 "Counting the bytes"] ---- */
void orc_int4_unpack(const uint32_t* packed, long n_words, uint8_t* nibbles);
void orc_int4_pack(const uint8_t* nibbles, long n_words, uint32_t* packed);

typedef struct {
    const uint32_t* q;   /* [out, in/8] */
    const uint16_t* s;   /* [out, in/64] fp16 */
    const uint16_t* b;   /* [out, in/64] fp16 */
    int out, in;
} orc_q4;

void orc_int4_dequant(const orc_q4* m, double* w /* [out, in] */);
void orc_int4_matvec(const orc_q4* m, const double* v, double* y);

/* dense fp16 weight [out, in] row-major with leading dimension ld (elements) */
void orc_f16_matvec(const uint16_t* W, int out, int in, int ld, const double* v, double* y);

double orc_gelu_erf(double z);
double orc_silu(double z);

/* SwiGLU expert, down(silu(gate(x)) * up(x)) [P1 S3.1 "Math contract"] */
void orc_expert_swiglu(const orc_q4* gate, const orc_q4* up, const orc_q4* down,
                       const double* x, double* y);

/* Unmerged LoRA delta dy = (alpha/r) * B (A v) [P1 S3.3; P2 eq.]
 * A [r, in], B [out, r] fp16 row-major. */
void orc_lora_delta(const uint16_t* A, const uint16_t* B, int r, int in, int out,
                    double alpha, const double* v, double* dy);

/* ---- routing [P1 App. A] ---- */
/* indices of the k largest scores, value descending, lower index first on ties */
void orc_topk(const float* score, int n, int k, int32_t* idx);

/* softmax-topK with renormalisation.  bias (nullable) is added in fp32 to the
 * logits before softmax and selection. */
void orc_route_softmax_topk(const float* logits, const float* bias, int E, int K,
                            int32_t* ids, float* w);

/* sigmoid-group: sigma = sigmoid(l) in fp32; selection score = sigma + bias
 * (fp32); group score = sum of the two largest selection scores in the group;
 * keep the best G of n_groups; top-K within survivors; weights use raw sigma:
 * w = scale * sigma / (sum sigma + 1e-20). */
void orc_route_sigmoid_group(const float* logits, const float* bias, int E, int K,
                             int n_groups, int G, float scale, int32_t* ids, float* w);

/* route_kind values */
#define ORC_ROUTE_SOFTMAX_TOPK 0
#define ORC_ROUTE_SIGMOID_GROUP 1

typedef struct {
    int kind;            /* ORC_ROUTE_* */
    int n_groups, topk_groups;
    float scale;
    const float* bias;   /* [E] or NULL */
} orc_route;

void orc_apply_route(const orc_route* r, const float* logits, int E, int K, int32_t* ids, float* w);

/* ---- prerouter head [P1 S3.2 "Head"; P2 eq.; P4 PrerouterHead] ----
 * fc1 [H, d+2E], fc2 [E, H], linit [E, d+2E], fp16, no bias.
 * feats = concat(x, exec_onehot, prev_onehot); logits = fc2 gelu(fc1 feats) + linit feats.
 * prev_ids may be NULL (no previous token: zero mask). */
void orc_prerouter_logits(const uint16_t* fc1, const uint16_t* fc2, const uint16_t* linit,
                          int d, int E, int H, const uint16_t* x,
                          const int32_t* exec_ids, const int32_t* prev_ids, int K,
                          float* logits);

/* x = fp16(h / sqrt(mean(h^2) + eps) * gamma); gamma NULL means unit gain */
void orc_rmsnorm(const uint16_t* h, const uint16_t* gamma, int d, double eps, uint16_t* x);

/* ---- MoE block ---- */
typedef struct {
    int d, I, Is, E, K;
    /* routed expert stacks: q [E, out, in/8], s/b [E, out, in/64] */
    const uint32_t *gate_q, *up_q, *down_q;
    const uint16_t *gate_s, *gate_b, *up_s, *up_b, *down_s, *down_b;
    /* shared expert (one expert, intermediate Is); gate_q NULL = none */
    const uint32_t *sh_gate_q, *sh_up_q, *sh_down_q;
    const uint16_t *sh_gate_s, *sh_gate_b, *sh_up_s, *sh_up_b, *sh_down_s, *sh_down_b;
} orc_moe;

/* y_b = sum_k w[b,k] * expert_{ids[b,k]}(x_b) + shared(x_b); no LoRA.
 * x [B,d] fp16; y16 [B,d] fp16 (nullable); y [B,d] fp64 (nullable). */
void orc_moe_forward(const orc_moe* m, const uint16_t* x, const int32_t* ids, const float* w,
                     int B, uint16_t* y16, double* y);

/* ---- one decode layer and one decode step over a stack ---- */
typedef struct {
    orc_moe moe;
    /* LoRA on the shared-expert projections (NULL A = none) */
    const uint16_t *lora_Ag, *lora_Bg, *lora_Au, *lora_Bu, *lora_Ad, *lora_Bd;
    int r; double alpha;
    const uint16_t* router;   /* [E, d] fp16 */
    const uint16_t* gamma;    /* [d] fp16 or NULL */
    double eps;
    orc_route route;          /* this layer's routing function */
    int prerouted;            /* consumes the upstream head's prediction when t > 0 */
    /* head owned by this layer (fc1 NULL = none) */
    const uint16_t *fc1, *fc2, *linit;
    int H;
    int head_target;          /* layer index whose routing the head predicts */
} orc_layer;

typedef struct {
    int L, B, K;
    int32_t* pred_ids;   /* [2][L][B][K], slot (t&1) written at step t */
    float*   pred_w;     /* [2][L][B][K] */
    int32_t* exec_ids;   /* [2][L][B][K], slot (t&1) = ids executed at step t */
} orc_state;

/* Optional per-layer record of one step (all nullable):
 * x [L][B][d] fp16, ids/w [L][B][K] used by each layer, hout [L][B][d] fp16,
 * head_logits [L][B][E] (rows of layers without a head are left untouched),
 * router_logits [L][B][E] (rows of layers that did not run their router are
 * left untouched). */
typedef struct {
    uint16_t* x; int32_t* ids; float* w; uint16_t* hout; float* head_logits;
    float* router_logits;
} orc_record;

/* run layer l of `layers` at step t on h [B,d] fp16 (in place) */
void orc_decode_layer(const orc_layer* layers, int l, orc_state* st, uint16_t* h, int t,
                      orc_record* rec);
/* run all L layers at step t */
void orc_decode_step(const orc_layer* layers, orc_state* st, uint16_t* h, int t, orc_record* rec);

#ifdef __cplusplus
}
#endif
#endif
