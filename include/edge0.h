/*
 * libedge0 -- C ABI of the prerouted int4 MoE decode path on GB300 (sm_103a).
 *
 * What the path computes (page titles and sections):
 *   "The Other Half of the Memory Wall: Serving 35B MoEs from SSD with Trained
 *    Routing Prediction":
 *     S3.1 "Math contract"  expert(x) = down(silu(gate(x)) * up(x)), int4 affine
 *                            group-64 weights;
 *     S3.2 "Head"           head(feats) = fc2(erf-gelu(fc1 feats)) + linear_init(feats),
 *                            feats = [x, executed one-hot, previous one-hot],
 *                            f_in = d_model + 2E; no biases;
 *     S3.2 "Motivation", "Prediction-as-routing"
 *                            the head owned by layer N runs at token t and its
 *                            prediction is layer N+1's routing at t+1;
 *     S3.3                   unmerged LoRA, y = W_int4 x + (alpha/r) B A x, on the
 *                            shared-expert projections;
 *     App. A                 softmax-topk (renormalised) and sigmoid-group routing.
 *   "Inside Edge0-35B", "Architectural Deep Dive": packed uint32 [E, out, in/8]
 *    weights with one scale and bias per 64 inputs.
 *
 * Conventions for every call
 *   - Pointers are DEVICE pointers unless the argument says HOST.  The caller
 *     owns every buffer; the library borrows them for the call and never frees
 *     them.  Its only state of its own: caches of tables it derives from the
 *     shapes and descriptors (the batch-1 kernel's per-shape plan table and its
 *     device copy of the layer descriptors), allocated and uploaded on the first
 *     call that needs them and kept for the process; the expert pool's device
 *     state (owned by its handle); and edge0_moe_int4_forward_noalloc's fixed
 *     scratch array (see its section; its device-side status is read with
 *     edge0_noalloc_error).
 *   - fp16 tensors are IEEE binary16 (passed as uint16_t); fp32 as float.
 *   - Every call enqueues work on `stream` and returns without synchronising,
 *     except where its section says otherwise (edge0_state_error, the pool's
 *     read-outs and set-up) and the first-use uploads above.  Arguments are
 *     validated on the host before anything is launched; an invalid argument
 *     returns EDGE0_EINVAL and launches nothing.
 *   - Stream capture into CUDA graphs is supported only for the allocation-free
 *     call (see its section): the first-use uploads above are synchronous, and
 *     the batched path (B > 4) and prefill upload a small per-call table from
 *     host memory.
 *   - Kernels never trap: a wait that runs out of time records EDGE0_ETIMEOUT in
 *     the route state's control block (read it with edge0_state_error) and the
 *     kernel returns.
 *
 * Weight layouts
 *   Canonical (the pages'): int4 matrix [out, in] = q uint32 [out, in/8] (nibble i
 *   of word j is input 8j+i, low nibble first), s and b fp16 [out, in/64],
 *   w = s*q + b; experts stacked on a leading [E] axis.  Dense fp16 weights are
 *   nn.Linear [out, in] row-major.
 *   Packed (this library's HBM layout, written by edge0_pack_*): rows are taken 16
 *   at a time ("row tile", padded with zero rows) and inputs 16 at a time
 *   ("step"); a (row tile, step) block is stored in the order the 32 lanes of a
 *   warp read it as the A operand of one m16n8k16 tensor-core step (int4: 4
 *   bytes per lane, 128 bytes; fp16: 16 bytes per lane, 512 bytes).  int4 scale
 *   and bias pairs of a row tile and group of 64 inputs take 64 bytes.
 *     gate/up  (edge0_pack_q4_gate_up): one interleaved matrix per expert whose
 *              row tile j holds gate rows 8j..8j+7 then up rows 8j..8j+7;
 *              per row tile and group a 576-byte unit (4 step blocks + scales).
 *     down     (edge0_pack_q4_down): K-major; per group of 64 inputs, the four
 *              step blocks of every row tile, then the scales of every row tile.
 *     fp16     (edge0_pack_f16): row-tile major, 2048 bytes per row tile and
 *              group; (edge0_pack_f16_kmajor): step major.
 *   Experts follow each other in the stacks.
 */
#ifndef EDGE0_H
#define EDGE0_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---- */
#define EDGE0_OK 0
#define EDGE0_EINVAL 1      /* bad argument: NULL, shape, K > E, in % 64, misalignment */
#define EDGE0_ECUDA 2       /* a CUDA runtime call failed */
#define EDGE0_ETIMEOUT 3    /* a bounded device wait ran out (reported by the kernel) */
#define EDGE0_EUNSUPPORTED 4/* shape outside what this build handles (see limits) */

const char* edge0_status_string(int status);

/* ---- limits of this build ---- */
#define EDGE0_MAX_LAYERS 48
#define EDGE0_MAX_BATCH 4     /* sequences per call of the persistent batch-1 engine */
#define EDGE0_MAX_BATCHED 256 /* sequences per decode call on the batched path */
#define EDGE0_MAX_K 8
#define EDGE0_MAX_E 512

/* ---- routing rule [App. A] ---- */
#define EDGE0_ROUTE_SOFTMAX_TOPK 0
#define EDGE0_ROUTE_SIGMOID_GROUP 1
typedef struct {
    int kind;            /* EDGE0_ROUTE_* */
    int n_groups;        /* sigmoid-group: number of groups n (E % n == 0) */
    int topk_groups;     /* sigmoid-group: groups kept G */
    float scale;         /* sigmoid-group: routed scale s */
    const float* bias;   /* [E] fp32 selection bias or NULL.  softmax-topk adds it to the
                            logits before softmax and selection; sigmoid-group adds it to
                            sigmoid(logit) for selection only (weights use raw sigmoid). */
} edge0_route;

/* ---- routed + shared int4 experts ---- */
typedef struct {
    int d, E, K, I, Is;        /* d_model, experts, top-k, expert and shared intermediate */
    const void* gate_up;       /* packed int4 [E][gate | up interleaved]  (edge0_pack_q4_gate_up) */
    const void* down;          /* packed int4 [E][d x I] K-major          (edge0_pack_q4_down)    */
    const void* sh_gate_up;    /* shared expert, same layouts, or NULL for no shared expert     */
    const void* sh_down;
    const int32_t* slot_table; /* [E] expert id -> slot in the stacks above, or NULL   */
    int n_slots;               /* slots in the stacks when slot_table != NULL (a slot
                                  outside [0, n_slots) makes the kernel record EDGE0_EINVAL,
                                  except -1 with a host tier below)                    */
    const void* host_gate_up;  /* host tier (batched decode path only): all E experts'
                                  packed gate/up and down stacks in pinned host memory the
                                  device can read; an expert whose slot_table entry is -1
                                  is read from here.  NULL: no host tier.              */
    const void* host_down;
    const void* down_rows;     /* down again in row-tile major units (edge0_pack_q4_rows),
                                  experts stacked, or NULL: the batch-1 kernel reads
                                  down by output row tiles from here               */
    const void* sh_down_rows;  /* the shared expert's down, same layout, or NULL    */
    unsigned long long* tier_counts; /* batched path with a slot table: device [2] u64,
                                  or NULL.  Each layer adds its active routed experts
                                  to [0] and those of them read from the host tier
                                  (published slot -1 when the layer dispatched) to [1] */
} edge0_moe_desc;

/* ---- one unmerged LoRA projection [S3.3]: y += (alpha/r) B (A v) ---- */
typedef struct {
    int r, in, out;            /* rank (at most 16), input and output width            */
    float alpha;
    const void* A;             /* packed fp16 [r x in]  (edge0_pack_f16); used for the
                                  shared expert's gate and up projections, and for its
                                  down projection by the batch-1 decode kernel (which
                                  is not used when lora_down.A is NULL)                */
    const uint16_t* A_T;       /* fp16 [in, r] = A transposed, row-major; used for the
                                  shared expert's down projection and edge0_lora_delta */
    const uint16_t* B;         /* fp16 [out, r] row-major                              */
} edge0_lora_desc;

/* ---- prerouter head [S3.2 "Head"] ---- */
typedef struct {
    int d, E, H, K;
    const void* fc1_dense;     /* packed fp16 [H x d]: fc1[:, :d]                      */
    const uint16_t* fc1_oh_T;  /* fp16 [2E, H]: row j = fc1[:, d + j] (edge0_pack_cols_T) */
    const void* fc2;           /* packed fp16 [E x H] K-major (edge0_pack_f16_kmajor)  */
    const void* linit_dense;   /* packed fp16 [E x d]: linear_init[:, :d]              */
    const uint16_t* linit_oh_T;/* fp16 [2E, E]: row j = linear_init[:, d + j]          */
    edge0_route route;         /* routing rule of the layer whose routing it predicts  */
} edge0_head_desc;

/* ---- one decode layer ---- */
typedef struct {
    edge0_moe_desc moe;
    edge0_lora_desc lora_gate, lora_up, lora_down; /* shared expert; A == NULL: no LoRA */
    const void* router;        /* packed fp16 [E x d] own router                       */
    edge0_route route;         /* this layer's routing rule                            */
    const uint16_t* gamma;     /* [d] RMSNorm gain, or NULL for unit gain              */
    float eps;                 /* RMSNorm epsilon                                      */
    int prerouted;             /* 1: at step > 0 route by the upstream head's prediction */
    int has_head;              /* 1: this layer owns `head`                            */
    edge0_head_desc head;
    int head_target;           /* state row the head's prediction is written to        */
    int index;                 /* this layer's row in the route state                  */
    cudaEvent_t ready;         /* batched path: the layer's kernels wait for this event
                                  (e.g. its expert-pool prefetch) when not NULL        */
} edge0_layer_desc;

/* ---- routing state carried across steps and the kernels' scratch ----
 * pred_ids/pred_w [2][L][B][K]: slot (t & 1) holds the predictions made at step t
 *   (consumed at t + 1); exec_ids [2][L][B][K]: slot (t & 1) holds the ids each
 *   layer executed at step t (the head's executed mask at t, previous mask at t+1).
 * workspace: device scratch of edge0_workspace_bytes(L, B, d, E) bytes, zeroed by
 *   edge0_state_init before first use; it holds the layer outputs and logits of
 *   two step parities, the launch counters and the error word.  A
 *   workspace belongs to one kind of call (decode on this state,
 *   edge0_moe_int4_forward, or edge0_prerouter_topk): calls of different kinds
 *   must not share one. */
typedef struct {
    int L, B, K;
    int32_t* pred_ids;
    float* pred_w;
    int32_t* exec_ids;
    void* workspace;
    size_t workspace_bytes;
    /* Optional records of a batch-1 decode call (B == 1; NULL: not recorded;
     * ignored for B > 1).  For checking a whole decode step against a reference
     * layer by layer, and for diagnosis.
     *   record_h      fp16 [L][d]: row l = the output h of the call's layer l;
     *   record_logits fp32 [L][E]: row l = the logits of the head owned by the
     *                 call's layer l (rows of layers without a head untouched). */
    uint16_t* record_h;
    float* record_logits;
} edge0_route_state;

/* ---- packing (device -> device, enqueued on stream) ---- */
size_t edge0_q4_gate_up_packed_bytes(int E, int I, int d);
/* gate and up q [E, I, d/8] uint32, s/b [E, I, d/64] fp16 -> one interleaved matrix per expert */
int edge0_pack_q4_gate_up(const uint32_t* q_gate, const uint16_t* s_gate, const uint16_t* b_gate,
                          const uint32_t* q_up, const uint16_t* s_up, const uint16_t* b_up, int E,
                          int I, int d, void* packed, cudaStream_t stream);
size_t edge0_q4_down_packed_bytes(int E, int out, int in);
/* q [E, out, in/8] uint32, s/b [E, out, in/64] fp16 -> K-major packed int4 */
int edge0_pack_q4_down(const uint32_t* q, const uint16_t* s, const uint16_t* b, int E, int out,
                       int in, void* packed, cudaStream_t stream);
/* q [E, out, in/8] uint32, s/b [E, out, in/64] fp16 -> row-tile major int4 units
 * [E][out/16][in/64][576] (edge0_q4_down_packed_bytes(E, out, in) bytes) */
int edge0_pack_q4_rows(const uint32_t* q, const uint16_t* s, const uint16_t* b, int E, int out,
                       int in, void* packed, cudaStream_t stream);
size_t edge0_f16_packed_bytes(int out, int in);
/* W [out, in] fp16 with row stride ld elements (use ld > in for a column slice) */
int edge0_pack_f16(const uint16_t* W, int out, int in, int ld, void* packed, cudaStream_t stream);
int edge0_pack_f16_kmajor(const uint16_t* W, int out, int in, int ld, void* packed,
                          cudaStream_t stream);
/* dst [ncols, out] = transpose of W[:, col0 : col0 + ncols] (W row stride ld) */
int edge0_pack_cols_T(const uint16_t* W, int out, int ld, int col0, int ncols, uint16_t* dst,
                      cudaStream_t stream);

/* ---- state ---- */
/* workspace of a state of L layers (L = 1 for edge0_moe_int4_forward and
 * edge0_prerouter_topk) for B <= EDGE0_MAX_BATCH sequences */
size_t edge0_workspace_bytes(int L, int B, int d, int E);
/* workspace of a decode state of L layers for any B <= EDGE0_MAX_BATCHED:
 * edge0_workspace_bytes for B <= EDGE0_MAX_BATCH, else the batched path's
 * (layer output, x of every layer, dispatch lists, act of every (token, expert)
 * pair); K top-k, I and Is the expert and shared intermediate, H the head width */
size_t edge0_decode_workspace_bytes(int L, int B, int d, int E, int K, int I, int Is, int H);
/* zero pred/exec/workspace; must precede the first decode call on a state */
int edge0_state_init(edge0_route_state* st, cudaStream_t stream);
/* HOST call: synchronises `stream`, returns the kernels' recorded status (EDGE0_OK,
 * EDGE0_ETIMEOUT, EDGE0_EINVAL for a routing id outside [0, E) in the state,
 * EDGE0_EUNSUPPORTED for a launch without its cluster shape) in *status.  After
 * a non-zero status the state is re-initialised as by edge0_state_init (a launch
 * that gave up leaves its accumulators part-way), which also resets the wait
 * limit. */
int edge0_state_error(const edge0_route_state* st, cudaStream_t stream, int* status);
/* HOST call (synchronises `stream`): the limit, in nanoseconds, of every bounded
 * wait of the persistent kernels on this state (0: the default of 2 s).  A wait
 * that runs out records EDGE0_ETIMEOUT, every CTA of the launch leaves, and the
 * next edge0_state_error reports it. */
int edge0_state_set_wait_limit(edge0_route_state* st, unsigned long long wait_ns, cudaStream_t stream);

/* ---- the four operations of the path ---- */

/* Prerouter head + top-K [S3.2 "Head", App. A].
 * x [B, d] fp16 post-attention-norm hidden state; exec_ids [B, K] the experts this
 * layer executed at this token; prev_ids [B, K] those of the previous token, or
 * NULL (no previous token: zero mask).  Writes the predicted routing for the
 * head's target layer: out_ids [B, K] (score-descending, lower id first on ties),
 * out_w [B, K]; out_logits [B, E] (optional, NULL to skip) the head's fp32 logits.
 * workspace: scratch of edge0_workspace_bytes(1, B, d, E) bytes, zeroed before its
 * first use (cudaMemset). */
int edge0_prerouter_topk(const edge0_head_desc* head, const uint16_t* x, const int32_t* exec_ids,
                         const int32_t* prev_ids, int B, int32_t* out_ids, float* out_w,
                         float* out_logits, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/* Routed + shared int4 SwiGLU experts [S3.1 "Math contract"], no LoRA:
 * y_b = sum_k w[b,k] expert_{ids[b,k]}(x_b) + shared(x_b).
 * x [B, d] fp16; ids [B, K] int32 (0 <= id < E); w [B, K] fp32; y [B, d] fp16.
 * workspace as for edge0_prerouter_topk (edge0_workspace_bytes(1, B, d, E)). */
int edge0_moe_int4_forward(const edge0_moe_desc* moe, const uint16_t* x, const int32_t* ids,
                           const float* w, int B, uint16_t* y, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream);

/* Unmerged LoRA delta [S3.3]: y[b] += (alpha/r) B (A v[b]) for v [B, in] fp16,
 * y [B, out] fp16 (read, add in fp32, round to fp16); reads lora->A_T and lora->B.
 * Needs no workspace. */
int edge0_lora_delta(const edge0_lora_desc* lora, const uint16_t* v, int B, uint16_t* y_inout,
                     cudaStream_t stream);

/* Dense fp16 GEMM on the fifth-generation tensor cores (tcgen05.mma with a TMEM
 * accumulator): D [M, N] fp32 = A [M, K] fp16 x B [N, K]^T fp16, all row-major
 * and 16-byte aligned on the device; M % 128 == 0, 16 <= N <= 256 with N % 16
 * == 0, K % 64 == 0.  *status (device int, set to 0 by the caller) receives
 * EDGE0_ETIMEOUT if a tensor-core wait ran past its limit.  The building block
 * of the grouped int4 kernels; enqueued on `stream`. */
int edge0_tc_gemm_f16(const uint16_t* A, const uint16_t* B, float* D, int M, int N, int K, int* status,
                      cudaStream_t stream);

/* One decode layer at step `step` for B sequences: h_inout [B, d] fp16 is the
 * layer input (residual stream) and receives the layer output
 *   h + routed experts + shared expert (with LoRA),
 * with routing from the upstream head's prediction (prerouted layers, step > 0)
 * or the layer's own router; if the layer owns a head, its prediction for
 * head_target at step + 1 is written to the state.  step < 0 uses and advances
 * the step counter kept in the workspace. */
int edge0_decode_layer(const edge0_layer_desc* layer, uint16_t* h_inout, edge0_route_state* st,
                       int B, int step, cudaStream_t stream);

/* All L layers of one decode step (same semantics as L successive
 * edge0_decode_layer calls).  B == 1: one launch of the batch-1 kernel when the
 * shapes are within its limits (d <= 2048, d % 128 == 0, K I + Is <= 4608,
 * every layer with the same shared-expert / LoRA parts, down_rows (and
 * sh_down_rows, lora_down.A) given, no slot table, one layer per state row),
 * else of the persistent engine; B <= EDGE0_MAX_BATCH: one persistent launch;
 * EDGE0_MAX_BATCH < B <= EDGE0_MAX_BATCHED: the batched path, a sequence of
 * kernels per layer in which every active expert's weights are read once for
 * all of its tokens, then every head of the step; it needs step >= 0 and a
 * workspace of edge0_decode_workspace_bytes. */
int edge0_decode_step(const edge0_layer_desc* layers, int L, uint16_t* h_inout,
                      edge0_route_state* st, int B, int step, cudaStream_t stream);
/* Calls on one state step through the step parities in order (step, step + 1,
 * ...): a call clears the accumulators of the other parity for the next one. */

/* ---- whole-layer prefill [S3.1 "Executor paths" (whole-layer), S5.1 Table 1
 * caption: prompt processing reads every expert of a layer once for all the
 * prompt's tokens; the prerouter is not used at prefill] ----
 * The L layers over a prompt of T tokens (1 <= T <= 8192): h_inout [T, d] fp16
 * (device, 16-byte aligned, updated in place).  Every layer routes every token
 * with its own router and routing rule (App. A) -- heads and route state are
 * not used -- then runs the routed experts grouped by expert (each active
 * expert's weights read once per block of its tokens) and the shared expert
 * with its LoRA over all tokens; h = fp16(h + y) per layer, as in
 * edge0_decode_step.  ids_out: NULL, or [L][T][K] int32 (device) that receives
 * every layer's executed ids.  workspace: device scratch of at least
 * edge0_prefill_workspace_bytes(T, ...) bytes (16-byte aligned, owned by the
 * caller, not zeroed beforehand; the call clears what it needs).  The shapes of
 * every layer are those of layers[0]; d % 128 == 0.  No slot table, no host
 * tier.  Returns EDGE0_EINVAL on bad arguments, EDGE0_ECUDA when a launch
 * fails; enqueued on `stream` (asynchronous). */
size_t edge0_prefill_workspace_bytes(int T, int d, int E, int K, int I, int Is);
#define EDGE0_PREFILL_TCGEN05_GATE_UP 1u  /* flags: gate/up on the tcgen05 kernel (dequantized
                                             fp16 tiles, TMEM accumulator) instead of the
                                             mma.sync kernel (int4 nibbles as fp16
                                             subnormals, scales in the epilogue); the
                                             results agree within the parity tolerance */
int edge0_prefill(const edge0_layer_desc* layers, int L, uint16_t* h_inout, int T, int32_t* ids_out,
                  unsigned flags, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---- expert pool with a host tier [S3.1 "SSD Streaming Expert Layers", S3.2
 * "Motivation", S5.3]: n_slots device slots per layer in front of every
 * expert's packed weights in pinned host memory.  The published slot table
 * (edge0_moe_desc.slot_table, [E] int32, device) maps an expert to its slot or
 * -1; the batched kernels read an expert whose entry is -1 from the host tier.
 *
 * Policy (edge0_pool_plan): a request marks experts as requested now; each
 * requested expert that is not in the planner's map takes a free slot, else the
 * least recently requested slot whose expert is not requested now (lowest
 * index on equal recency); experts left without a slot stay in the host tier.
 *
 * edge0_pool_create: L <= EDGE0_MAX_LAYERS layers of E <= EDGE0_MAX_E experts,
 *   1 <= n_slots <= E; one expert's packed gate/up and down take gu_bytes and
 *   dn_bytes (multiples of 16).  edge0_pool_set_layer: the layer's host stacks
 *   [E][..], its slot stacks [n_slots][..] and its slot table (16-byte aligned).
 * Device mode (the product path), after edge0_pool_device_init (every layer set;
 *   allocates the pool's device state, empties every slot table):
 *   edge0_pool_prefetch_async(ids, n, stream, copy_stream): ids[l] is a device
 *     pointer to n expert ids of layer l (e.g. its prediction for the next
 *     step), or NULL to leave layer l alone.  Enqueues on `stream` one planner
 *     CTA per layer; an evicted expert leaves the published table before any
 *     later work of `stream` reads it.  Then on `copy_stream` (after the
 *     planner) one copy kernel moves the planned experts from host memory into
 *     their slots and publishes each (release store of its table entry) once
 *     all of its bytes are in place.  Neither the host nor `stream` waits for a
 *     copy: an expert whose copy has not been published is read from the host
 *     tier.  A layer whose previous copies are still in flight skips this plan
 *     (counted).  Asynchronous; returns EDGE0_EINVAL on bad arguments.
 *   edge0_pool_wait(timeout_ns): polls from the host until the last copy pass
 *     enqueued has ended, at most timeout_ns; EDGE0_ETIMEOUT when it has not
 *     (the copies go on; nothing is cancelled).  For callers that want the
 *     published map settled, e.g. before reading it; the decode path never
 *     calls it.
 *   edge0_pool_inject(fail_every, delay_ns): host-side fault injection for the
 *     following copy passes: copy number q fails when fail_every > 0 and
 *     q % fail_every == fail_every - 1 (its bytes are not moved, it is not
 *     published, the next plan frees its slot); every copy pass first waits
 *     delay_ns (at most 1e9, else EDGE0_EINVAL).  0, 0 turns both off.
 *   edge0_pool_stats_ex / edge0_pool_stats / edge0_pool_resident wait for the
 *     device (cudaDeviceSynchronize) and read the device counters and the
 *     published table of layer l.
 * Host mode (no GPU: the same planner and publication steps over host
 * buffers; set_layer then takes host buffers for the slots and the table):
 *   edge0_pool_plan           one request of layer l; returns the copies to make
 *                             (expert, slot) without making them.
 *   edge0_pool_host_prefetch  as edge0_pool_prefetch_async's planner: ids[l] host
 *                             pointers, evicted experts leave the table.
 *   edge0_pool_host_copy      as the copy kernel: completes every copy in flight
 *                             (memcpy, publish, or mark failed under injection).
 * Counters (edge0_pool_stats_ex, out[8]): requests, hits, copies planned,
 * copies published, copies failed, layer plans skipped, bytes published,
 * requested ids outside [0, E).  edge0_pool_stats gives hits and copies planned.
 * Not thread-safe; one pool per device. */
typedef struct edge0_pool edge0_pool;
int edge0_pool_create(int L, int E, int n_slots, size_t gu_bytes, size_t dn_bytes, edge0_pool** out);
int edge0_pool_set_layer(edge0_pool* pool, int l, const void* host_gu, const void* host_dn, void* dev_gu,
                         void* dev_dn, int32_t* dev_slot_table);
int edge0_pool_plan(edge0_pool* pool, int l, const int32_t* ids, int n, int32_t* out_expert,
                    int32_t* out_slot, int* n_copy);
int edge0_pool_host_prefetch(edge0_pool* pool, const int32_t* const* ids, int n);
int edge0_pool_host_copy(edge0_pool* pool);
int edge0_pool_device_init(edge0_pool* pool);
int edge0_pool_prefetch_async(edge0_pool* pool, const int32_t* const* ids, int n, cudaStream_t stream,
                              cudaStream_t copy_stream);
int edge0_pool_wait(edge0_pool* pool, unsigned long long timeout_ns);
int edge0_pool_inject(edge0_pool* pool, int fail_every, unsigned long long delay_ns);
int edge0_pool_stats_ex(const edge0_pool* pool, long long* out, int n);
int edge0_pool_stats(const edge0_pool* pool, long long* hits, long long* copies);
int edge0_pool_resident(const edge0_pool* pool, int l, int32_t* slot_of);
void edge0_pool_destroy(edge0_pool* pool);

/* ---- allocation-free variant (the paper has no counterpart to this call) ----
 * edge0_moe_int4_forward for callers that cannot allocate memory: code running
 * in an allocator-free part of a serving loop, code whose memory budget was fixed
 * at start-up, or hosts that pass this library only buffers they already own.
 * Same arguments and result as edge0_moe_int4_forward minus the workspace: the
 * kernel's scratch is a fixed array of EDGE0_NOALLOC_SCRATCH_BYTES bytes inside
 * the library, present in every GPU that loads it until the process exits.  The
 * call allocates nothing (no cudaMalloc, no host heap); it clears the part of
 * the array it uses before launching.
 *   - The call needs 512 + 10 B d + 16 B E + 384 B bytes of it (about 98 KB at d=2048,
 *     E=256, B=4); shapes whose need exceeds the array (d=4096, E=512, B=4)
 *     return EDGE0_EUNSUPPORTED.
 *   - The first call on a device looks up the array's device address for that
 *     device (cudaGetSymbolAddress); make that first call before any stream
 *     capture.
 *   - All calls share the array: two calls whose kernels overlap on the GPU (for
 *     instance on different streams) race and give wrong results.
 *   - The cached address belongs to the device's primary context: it is no longer
 *     valid after cudaDeviceReset on that device.
 *   - The call builds the kernel's parameter block (up to 32 KB) on the calling
 *     thread's stack: threads with small stacks must allow for it.
 *   - A shape refused on the host (EDGE0_EINVAL, EDGE0_EUNSUPPORTED) queues
 *     nothing.  What the kernel itself records (EDGE0_EINVAL for a slot_table
 *     entry outside [0, n_slots), EDGE0_ETIMEOUT for a wait that ran out) stays
 *     in the array's header until the next call clears it: read it with
 *     edge0_noalloc_error before that call. */
#define EDGE0_NOALLOC_SCRATCH_BYTES (1 << 17)
int edge0_moe_int4_forward_noalloc(const edge0_moe_desc* moe, const uint16_t* x,
                                   const int32_t* ids, const float* w, int B, uint16_t* y,
                                   cudaStream_t stream);
/* HOST call: synchronises `stream`, writes the status the last
 * edge0_moe_int4_forward_noalloc kernel on the current device recorded
 * (EDGE0_OK, EDGE0_EINVAL, EDGE0_ETIMEOUT) to *status and clears it.  Allocates
 * nothing. */
int edge0_noalloc_error(cudaStream_t stream, int* status);

#ifdef __cplusplus
}
#endif
#endif
