// Internal definitions of libedge0 (CUDA sources only).
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "edge0.h"

namespace edge0 {

// ---------------------------------------------------------------- layout ----
constexpr int kGroup = 64;           // inputs per affine group (int4 group-64)
constexpr int kRowTile = 16;         // rows per tensor-core row tile
constexpr int kQ4Unit = 576;         // int4 unit: 512 B nibbles + 64 B scale/bias pairs
constexpr int kQ4Quarter = 128;      // int4 block of one 16-input step of one row tile
constexpr int kQ4Scales = 64;        // scale/bias pairs of one row tile and group
constexpr int kF16Unit = 2048;       // fp16 unit: 16 rows x 64 inputs
constexpr int kF16Step = 512;        // fp16 block of one 16-input step of one row tile
constexpr int kHalfRow = 8;          // act rows per interleaved gate/up tile

inline __host__ __device__ int ceil_div(int a, int b) { return (a + b - 1) / b; }
// packed bytes of an int4 matrix [out, in] (row tiles x groups x 576)
inline __host__ __device__ long long q4_bytes(int out, int in) {
    return (long long)ceil_div(out, kRowTile) * (in / kGroup) * kQ4Unit;
}
// packed bytes of an fp16 matrix [out, in] (row tiles x 16-input steps x 512)
inline __host__ __device__ long long f16_bytes(int out, int in) {
    return (long long)ceil_div(out, kRowTile) * (in / 16) * kF16Step;
}

// --------------------------------------------------------------- engine ----
constexpr int kConsumerWarps = 16;
constexpr int kThreads = (kConsumerWarps + 1) * 32;   // + one producer warp
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kClusterCtas = 2;                        // CTA pairs share gate/up partial sums

enum Mode : int { MODE_DECODE = 0, MODE_MOE = 1, MODE_HEAD = 2, MODE_PREFILL = 3 };

enum LayerFlags : int {
    LF_PREROUTED = 1,
    LF_HEAD = 2,
    LF_LORA = 4,
    LF_SHARED = 8,
};

struct LayerP {
    const char* gu;          // packed interleaved gate/up, experts stacked (stride q4_bytes(2I, d))
    const char* down;        // packed K-major down, experts stacked (stride q4_bytes(d, I))
    const char* sh_gu;       // shared expert, same layouts
    const char* sh_down;
    const int* slot_table;   // expert id -> slot of the stacks (or null: slot = id)
    int n_slots;
    const char* gu_host;     // host tier: all experts (slot -1), batched path only
    const char* down_host;
    const char* down_rows;   // down in row-tile major units (batch-1 kernel), or null
    const char* sh_down_rows;
    void* ready;             // host: event the batched path waits for before the layer
    unsigned long long* tier_counts;   // [2] += active routed experts, += of them read from the host tier
    const char* router;      // packed fp16 [E x d]
    const char* lora_Ag;     // packed fp16 [r x d] (one row tile)
    const char* lora_Au;
    const char* lora_Ad;     // packed fp16 [r x Is] (one row tile), or null
    const __half* lora_AdT;  // [Is, r]: A_down transposed
    const __half* lora_Bg;   // [Is, r]
    const __half* lora_Bu;
    const __half* lora_Bd;   // [d, r]
    const char* fc1;         // packed fp16 [H x d]
    const __half* fc1_oh;    // [2E, H]
    const char* fc2;         // packed fp16 K-major [E x H]
    const char* linit;       // packed fp16 [E x d]
    const __half* linit_oh;  // [2E, E]
    const __half* gamma;
    const float* bias;       // this layer's routing bias (or null)
    const float* head_bias;  // head target's routing bias (or null)
    float eps;
    float lora_scale;        // alpha / r
    float route_scale, head_route_scale;
    int route_kind, n_groups, topk_groups;
    int head_route_kind, head_n_groups, head_topk_groups;
    int flags;
    int head_target;         // state row
    int sidx;                // state row of this layer
};

struct Prog {
    int mode;
    int L, B, K, d, E, I, Is, H, r;
    int step;                 // >= 0: explicit; < 0: read and advance the workspace counter
    // decode
    __half* h_io;             // [B, d]
    int32_t* pred_ids;        // [2][Ls][B][K]
    float* pred_w;
    int32_t* exec_ids;
    int Ls;                   // rows of the route state
    // moe / head modes
    const __half* x_in;       // [B, d]
    const int32_t* ids_in;    // [B, K]
    const float* w_in;
    __half* y_out;            // [B, d]
    const int32_t* exec_in;   // [B, K]
    const int32_t* prev_in;   // [B, K] or null
    int32_t* out_ids;
    float* out_w;
    float* out_logits;
    // workspace
    char* ws;
    // derived by engine_check for the launch's grid
    int slots_max;            // routed expert slots of a layer: min(B K, E)
    int ps[2];                // CTA pairs that own shared-expert rows (without, with LoRA)
    int hr_max, q_max;        // most half-row tiles / act quarters one CTA pair owns
    int ring_bytes;           // shared-memory ring of streamed weights
    int ft;                   // most head tasks in one table of the head flush
    // batch-1 decode kernel (decode1.cu), filled by decode1_check
    int grid1[2];             // CTAs of the launch, LoRA-A CTAs per LoRA matrix
    int ring1;                // bytes of its shared-memory ring
    const char* tab1;         // device table of every CTA's plan and block layout
    const LayerP* ly1;        // device copy of layers[0..L) (the batch-1 kernel reads it there)
    int tc_gu;                // prefill: gate/up on the tcgen05 kernel
    int n_heads1;             // layers that own a head, in order (batch-1 kernel)
    int heads1[EDGE0_MAX_LAYERS];
    long long ws_bytes;       // workspace bytes (the trace area is at its end)
    __half* dbg_h;            // [L][d] or null: each layer's output h (batch 1)
    float* dbg_logits;        // [L][E] or null: each head's logits, at its owner layer's row
    LayerP layers[EDGE0_MAX_LAYERS];
};

// Workspace header (first 256 bytes)
struct WsHeader {
    unsigned long long barrier;   // monotonically increasing arrival counter
    unsigned int serial;          // launches of the batch-1 kernel on this workspace
    int step;                     // auto step counter
    int error;                    // EDGE0_* status recorded by a kernel
    int abort;                    // set with error: every wait gives up
    int trace;                    // non-zero: record phase timestamps in the trace area
    int hold;                     // test hook (> 0): the first wait of each CTA of a launch
                                  // cannot complete (the engine's first grid barrier waits
                                  // for arrivals beyond the grid, the batch-1 kernel's first
                                  // poll for a tag that is never written)
    unsigned long long wait_ns;   // limit of every bounded wait (0: kDefaultWaitNs)
    unsigned long long barrier_r; // arrival counter of the batch-1 kernel's router barriers
};
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;   // 2 s
constexpr int kWsHeaderBytes = 256;
// trace area (at the end of the workspace): per CTA kTraceSlots u64
constexpr int kTraceCtas = 160;
constexpr int kTraceSlots = 4096;   // u64 words: (tag, globaltimer, clock) triples

// Workspace after the header, per step parity p in {0, 1} and state row s:
//   y        [2][Ls][B][d]   fp32  layer output accumulators (red.add)
//   logits_r [2][Ls][B][E]   fp32  own-router logits
//   logits_h [2][Ls][B][E]   fp32  head logits (row of the head's owner)
//   lora     [2][Ls][B][48]  fp32  the shared expert's LoRA sums: A_gate x, A_up x
//                                  (2 x 16 per token), v = A_down act (16)
//   count    [2][Ls][4]      u32   arrival counters: head tasks, LoRA A units,
//                                  shared act rows
//   xs       [Ls][B][d]      fp16  x of each head layer, for the head flush
constexpr int kLoraAcc = 48;
constexpr int kLayerCounters = 4;
enum { CNT_HEAD = 0, CNT_LORA_A = 1, CNT_LORA_V = 2 };

struct WsLayout {
    long long y, logr, logh, lora, cnt, xs, trace, total;   // byte offsets
};
inline __host__ __device__ WsLayout ws_layout(int Ls, int B, int d, int E) {
    WsLayout w;
    long long o = kWsHeaderBytes;
    w.y = o;     o += 2LL * Ls * B * d * 4;
    w.logr = o;  o += 2LL * Ls * B * E * 4;
    w.logh = o;  o += 2LL * Ls * B * E * 4;
    w.lora = o;  o += 2LL * Ls * B * kLoraAcc * 4;
    w.cnt = o;   o += (2LL * Ls * kLayerCounters * 4 + 255) / 256 * 256;
    w.xs = o;    o += ((long long)Ls * B * d * 2 + 255) / 256 * 256;
    w.trace = o; o += (long long)kTraceCtas * kTraceSlots * 8;
    w.total = o;
    return w;
}

// Workspace of the batched decode path (B > EDGE0_MAX_BATCH), after the header:
//   y [B][d] fp32 layer output, xs [Ls][B][d] fp16 x of every layer (heads),
//   xsum [B][d/64] group sums of x, lg [B][E] logits, z [B][H] head hidden,
//   la [B][32] LoRA A x, wsel [B][K] own-router weights, disp (dispatch of a
//   layer), tok / wt [B K] (token, weight) per position, act [B K + B][Imax].
struct BatchWs {
    long long y, xs, xsum, lg, z, la, wsel, exec, disp, tok, wt, act, total;
};
BatchWs batch_ws_layout(int L, int B, int d, int E, int K, int I, int H);
// prompt tokens of one whole-layer prefill call
constexpr int kMaxPrefill = 8192;
// the layers of a prompt of p.B tokens (p.mode == MODE_PREFILL), every layer on
// its own router; enqueued on `st`
int batch_prefill(const Prog& p, int32_t* ids_out, cudaStream_t st);

// --------------------------------------------------------------- PTX -----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mma_16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;\n" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
// `count` arrivals at once (one thread standing for several)
__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar))
                 : "memory");
}
// parity wait with cluster-scope acquire: also orders the data that the other CTA
// of the cluster wrote with st.async before completing the transaction
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// bulk global -> shared copy completing on an mbarrier, streamed with evict-first
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;\n" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(p));
    return p;
}

// ---- thread-block cluster (CTA pairs) ----
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
// shared::cluster address of the same shared variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// 16-byte store into another CTA's shared memory that completes `bytes` on its mbarrier
__device__ __forceinline__ void st_async_v4(uint32_t raddr, uint4 v, uint32_t rbar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1,%2,%3,%4}, [%5];\n"
        ::"r"(raddr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(rbar)
        : "memory");
}
// 4-byte store into another CTA's shared memory that completes 4 bytes on its mbarrier
__device__ __forceinline__ void st_async_b32(uint32_t raddr, float v, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];\n"
                 ::"r"(raddr), "r"(__float_as_uint(v)), "r"(rbar)
                 : "memory");
}
// generic-proxy accesses of shared memory ordered before later bulk copies into it
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
// single-copy-atomic 64-bit global accesses at GPU scope (value and tag travel together)
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;\n" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];\n" : "=l"(v) : "l"(p) : "memory");
    return v;
}
// two single-copy-atomic 64-bit loads at GPU scope (16-byte aligned pair)
__device__ __forceinline__ ulonglong2 ld_relaxed_u64x2(const unsigned long long* p) {
    ulonglong2 v;
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];\n" : "=l"(v.x), "=l"(v.y) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" :::
                     "memory");
}

__device__ __forceinline__ void red_add_f32(float* p, float v) {
    asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;\n" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ void red_add_v4_f32(float* p, float a, float b, float c, float d) {
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1,%2,%3,%4};\n" ::"l"(p), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}
__device__ __forceinline__ void red_release_add_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;\n" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long atom_acq_rel_add_u64(unsigned long long* p, unsigned long long v) {
    unsigned long long old;
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;\n" : "=l"(old) : "l"(p), "l"(v) : "memory");
    return old;
}
__device__ __forceinline__ void red_release_add_u32(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned atom_acq_rel_add_u32(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;\n" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];\n" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_volatile_s32(const int* p) {
    int v;
    asm volatile("ld.volatile.global.s32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + __expf(-z)); }

__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
    for (int k = 16; k; k >>= 1) s += __shfl_xor_sync(0xffffffffu, s, k);
    return s;
}

// Activation sources are split v = hi + lo * 2^-11 (hi = fp16(v), lo =
// fp16((v - hi) * 2^11)) and the halves go to two tensor-core columns, so the
// products keep ~22 bits of the fp32 value.
constexpr float kLoScale = 2048.0f;
constexpr float kLoInv = 1.0f / 2048.0f;
constexpr float kTwo24 = 16777216.0f;   // int4 nibbles enter the tensor cores as q * 2^-24

// batch-1 decode kernel (decode1.cu): one launch per decode step of B = 1
// workspace bytes it needs for Ls state rows
long long decode1_ws_bytes(int Ls, int d, int E, int K, int I, int Is);
// fills p's batch-1 fields for the current device and checks that the kernel
// takes the call (EDGE0_OK) or not (EDGE0_EUNSUPPORTED: use the engine)
int decode1_check(Prog& p);
int decode1_launch(Prog& p, cudaStream_t stream);

// engine (engine.cu)
__global__ void engine_kernel(const __grid_constant__ Prog prog);
// grid size (CTAs, a multiple of the cluster size) the engine runs with on the current device
int engine_grid(int* nct);
// fills p's derived fields for a grid of nct CTAs and checks the shapes against the
// engine's limits; *smem_bytes <- dynamic shared memory.  0 or an EDGE0_* status.
int engine_check(Prog& p, int nct, int smem_max, int* smem_bytes);
// dynamic shared memory the engine can use on the current device (after engine_grid)
int engine_smem_max();
// launch the engine for `p` on `stream` (cooperative, CTA pairs); fills p's derived
// fields.  Allocates nothing.
int engine_launch(Prog& p, cudaStream_t stream);

// the batched decode path (batch.cu): one step of p.L layers for p.B sequences
struct Prog;
int batch_decode(const Prog& p, cudaStream_t stream);

}  // namespace edge0
