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
constexpr int kF16Unit = 2048;       // fp16 unit: 16 rows x 64 inputs
constexpr int kFragPerGroup = 64;    // halves of one token's B fragments per group

inline __host__ __device__ int ceil_div(int a, int b) { return (a + b - 1) / b; }
inline __host__ __device__ long long q4_bytes(int out, int in) {
    return (long long)ceil_div(out, kRowTile) * (in / kGroup) * kQ4Unit;
}
inline __host__ __device__ long long f16_bytes(int out, int in) {
    return (long long)ceil_div(out, kRowTile) * (in / kGroup) * kF16Unit;
}

// --------------------------------------------------------------- engine ----
constexpr int kConsumerWarps = 16;
constexpr int kThreads = (kConsumerWarps + 1) * 32;   // + one producer warp
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kStageBytes = 16384;
constexpr int kStages = 8;
constexpr int kMaxSeg = 40;
constexpr int kSaccRows = 32 * kRowTile;               // rows one chunk can touch

enum Mode : int { MODE_DECODE = 0, MODE_MOE = 1, MODE_HEAD = 2 };

enum LayerFlags : int {
    LF_PREROUTED = 1,
    LF_HEAD = 2,
    LF_LORA = 4,
    LF_SHARED = 8,
};

struct LayerP {
    const char* gate;       // packed int4 stacks (expert stride q4_bytes)
    const char* up;
    const char* down;
    const char* sh_gate;
    const char* sh_up;
    const char* sh_down;
    const int* slot_table;
    int n_slots;
    const char* router;     // packed fp16 [E x d]
    const char* lora_Ag;    // packed fp16 [r x d]
    const char* lora_Au;
    const char* lora_Ad;    // packed fp16 [r x Is]
    const __half* lora_Bg;  // [Is, r]
    const __half* lora_Bu;
    const __half* lora_Bd;  // [d, r]
    const char* fc1;        // packed fp16 [H x d]
    const __half* fc1_oh;   // [2E, H]
    const char* fc2;        // packed fp16 [E x H]
    const char* linit;      // packed fp16 [E x d]
    const __half* linit_oh; // [2E, E]
    const __half* gamma;
    const float* bias;      // this layer's routing bias (or null)
    const float* head_bias; // head target's routing bias (or null)
    float eps;
    float lora_scale;       // alpha / r
    float route_scale, head_route_scale;
    int route_kind, n_groups, topk_groups;
    int head_route_kind, head_n_groups, head_topk_groups;
    int flags;
    int head_target;        // state row
    int sidx;               // state row of this layer
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
    long long ws_set_floats;  // floats per accumulator set
    LayerP layers[EDGE0_MAX_LAYERS];
};

// Workspace header (first 256 bytes)
struct WsHeader {
    unsigned long long barrier;   // monotonically increasing arrival counter
    unsigned int pc;              // phase counter (accumulator ring position)
    int step;                     // auto step counter
    int error;                    // EDGE0_* status recorded by a kernel
    int abort;                    // set with error: every wait gives up
    int trace;                    // non-zero: record phase timestamps in the trace area
};
constexpr int kWsHeaderBytes = 256;
// trace area (after the residual buffers): per CTA kTraceSlots u64 globaltimer stamps
constexpr int kTraceCtas = 160;
constexpr int kTraceSlots = 1024;   // (tag, time) pairs

// Accumulator set layout (floats), per token b:
struct AccLayout {
    long long gu, gus, aacc, z, lin, y, logr, logh, total;   // offsets of [B] blocks
};
inline __host__ __device__ AccLayout acc_layout(int B, int K, int I, int Is, int r, int H, int E, int d) {
    AccLayout a;
    long long o = 0;
    a.gu = o;   o += (long long)B * K * 2 * I;
    a.gus = o;  o += (long long)B * 2 * Is;
    a.aacc = o; o += (long long)B * 2 * ceil_div(r, 16) * 16;
    a.z = o;    o += (long long)B * H;
    a.lin = o;  o += (long long)B * E;
    a.y = o;    o += (long long)B * d;
    a.logr = o; o += (long long)B * E;
    a.logh = o; o += (long long)B * E;
    a.total = (o + 63) / 64 * 64;
    return a;
}
// workspace: header | 3 accumulator sets | 2 residual buffers [B, d] fp16
inline __host__ __device__ long long ws_bytes(int B, int K, int I, int Is, int r, int H, int E, int d) {
    AccLayout a = acc_layout(B, K, I, Is, r, H, E, d);
    return kWsHeaderBytes + 3 * a.total * 4 + 2LL * B * d * 2 + 256 +
           (long long)kTraceCtas * kTraceSlots * 8;
}

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
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::);
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;\n" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
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

__device__ __forceinline__ void red_add_f32(float* p, float v) {
    asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;\n" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ void red_release_add_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;\n" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];\n" : "=l"(v) : "l"(p) : "memory");
    return v;
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

// position of group-local input o (0..15 within a 16-input quarter) in the
// lane's 16 B-fragment halves; the map is its own inverse
__device__ __forceinline__ int frag_pos(int o) {
    const int lo = o & 7;
    const int m = (lo == 1) ? 4 : (lo == 4) ? 1 : (lo == 3) ? 6 : (lo == 6) ? 3 : lo;
    return (o & 8) | m;
}

// Write one group (64 inputs) of B fragments: lane holds inputs lane and lane+32.
// Odd inputs (those the int4 masks deliver as 16 q 2^-24) are stored divided by 16.
// With `lo` non-null the value is split v = hi + lo * 2^-11 (hi = fp16(v), lo =
// fp16((v - hi) * 2^11)); the two halves go to two tensor-core columns so the
// products keep ~22 bits of the fp32 activation.  Sums are of the represented
// values (hi, and v - hi).
constexpr float kLoScale = 2048.0f;
constexpr float kLoInv = 1.0f / 2048.0f;

__device__ __forceinline__ void put_one(__half* frag, int j, __half h) {
    const int o = j & 15;
    frag[(j >> 4) * 16 + frag_pos(o)] = (o & 1) ? __float2half_rn(__half2float(h) * 0.0625f) : h;
}

__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
    for (int k = 16; k; k >>= 1) s += __shfl_xor_sync(0xffffffffu, s, k);
    return s;
}

__device__ __forceinline__ void put_group(__half* frag, float* sum_out, float v0, float v1,
                                          int lane, __half* lo = nullptr,
                                          float* lo_sum_out = nullptr) {
    const __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1);
    put_one(frag, lane, h0);
    put_one(frag, lane + 32, h1);
    const float s = warp_sum(__half2float(h0) + __half2float(h1));
    if (lane == 0) *sum_out = s;
    if (lo) {
        const float r0 = v0 - __half2float(h0), r1 = v1 - __half2float(h1);
        put_one(lo, lane, __float2half_rn(r0 * kLoScale));
        put_one(lo, lane + 32, __float2half_rn(r1 * kLoScale));
        const float sl = warp_sum(r0 + r1);
        if (lane == 0) *lo_sum_out = sl;
    }
}

// engine entry (engine.cu)
__global__ void engine_kernel(const __grid_constant__ Prog prog);
int engine_smem_bytes(const Prog& p);

}  // namespace edge0
