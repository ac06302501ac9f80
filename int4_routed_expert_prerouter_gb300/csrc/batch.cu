// Batched decode path: one decode step for many independent sequences (B from
// EDGE0_MAX_BATCH + 1 up to EDGE0_MAX_BATCHED), the shape of the batched
// configurations (64 sequences on the 8B tier, 256 on the 35B tier).
//
// Per layer ("The Other Half of the Memory Wall", S3.1 "Math contract", S3.2
// "Prediction-as-routing", S3.3, App. A), as stream-ordered kernels:
//   k_norm      h = fp16(h + y_prev), x = fp16(RMSNorm(h) gamma), x group sums
//   routing     prediction (prerouted layers, step > 0) or own router
//               (k_dense + k_route)
//   k_dispatch  tokens grouped by expert: the active experts in id order, each
//               with its token list and routing weights
//   k_dense_pair  LoRA A_gate x, A_up x (shared expert), one launch
//   k_gu        gate/up of every active expert and the shared expert over
//               blocks of up to 32 of its tokens -> act = silu(g) up (fp32)
//   k_down      down of the same -> y += w act (fp32 reductions)
//   k_lora_vd   y += (alpha/r) B_down (A_down act_shared)
// and after the last layer h = fp16(h + y), then every head of the step (one
// flush per step: a head's prediction is consumed only at the next token):
//   z = fc1 x + executed / previous one-hot columns, GELU, logits = fc2 g +
//   linear_init x + its one-hot columns, top-K -> prediction for the next step,
// each stage one launch over all heads (k_dense_heads, k_onehot_heads,
// k_route_heads).
//
// The weights are the same packed layouts as the persistent engine's (int4
// nibbles enter mma.sync as fp16 subnormals q 2^-24, the epilogue rescales by
// s 2^24 and adds b times the group sum of the input; fp32 inputs enter as a
// hi + lo pair of fp16).  An expert's weights are read once per block of its
// tokens (32 for gate/up, 16 for down), not once per token: the contraction
// becomes a skinny GEMM over the block.
#include <string.h>

#include <vector>

#include "internal.cuh"
#include "common.cuh"
#include "tc05.cuh"

namespace edge0 {

// ---------------------------------------------------------------- layout ----
// work items of the expert kernels in the dispatch record (see Disp): at most
// B K / 8 (blocks of at least 8 positions) + one partial block per active
// expert + the shared expert's blocks, per kernel
__host__ __device__ inline int disp_cap(int B, int K, int E) {
    return (B * K + 7) / 8 + (B * K < E ? B * K : E) + (B + 7) / 8 + 2;
}
// bytes of the dispatch record's fixed part (Disp); the work items follow it
constexpr long long kDispHead = 8448;
// room for one head's job of the head flush (HeadJob)
constexpr long long kHeadJobBytes = 128;
BatchWs batch_ws_layout(int L, int B, int d, int E, int K, int I, int H) {
    BatchWs w;
    auto al = [](long long x) { return (x + 255) / 256 * 256; };
    long long o = kWsHeaderBytes;
    w.y = o;     o += al((long long)B * d * 4);
    w.xs = o;    o += al((long long)L * B * d * 2);
    w.xsum = o;  o += al((long long)B * (d / kGroup) * 4);
    w.lg = o;    o += al((long long)B * E * 4);
    // head flush: per head its fc1 output [B][H] then its logits [B][E] (the
    // heads of a step one run: one memset), then the heads' job table
    w.z = o;     o += al((long long)L * B * (H + E) * 4) + al((long long)L * kHeadJobBytes);
    w.la = o;    o += al((long long)B * 32 * 4);
    w.wsel = o;  o += al((long long)B * K * 4);
    w.exec = o;  o += al((long long)B * K * 4);
    w.disp = o;  o += al(kDispHead + 2LL * disp_cap(B, K, E) * 8);
    w.tok = o;   o += al((long long)B * K * 4);
    w.wt = o;    o += al((long long)B * K * 4);
    w.act = o;   o += al((long long)(B * K + B) * I * 4);
    w.total = o;
    return w;
}

namespace {

struct Disp {   // dispatch of one layer (device); fits the workspace's dispatch record
    int nact;
    int sexp[EDGE0_MAX_E + 1];
    int soff[EDGE0_MAX_E + 1];
    int scnt[EDGE0_MAX_E + 1];
    int sslot[EDGE0_MAX_E + 1];       // slot of each active expert (-1: host tier), read once per layer
    int n_gu, n_dn;                   // work items of k_gu / k_down
    int cap;                          // room for the items of each kernel
    // then, kDispHead bytes from the record's start, the work items (slot, first
    // position of a block): cap for k_gu, cap for k_down
};
static_assert(sizeof(Disp) <= kDispHead && kDispHead % 16 == 0, "the work items start 16-byte aligned after Disp");
__device__ __forceinline__ int2* gu_items(Disp* D) {
    return reinterpret_cast<int2*>(reinterpret_cast<char*>(D) + kDispHead);
}
__device__ __forceinline__ int2* dn_items(Disp* D) { return gu_items(D) + D->cap; }
__device__ __forceinline__ const int2* gu_items(const Disp* D) {
    return reinterpret_cast<const int2*>(reinterpret_cast<const char*>(D) + kDispHead);
}
__device__ __forceinline__ const int2* dn_items(const Disp* D) { return gu_items(D) + D->cap; }

__device__ __forceinline__ void record_error(WsHeader* hdr, int code) {
    atomicCAS(&hdr->error, 0, code);
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    const __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// ------------------------------------------------------------- k_norm -------
// One CTA per token.  add_y: h = fp16(h + y) and y = 0 (the previous layer's
// output); want_x: x = fp16(h rsqrt(mean h^2 + eps) gamma) into x_out and the
// sums of each 64-input group of x into xsum.
__global__ void __launch_bounds__(256) k_norm(__half* h, float* y, int add_y, const __half* gamma, float eps,
                                              int d, __half* x_out, float* xsum, int want_x, float* la) {
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (la && tid < 32) la[(long long)b * 32 + tid] = 0.f;   // the layer's LoRA A sums start at zero
    __half* hb = h + (long long)b * d;
    float* yb = y + (long long)b * d;
    float ss = 0.f;
    for (int i = 2 * tid; i < d; i += 512) {
        __half2 hv = *reinterpret_cast<const __half2*>(hb + i);
        if (add_y) {
            const float2 f = __half22float2(hv);
            const float2 yv = *reinterpret_cast<const float2*>(yb + i);
            hv = __floats2half2_rn(f.x + yv.x, f.y + yv.y);
            *reinterpret_cast<__half2*>(hb + i) = hv;
            *reinterpret_cast<float2*>(yb + i) = make_float2(0.f, 0.f);
        }
        const float2 f = __half22float2(hv);
        ss += f.x * f.x + f.y * f.y;
    }
    if (!want_x) return;
    __shared__ float red[8];
    __shared__ float rs;
    ss = warp_sum(ss);
    if (lane == 0) red[wid] = ss;
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        for (int w = 0; w < 8; ++w) s += red[w];
        rs = rsqrtf(s / (float)d + eps);
    }
    __syncthreads();
    const float r = rs;
    // 512 inputs per pass: warp w covers inputs [64 w, 64 w + 64) of the pass,
    // exactly one group
    for (int i = 2 * tid; i < d; i += 512) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(hb + i));
        float g0 = 1.f, g1 = 1.f;
        if (gamma) {
            const float2 gg = __half22float2(*reinterpret_cast<const __half2*>(gamma + i));
            g0 = gg.x;
            g1 = gg.y;
        }
        const __half2 xv = __floats2half2_rn(f.x * r * g0, f.y * r * g1);
        *reinterpret_cast<__half2*>(x_out + (long long)b * d + i) = xv;
        const float2 xf = __half22float2(xv);
        const float s = warp_sum(xf.x + xf.y);
        if (lane == 0) xsum[(long long)b * (d / kGroup) + i / kGroup] = s;
    }
}

// ------------------------------------------------------------- k_dense ------
// out[b][o] += sum_k W[o][k] X[b][k] for rows o < N and tokens b < B (the caller
// zeroes `out` where it does not accumulate).  W packed fp16: kmajor = 0:
// [half][16-row tile][group of the half][4 steps x 512 B] (2 KB units);
// kmajor = 1: [16-input step][row tile] x 512 B.  X: fp16 [B][ldx] (xh) or fp32
// (xf, entered as hi + lo fp16).  One CTA per (row tile, 32 tokens, 256-input
// chunk); its 4 warps split the chunk's 16 steps; fp32 reductions into out.
template <bool F32IN>
__device__ __forceinline__ void dense_tile(const char* __restrict__ W, int kmajor, int N, int Kin,
                                           const __half* __restrict__ xh, const float* __restrict__ xf, int ldx,
                                           int B, float* out, int ldo, int rt, int tb, int kc) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, g = lane >> 2, t = lane & 3;
    const int nks = Kin / 16, RT = (N + 15) / 16, hn = Kin / kGroup / 2;
    const int ks1 = nks < kc * 16 + 16 ? nks : kc * 16 + 16;
    float acc[4][4], accl[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[n][e] = accl[n][e] = 0.f;
#pragma unroll 4
    for (int ks = kc * 16 + wid; ks < ks1; ks += 4) {
        const char* ap;
        if (kmajor) {
            ap = W + ((long long)ks * RT + rt) * kF16Step;
        } else {
            const int gg = ks >> 2, s = ks & 3, h = gg / hn, gl = gg - h * hn;
            ap = W + ((long long)(h * RT + rt) * hn + gl) * kF16Unit + s * kF16Step;
        }
        const uint4 av = __ldg(reinterpret_cast<const uint4*>(ap + 16 * lane));
        const uint32_t A[4] = {av.x, av.y, av.z, av.w};
        const int k0 = ks * 16 + 2 * t;
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const int tok = tb + n * 8 + g;
            uint32_t b0 = 0u, b1 = 0u, l0 = 0u, l1 = 0u;
            if (tok < B) {
                if (!F32IN) {
                    b0 = __ldg(reinterpret_cast<const uint32_t*>(xh + (long long)tok * ldx + k0));
                    b1 = __ldg(reinterpret_cast<const uint32_t*>(xh + (long long)tok * ldx + k0 + 8));
                } else {
                    const float2 f0 = __ldg(reinterpret_cast<const float2*>(xf + (long long)tok * ldx + k0));
                    const float2 f1 = __ldg(reinterpret_cast<const float2*>(xf + (long long)tok * ldx + k0 + 8));
                    const __half2 h0 = __floats2half2_rn(f0.x, f0.y), h1 = __floats2half2_rn(f1.x, f1.y);
                    const float2 r0 = __half22float2(h0), r1 = __half22float2(h1);
                    b0 = *reinterpret_cast<const uint32_t*>(&h0);
                    b1 = *reinterpret_cast<const uint32_t*>(&h1);
                    l0 = pack_h2((f0.x - r0.x) * kLoScale, (f0.y - r0.y) * kLoScale);
                    l1 = pack_h2((f1.x - r1.x) * kLoScale, (f1.y - r1.y) * kLoScale);
                }
            }
            mma_16816(acc[n], A, b0, b1);
            if (F32IN) mma_16816(accl[n], A, l0, l1);
        }
    }
    __shared__ float red[4][16][33];
#pragma unroll
    for (int n = 0; n < 4; ++n) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = F32IN ? acc[n][e] + accl[n][e] * kLoInv : acc[n][e];
        red[wid][g][n * 8 + 2 * t] = v[0];
        red[wid][g][n * 8 + 2 * t + 1] = v[1];
        red[wid][g + 8][n * 8 + 2 * t] = v[2];
        red[wid][g + 8][n * 8 + 2 * t + 1] = v[3];
    }
    __syncthreads();
    for (int i = tid; i < 16 * 32; i += 128) {
        const int r = i >> 5, c = i & 31;
        const int row = rt * 16 + r, tok = tb + c;
        if (row < N && tok < B)
            red_add_f32(out + (long long)tok * ldo + row, (red[0][r][c] + red[1][r][c]) + (red[2][r][c] + red[3][r][c]));
    }
}


template <bool F32IN>
__global__ void __launch_bounds__(128) k_dense(const char* __restrict__ W, int kmajor, int N, int Kin,
                                               const __half* __restrict__ xh, const float* __restrict__ xf,
                                               int ldx, int B, float* out, int ldo) {
    dense_tile<F32IN>(W, kmajor, N, Kin, xh, xf, ldx, B, out, ldo, blockIdx.x, blockIdx.y * 32, blockIdx.z);
}

// Two fp16-input matrices of the same shape against the same x in one launch:
// row tiles [0, RT) of W0 into out, row tiles [RT, 2 RT) of W1 into out + off1
// (the shared expert's A_gate x and A_up x).
__global__ void __launch_bounds__(128) k_dense_pair(const char* __restrict__ W0, const char* __restrict__ W1,
                                                    int N, int Kin, const __half* __restrict__ xh, int ldx, int B,
                                                    float* out, int ldo, int off1) {
    const int RT = (N + 15) / 16, second = blockIdx.x >= RT;
    dense_tile<false>(second ? W1 : W0, 0, N, Kin, xh, nullptr, ldx, B, second ? out + off1 : out, ldo,
                      blockIdx.x - (second ? RT : 0), blockIdx.y * 32, blockIdx.z);
}

// ------------------------------------------------------------ head flush ----
// Every head of a step runs in one launch per stage (fc1, one-hot + GELU, fc2,
// linear_init, one-hot, routing): blockIdx.z (or .y) selects the head's job.
struct HeadJob;
struct HeadJob {
    const char* fc1;
    const __half* fc1_oh;
    const char* fc2;
    const char* linit;
    const __half* linit_oh;
    const __half* x;           // the head layer's x [B][d]
    const int32_t* exec;       // its executed ids [B][K]
    const int32_t* prev;       // the previous step's (or null)
    int32_t* pred_ids;         // the prediction's rows [B][K]
    float* pred_w;
    const float* bias;         // the target layer's routing bias (or null)
    float scale;
    int kind, ng, G;
};
static_assert(sizeof(HeadJob) <= kHeadJobBytes, "a head job fits its room in the workspace");
enum HeadStage : int { HS_FC1 = 0, HS_FC2 = 1, HS_LINIT = 2 };
template <bool F32IN>
__global__ void __launch_bounds__(128) k_dense_heads(const HeadJob* __restrict__ jobs, int stage, int nkc, int N,
                                                     int Kin, int B, const float* zbase, long long zstride,
                                                     float* obase, int ldo, long long ostride) {
    const int h = blockIdx.z / nkc, kc = blockIdx.z - h * nkc;
    const HeadJob& J = jobs[h];
    const char* W = stage == HS_FC1 ? J.fc1 : stage == HS_FC2 ? J.fc2 : J.linit;
    dense_tile<F32IN>(W, stage == HS_FC2 ? 1 : 0, N, Kin, F32IN ? nullptr : J.x,
                      F32IN ? zbase + h * zstride : nullptr, Kin, B, obase + h * ostride, ldo, blockIdx.x,
                      blockIdx.y * 32, kc);
}

// ----------------------------------------------------------- k_onehot -------
// z[b][n] += sum over executed e of M[e][n] + sum over previous e of M[E + e][n]
// (M = [2E][N] fp16: the one-hot columns of a head matrix, transposed), then
// GELU (erf form) if `gelu`.
__device__ __forceinline__ void onehot_col(float* z, int ldz, int N, const __half* __restrict__ M,
                                           const int32_t* ids, const int32_t* prev, int K, int E, int gelu, int b,
                                           int n) {
    if (n >= N) return;
    // (ids outside [0, E) were recorded as errors by the dispatch; read column 0)
    auto col = [E](int e) { return e >= 0 && e < E ? e : 0; };
    float oh = 0.f;
    for (int k = 0; k < K; ++k) oh += __half2float(M[(long long)col(ids[b * K + k]) * N + n]);
    if (prev)
        for (int k = 0; k < K; ++k) oh += __half2float(M[(long long)(E + col(prev[b * K + k])) * N + n]);
    float v = z[(long long)b * ldz + n] + oh;
    if (gelu) v = 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
    z[(long long)b * ldz + n] = v;
}
// the heads' one-hot columns: of fc1 with GELU (linit = 0) or of linear_init
__global__ void k_onehot_heads(const HeadJob* __restrict__ jobs, int linit, float* zbase, long long zstride, int N,
                               int K, int E) {
    const HeadJob& J = jobs[blockIdx.z];
    onehot_col(zbase + blockIdx.z * zstride, N, N, linit ? J.linit_oh : J.fc1_oh, J.exec, J.prev, K, E, !linit,
               blockIdx.y, blockIdx.x * blockDim.x + threadIdx.x);
}

// ------------------------------------------------------------ k_route -------
// Routing rule of App. A, one token per warp, 8 warps per CTA.
__device__ __forceinline__ void route_rows(const float* logits, int ldl, int B, int E, int K, int kind, int ng,
                                           int G, float scale, const float* bias, int32_t* ids_out, float* w_out) {
    extern __shared__ float sm[];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, b = blockIdx.x * 8 + wid;
    float* lg = sm + wid * 3 * E;
    int* rid = reinterpret_cast<int*>(sm + 8 * 3 * E) + wid * EDGE0_MAX_K;
    float* rw = sm + 8 * 3 * E + 8 * EDGE0_MAX_K + wid * EDGE0_MAX_K;
    if (b >= B) return;
    float v[EDGE0_MAX_E / 32];   // all of the warp's loads in flight at once
#pragma unroll
    for (int i = 0; i < EDGE0_MAX_E / 32; ++i)
        if (lane + 32 * i < E) v[i] = logits[(long long)b * ldl + lane + 32 * i];
#pragma unroll
    for (int i = 0; i < EDGE0_MAX_E / 32; ++i)
        if (lane + 32 * i < E) lg[lane + 32 * i] = v[i];
    __syncwarp();
    warp_route(lg, E, K, kind, ng, G, scale, bias, lg + E, rid, rw, lane);
    if (lane < K) {
        ids_out[b * K + lane] = rid[lane];
        w_out[b * K + lane] = rw[lane];
    }
}
__global__ void __launch_bounds__(256) k_route(const float* logits, int ldl, int B, int E, int K, int kind,
                                               int ng, int G, float scale, const float* bias, int32_t* ids_out,
                                               float* w_out) {
    route_rows(logits, ldl, B, E, K, kind, ng, G, scale, bias, ids_out, w_out);
}
__global__ void __launch_bounds__(256) k_route_heads(const HeadJob* __restrict__ jobs, const float* lbase,
                                                     long long lstride, int B, int E, int K) {
    const HeadJob& J = jobs[blockIdx.y];
    route_rows(lbase + blockIdx.y * lstride, E, B, E, K, J.kind, J.ng, J.G, J.scale, J.bias, J.pred_ids, J.pred_w);
}

// --------------------------------------------------------- k_dispatch -------
// The active experts of a layer in id order, each with the positions of its
// (token, weight) pairs; one CTA.  An id outside [0, E) records EDGE0_EINVAL
// and counts as expert 0.
__global__ void __launch_bounds__(1024) k_dispatch(const int32_t* ids, int32_t* ids_copy, const float* w, int B,
                                                   int K, int E, int shared, int blk_gu, int blk_dn, int cap,
                                                   const int* table, unsigned long long* tier, Disp* D, int* tok,
                                                   float* wt, WsHeader* hdr) {
    __shared__ int cnt[EDGE0_MAX_E], off[EDGE0_MAX_E], fill[EDGE0_MAX_E];
    __shared__ int n_host;
    const int tid = threadIdx.x, n = B * K;
    if (tid == 0) {
        D->cap = cap;
        n_host = 0;
    }
    for (int e = tid; e < E; e += blockDim.x) cnt[e] = fill[e] = 0;
    __syncthreads();
    for (int p = tid; p < n; p += blockDim.x) {
        int e = ids[p];
        if (ids_copy) ids_copy[p] = e;   // a prediction becomes the layer's executed ids
        if (e < 0 || e >= E) { record_error(hdr, EDGE0_EINVAL); e = 0; }
        atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    // exclusive scans over the experts (thread e owns expert e): position offset,
    // slot index, and the first work item of each kernel
    __shared__ int sc_wsum[4][32];
    const int e = tid;
    const int c_e = e < E ? cnt[e] : 0;
    int v[4] = {c_e, c_e > 0 ? 1 : 0, (c_e + blk_gu - 1) / blk_gu, (c_e + blk_dn - 1) / blk_dn};
    int incl[4];
    const int lane = tid & 31, wid = tid >> 5;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        int x = v[q];
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        incl[q] = x;
        if (lane == 31) sc_wsum[q][wid] = x;
    }
    __syncthreads();
    if (wid == 0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            int x = lane < (int)(blockDim.x >> 5) ? sc_wsum[q][lane] : 0;
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            sc_wsum[q][lane] = x;   // inclusive over warps
        }
    }
    __syncthreads();
    int ex[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) ex[q] = incl[q] - v[q] + (wid > 0 ? sc_wsum[q][wid - 1] : 0);
    const int nwarps = blockDim.x >> 5;
    const int a = sc_wsum[1][nwarps - 1];   // active experts
    if (e < E) {
        off[e] = ex[0];
        if (c_e > 0) {
            const int j = ex[1];
            D->sexp[j] = e;
            D->soff[j] = ex[0];
            D->scnt[j] = c_e;
            // the slot table is read once per layer: a copy published later in
            // the layer does not change where its kernels read the expert
            int sl = e;
            if (table) {
                sl = (int)ld_acquire_u32(reinterpret_cast<const unsigned*>(table + e));
                if (sl == -1) atomicAdd(&n_host, 1);
            }
            D->sslot[j] = sl;
            for (int i = 0; i < v[2]; ++i) gu_items(D)[ex[2] + i] = make_int2(j, i * blk_gu);
            for (int i = 0; i < v[3]; ++i) dn_items(D)[ex[3] + i] = make_int2(j, i * blk_dn);
        }
    }
    if (tid == 0) {
        // the shared expert's work items after the routed ones (slot a)
        int ng = sc_wsum[2][nwarps - 1], nd = sc_wsum[3][nwarps - 1];
        if (shared) {
            for (int tb = 0; tb < B; tb += blk_gu) gu_items(D)[ng++] = make_int2(a, tb);
            for (int tb = 0; tb < B; tb += blk_dn) dn_items(D)[nd++] = make_int2(a, tb);
        }
        D->nact = a;
        D->n_gu = ng;
        D->n_dn = nd;
    }
    __syncthreads();
    if (tid == 0 && tier && table) {   // residency counters: active routed experts, of them in the host tier
        atomicAdd(&tier[0], (unsigned long long)a);
        atomicAdd(&tier[1], (unsigned long long)n_host);
    }
    for (int p = tid; p < n; p += blockDim.x) {
        int e = ids[p];
        if (e < 0 || e >= E) e = 0;
        const int pos = off[e] + atomicAdd(&fill[e], 1);
        tok[pos] = p / K;
        wt[pos] = w[p];
    }
}

// One expert of a layer for a CTA: blockIdx.y < nact is a routed expert (its
// weights through the slot table), blockIdx.y == nact the shared expert (every
// token, weight 1).  False: nothing to do.
struct Slot {
    const char* gu;
    const char* dn;
    int I, m, pos0;
    const int* toks;     // token of each position (null: position = token)
    const float* wts;    // weight of each position (null: 1)
    bool shared;
    bool host;           // weights in the host tier
};
__device__ __forceinline__ bool slot_of(int j, const Disp* D, const LayerP& Ly, int B, int K, int d, int I,
                                        int Is, const int* tok, const float* wt, WsHeader* hdr, Slot& s) {
    const int nact = D->nact;
    if (j < nact) {
        const int e = D->sexp[j];
        const int sl = D->sslot[j];
        s.host = false;
        if (sl == -1 && Ly.gu_host) {
            // host tier: the expert's weights are read from pinned host memory
            s.gu = Ly.gu_host + (long long)e * q4_bytes(2 * I, d);
            s.dn = Ly.down_host + (long long)e * q4_bytes(d, I);
            s.host = true;
        } else if (sl < 0 || sl >= Ly.n_slots) {
            if (threadIdx.x == 0) record_error(hdr, EDGE0_EINVAL);
            return false;
        } else {
            s.gu = Ly.gu + (long long)sl * q4_bytes(2 * I, d);
            s.dn = Ly.down + (long long)sl * q4_bytes(d, I);
        }
        s.I = I;
        s.m = D->scnt[j];
        s.pos0 = D->soff[j];
        s.toks = tok + s.pos0;
        s.wts = wt + s.pos0;
        s.shared = false;
        return true;
    }
    if (j == nact && Ly.sh_gu) {
        s.gu = Ly.sh_gu;
        s.dn = Ly.sh_down;
        s.I = Is;
        s.m = B;
        s.pos0 = B * K;
        s.toks = nullptr;
        s.wts = nullptr;
        s.shared = true;
        s.host = false;
        return true;
    }
    return false;
}

// Experts run in CTAs of 8 warps, one 16-row tile each, over blocks of tokens
// of one expert: the block's B operand (x rows, or act fragments as hi + lo
// fp16) is staged in shared memory once per CTA; each warp streams its tile's
// 576-byte int4 slices group by group through a 4-stage ring in shared memory
// (cp.async for device-resident experts, plain loads for host-tier ones), three
// groups in flight.
constexpr int kExpWarps = 8;   // warps of a down CTA
constexpr int kGuWarps = 16;   // warps of a gate/up CTA
constexpr int kGuTok = 32;     // tokens per gate/up block (4 mma column tiles)
constexpr int kGuNt = kGuTok / 8;
constexpr int kGuStages = 8;   // gate/up ring depth per warp: 7 groups in flight
constexpr int kDnTok = 16;     // tokens per down block (4 tiles of 4 tokens x hi/lo)
constexpr int kStages = 4;
constexpr int kSlice = 576;   // one group of one row tile: 512 B of nibbles + 64 B of (s, b)

__device__ __forceinline__ void cp16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// four 8x8 b16 matrices from shared memory (lane l gives the row address of
// matrix l / 8, row l % 8; register i holds matrix i's fragment)
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t r[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_wait_1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }
__device__ __forceinline__ void cp_wait_2() { asm volatile("cp.async.wait_group 2;\n" ::: "memory"); }
__device__ __forceinline__ void cp_wait_6() { asm volatile("cp.async.wait_group 6;\n" ::: "memory"); }
__device__ __forceinline__ void cp_wait_0() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// one 16-byte piece of a slice into the ring: asynchronous from device memory,
// a plain load + store from the host tier
__device__ __forceinline__ void piece(void* dst, const char* src, bool host) {
    if (!host) cp16(dst, src);
    else *reinterpret_cast<uint4*>(dst) = __ldg(reinterpret_cast<const uint4*>(src));
}

// --------------------------------------------------------------- k_gu -------
// gate/up of one expert for a block of up to 32 of its tokens: warp w of CTA x
// takes the interleaved 16-row tile 16 x + w (gate rows of act rows
// 8 (16 x + w) .. + 7 and the same up rows) over all of d, and runs each int4
// fragment against the block's 4 token column tiles (the nibble masks are taken
// once per fragment).  act[position][row] = silu(gate) up (the shared expert's
// gate and up with their LoRA terms (alpha/r) B (A x), A x precomputed in la).
// Each warp streams its tile's 576-byte slices group by group through an
// 8-stage ring (7 groups in flight), started before the token rows are staged.
// Dynamic shared memory: x rows [kGuTok][d + 8] fp16 (padded: conflict-free
// fragment reads), x group sums [kGuTok][d/64], ring [16 warps][8][576 B].
__global__ void __launch_bounds__(kGuWarps * 32) k_gu(const LayerP Ly, const Disp* D, const int* tok,
                                                      const float* wt, const __half* __restrict__ x,
                                                      const float* __restrict__ xsum, const float* la, int lora,
                                                      int r, int B, int K, int d, int I, int Is, int Imax,
                                                      float* act, WsHeader* hdr) {
    extern __shared__ __align__(16) char gsm[];
    auto run_item = [&](const int2 item, const Slot& S) {
    constexpr int NT = kGuWarps * 32;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, g = lane >> 2, t = lane & 3;
    const int n_gd = d / kGroup, hn = n_gd / 2, RTI = S.I / kHalfRow, ld = d + 8;
    __half* xrow = reinterpret_cast<__half*>(gsm);
    float* xss = reinterpret_cast<float*>(gsm + kGuTok * ld * 2);
    char* ring = gsm + kGuTok * ld * 2 + kGuTok * n_gd * 4 + wid * kGuStages * kSlice;
    const int rt = blockIdx.x * kGuWarps + wid;
    const bool live = rt < RTI;
    // the tile's units in group order: half 0's groups, then half 1's (the source
    // advances by one unit, and jumps to the other half once)
    const char* nxt = S.gu + (long long)rt * hn * kQ4Unit;
    int gn = 0;   // groups filled so far
    auto fill = [&]() {
        if (gn < n_gd) {
            char* dst = ring + (gn & (kGuStages - 1)) * kSlice;
            piece(dst + 16 * lane, nxt + 16 * lane, S.host);
            if (lane < 4) piece(dst + 512 + 16 * lane, nxt + 512 + 16 * lane, S.host);
            nxt += kQ4Unit;
            if (++gn == hn) nxt += (long long)(RTI - 1) * hn * kQ4Unit;
        }
        cp_commit();
    };
    // the weight stream first: it does not depend on the token rows
    if (live)
        for (int j = 0; j < kGuStages - 1; ++j) fill();
    const int tb = item.y;
    {
        // the block's token rows and group sums: 16 threads per token, every load
        // of a pass issued before any store (one round trip per pass)
        static_assert(kGuTok * 16 == NT, "16 threads per token");
        const int q = tid >> 4, j = tid & 15, p = tb + q;
        const bool valid = p < S.m;
        const long long row = valid ? (S.toks ? S.toks[p] : p) : 0;
        const uint4* src = reinterpret_cast<const uint4*>(x + row * d);
        const int nc = d / 8;
        for (int c0 = 0; c0 < nc; c0 += 16 * 16) {
            uint4 v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int c = c0 + j + 16 * i;
                v[i] = valid && c < nc ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
            }
            float xv[2] = {0.f, 0.f};
            if (c0 == 0)
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    if (valid && j + 16 * i < n_gd) xv[i] = __ldg(xsum + row * n_gd + j + 16 * i);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int c = c0 + j + 16 * i;
                if (c < nc) *reinterpret_cast<uint4*>(xrow + q * ld + c * 8) = v[i];
            }
            if (c0 == 0)
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    if (j + 16 * i < n_gd) xss[q * n_gd + j + 16 * i] = xv[i];
        }
        for (int gg = j + 32; gg < n_gd; gg += 16)   // d > 2048 only
            xss[q * n_gd + gg] = valid ? __ldg(xsum + row * n_gd + gg) : 0.f;
    }
    __syncthreads();
    if (!live) return;
    float racc[kGuNt][4];
#pragma unroll
    for (int n = 0; n < kGuNt; ++n) racc[n][0] = racc[n][1] = racc[n][2] = racc[n][3] = 0.f;
    // B fragments by ldmatrix: lane l addresses row l % 8 of 8x8 matrix l / 8;
    // matrices (tokens 8 n .. + 7) x (k 0..7 | 8..15) for n-tile pairs
    const uint32_t xl = smem_u32(xrow + (8 * ((lane >> 3) >> 1) + (lane & 7)) * ld + 8 * ((lane >> 3) & 1));
    for (int gg = 0; gg < n_gd; ++gg) {
        cp_wait_6();
        __syncwarp();
        const char* u = ring + (gg & (kGuStages - 1)) * kSlice;
        const uint4 wv = *reinterpret_cast<const uint4*>(u + 16 * lane);
        const uint2 sc = *reinterpret_cast<const uint2*>(u + 512 + 8 * g);
        __syncwarp();
        fill();
        const uint32_t wq[4] = {wv.x, wv.y, wv.z, wv.w};
        float acc[kGuNt][4];
#pragma unroll
        for (int n = 0; n < kGuNt; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            uint32_t A[4];
            q4_masks(wq[s], A);
#pragma unroll
            for (int n2 = 0; n2 < kGuNt / 2; ++n2) {
                uint32_t b[4];
                ldsm_x4(xl + (uint32_t)((16 * n2 * ld + gg * kGroup + s * 16) * 2), b);
                mma_16816(acc[2 * n2], A, b[0], b[1]);
                mma_16816(acc[2 * n2 + 1], A, b[2], b[3]);
            }
        }
        const __half2 s0 = *reinterpret_cast<const __half2*>(&sc.x);   // (s, b) of row g
        const __half2 s1 = *reinterpret_cast<const __half2*>(&sc.y);   // (s, b) of row g + 8
        const float a0 = __low2float(s0) * kTwo24, b0 = __high2float(s0);
        const float a1 = __low2float(s1) * (kTwo24 / 16.0f), b1 = __high2float(s1);
#pragma unroll
        for (int n = 0; n < kGuNt; ++n) {
            const float xs0 = xss[(8 * n + 2 * t) * n_gd + gg], xs1 = xss[(8 * n + 2 * t + 1) * n_gd + gg];
            racc[n][0] += a0 * acc[n][0] + b0 * xs0;
            racc[n][1] += a0 * acc[n][1] + b0 * xs1;
            racc[n][2] += a1 * acc[n][2] + b1 * xs0;
            racc[n][3] += a1 * acc[n][3] + b1 * xs1;
        }
    }
    cp_wait_0();
    const int arow = rt * kHalfRow + g;
#pragma unroll
    for (int n = 0; n < kGuNt; ++n)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int q = tb + 8 * n + 2 * t + c;
            if (q >= S.m) continue;
            float gate = racc[n][c], up = racc[n][2 + c];
            if (S.shared && lora) {
                const int b = S.toks ? S.toks[q] : q;
                const __half* bg = Ly.lora_Bg + (long long)arow * r;
                const __half* bu = Ly.lora_Bu + (long long)arow * r;
                float dg = 0.f, du = 0.f;
                for (int qq = 0; qq < r; ++qq) {
                    dg += __half2float(bg[qq]) * la[b * 32 + qq];
                    du += __half2float(bu[qq]) * la[b * 32 + 16 + qq];
                }
                gate += Ly.lora_scale * dg;
                up += Ly.lora_scale * du;
            }
            act[(long long)(S.pos0 + q) * Imax + arow] = silu_f(gate) * up;
        }
    };
    // the CTAs of a column take the work items in turn (the grid is sized to the
    // GPU, not to the most items a layer can have)
    for (int yi = blockIdx.y; yi < D->n_gu; yi += gridDim.y) {   // CTA-uniform
        Slot S;
        const int2 item = gu_items(D)[yi];
        if (!slot_of(item.x, D, Ly, B, K, d, I, Is, tok, wt, hdr, S)) continue;
        run_item(item, S);
        __syncthreads();   // the staged token rows are reused by the next item
    }
}

// ------------------------------------------------------------ k_gu_tc -------
// gate/up of one expert for a block of up to 128 of its tokens on the fifth-
// generation tensor cores (prefill): CTA x takes the expert's 128-row tile x of
// interleaved gate/up rows (8 packed 16-row tiles: the gate rows of act rows
// 8 p .. 8 p + 7, then the same up rows, for p = 8 x .. 8 x + 7) over all of
// d, one group of 64 inputs (one K chunk) at a time:
//   * cp.async brings the chunk's 8 packed units and the block's token rows of
//     x (straight into the canonical K-major layout, zero rows past the
//     block's tokens) into one of three slots, two chunks ahead;
//   * every thread dequantizes one unit's lane slice (s q + b, rounded to fp16
//     once) from the slot into one of two A stages (canonical K-major layout);
//   * one thread issues four tcgen05.mma K-steps (M 128, N = the block's tokens
//     rounded up to 16, K 16) into a TMEM accumulator and commits to the A
//     stage's mbarrier, which frees the stage and the slot.
// The epilogue reads the accumulator (lane = row, column = token), pairs each
// gate row with its up row (8 lanes apart) and writes act[position][row] =
// silu(gate) up (the shared expert with its LoRA terms (alpha/r) B (A x), A x
// precomputed in la).
constexpr int kTcTok = 128;                  // tokens per block (MMA N at most)
constexpr int kTcThreads = 256;
constexpr int kTcA = 4 * 128 * 32;           // dequantized A of one K chunk (4 K-steps x 128 rows x 32 B)
constexpr int kTcB = 4 * kTcTok * 32;        // B of one K chunk
constexpr int kTcRaw = 8 * kQ4Unit;          // the chunk's 8 packed units
constexpr int kTcSlots = 4;                  // raw + B slots (chunks in flight)
constexpr int kTcSlot = kTcB + kTcRaw;       // B first: 1 KB aligned
constexpr int kTcSmem = kTcSlots * kTcSlot + 2 * kTcA;
constexpr unsigned long long kTcWait = 2000000000ull;

__device__ __forceinline__ unsigned long long tc_time() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// every thread: the barrier's phase of parity `par` has completed (bounded)
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t par) {
    if (mbar_try_wait(bar, par)) return true;
    const unsigned long long t0 = tc_time();
    while (!mbar_try_wait(bar, par))
        if (tc_time() - t0 > kTcWait) return false;
    return true;
}
// 16 bytes by cp.async, or 16 zero bytes (src_size 0)
__device__ __forceinline__ void cp16z(void* dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
// (s q + b) for the nibble pair (bits 0-3 and 16-19 of v): each nibble with
// exponent bits of 1024 is the fp16 1024 + q, exact; minus 1024 gives q; one
// fused multiply-add with the row's (s, b) rounds s q + b to fp16 once
__device__ __forceinline__ uint32_t deq2(uint32_t v, __half2 s2, __half2 b2) {
    const uint32_t m = (v & 0x000F000Fu) | 0x64006400u;
    const __half2 q = __hsub2(*reinterpret_cast<const __half2*>(&m), __float2half2_rn(1024.f));
    const __half2 h = __hfma2(q, s2, b2);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(kTcThreads) k_gu_tc(const LayerP Ly, const Disp* D, const int* tok, const float* wt,
                                                      const __half* __restrict__ x, const float* la, int lora, int r,
                                                      int B, int K, int d, int I, int Is, int Imax, float* act,
                                                      WsHeader* hdr) {
    extern __shared__ __align__(1024) char tsm[];
    __shared__ uint64_t bar[2];
    __shared__ uint32_t taddr_s;
    __shared__ int bad;
    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    const int mt = blockIdx.x, n_gd = d / kGroup, ng0 = n_gd / 2, ng1 = n_gd - ng0;
    char* slots = tsm;
    char* astage = tsm + kTcSlots * kTcSlot;
    if (wid == 0) {
        tc::tmem_alloc(&taddr_s, kTcTok);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
        bad = 0;
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t taddr = taddr_s;
    int cc = 0;   // K chunks whose MMAs this CTA issued (A stage = cc & 1; commit count of bar[s] = cc >> 1)
    for (int yi = blockIdx.y; yi < D->n_gu && !bad; yi += gridDim.y) {   // CTA-uniform
        Slot S;
        const int2 item = gu_items(D)[yi];
        if (!slot_of(item.x, D, Ly, B, K, d, I, Is, tok, wt, hdr, S) || S.host) continue;
        const int RT = S.I / kHalfRow;          // packed 16-row tiles of the expert
        if (mt * 8 >= RT) continue;             // this row tile lies beyond a narrower expert
        const int tb = item.y, m = min(kTcTok, S.m - tb), nb = (m + 15) & ~15;
        const uint32_t idesc = tc::idesc_f16(128, nb);
        // this thread's token pieces: token q = tid / 8 + 32 j, inputs 8 (tid % 8)
        // of the chunk; their x rows (fixed for the item) and shared-memory places
        const int c8 = tid & 7;
        long long xrow[4];
        uint32_t boff[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int q = (tid >> 3) + 32 * j;
            xrow[j] = q < m ? (long long)(S.toks ? S.toks[tb + q] : tb + q) * d : -1;
            boff[j] = (uint32_t)((c8 >> 1) * kTcTok * 32) + tc::kstep_off(q, (c8 & 1) * 8);
        }
        // the prefetch of chunk kc into slot kc % kTcSlots: the 8 units (288
        // pieces of 16 bytes) and the block's token rows (zeros past them)
        auto prefetch = [&](int kc) {
            if (kc < n_gd) {
                char* sl = slots + (kc % kTcSlots) * kTcSlot;
                const int h = kc >= ng0, gh = kc - h * ng0, ngh = h ? ng1 : ng0;
                const char* u0 = S.gu + (h ? (long long)RT * ng0 * kQ4Unit : 0LL) +
                                 ((long long)(mt * 8) * ngh + gh) * kQ4Unit;
                for (int i = tid; i < kTcRaw / 16; i += kTcThreads) {
                    const int uu = i / (kQ4Unit / 16), o = (i - uu * (kQ4Unit / 16)) * 16;
                    cp16(sl + kTcB + uu * kQ4Unit + o, u0 + (long long)uu * ngh * kQ4Unit + o);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int q = (tid >> 3) + 32 * j;
                    if (q < nb)
                        cp16z(sl + boff[j], x + (xrow[j] < 0 ? 0 : xrow[j]) + kc * kGroup + c8 * 8, xrow[j] >= 0);
                }
            }
            cp_commit();
        };
        prefetch(0);
        prefetch(1);
        const int u = tid >> 5, g8 = lane >> 2, t = lane & 3;
        const int row0 = u * 16 + g8, row1 = row0 + 8;
        const uint32_t o00 = tc::kstep_off(row0, 2 * t), o01 = tc::kstep_off(row0, 2 * t + 8);
        const uint32_t o10 = tc::kstep_off(row1, 2 * t), o11 = tc::kstep_off(row1, 2 * t + 8);
        for (int kc = 0; kc < n_gd; ++kc, ++cc) {
            const int st = cc & 1;
            char* sl = slots + (kc % kTcSlots) * kTcSlot;
            char* sA = astage + st * kTcA;
            // chunk kc's copies landed (every thread's, after the barrier); the A
            // stage and the slot of chunk kc + 2 (that of chunk kc - 2) are free
            // once the MMAs of the chunk two before completed (one thread waits)
            cp_wait_1();
            if (tid == 0 && cc >= 2 && !tc_wait(&bar[st], (uint32_t)(((cc - 2) >> 1) & 1))) bad = 1;
            __syncthreads();
            if (bad) break;
            {
                const char* unit = sl + kTcB + u * kQ4Unit;
                const uint4 wv = *reinterpret_cast<const uint4*>(unit + 16 * lane);
                const uint2 sc = *reinterpret_cast<const uint2*>(unit + 512 + 8 * g8);
                const __half2 sb0 = *reinterpret_cast<const __half2*>(&sc.x);   // (s, b) row g8
                const __half2 sb1 = *reinterpret_cast<const __half2*>(&sc.y);   // (s, b) row g8 + 8
                const __half2 s20 = __low2half2(sb0), b20 = __high2half2(sb0);
                const __half2 s21 = __low2half2(sb1), b21 = __high2half2(sb1);
                const uint32_t wq[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    char* a = sA + ks * 128 * 32;
                    const uint32_t w = wq[ks];
                    *reinterpret_cast<uint32_t*>(a + o00) = deq2(w, s20, b20);          // k 2t, 2t+1 of row g8
                    *reinterpret_cast<uint32_t*>(a + o01) = deq2(w >> 8, s20, b20);     // k 2t+8, 2t+9
                    *reinterpret_cast<uint32_t*>(a + o10) = deq2(w >> 4, s21, b21);     // row g8 + 8
                    *reinterpret_cast<uint32_t*>(a + o11) = deq2(w >> 12, s21, b21);
                }
            }
            tc::fence_async_smem();   // the generic-proxy writes (A) and the copies (B) to the tensor core
            prefetch(kc + 2);
            __syncthreads();
            if (tid == 0) {
                tc::fence_after_sync();
                const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sl);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_f16(taddr, tc::smem_desc(a0 + ks * 128 * 32), tc::smem_desc(b0 + ks * kTcTok * 32), idesc,
                                kc > 0 || ks > 0);
                tc::mma_commit(&bar[st]);
            }
        }
        cp_wait_0();   // the item's trailing (empty) copy groups
        if (bad) break;
        // the accumulator is complete once the last chunk's commit arrived
        if (tid == 0 && !tc_wait(&bar[(cc - 1) & 1], (uint32_t)(((cc - 1) >> 1) & 1))) bad = 1;
        __syncthreads();
        if (bad) break;
        tc::fence_after_sync();
        {
            // warp w: TMEM lanes 32 (w % 4) .. (rows: packed tiles 2 (w % 4), + 1),
            // columns (tokens) of half w / 4 of the block
            const int qd = wid & 3, c_lo = (wid >> 2) * (kTcTok / 2);
            const int tile = mt * 8 + 2 * qd + (lane >> 4);
            const int arow = tile * kHalfRow + (lane & 7);
            const bool gate_lane = (lane & 8) == 0;
            for (int c0 = c_lo; c0 < c_lo + kTcTok / 2 && c0 < nb; c0 += 8) {
                float v[8];
                tc::tmem_ld8(taddr + ((uint32_t)(32 * qd) << 16) + (uint32_t)c0, v);
                tc::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float other = __shfl_xor_sync(0xffffffffu, v[j], 8);
                    const int q = c0 + j;
                    if (!gate_lane || q >= m) continue;
                    float gate = v[j], up = other;
                    if (S.shared && lora) {
                        const int b = S.toks ? S.toks[tb + q] : tb + q;
                        const __half* bg = Ly.lora_Bg + (long long)arow * r;
                        const __half* bu = Ly.lora_Bu + (long long)arow * r;
                        float dg = 0.f, du = 0.f;
                        for (int qq = 0; qq < r; ++qq) {
                            dg += __half2float(bg[qq]) * la[b * 32 + qq];
                            du += __half2float(bu[qq]) * la[b * 32 + 16 + qq];
                        }
                        gate += Ly.lora_scale * dg;
                        up += Ly.lora_scale * du;
                    }
                    act[(long long)(S.pos0 + tb + q) * Imax + arow] = silu_f(gate) * up;
                }
            }
        }
        // every read of the accumulator done before the next item's MMAs overwrite it
        tc::fence_before_sync();
        __syncthreads();
    }
    cp_wait_0();
    if (bad && tid == 0) record_error(hdr, EDGE0_ETIMEOUT);
    tc::fence_before_sync();
    __syncthreads();
    if (wid == 0) tc::tmem_dealloc(taddr, kTcTok);
}

// ------------------------------------------------------------- k_down -------
// down of one expert for all of its tokens: warp w of CTA x takes the 16 output
// rows of row tile 8 x + w over all of the expert's act rows, 16 tokens per
// block (4 mma column tiles of 4 tokens x hi/lo); y[token] += w act_out (fp32
// reductions).  A warp's slice of group gg (its 4 step blocks of 128 B and its
// 64 B of scales) is gathered into the ring in the unit layout of gate/up.
// Dynamic shared memory: act fragments [I/64][4 steps][4 tiles][32 lanes] uint2,
// act group sums [kDnTok][I/64], ring [8 warps][4][576 B].
__global__ void __launch_bounds__(256, 3) k_down(const LayerP Ly, const Disp* D, const int* tok, const float* wt,
                                              const float* __restrict__ act, int B, int K, int d, int I, int Is,
                                              int Imax, float* y, WsHeader* hdr) {
    extern __shared__ __align__(16) char dsm[];
    auto run_item = [&](const int2 item, const Slot& S) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, g = lane >> 2, t = lane & 3;
    const int n_rtd = d / kRowTile, nh = n_rtd / 2, ngi = S.I / kGroup, ngmax = Imax / kGroup;
    uint2* afr = reinterpret_cast<uint2*>(dsm);
    float* qsm = reinterpret_cast<float*>(dsm + ngmax * 512 * 8);
    char* ring = dsm + ngmax * 512 * 8 + kDnTok * ngmax * 4 + wid * kStages * kSlice;
    const int rt = blockIdx.x * kExpWarps + wid;
    const bool live = rt < n_rtd;
    const int h = rt >= nh ? 1 : 0, i = rt - h * nh;
    auto fill = [&](int gg) {
        if (gg < ngi) {
            char* dst = ring + (gg & (kStages - 1)) * kSlice;
            const char* grp = S.dn + (long long)gg * n_rtd * kQ4Unit + (long long)h * nh * kQ4Unit;
            piece(dst + 16 * lane, grp + ((lane >> 3) * nh + i) * kQ4Quarter + 16 * (lane & 7), S.host);
            if (lane < 4) piece(dst + 512 + 16 * lane, grp + 4 * nh * kQ4Quarter + i * kQ4Scales + 16 * lane, S.host);
        }
        cp_commit();
    };
    // the weight stream first: it does not depend on the act rows
    if (live)
        for (int j = 0; j < kStages - 1; ++j) fill(j);
    {
        const int tb = item.y;
        // act fragments, 8 per thread and pass with every load of a pass issued
        // before any conversion (one round trip per pass)
        for (int e0 = 0; e0 < ngi * 512; e0 += 8 * 256) {
            float2 a0[8], a1[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = e0 + tid + 256 * i;
                const int ln = e & 31, n = (e >> 5) & 3, s = (e >> 7) & 3, gg = e >> 9;
                const int p = tb + n * 4 + (ln >> 3);
                a0[i] = a1[i] = make_float2(0.f, 0.f);
                if (e < ngi * 512 && p < S.m) {
                    const float* ar = act + (long long)(S.pos0 + p) * Imax + gg * kGroup + s * 16 + 2 * (ln & 3);
                    a0[i] = *reinterpret_cast<const float2*>(ar);
                    a1[i] = *reinterpret_cast<const float2*>(ar + 8);
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = e0 + tid + 256 * i;
                if (e >= ngi * 512) continue;
                const int part = ((e & 31) >> 2) & 1;
                const __half2 h0 = __floats2half2_rn(a0[i].x, a0[i].y), h1 = __floats2half2_rn(a1[i].x, a1[i].y);
                uint2 v;
                if (!part) {
                    v.x = *reinterpret_cast<const uint32_t*>(&h0);
                    v.y = *reinterpret_cast<const uint32_t*>(&h1);
                } else {
                    const float2 r0 = __half22float2(h0), r1 = __half22float2(h1);
                    v.x = pack_h2((a0[i].x - r0.x) * kLoScale, (a0[i].y - r0.y) * kLoScale);
                    v.y = pack_h2((a1[i].x - r1.x) * kLoScale, (a1[i].y - r1.y) * kLoScale);
                }
                afr[e] = v;
            }
        }
        for (int e = tid; e < kDnTok * ngi; e += 256) {
            const int q = e / ngi, gg = e - q * ngi, p = tb + q;
            float sum = 0.f;
            if (p < S.m) {
                const float4* ar = reinterpret_cast<const float4*>(act + (long long)(S.pos0 + p) * Imax + gg * kGroup);
                for (int k = 0; k < kGroup / 4; ++k) {
                    const float4 a = ar[k];
                    sum += (a.x + a.y) + (a.z + a.w);
                }
            }
            qsm[e] = sum;
        }
        __syncthreads();
        if (!live) return;
        float o[4][2];
#pragma unroll
        for (int n = 0; n < 4; ++n) o[n][0] = o[n][1] = 0.f;
        for (int gg = 0; gg < ngi; ++gg) {
            cp_wait_2();
            __syncwarp();
            const char* u = ring + (gg & (kStages - 1)) * kSlice;
            uint32_t wq[4];
#pragma unroll
            for (int s = 0; s < 4; ++s) wq[s] = *reinterpret_cast<const uint32_t*>(u + s * kQ4Quarter + 4 * lane);
            const uint2 sc = *reinterpret_cast<const uint2*>(u + 512 + 8 * g);
            __syncwarp();
            fill(gg + kStages - 1);
            float acc[4][4];
#pragma unroll
            for (int n = 0; n < 4; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                uint32_t A[4];
                q4_masks(wq[s], A);
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    const uint2 bb = afr[((gg * 4 + s) * 4 + n) * 32 + lane];
                    mma_16816(acc[n], A, bb.x, bb.y);
                }
            }
            const __half2 s0 = *reinterpret_cast<const __half2*>(&sc.x);
            const __half2 s1 = *reinterpret_cast<const __half2*>(&sc.y);
            const float sg0 = __low2float(s0) * kTwo24, bg0 = __high2float(s0);
            const float sg1 = __low2float(s1) * (kTwo24 / 16.0f), bg1 = __high2float(s1);
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const float qt = qsm[(n * 4 + t) * ngi + gg];   // group sum of the lane's C-column token
                o[n][0] += sg0 * (acc[n][0] + acc[n][1] * kLoInv) + bg0 * qt;
                o[n][1] += sg1 * (acc[n][2] + acc[n][3] * kLoInv) + bg1 * qt;
            }
        }
        cp_wait_0();
        const int row = rt * kRowTile + g;
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const int p = tb + n * 4 + t;
            if (p >= S.m) continue;
            const int b = S.toks ? S.toks[p] : p;
            const float w = S.wts ? S.wts[p] : 1.f;
            red_add_f32(y + (long long)b * d + row, w * o[n][0]);
            red_add_f32(y + (long long)b * d + row + 8, w * o[n][1]);
        }
    }
    };
    for (int yi = blockIdx.y; yi < D->n_dn; yi += gridDim.y) {   // CTA-uniform, as in k_gu
        Slot S;
        const int2 item = dn_items(D)[yi];
        if (!slot_of(item.x, D, Ly, B, K, d, I, Is, tok, wt, hdr, S)) continue;
        run_item(item, S);
        __syncthreads();   // the staged act fragments are reused by the next item
    }
}

// ---------------------------------------------------------- k_lora_vd -------
// One CTA per block of 8 tokens and 128 output rows.  A_down (transposed back
// to [r][Is], rows padded by one word) and the block's shared-expert act rows
// are staged in shared memory; warp j forms v = A_down act of token j of the
// block (r values, lanes over Is without bank conflicts); then thread t takes
// output row t mod 128 for four of the block's tokens and adds (alpha/r)
// B_down[row] v (one read of a B_down row serves four tokens).
constexpr int kLoraTok = 8;
constexpr int kLoraRows = 128;
__host__ __device__ inline int lora_vd_lda(int Is) { return Is + 2; }
__host__ __device__ inline size_t lora_vd_smem(int Is, int r) {
    (void)r;
    return (size_t)16 * lora_vd_lda(Is) * 2 + (size_t)kLoraTok * Is * 4;
}
__global__ void __launch_bounds__(256) k_lora_vd(const float* __restrict__ act, int Imax, int pos0,
                                                 const __half* __restrict__ AdT, const __half* __restrict__ Bd,
                                                 int r, int Is, int d, int B, float scale, float* __restrict__ y) {
    extern __shared__ __align__(16) char lsm[];
    const int lda = lora_vd_lda(Is);
    __half* sA = reinterpret_cast<__half*>(lsm);                               // [16][lda]
    float* sx = reinterpret_cast<float*>(lsm + (size_t)16 * lda * 2);         // [kLoraTok][Is]
    __shared__ float vs[kLoraTok][16];
    const int b0 = blockIdx.x * kLoraTok, row0 = blockIdx.y * kLoraRows;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nb = min(kLoraTok, B - b0);
    for (int i = tid; i < Is * r; i += 256) {
        const int k = i / r, q = i - k * r;
        sA[q * lda + k] = AdT[i];
    }
    for (int i = tid; i < nb * (Is / 4); i += 256) {
        const int j = i / (Is / 4), k4 = i - j * (Is / 4);
        reinterpret_cast<float4*>(sx + j * Is)[k4] =
            reinterpret_cast<const float4*>(act + (long long)(pos0 + b0 + j) * Imax)[k4];
    }
    __syncthreads();
    if (wid < nb) {
        float acc[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) acc[q] = 0.f;
        for (int k = lane; k < Is; k += 32) {
            const float av = sx[wid * Is + k];
#pragma unroll
            for (int q = 0; q < 16; ++q)
                if (q < r) acc[q] += __half2float(sA[q * lda + k]) * av;
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const float sq = warp_sum(acc[q]);
            if (lane == 0) vs[wid][q] = sq;
        }
    }
    __syncthreads();
    const int row = row0 + (tid & (kLoraRows - 1)), j0 = (tid / kLoraRows) * (kLoraTok / 2);
    if (row < d && j0 < nb) {
        float bd[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) bd[q] = q < r ? __half2float(Bd[(long long)row * r + q]) : 0.f;
#pragma unroll
        for (int jj = 0; jj < kLoraTok / 2; ++jj) {
            const int j = j0 + jj;
            if (j >= nb) break;
            float sj = 0.f;
#pragma unroll
            for (int q = 0; q < 16; ++q) sj += bd[q] * vs[j][q];
            y[(long long)(b0 + j) * d + row] += scale * sj;
        }
    }
}

// launch helpers
// out [B][ldo] += W X^T (zero out first unless accumulating into it)
template <bool F32IN>
int dense(const char* W, int kmajor, int N, int Kin, const __half* xh, const float* xf, int ldx, int B,
          float* out, int ldo, bool zero, cudaStream_t st) {
    if (zero && cudaMemsetAsync(out, 0, (size_t)B * ldo * 4, st) != cudaSuccess) return EDGE0_ECUDA;
    const dim3 grid((N + 15) / 16, (B + 31) / 32, (Kin / 16 + 15) / 16);
    k_dense<F32IN><<<grid, 128, 0, st>>>(W, kmajor, N, Kin, xh, xf, ldx, B, out, ldo);
    return cudaGetLastError() == cudaSuccess ? EDGE0_OK : EDGE0_ECUDA;
}

// opt in to `smem` bytes of dynamic shared memory for `f` (once per size reached)
template <class F>
bool smem_opt_in(F f, size_t smem, size_t* done) {
    if (smem <= 48 * 1024 || smem <= *done) return true;
    if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return false;
    *done = smem;
    return true;
}

int route(const float* lg, int B, int E, int K, int kind, int ng, int G, float scale, const float* bias,
          int32_t* ids, float* w, cudaStream_t st) {
    const size_t smem = (size_t)8 * 3 * E * 4 + 2 * 8 * EDGE0_MAX_K * 4;
    if (smem > 48 * 1024) {   // E > 496: opt in to more dynamic shared memory
        static int done = 0;
        if (!done) {
            if (cudaFuncSetAttribute(k_route, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
                return EDGE0_ECUDA;
            done = 1;
        }
    }
    k_route<<<(B + 7) / 8, 256, smem, st>>>(lg, E, B, E, K, kind, ng, G, scale, bias, ids, w);
    return cudaGetLastError() == cudaSuccess ? EDGE0_OK : EDGE0_ECUDA;
}

}  // namespace

namespace {
// One decode step of L layers for B > EDGE0_MAX_BATCH sequences, or (prefill)
// the L layers over a prompt of B tokens, every layer on its own router and no
// head (the prerouter is not used at prefill), the executed ids into ids_out
// ([L][B][K], or the workspace when null).  Validates nothing beyond what the
// caller checked; enqueues on `st`.
int run_batched(const Prog& p, int32_t* ids_out, cudaStream_t st) {
    const bool prefill = p.mode == MODE_PREFILL, tcgu = prefill && p.tc_gu;
    const int L = p.L, B = p.B, K = p.K, d = p.d, E = p.E, I = p.I, Is = p.Is, H = p.H, r = p.r;
    const int Imax = I > Is ? I : Is;
    const BatchWs W = prefill ? batch_ws_layout(1, B, d, E, K, Imax, 16) : batch_ws_layout(p.Ls, B, d, E, K, Imax, H);
    char* ws = p.ws;
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
    float* y = reinterpret_cast<float*>(ws + W.y);
    __half* xs = reinterpret_cast<__half*>(ws + W.xs);
    float* xsum = reinterpret_cast<float*>(ws + W.xsum);
    float* lg = reinterpret_cast<float*>(ws + W.lg);
    float* la = reinterpret_cast<float*>(ws + W.la);
    float* wsel = reinterpret_cast<float*>(ws + W.wsel);
    Disp* D = reinterpret_cast<Disp*>(ws + W.disp);
    int* tok = reinterpret_cast<int*>(ws + W.tok);
    float* wt = reinterpret_cast<float*>(ws + W.wt);
    float* act = reinterpret_cast<float*>(ws + W.act);
    const int step = prefill ? 0 : p.step, par = step & 1;
    const int slots = (B * K < E ? B * K : E) + 1;
    const int cap = disp_cap(B, K, E);
    // gate/up on the tcgen05 kernel (prefill, when asked): blocks of kTcTok tokens
    const int blk_gu = tcgu ? kTcTok : kGuTok;
    const int items_gu = (B * K + blk_gu - 1) / blk_gu + slots + (B + blk_gu - 1) / blk_gu;
    const int items_dn = (B * K + kDnTok - 1) / kDnTok + slots + (B + kDnTok - 1) / kDnTok;
    auto ok = [] { return cudaGetLastError() == cudaSuccess; };
    // staged B fragments (+ group sums) of one token block
    const size_t ring = (size_t)kExpWarps * kStages * kSlice;
    const size_t smem_gu = (size_t)kGuTok * (d + 8) * 2 + (size_t)kGuTok * (d / kGroup) * 4 +
                           (size_t)kGuWarps * kGuStages * kSlice;
    const size_t smem_dn = (size_t)(Imax / kGroup) * 512 * 8 + (size_t)kDnTok * (Imax / kGroup) * 4 + ring;
    int dev = 0, smem_max = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return EDGE0_ECUDA;
    if (smem_gu > (size_t)smem_max || smem_dn > (size_t)smem_max) return EDGE0_EUNSUPPORTED;   // d or I too large
    static size_t done_gu = 0, done_dn = 0, done_tc = 0;
    if (!smem_opt_in(k_gu, smem_gu, &done_gu) || !smem_opt_in(k_down, smem_dn, &done_dn)) return EDGE0_ECUDA;
    if (tcgu && !smem_opt_in(k_gu_tc, kTcSmem, &done_tc)) return EDGE0_ECUDA;
    static size_t done_lv = 0;
    if (lora_vd_smem(Is, r) > (size_t)smem_max) return EDGE0_EUNSUPPORTED;
    if (!smem_opt_in(k_lora_vd, lora_vd_smem(Is, r), &done_lv)) return EDGE0_ECUDA;
    // expert grids: the CTAs that fit on the GPU at once, each looping over items
    int nsm = 0, occ_gu = 0, occ_dn = 0;
    if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_gu, k_gu, kGuWarps * 32, smem_gu) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_dn, k_down, 256, smem_dn) != cudaSuccess)
        return EDGE0_ECUDA;
    int occ_tc = 1;
    if (tcgu && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_tc, k_gu_tc, kTcThreads, kTcSmem) != cudaSuccess)
        return EDGE0_ECUDA;
    const int gu_x = tcgu ? Imax / (8 * kHalfRow) : (Imax / kHalfRow + kGuWarps - 1) / kGuWarps;
    const int dn_x = (d / kRowTile + kExpWarps - 1) / kExpWarps;
    const int gu_y = std::max(1, std::min(items_gu, nsm * std::max(tcgu ? occ_tc : occ_gu, 1) / gu_x));
    const int dn_y = std::max(1, std::min(items_dn, nsm * std::max(occ_dn, 1) / dn_x));
    int rc = EDGE0_OK;
    for (int l = 0; l < L && rc == EDGE0_OK; ++l) {
        const LayerP& Ly = p.layers[l];
        const long long srow = (long long)Ly.sidx * B * K;
        __half* x = xs + (prefill ? 0LL : (long long)Ly.sidx * B * d);
        if (Ly.ready && cudaStreamWaitEvent(st, (cudaEvent_t)Ly.ready, 0) != cudaSuccess) return EDGE0_ECUDA;
        k_norm<<<B, 256, 0, st>>>(p.h_io, y, l > 0, Ly.gamma, Ly.eps, d, x, xsum, 1,
                                  (Ly.flags & LF_LORA) ? la : nullptr);
        if (!ok()) return EDGE0_ECUDA;
        int32_t* exec = prefill ? (ids_out ? ids_out + (long long)l * B * K : reinterpret_cast<int32_t*>(ws + W.exec))
                                : p.exec_ids + (long long)par * p.Ls * B * K + srow;
        const float* w;
        const int32_t* ids = exec;      // the routing the dispatch reads
        int32_t* ids_copy = nullptr;    // where it copies a prediction to
        if (!prefill && (Ly.flags & LF_PREROUTED) && step > 0) {
            const long long o = (long long)(par ^ 1) * p.Ls * B * K + srow;
            ids = p.pred_ids + o;
            ids_copy = exec;
            w = p.pred_w + o;
        } else {
            rc = dense<false>(Ly.router, 0, E, d, x, nullptr, d, B, lg, E, true, st);
            if (rc == EDGE0_OK)
                rc = route(lg, B, E, K, Ly.route_kind, Ly.n_groups, Ly.topk_groups, Ly.route_scale, Ly.bias, exec,
                           wsel, st);
            w = wsel;
        }
        if (rc) return rc;
        k_dispatch<<<1, 1024, 0, st>>>(ids, ids_copy, w, B, K, E, Ly.sh_gu ? 1 : 0, blk_gu, kDnTok, cap,
                                       Ly.slot_table, Ly.tier_counts, D, tok, wt, hdr);
        if (!ok()) return EDGE0_ECUDA;
        const int lora = (Ly.flags & LF_LORA) ? 1 : 0;
        if (lora) {
            k_dense_pair<<<dim3(2 * ((r + 15) / 16), (B + 31) / 32, (d / 16 + 15) / 16), 128, 0, st>>>(
                Ly.lora_Ag, Ly.lora_Au, r, d, x, d, B, la, 32, 16);
            if (!ok()) return EDGE0_ECUDA;
        }
        if (tcgu)
            k_gu_tc<<<dim3(gu_x, gu_y), kTcThreads, kTcSmem, st>>>(Ly, D, tok, wt, x, la, lora, r, B, K, d, I, Is,
                                                                 Imax, act, hdr);
        else
            k_gu<<<dim3(gu_x, gu_y), kGuWarps * 32, smem_gu, st>>>(
                Ly, D, tok, wt, x, xsum, la, lora, r, B, K, d, I, Is, Imax, act, hdr);
        if (!ok()) return EDGE0_ECUDA;
        k_down<<<dim3(dn_x, dn_y), 256, smem_dn, st>>>(
            Ly, D, tok, wt, act, B, K, d, I, Is, Imax, y, hdr);
        if (!ok()) return EDGE0_ECUDA;
        if (lora) {
            k_lora_vd<<<dim3((B + kLoraTok - 1) / kLoraTok, (d + kLoraRows - 1) / kLoraRows), 256,
                        lora_vd_smem(Is, r), st>>>(act, Imax, B * K, Ly.lora_AdT, Ly.lora_Bd, r, Is,
                                                                      d, B, Ly.lora_scale, y);
            if (!ok()) return EDGE0_ECUDA;
        }
    }
    // the last layer's output
    k_norm<<<B, 256, 0, st>>>(p.h_io, y, 1, nullptr, 0.f, d, nullptr, nullptr, 0, nullptr);
    if (!ok()) return EDGE0_ECUDA;
    if (prefill) return rc;
    // head flush: every head of the step, from its layer's x and routing, one
    // launch per stage over all heads (the job table goes to the workspace with
    // the step's parity and previous-step ids)
    std::vector<HeadJob> jobs;
    for (int l = 0; l < L; ++l) {
        const LayerP& Ly = p.layers[l];
        if (!(Ly.flags & LF_HEAD)) continue;
        const long long srow = (long long)Ly.sidx * B * K;
        const long long o = (long long)par * p.Ls * B * K + (long long)Ly.head_target * B * K;
        HeadJob J;
        J.fc1 = Ly.fc1;
        J.fc1_oh = Ly.fc1_oh;
        J.fc2 = Ly.fc2;
        J.linit = Ly.linit;
        J.linit_oh = Ly.linit_oh;
        J.x = xs + (long long)Ly.sidx * B * d;
        J.exec = p.exec_ids + (long long)par * p.Ls * B * K + srow;
        J.prev = step > 0 ? p.exec_ids + (long long)(par ^ 1) * p.Ls * B * K + srow : nullptr;
        J.pred_ids = p.pred_ids + o;
        J.pred_w = p.pred_w + o;
        J.bias = Ly.head_bias;
        J.scale = Ly.head_route_scale;
        J.kind = Ly.head_route_kind;
        J.ng = Ly.head_n_groups;
        J.G = Ly.head_topk_groups;
        jobs.push_back(J);
    }
    const int nh = (int)jobs.size();
    if (nh == 0) return rc;
    if (nh > p.Ls) return EDGE0_EINVAL;
    // head h: fc1 output at zh + h hs, logits at lgh + h hs; the job table after
    const long long hs = (long long)B * (H + E);
    HeadJob* dj = reinterpret_cast<HeadJob*>(ws + W.z + ((long long)p.Ls * hs * 4 + 255) / 256 * 256);
    float* zh = reinterpret_cast<float*>(ws + W.z);
    float* lgh = zh + (long long)B * H;
    const long long zs = hs, ls = hs;
    if (cudaMemcpyAsync(dj, jobs.data(), sizeof(HeadJob) * nh, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemsetAsync(zh, 0, (size_t)nh * hs * 4, st) != cudaSuccess)
        return EDGE0_ECUDA;
    const int nk_d = (d / 16 + 15) / 16, nk_h = (H / 16 + 15) / 16;
    k_dense_heads<false><<<dim3((H + 15) / 16, (B + 31) / 32, nk_d * nh), 128, 0, st>>>(
        dj, HS_FC1, nk_d, H, d, B, nullptr, 0, zh, H, zs);
    if (!ok()) return EDGE0_ECUDA;
    k_onehot_heads<<<dim3((H + 127) / 128, B, nh), 128, 0, st>>>(dj, 0, zh, zs, H, K, E);
    if (!ok()) return EDGE0_ECUDA;
    k_dense_heads<true><<<dim3((E + 15) / 16, (B + 31) / 32, nk_h * nh), 128, 0, st>>>(
        dj, HS_FC2, nk_h, E, H, B, zh, zs, lgh, E, ls);
    if (!ok()) return EDGE0_ECUDA;
    k_dense_heads<false><<<dim3((E + 15) / 16, (B + 31) / 32, nk_d * nh), 128, 0, st>>>(
        dj, HS_LINIT, nk_d, E, d, B, nullptr, 0, lgh, E, ls);
    if (!ok()) return EDGE0_ECUDA;
    k_onehot_heads<<<dim3((E + 127) / 128, B, nh), 128, 0, st>>>(dj, 1, lgh, ls, E, K, E);
    if (!ok()) return EDGE0_ECUDA;
    const size_t rsmem = (size_t)8 * 3 * E * 4 + 2 * 8 * EDGE0_MAX_K * 4;
    static size_t done_rh = 0;
    if (!smem_opt_in(k_route_heads, rsmem, &done_rh)) return EDGE0_ECUDA;
    k_route_heads<<<dim3((B + 7) / 8, nh), 256, rsmem, st>>>(dj, lgh, ls, B, E, K);
    if (!ok()) return EDGE0_ECUDA;
    return rc;
}
}  // namespace

int batch_decode(const Prog& p, cudaStream_t st) { return run_batched(p, nullptr, st); }

int batch_prefill(const Prog& p, int32_t* ids_out, cudaStream_t st) {
    if (p.mode != MODE_PREFILL || p.B < 1 || p.B > kMaxPrefill) return EDGE0_EINVAL;
    return run_batched(p, ids_out, st);
}

}  // namespace edge0
