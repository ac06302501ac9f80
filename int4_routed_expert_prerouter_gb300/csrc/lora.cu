// Standalone unmerged LoRA delta, y += (alpha/r) B (A v)  ("The Other Half of the
// Memory Wall", S3.3).  Inside a decode step the same delta is fused into the
// engine; this entry point exists for callers that apply one projection alone.
// One CTA per token: u = A v (r values) from A transposed [in, r], then the
// rank-r product with B on the CUDA cores, accumulated in fp32.
#include "internal.cuh"

namespace edge0 {

constexpr int kLoraThreads = 256;

__global__ void __launch_bounds__(kLoraThreads) lora_kernel(const __half* __restrict__ AT,
                                                            const __half* __restrict__ Bm, int r,
                                                            int in, int out, float scale,
                                                            const __half* __restrict__ v,
                                                            __half* __restrict__ y) {
    __shared__ float part[kLoraThreads / 32][16];
    __shared__ float u[16];
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const __half* vb = v + (long long)b * in;
    float acc[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) acc[q] = 0.f;
    for (int i = tid; i < in; i += kLoraThreads) {
        const float vi = __half2float(vb[i]);
        for (int q = 0; q < r; ++q) acc[q] += __half2float(AT[(long long)i * r + q]) * vi;
    }
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        const float s = warp_sum(acc[q]);
        if (lane == 0) part[wid][q] = s;
    }
    __syncthreads();
    if (tid < r) {
        float s = 0.f;
        for (int w = 0; w < kLoraThreads / 32; ++w) s += part[w][tid];
        u[tid] = s;
    }
    __syncthreads();
    for (int o = tid; o < out; o += kLoraThreads) {
        float s = 0.f;
        for (int q = 0; q < r; ++q) s += __half2float(Bm[(long long)o * r + q]) * u[q];
        const long long i = (long long)b * out + o;
        y[i] = __float2half_rn(__half2float(y[i]) + scale * s);
    }
}

}  // namespace edge0

using namespace edge0;

extern "C" int edge0_lora_delta(const edge0_lora_desc* lora, const uint16_t* v, int B,
                                uint16_t* y_inout, cudaStream_t stream) {
    if (!lora || !lora->A_T || !lora->B || !v || !y_inout || B <= 0) return EDGE0_EINVAL;
    if (lora->r <= 0 || lora->r > 16 || lora->in <= 0 || lora->out <= 0) return EDGE0_EINVAL;
    if (((uintptr_t)lora->A_T & 1) || ((uintptr_t)lora->B & 1) || ((uintptr_t)v & 1) ||
        ((uintptr_t)y_inout & 1))
        return EDGE0_EINVAL;
    lora_kernel<<<B, kLoraThreads, 0, stream>>>((const __half*)lora->A_T, (const __half*)lora->B,
                                               lora->r, lora->in, lora->out,
                                               lora->alpha / (float)lora->r, (const __half*)v,
                                               (__half*)y_inout);
    return cudaGetLastError() == cudaSuccess ? EDGE0_OK : EDGE0_ECUDA;
}
