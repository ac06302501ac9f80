// Standalone unmerged LoRA delta, y += (alpha/r) B (A v)  ("The Other Half of the
// Memory Wall", S3.3).  Inside a decode step the same delta is fused into the
// engine; this entry point exists for callers that apply one projection alone.
// One CTA per token: A v on the tensor cores from the packed fp16 units of A,
// then the rank-r B product on the CUDA cores.
#include "internal.cuh"

namespace edge0 {

constexpr int kLoraThreads = 256;

__global__ void __launch_bounds__(kLoraThreads) lora_kernel(const char* __restrict__ A,
                                                            const __half* __restrict__ Bm, int r,
                                                            int in, int out, float scale,
                                                            const __half* __restrict__ v,
                                                            __half* __restrict__ y) {
    extern __shared__ __align__(16) char sm[];
    const int ng = in / kGroup, n_rt = ceil_div(r, kRowTile), R16 = n_rt * kRowTile;
    __half* frag = reinterpret_cast<__half*>(sm);
    float* sums = reinterpret_cast<float*>(sm + in * 2);
    float* av = sums + ng;
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nw = kLoraThreads / 32;
    const __half* vb = v + (long long)b * in;
    for (int i = tid; i < R16; i += kLoraThreads) av[i] = 0.f;
    for (int grp = wid; grp < ng; grp += nw)
        put_group(frag + grp * kGroup, sums + grp, __half2float(vb[grp * kGroup + lane]),
                  __half2float(vb[grp * kGroup + lane + 32]), lane);
    __syncthreads();
    const int g = lane >> 2, t = lane & 3;
    for (int rt = 0; rt < n_rt; ++rt) {
        float lo[4] = {0.f, 0.f, 0.f, 0.f}, hi[4] = {0.f, 0.f, 0.f, 0.f};
        for (int grp = wid; grp < ng; grp += nw) {
            uint4 b0 = make_uint4(0, 0, 0, 0), b1 = make_uint4(0, 0, 0, 0);
            if (g == 0) {
                const uint4* bp = reinterpret_cast<const uint4*>(frag + (grp * 4 + t) * 16);
                b0 = bp[0];
                b1 = bp[1];
            }
            const char* unit = A + ((long long)rt * ng + grp) * kF16Unit;
            uint32_t a[4];
            const uint4 a0 = *reinterpret_cast<const uint4*>(unit + 0 * 512 + 16 * lane);
            const uint4 a1 = *reinterpret_cast<const uint4*>(unit + 1 * 512 + 16 * lane);
            const uint4 a2 = *reinterpret_cast<const uint4*>(unit + 2 * 512 + 16 * lane);
            const uint4 a3 = *reinterpret_cast<const uint4*>(unit + 3 * 512 + 16 * lane);
            a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
            mma_16816(lo, a, b0.x, b0.y);
            a[0] = a1.x; a[1] = a1.y; a[2] = a1.z; a[3] = a1.w;
            mma_16816(hi, a, b0.z, b0.w);
            a[0] = a2.x; a[1] = a2.y; a[2] = a2.z; a[3] = a2.w;
            mma_16816(lo, a, b1.x, b1.y);
            a[0] = a3.x; a[1] = a3.y; a[2] = a3.z; a[3] = a3.w;
            mma_16816(hi, a, b1.z, b1.w);
        }
        if (t == 0) {   // column 0 holds this token
            atomicAdd(&av[rt * kRowTile + g], lo[0] + 16.0f * hi[0]);
            atomicAdd(&av[rt * kRowTile + g + 8], lo[2] + 16.0f * hi[2]);
        }
    }
    __syncthreads();
    for (int o = tid; o < out; o += kLoraThreads) {
        float acc = 0.f;
        for (int j = 0; j < r; ++j) acc += __half2float(Bm[(long long)o * r + j]) * av[j];
        const long long i = (long long)b * out + o;
        y[i] = __float2half_rn(__half2float(y[i]) + scale * acc);
    }
}

}  // namespace edge0

using namespace edge0;

extern "C" int edge0_lora_delta(const edge0_lora_desc* lora, const uint16_t* v, int B,
                                uint16_t* y_inout, cudaStream_t stream) {
    if (!lora || !lora->A || !lora->B || !v || !y_inout || B <= 0) return EDGE0_EINVAL;
    if (lora->r <= 0 || lora->r > 64 || lora->in <= 0 || lora->in % kGroup || lora->out <= 0)
        return EDGE0_EINVAL;
    if (((uintptr_t)lora->A & 15) || ((uintptr_t)v & 1) || ((uintptr_t)y_inout & 1))
        return EDGE0_EINVAL;
    const int smem = lora->in * 2 + (lora->in / kGroup) * 4 + ceil_div(lora->r, kRowTile) * kRowTile * 4;
    if (smem > 48 * 1024) {
        if (cudaFuncSetAttribute(lora_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
            return EDGE0_EUNSUPPORTED;
    }
    lora_kernel<<<B, kLoraThreads, smem, stream>>>((const char*)lora->A, (const __half*)lora->B,
                                                   lora->r, lora->in, lora->out,
                                                   lora->alpha / (float)lora->r,
                                                   (const __half*)v, (__half*)y_inout);
    return cudaGetLastError() == cudaSuccess ? EDGE0_OK : EDGE0_ECUDA;
}
