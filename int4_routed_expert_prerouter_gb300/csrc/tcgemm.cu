// Dense fp16 GEMM on the fifth-generation tensor cores: D = A B^T with fp16 A
// [M x K] and B [N x K] (row-major, K contiguous) and fp32 D [M x N].  One CTA
// of four warps per 128-row tile of D: each 64-wide K chunk of A and B is staged
// in shared memory in the canonical K-major layout (tc05.cuh), one thread issues
// the four tcgen05.mma K-steps into a TMEM accumulator of N columns, and a
// commit to an mbarrier tells the CTA when the chunk may be overwritten; the
// four warps then read their 32 lanes (rows) of the accumulator out.
//
// This is the building block the grouped int4 kernels stage their tiles for;
// as an entry point it serves dense fp16 products (and the tests of the
// descriptors and the TMEM round trip).
#include <string.h>

#include "tc05.cuh"

namespace edge0 {
namespace {

constexpr int kTcM = 128;
constexpr int kTcKc = 64;                  // K per staged chunk (4 MMA K-steps of 16)
constexpr unsigned long long kTcWaitNs = 1000000000ull;

__device__ __forceinline__ unsigned long long gtime() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__global__ void __launch_bounds__(128) tc_gemm_kernel(const __half* __restrict__ A, const __half* __restrict__ B,
                                                      float* __restrict__ D, int M, int N, int K, int ncols,
                                                      int* err) {
    extern __shared__ __align__(128) char tsm[];
    __shared__ uint64_t bar;
    __shared__ uint32_t taddr_s;
    __shared__ int bad;
    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    const int m0 = blockIdx.x * kTcM;
    char* sA = tsm;                                  // 4 K-steps x 128 rows x 32 B
    char* sB = tsm + 4 * kTcM * 32;                  // 4 K-steps x N rows x 32 B
    if (wid == 0) {
        tc::tmem_alloc(&taddr_s, (uint32_t)ncols);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        bad = 0;
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t taddr = taddr_s;
    const uint32_t idesc = tc::idesc_f16(kTcM, N);
    uint32_t phase = 0;
    for (int kc = 0; kc < K; kc += kTcKc) {
        // stage: 16-byte pieces (8 values of one row and K-step half)
        for (int i = tid; i < kTcM * 8; i += 128) {
            const int row = i >> 3, c8 = i & 7;
            const uint4 v = *reinterpret_cast<const uint4*>(A + (long long)(m0 + row) * K + kc + c8 * 8);
            *reinterpret_cast<uint4*>(sA + (c8 >> 1) * kTcM * 32 + tc::kstep_off(row, (c8 & 1) * 8)) = v;
        }
        for (int i = tid; i < N * 8; i += 128) {
            const int row = i >> 3, c8 = i & 7;
            const uint4 v = *reinterpret_cast<const uint4*>(B + (long long)row * K + kc + c8 * 8);
            *reinterpret_cast<uint4*>(sB + (c8 >> 1) * N * 32 + tc::kstep_off(row, (c8 & 1) * 8)) = v;
        }
        tc::fence_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                tc::mma_f16(taddr, tc::smem_desc(a0 + ks * kTcM * 32), tc::smem_desc(b0 + ks * N * 32), idesc,
                            kc > 0 || ks > 0);
            tc::mma_commit(&bar);
            // the chunk's shared memory is free once its MMAs completed (bounded wait)
            const unsigned long long t0 = gtime();
            while (!mbar_try_wait(&bar, phase))
                if (gtime() - t0 > kTcWaitNs) {
                    bad = 1;
                    break;
                }
        }
        phase ^= 1u;
        __syncthreads();
        if (bad) break;
    }
    tc::fence_after_sync();
    if (!bad) {
        // warp w reads rows 32 w .. 32 w + 31 (its TMEM lanes)
        const int row = m0 + 32 * wid + lane;
        for (int c = 0; c < N; c += 8) {
            float v[8];
            tc::tmem_ld8(taddr + ((uint32_t)(32 * wid) << 16) + (uint32_t)c, v);
            tc::tmem_wait_ld();
            float4* dst = reinterpret_cast<float4*>(D + (long long)row * N + c);
            dst[0] = make_float4(v[0], v[1], v[2], v[3]);
            dst[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
    } else if (tid == 0) {
        atomicExch(err, EDGE0_ETIMEOUT);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (wid == 0) tc::tmem_dealloc(taddr, (uint32_t)ncols);
}

}  // namespace
}  // namespace edge0

using namespace edge0;

extern "C" int edge0_tc_gemm_f16(const uint16_t* A, const uint16_t* B, float* D, int M, int N, int K, int* status,
                                 cudaStream_t stream) {
    if (!A || !B || !D || !status) return EDGE0_EINVAL;
    if (M <= 0 || M % kTcM || N < 16 || N > 256 || N % 16 || K <= 0 || K % kTcKc) return EDGE0_EINVAL;
    if (((uintptr_t)A | (uintptr_t)B | (uintptr_t)D) & 15) return EDGE0_EINVAL;
    int ncols = 32;
    while (ncols < N) ncols <<= 1;
    const size_t smem = (size_t)4 * (kTcM + N) * 32;
    static bool opted = false;   // beyond the default 48 KB of dynamic shared memory
    if (!opted) {
        if (cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024) !=
            cudaSuccess)
            return EDGE0_ECUDA;
        opted = true;
    }
    tc_gemm_kernel<<<M / kTcM, 128, smem, stream>>>(reinterpret_cast<const __half*>(A),
                                                    reinterpret_cast<const __half*>(B), D, M, N, K, ncols, status);
    return cudaGetLastError() == cudaSuccess ? EDGE0_OK : EDGE0_ECUDA;
}
