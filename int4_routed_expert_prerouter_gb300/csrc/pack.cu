// Conversion of canonical weights into the packed fragment-ordered HBM layout.
//
// int4 unit (16 rows x 64 inputs of one matrix, 576 bytes):
//   bytes [16 L, 16 L + 16), L = 4 g + t (g = L / 4, t = L % 4), hold the packed
//   words (row g: words 2t, 2t+1 of the group; row g+8: words 2t, 2t+1), which is
//   exactly the 16 bytes lane L of a warp needs for four m16n8k16 tensor-core
//   steps over that group;
//   bytes [512 + 8 g, 520 + 8 g) hold (s, b) of row g then (s, b) of row g + 8.
// fp16 unit (2048 bytes): four 512-byte blocks, one per m16n8k16 step m; lane L's
//   16 bytes are its A registers a0..a3 for that step.  Step m pairs the inputs
//   (16 t + o, 16 t + o + 4) with o = (m & 1) + 8 (m >> 1) + 2 j, j = 0 (a0/a1) or
//   1 (a2/a3), the same input permutation the int4 nibble masks produce.
#include "internal.cuh"

namespace edge0 {

__global__ void pack_q4_kernel(const uint32_t* __restrict__ q, const uint16_t* __restrict__ s,
                               const uint16_t* __restrict__ b, int E, int out, int in,
                               char* __restrict__ dst) {
    const int n_rt = ceil_div(out, kRowTile), n_g = in / kGroup;
    const long long units = (long long)E * n_rt * n_g;
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (tid >= units * 32) return;
    const int lane = (int)(tid & 31);
    const long long unit = tid >> 5;
    const int c = (int)(unit % n_g);
    const int rt = (int)((unit / n_g) % n_rt);
    const int e = (int)(unit / ((long long)n_g * n_rt));
    const int g = lane >> 2, t = lane & 3;
    const int r0 = rt * kRowTile + g, r1 = r0 + 8;
    const long long wpr = in / 8, gpr = in / kGroup;
    const uint32_t* qe = q + (long long)e * out * wpr;
    uint4 v;
    v.x = r0 < out ? qe[r0 * wpr + 8 * c + 2 * t] : 0u;
    v.y = r0 < out ? qe[r0 * wpr + 8 * c + 2 * t + 1] : 0u;
    v.z = r1 < out ? qe[r1 * wpr + 8 * c + 2 * t] : 0u;
    v.w = r1 < out ? qe[r1 * wpr + 8 * c + 2 * t + 1] : 0u;
    char* u = dst + unit * kQ4Unit;
    *reinterpret_cast<uint4*>(u + 16 * lane) = v;
    if (t == 0) {
        const uint16_t* se = s + (long long)e * out * gpr;
        const uint16_t* be = b + (long long)e * out * gpr;
        ushort4 sb;
        sb.x = r0 < out ? se[r0 * gpr + c] : 0;
        sb.y = r0 < out ? be[r0 * gpr + c] : 0;
        sb.z = r1 < out ? se[r1 * gpr + c] : 0;
        sb.w = r1 < out ? be[r1 * gpr + c] : 0;
        *reinterpret_cast<ushort4*>(u + 512 + 8 * g) = sb;
    }
}

__global__ void pack_f16_kernel(const uint16_t* __restrict__ W, int out, int in, int ld,
                                char* __restrict__ dst) {
    const int n_rt = ceil_div(out, kRowTile), n_g = in / kGroup;
    const long long units = (long long)n_rt * n_g;
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (tid >= units * 128) return;
    const int lane = (int)(tid & 31);
    const int m = (int)((tid >> 5) & 3);
    const long long unit = tid >> 7;
    const int c = (int)(unit % n_g);
    const int rt = (int)(unit / n_g);
    const int g = lane >> 2, t = lane & 3;
    const int r0 = rt * kRowTile + g, r1 = r0 + 8;
    uint32_t a[4];
    for (int j = 0; j < 2; ++j) {
        const int k = kGroup * c + 16 * t + (m & 1) + 8 * (m >> 1) + 2 * j;
        const uint32_t lo0 = r0 < out ? W[(long long)r0 * ld + k] : 0u;
        const uint32_t hi0 = r0 < out ? W[(long long)r0 * ld + k + 4] : 0u;
        const uint32_t lo1 = r1 < out ? W[(long long)r1 * ld + k] : 0u;
        const uint32_t hi1 = r1 < out ? W[(long long)r1 * ld + k + 4] : 0u;
        a[2 * j] = lo0 | (hi0 << 16);       // a0 / a2: row g
        a[2 * j + 1] = lo1 | (hi1 << 16);   // a1 / a3: row g + 8
    }
    uint4 v = make_uint4(a[0], a[1], a[2], a[3]);
    *reinterpret_cast<uint4*>(dst + unit * kF16Unit + m * 512 + 16 * lane) = v;
}

__global__ void pack_cols_T_kernel(const uint16_t* __restrict__ W, int out, int ld, int col0,
                                   int ncols, uint16_t* __restrict__ dst) {
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (tid >= (long long)out * ncols) return;
    const int o = (int)(tid % out), j = (int)(tid / out);
    dst[(long long)j * out + o] = W[(long long)o * ld + col0 + j];
}

static bool aligned(const void* p, int a) { return ((uintptr_t)p % a) == 0; }

}  // namespace edge0

using namespace edge0;

extern "C" size_t edge0_q4_packed_bytes(int E, int out, int in) {
    if (E <= 0 || out <= 0 || in <= 0 || in % kGroup) return 0;
    return (size_t)E * (size_t)q4_bytes(out, in);
}

extern "C" int edge0_pack_q4(const uint32_t* q, const uint16_t* s, const uint16_t* b, int E,
                             int out, int in, void* packed, cudaStream_t stream) {
    if (!q || !s || !b || !packed || E <= 0 || out <= 0 || in <= 0 || in % kGroup)
        return EDGE0_EINVAL;
    if (!aligned(q, 4) || !aligned(s, 2) || !aligned(b, 2) || !aligned(packed, 16))
        return EDGE0_EINVAL;
    const long long threads = (long long)E * ceil_div(out, kRowTile) * (in / kGroup) * 32;
    const int bs = 256;
    pack_q4_kernel<<<(unsigned)((threads + bs - 1) / bs), bs, 0, stream>>>(q, s, b, E, out, in,
                                                                           (char*)packed);
    return cudaGetLastError() == cudaSuccess ? EDGE0_OK : EDGE0_ECUDA;
}

extern "C" size_t edge0_f16_packed_bytes(int out, int in) {
    if (out <= 0 || in <= 0 || in % kGroup) return 0;
    return (size_t)f16_bytes(out, in);
}

extern "C" int edge0_pack_f16(const uint16_t* W, int out, int in, int ld, void* packed,
                              cudaStream_t stream) {
    if (!W || !packed || out <= 0 || in <= 0 || in % kGroup || ld < in) return EDGE0_EINVAL;
    if (!aligned(W, 2) || !aligned(packed, 16)) return EDGE0_EINVAL;
    const long long threads = (long long)ceil_div(out, kRowTile) * (in / kGroup) * 128;
    const int bs = 256;
    pack_f16_kernel<<<(unsigned)((threads + bs - 1) / bs), bs, 0, stream>>>(W, out, in, ld,
                                                                            (char*)packed);
    return cudaGetLastError() == cudaSuccess ? EDGE0_OK : EDGE0_ECUDA;
}

extern "C" int edge0_pack_cols_T(const uint16_t* W, int out, int ld, int col0, int ncols,
                                 uint16_t* dst, cudaStream_t stream) {
    if (!W || !dst || out <= 0 || ncols <= 0 || col0 < 0 || col0 + ncols > ld) return EDGE0_EINVAL;
    const long long n = (long long)out * ncols;
    const int bs = 256;
    pack_cols_T_kernel<<<(unsigned)((n + bs - 1) / bs), bs, 0, stream>>>(W, out, ld, col0, ncols, dst);
    return cudaGetLastError() == cudaSuccess ? EDGE0_OK : EDGE0_ECUDA;
}
