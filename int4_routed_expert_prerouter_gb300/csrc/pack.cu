// Conversion of canonical weights into the packed, fragment-ordered HBM layouts.
//
// Every packed block holds what one warp's m16n8k16 tensor-core step reads:
// lane L = 4 g + t (g = L / 4, t = L % 4) owns the A elements of rows g and g + 8
// at step-local inputs k in {2t, 2t+1, 2t+8, 2t+9}.
//
// int4 step word (4 bytes per lane, 128 bytes per row tile and step): nibble
// positions (bits 4p..4p+3) hold
//     p = 0: (g, 2t)    p = 1: (g+8, 2t)    p = 2: (g, 2t+8)    p = 3: (g+8, 2t+8)
//     p = 4: (g, 2t+1)  p = 5: (g+8, 2t+1)  p = 6: (g, 2t+9)    p = 7: (g+8, 2t+9)
// so that word & 0x000F000F, word & 0x00F000F0, (word >> 8) & 0x000F000F and
// (word >> 8) & 0x00F000F0 are the four A registers as fp16 subnormals
// (q * 2^-24, rows g+8 scaled by 16).
// fp16 step block (16 bytes per lane, 512 per row tile and step): the lane's A
// registers a0..a3 = (g, 2t|2t+1), (g+8, 2t|2t+1), (g, 2t+8|2t+9), (g+8, 2t+8|2t+9).
//
// Packed matrices.  The decode engine splits the input groups of a matrix that
// multiplies x, and the output rows of down, into two halves (half 0: the first
// n/2, half 1: the rest), one per CTA of a pair; each half is stored contiguously
// so that a CTA's share of consecutive row tiles is one run of bytes.
//   gate/up  [E][half][I/8 tiles][groups of the half][576]: tile j interleaves
//            gate rows 8j..8j+7 (tile rows 0..7) with up rows 8j..8j+7 (tile rows
//            8..15); a 576-byte unit = 4 step words per lane (512 B) + (s, b) of
//            rows g and g + 8 at 512 + 8 g.
//   down     [E][I/64 groups][half of the d/16 row tiles]: 4 step blocks of 128 B
//            per row tile of the half (step major), then the half's 64-byte
//            scale/bias blocks; one 16-input slice of the intermediate over a
//            half of the output rows is contiguous.
//   rows     [E][out/16 row tiles][in/64 groups][576]: the gate/up unit format with
//            the rows in order (down, for the batch-1 kernel's output row tiles).
//   fp16     [half][out/16 row tiles][groups of the half][4 steps][512] (row
//            tiles x input groups; every matrix that multiplies x) or
//            [in/16 steps][out/16 row tiles][512] (K-major, for the head's fc2).
#include "internal.cuh"

namespace edge0 {

__device__ __forceinline__ uint32_t nib(const uint32_t* row_words, int i) {
    return (row_words[i >> 3] >> (4 * (i & 7))) & 0xFu;
}

// one step word for lane (g, t): rows r0 (tile row g) and r1 (tile row g + 8) of
// the canonical words, inputs k0 + {2t, 2t+1, 2t+8, 2t+9}; null rows are zero
__device__ __forceinline__ uint32_t step_word(const uint32_t* r0, const uint32_t* r1, int k0, int t) {
    const int k = k0 + 2 * t;
    uint32_t w = 0;
    if (r0) w |= nib(r0, k) | (nib(r0, k + 8) << 8) | (nib(r0, k + 1) << 16) | (nib(r0, k + 9) << 24);
    if (r1) w |= (nib(r1, k) << 4) | (nib(r1, k + 8) << 12) | (nib(r1, k + 1) << 20) | (nib(r1, k + 9) << 28);
    return w;
}

// gate/up interleaved: one thread per (expert, tile, group, lane)
__global__ void pack_gu_kernel(const uint32_t* __restrict__ qg, const uint16_t* __restrict__ sg,
                               const uint16_t* __restrict__ bg, const uint32_t* __restrict__ qu,
                               const uint16_t* __restrict__ su, const uint16_t* __restrict__ bu,
                               int E, int I, int d, char* __restrict__ dst) {
    const int n_t = I / kHalfRow, n_g = d / kGroup;
    const long long units = (long long)E * n_t * n_g;
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (tid >= units * 32) return;
    const int lane = (int)(tid & 31);
    const long long unit = tid >> 5;
    const int c = (int)(unit % n_g);
    const int j = (int)((unit / n_g) % n_t);
    const int e = (int)(unit / ((long long)n_g * n_t));
    const int g = lane >> 2, t = lane & 3;
    const int row = j * kHalfRow + g;
    const long long wpr = d / 8, gpr = d / kGroup;
    const uint32_t* rg = qg + ((long long)e * I + row) * wpr;
    const uint32_t* ru = qu + ((long long)e * I + row) * wpr;
    uint4 v;
    v.x = step_word(rg, ru, kGroup * c + 0, t);
    v.y = step_word(rg, ru, kGroup * c + 16, t);
    v.z = step_word(rg, ru, kGroup * c + 32, t);
    v.w = step_word(rg, ru, kGroup * c + 48, t);
    // half-major position of unit (j, c) of expert e
    const int n0 = n_g / 2, h = c >= n0 ? 1 : 0, nh = h ? n_g - n0 : n0;
    const long long pos = (long long)e * n_t * n_g + (long long)h * n_t * n0 + (long long)j * nh + (c - h * n0);
    char* u = dst + pos * kQ4Unit;
    *reinterpret_cast<uint4*>(u + 16 * lane) = v;
    if (t == 0) {
        const long long o = ((long long)e * I + row) * gpr + c;
        ushort4 sb;
        sb.x = sg[o];
        sb.y = bg[o];
        sb.z = su[o];
        sb.w = bu[o];
        *reinterpret_cast<ushort4*>(u + 512 + 8 * g) = sb;
    }
}

// down, K-major: one thread per (expert, group, row tile, lane)
__global__ void pack_down_kernel(const uint32_t* __restrict__ q, const uint16_t* __restrict__ s,
                                 const uint16_t* __restrict__ b, int E, int out, int in,
                                 char* __restrict__ dst) {
    const int n_rt = ceil_div(out, kRowTile), n_g = in / kGroup;
    const long long items = (long long)E * n_g * n_rt;
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (tid >= items * 32) return;
    const int lane = (int)(tid & 31);
    const long long it = tid >> 5;
    const int i = (int)(it % n_rt);
    const int c = (int)((it / n_rt) % n_g);
    const int e = (int)(it / ((long long)n_rt * n_g));
    const int g = lane >> 2, t = lane & 3;
    const int r0 = i * kRowTile + g, r1 = r0 + 8;
    const long long wpr = in / 8, gpr = in / kGroup;
    const uint32_t* w0 = r0 < out ? q + ((long long)e * out + r0) * wpr : nullptr;
    const uint32_t* w1 = r1 < out ? q + ((long long)e * out + r1) * wpr : nullptr;
    // half h of the row tiles: [4 steps][row tiles of the half][128] then [row tiles of the half][64]
    const int n0 = n_rt / 2, h = i >= n0 ? 1 : 0, nh = h ? n_rt - n0 : n0, il = i - h * n0;
    char* base = dst + ((long long)e * n_g + c) * n_rt * kQ4Unit + (long long)h * n0 * kQ4Unit;
    for (int st = 0; st < 4; ++st)
        *reinterpret_cast<uint32_t*>(base + ((long long)st * nh + il) * kQ4Quarter + 4 * lane) =
            step_word(w0, w1, kGroup * c + 16 * st, t);
    if (t == 0) {
        ushort4 sb;
        const long long o0 = ((long long)e * out + r0) * gpr + c, o1 = ((long long)e * out + r1) * gpr + c;
        sb.x = r0 < out ? s[o0] : 0;
        sb.y = r0 < out ? b[o0] : 0;
        sb.z = r1 < out ? s[o1] : 0;
        sb.w = r1 < out ? b[o1] : 0;
        *reinterpret_cast<ushort4*>(base + 4LL * nh * kQ4Quarter + (long long)il * kQ4Scales + 8 * g) = sb;
    }
}

// int4 row-tile major: [E][row tile][group][576] (the unit format of gate/up,
// rows in order); one thread per (expert, row tile, group, lane)
__global__ void pack_rows_kernel(const uint32_t* __restrict__ q, const uint16_t* __restrict__ s,
                                 const uint16_t* __restrict__ b, int E, int out, int in,
                                 char* __restrict__ dst) {
    const int n_rt = ceil_div(out, kRowTile), n_g = in / kGroup;
    const long long units = (long long)E * n_rt * n_g;
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (tid >= units * 32) return;
    const int lane = (int)(tid & 31);
    const long long unit = tid >> 5;
    const int c = (int)(unit % n_g);
    const int i = (int)((unit / n_g) % n_rt);
    const int e = (int)(unit / ((long long)n_g * n_rt));
    const int g = lane >> 2, t = lane & 3;
    const int r0 = i * kRowTile + g, r1 = r0 + 8;
    const long long wpr = in / 8, gpr = in / kGroup;
    const uint32_t* w0 = r0 < out ? q + ((long long)e * out + r0) * wpr : nullptr;
    const uint32_t* w1 = r1 < out ? q + ((long long)e * out + r1) * wpr : nullptr;
    uint4 v;
    v.x = step_word(w0, w1, kGroup * c + 0, t);
    v.y = step_word(w0, w1, kGroup * c + 16, t);
    v.z = step_word(w0, w1, kGroup * c + 32, t);
    v.w = step_word(w0, w1, kGroup * c + 48, t);
    char* u = dst + unit * kQ4Unit;
    *reinterpret_cast<uint4*>(u + 16 * lane) = v;
    if (t == 0) {
        ushort4 sb;
        const long long o0 = ((long long)e * out + r0) * gpr + c, o1 = ((long long)e * out + r1) * gpr + c;
        sb.x = r0 < out ? s[o0] : 0;
        sb.y = r0 < out ? b[o0] : 0;
        sb.z = r1 < out ? s[o1] : 0;
        sb.w = r1 < out ? b[o1] : 0;
        *reinterpret_cast<ushort4*>(u + 512 + 8 * g) = sb;
    }
}

// fp16 step block of lane (g, t) for row tile i, inputs k0 + {2t, 2t+1, 2t+8, 2t+9}
__device__ __forceinline__ uint4 f16_block(const uint16_t* W, int out, int ld, int i, int k0, int g, int t) {
    const int r0 = i * kRowTile + g, r1 = r0 + 8, k = k0 + 2 * t;
    auto at = [&](int r, int c) -> uint32_t { return r < out ? W[(long long)r * ld + c] : 0u; };
    uint4 v;
    v.x = at(r0, k) | (at(r0, k + 1) << 16);
    v.y = at(r1, k) | (at(r1, k + 1) << 16);
    v.z = at(r0, k + 8) | (at(r0, k + 9) << 16);
    v.w = at(r1, k + 8) | (at(r1, k + 9) << 16);
    return v;
}

// kmajor = 0: [row tile][step]; 1: [step][row tile].  One thread per (block, lane).
__global__ void pack_f16_kernel(const uint16_t* __restrict__ W, int out, int in, int ld, int kmajor,
                                char* __restrict__ dst) {
    const int n_rt = ceil_div(out, kRowTile), n_s = in / 16;
    const long long blocks = (long long)n_rt * n_s;
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (tid >= blocks * 32) return;
    const int lane = (int)(tid & 31);
    const long long blk = tid >> 5;
    int i, st;
    long long pos = blk;
    if (kmajor) {
        i = (int)(blk % n_rt);
        st = (int)(blk / n_rt);
    } else {
        // half-major over the input groups: [half][row tile][group of the half][step]
        st = (int)(blk % n_s);
        i = (int)(blk / n_s);
        const int n_g = n_s / 4, n0 = n_g / 2, c = st / 4, h = c >= n0 ? 1 : 0, nh = h ? n_g - n0 : n0;
        pos = ((long long)h * n_rt * n0 + (long long)i * nh + (c - h * n0)) * 4 + st % 4;
    }
    *reinterpret_cast<uint4*>(dst + pos * kF16Step + 16 * lane) =
        f16_block(W, out, ld, i, 16 * st, lane >> 2, lane & 3);
}

__global__ void pack_cols_T_kernel(const uint16_t* __restrict__ W, int out, int ld, int col0,
                                   int ncols, uint16_t* __restrict__ dst) {
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (tid >= (long long)out * ncols) return;
    const int o = (int)(tid % out), j = (int)(tid / out);
    dst[(long long)j * out + o] = W[(long long)o * ld + col0 + j];
}

static bool aligned(const void* p, int a) { return ((uintptr_t)p % a) == 0; }

int launch_1d(long long threads) {
    return (int)((threads + 255) / 256);
}

}  // namespace edge0

using namespace edge0;

extern "C" size_t edge0_q4_gate_up_packed_bytes(int E, int I, int d) {
    if (E <= 0 || I <= 0 || d <= 0 || I % kGroup || d % kGroup) return 0;
    return (size_t)E * (size_t)q4_bytes(2 * I, d);
}

extern "C" int edge0_pack_q4_gate_up(const uint32_t* q_gate, const uint16_t* s_gate,
                                     const uint16_t* b_gate, const uint32_t* q_up,
                                     const uint16_t* s_up, const uint16_t* b_up, int E, int I, int d,
                                     void* packed, cudaStream_t stream) {
    if (!q_gate || !s_gate || !b_gate || !q_up || !s_up || !b_up || !packed) return EDGE0_EINVAL;
    if (E <= 0 || I <= 0 || d <= 0 || I % kGroup || d % kGroup) return EDGE0_EINVAL;
    if (!aligned(q_gate, 4) || !aligned(q_up, 4) || !aligned(s_gate, 2) || !aligned(b_gate, 2) ||
        !aligned(s_up, 2) || !aligned(b_up, 2) || !aligned(packed, 16))
        return EDGE0_EINVAL;
    const long long threads = (long long)E * (I / kHalfRow) * (d / kGroup) * 32;
    pack_gu_kernel<<<launch_1d(threads), 256, 0, stream>>>(q_gate, s_gate, b_gate, q_up, s_up, b_up,
                                                           E, I, d, (char*)packed);
    return cudaGetLastError() == cudaSuccess ? EDGE0_OK : EDGE0_ECUDA;
}

extern "C" size_t edge0_q4_down_packed_bytes(int E, int out, int in) {
    if (E <= 0 || out <= 0 || in <= 0 || in % kGroup) return 0;
    return (size_t)E * (size_t)q4_bytes(out, in);
}

extern "C" int edge0_pack_q4_down(const uint32_t* q, const uint16_t* s, const uint16_t* b, int E,
                                  int out, int in, void* packed, cudaStream_t stream) {
    if (!q || !s || !b || !packed || E <= 0 || out <= 0 || in <= 0 || in % kGroup)
        return EDGE0_EINVAL;
    if (!aligned(q, 4) || !aligned(s, 2) || !aligned(b, 2) || !aligned(packed, 16))
        return EDGE0_EINVAL;
    const long long threads = (long long)E * (in / kGroup) * ceil_div(out, kRowTile) * 32;
    pack_down_kernel<<<launch_1d(threads), 256, 0, stream>>>(q, s, b, E, out, in, (char*)packed);
    return cudaGetLastError() == cudaSuccess ? EDGE0_OK : EDGE0_ECUDA;
}

extern "C" int edge0_pack_q4_rows(const uint32_t* q, const uint16_t* s, const uint16_t* b, int E,
                                  int out, int in, void* packed, cudaStream_t stream) {
    if (!q || !s || !b || !packed || E <= 0 || out <= 0 || in <= 0 || in % kGroup)
        return EDGE0_EINVAL;
    if (!aligned(q, 4) || !aligned(s, 2) || !aligned(b, 2) || !aligned(packed, 16))
        return EDGE0_EINVAL;
    const long long threads = (long long)E * ceil_div(out, kRowTile) * (in / kGroup) * 32;
    pack_rows_kernel<<<launch_1d(threads), 256, 0, stream>>>(q, s, b, E, out, in, (char*)packed);
    return cudaGetLastError() == cudaSuccess ? EDGE0_OK : EDGE0_ECUDA;
}

extern "C" size_t edge0_f16_packed_bytes(int out, int in) {
    if (out <= 0 || in <= 0 || in % kGroup) return 0;
    return (size_t)f16_bytes(out, in);
}

static int pack_f16_common(const uint16_t* W, int out, int in, int ld, void* packed, int kmajor,
                           cudaStream_t stream) {
    if (!W || !packed || out <= 0 || in <= 0 || in % kGroup || ld < in) return EDGE0_EINVAL;
    if (!aligned(W, 2) || !aligned(packed, 16)) return EDGE0_EINVAL;
    const long long threads = (long long)ceil_div(out, kRowTile) * (in / 16) * 32;
    pack_f16_kernel<<<launch_1d(threads), 256, 0, stream>>>(W, out, in, ld, kmajor, (char*)packed);
    return cudaGetLastError() == cudaSuccess ? EDGE0_OK : EDGE0_ECUDA;
}

extern "C" int edge0_pack_f16(const uint16_t* W, int out, int in, int ld, void* packed,
                              cudaStream_t stream) {
    return pack_f16_common(W, out, in, ld, packed, 0, stream);
}

extern "C" int edge0_pack_f16_kmajor(const uint16_t* W, int out, int in, int ld, void* packed,
                                     cudaStream_t stream) {
    return pack_f16_common(W, out, in, ld, packed, 1, stream);
}

extern "C" int edge0_pack_cols_T(const uint16_t* W, int out, int ld, int col0, int ncols,
                                 uint16_t* dst, cudaStream_t stream) {
    if (!W || !dst || out <= 0 || ncols <= 0 || col0 < 0 || col0 + ncols > ld) return EDGE0_EINVAL;
    const long long n = (long long)out * ncols;
    pack_cols_T_kernel<<<launch_1d(n), 256, 0, stream>>>(W, out, ld, col0, ncols, dst);
    return cudaGetLastError() == cudaSuccess ? EDGE0_OK : EDGE0_ECUDA;
}
