// edge0_moe_int4_forward_noalloc: the routed + shared int4 expert forward for
// callers that cannot allocate memory.
//
// Some callers must not call cudaMalloc (or anything else that allocates) at the
// point where they run the MoE block: code inside an allocator-free region of a
// serving loop, code whose memory budget was fixed when the process started, or
// a host that hands this library only the input and output buffers it already
// owns.  For them this entry point keeps the kernel's scratch (its accumulators,
// grid-barrier word and error word) in a fixed array compiled into the library,
// builds the kernel's parameter block on the stack, and needs nothing from the
// caller beyond its inputs and outputs.
//
// The array is allocated in each GPU's memory when the library is loaded there
// and stays until the process exits.  Every call on a device uses the same array;
// two calls whose kernels overlap on the GPU (for instance on two streams) race on
// it and produce wrong results.
#include <string.h>

#include <mutex>

#include "internal.cuh"

using namespace edge0;

namespace {

// fixed scratch of the allocation-free entry point
static __device__ __align__(256) unsigned char g_noalloc_scratch[EDGE0_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code the
// array's name is only a stand-in, so the address is looked up once per device
// (with that device current) and kept.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return EDGE0_ECUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return EDGE0_ECUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return EDGE0_OK;
}

bool a16(const void* p) { return ((uintptr_t)p & 15) == 0; }

}  // namespace

extern "C" int edge0_moe_int4_forward_noalloc(const edge0_moe_desc* moe, const uint16_t* x,
                                              const int32_t* ids, const float* w, int B,
                                              uint16_t* y, cudaStream_t stream) {
    // the same argument rules as edge0_moe_int4_forward
    if (!moe || !x || !ids || !w || !y) return EDGE0_EINVAL;
    const edge0_moe_desc& m = *moe;
    if (!m.gate_up || !m.down || !a16(m.gate_up) || !a16(m.down)) return EDGE0_EINVAL;
    if (!a16(x) || !a16(y)) return EDGE0_EINVAL;
    const bool shared = m.sh_gate_up || m.sh_down;
    if (shared && (!m.sh_gate_up || !m.sh_down || !a16(m.sh_gate_up) || !a16(m.sh_down)))
        return EDGE0_EINVAL;
    const int Is = m.Is > 0 ? m.Is : 64;
    if (B <= 0 || B > EDGE0_MAX_BATCH) return EDGE0_EINVAL;
    if (m.d <= 0 || m.d % kGroup || m.I <= 0 || m.I % kGroup || Is % kGroup) return EDGE0_EINVAL;
    if (m.E <= 0 || m.E > EDGE0_MAX_E || m.E % 16 || m.K <= 0 || m.K > EDGE0_MAX_K || m.K > m.E)
        return EDGE0_EINVAL;
    if (m.slot_table && m.n_slots <= 0) return EDGE0_EINVAL;
    // scratch: header and the accumulators of one layer in two step parities (the
    // trace area at the end of a workspace is never switched on here)
    const WsLayout wl = ws_layout(1, B, m.d, m.E);
    const long long need = wl.trace;
    if (need > (long long)EDGE0_NOALLOC_SCRATCH_BYTES) return EDGE0_EUNSUPPORTED;
    void* scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc) return rc;

    Prog p;   // kernel parameter block, on the stack
    memset(&p, 0, sizeof(p));
    p.mode = MODE_MOE;
    p.L = 1;
    p.B = B;
    p.d = m.d;
    p.E = m.E;
    p.K = m.K;
    p.I = m.I;
    p.Is = Is;
    p.H = 64;
    p.r = 16;
    p.step = 0;
    p.x_in = (const __half*)x;
    p.ids_in = ids;
    p.w_in = w;
    p.y_out = (__half*)y;
    p.Ls = 1;
    p.ws = (char*)scratch;
    LayerP& P = p.layers[0];
    P.gu = (const char*)m.gate_up;
    P.down = (const char*)m.down;
    P.slot_table = m.slot_table;
    P.n_slots = m.slot_table ? m.n_slots : m.E;
    if (shared) {
        P.sh_gu = (const char*)m.sh_gate_up;
        P.sh_down = (const char*)m.sh_down;
        P.flags = LF_SHARED;
    }
    P.n_groups = P.topk_groups = P.head_n_groups = P.head_topk_groups = 1;
    // the shapes are checked before anything is queued: a refused call leaves
    // the array (and a kernel still using it) alone
    int nct = 0, smem = 0;
    rc = engine_grid(&nct);
    if (rc) return rc;
    rc = engine_check(p, nct, engine_smem_max(), &smem);
    if (rc) return rc;
    // every call starts from a cleared header and cleared accumulators: the
    // previous call may have used other shapes
    if (cudaMemsetAsync(scratch, 0, (size_t)need, stream) != cudaSuccess) return EDGE0_ECUDA;
    return engine_launch(p, stream);
}

extern "C" int edge0_noalloc_error(cudaStream_t stream, int* status) {
    if (!status) return EDGE0_EINVAL;
    void* scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc) return rc;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return EDGE0_ECUDA;
    WsHeader h;
    if (cudaMemcpyFromSymbol(&h, g_noalloc_scratch, sizeof(h), 0, cudaMemcpyDeviceToHost) != cudaSuccess)
        return EDGE0_ECUDA;
    *status = h.error;
    if (h.error || h.abort) {
        h.error = 0;
        h.abort = 0;
        if (cudaMemcpyToSymbol(g_noalloc_scratch, &h, sizeof(h), 0, cudaMemcpyHostToDevice) != cudaSuccess)
            return EDGE0_ECUDA;
    }
    return EDGE0_OK;
}
