// decode_static.cu -- lrkv_decode for callers that cannot allocate device memory.
//
// lrkv_decode needs a scratch workspace (one partial softmax state per split
// and head).  Some callers cannot hand one over: cudaMalloc / cudaFree may
// synchronise the whole device and stall every other stream, some host
// frameworks own the GPU allocator and forbid allocations behind their back,
// and some deployments fix their device-memory budget once at start-up.
// lrkv_decode_static_ws gives them the same decode with its scratch in a
// fixed-size array that lives in this library's device image: every GPU that
// loads the library holds LRKV_STATIC_WS_BYTES for it until the process exits.
//
// The array's name seen from host code is only a host-side stand-in, never a
// device address, so its device address is looked up with cudaGetSymbolAddress
// (with the device current) and cached per device together with the id of the
// context it was found in: a context that is destroyed and created again (e.g.
// after cudaDeviceReset) loads the module afresh, and the address is looked up again.
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "lrkv_internal.cuh"

namespace lrkv {
lrkv_status report_error(lrkv_status s, const char* msg);
}

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[LRKV_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

// Id of the calling thread's current context (0 if the driver cannot tell).
unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_cur && get_id && get_cur(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, &id) == CUDA_SUCCESS) return id;
    return 0;
}

}  // namespace

extern "C" lrkv_status lrkv_decode_static_ws(const lrkv_dims* dims, const void* q, const void* BK, const void* BV,
                                             const lrkv_cache* cache, const int32_t* block_table,
                                             int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t batch,
                                             void* out, uint32_t* status_dev, void* stream) {
    const size_t need = lrkv_decode_workspace_bytes(dims, batch);
    if (need > LRKV_STATIC_WS_BYTES) {
        char msg[256];
        std::snprintf(msg, sizeof msg,
                      "lrkv_decode_static_ws: this batch needs %zu bytes of scratch but the static area holds %zu "
                      "(LRKV_STATIC_WS_BYTES); call lrkv_decode with a workspace instead",
                      need, (size_t)LRKV_STATIC_WS_BYTES);
        return lrkv::report_error(LRKV_ERR_WORKSPACE, msg);
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return lrkv::report_error(LRKV_ERR_CUDA, "lrkv_decode_static_ws: no usable current device");
    void* ws = nullptr;
    {
        // (0 before the runtime has made a context current: the lookup below does that, and
        // the id is read again after it)
        unsigned long long ctx = current_context_id();
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (!g_scratch_addr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
            void* p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
            if (e != cudaSuccess || !p) {
                char msg[256];
                std::snprintf(msg, sizeof msg, "lrkv_decode_static_ws: cudaGetSymbolAddress failed: %s",
                              cudaGetErrorString(e));
                return lrkv::report_error(LRKV_ERR_CUDA, msg);
            }
            g_scratch_addr[dev] = p;
            g_scratch_ctx[dev] = current_context_id();
        }
        ws = g_scratch_addr[dev];
    }
    // Every scratch byte the decode kernels read was written earlier in the same
    // call, so nothing left over from a previous call needs clearing.
    return lrkv_decode(dims, q, BK, BV, cache, block_table, max_blocks_per_seq, seq_lens, batch, out, ws,
                       (size_t)LRKV_STATIC_WS_BYTES, status_dev, stream);
}
