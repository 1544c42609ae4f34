// gdn_chunk_fwd_noalloc: the chunked prefill for callers that cannot allocate.
//
// Some callers have no way to hand the library a workspace: code that runs
// where cudaMalloc is off limits (inside a host callback or a custom memory
// pool's own hooks, or a runtime that forbids allocations after start-up so
// that its memory footprint stays fixed). For them this entry point keeps its
// scratch in one statically sized device array that is part of the loaded
// module, so a call never allocates or frees anything.
//
// The array holds GDN_NOALLOC_SCRATCH_BYTES bytes. Every GPU that loads the
// library keeps that much device memory for the life of the process, which
// is why the size is modest; a problem whose workspace
// (gdn_chunk_fwd_workspace_size) is larger is rejected with GDN_ETOOBIG.
//
// In host code the array's name is only a host-side stand-in, never a device
// address. The device address is looked up once per device, with that device
// current, by cudaGetSymbolAddress on the first call made on that device, and
// cached with the id of the context it belongs to: a cudaDeviceReset unloads
// the module, and the first call in the new context looks the address up
// again instead of handing the kernels a stale pointer.
#include <mutex>

#include "gdn_common.cuh"
#include "tma_host.cuh"

namespace gdn {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxNoallocDevices = 64;
void *g_scratch_addr[kMaxNoallocDevices];
unsigned long long g_scratch_ctx[kMaxNoallocDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (set-up on the
// first call per device and context; later calls only read the cache).
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxNoallocDevices) return GDN_ECUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    unsigned long long ctx = 0;
    const bool have_ctx = current_context_id(&ctx);
    if (!g_scratch_addr[dev] || !have_ctx || g_scratch_ctx[dev] != ctx) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return GDN_ECUDA;
        g_scratch_addr[dev] = ptr;
        g_scratch_ctx[dev] = (have_ctx || current_context_id(&ctx)) ? ctx : 0;
    }
    *out = g_scratch_addr[dev];
    return GDN_OK;
}

}  // namespace
}  // namespace gdn

extern "C" int gdn_chunk_fwd_noalloc(const gdn_problem *p, const void *q, const void *k, const void *v,
                                     const float *g, const float *beta, float scale, const float *initial_state,
                                     const int32_t *cu_seqlens, void *out, float *final_state, void *stream) {
    const size_t need = gdn_chunk_fwd_workspace_size(p);
    if (need == 0) {
        // invalid problem: let the regular entry point name the error; it
        // returns before any CUDA call because the descriptor is rejected
        return gdn_chunk_fwd(p, q, k, v, g, beta, scale, initial_state, cu_seqlens, out, final_state, nullptr, 0,
                             stream);
    }
    if (need > size_t(GDN_NOALLOC_SCRATCH_BYTES)) return GDN_ETOOBIG;
    void *scratch = nullptr;
    const int st = gdn::scratch_address(&scratch);
    if (st != GDN_OK) return st;
    // The workspace contents need no initialisation (every kernel of the
    // forward writes what it later reads), so nothing is cleared here.
    return gdn_chunk_fwd(p, q, k, v, g, beta, scale, initial_state, cu_seqlens, out, final_state, scratch,
                         size_t(GDN_NOALLOC_SCRATCH_BYTES), stream);
}
