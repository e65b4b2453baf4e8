// Allocation-free entry point: gdn2_chunk_fwd with its workspace taken from a
// fixed device array that lives in this library, for callers that cannot
// allocate device memory (see include/gdn2.h, gdn2_chunk_fwd_noalloc).
#include <mutex>

#include "gdn2_internal.cuh"

namespace {

constexpr int kMaxDevices = 64;

// The scratch every call of gdn2_chunk_fwd_noalloc uses.  A file-scope device
// array: each GPU that loads the library holds GDN2_NOALLOC_SCRATCH_BYTES of
// it until the process exits.  Host code must never pass the symbol itself to
// a kernel (on the host it is a stand-in, not a device address); its device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN2_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void *g_scratch[kMaxDevices] = {};

// Device address of the scratch on `dev` (the current device), looked up once
// per device; nullptr if the lookup fails.  The address belongs to the context
// current at the lookup (it does not survive cudaDeviceReset).
void *scratch_address(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch[dev]) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_scratch[dev] = ptr;
    }
    return g_scratch[dev];
}

// The scratch of the current device after the architecture check: the image
// holds sm_103a code only, so on another device the lookup itself would fail
// with a CUDA error instead of GDN2_ERR_ARCH.
gdn2_status current_scratch(void **ws) {
    int dev = 0;
    if (!gdn2::device_is_sm103(&dev)) return GDN2_ERR_ARCH;
    *ws = scratch_address(dev);
    return *ws ? GDN2_OK : GDN2_ERR_CUDA;
}

}  // namespace

extern "C" gdn2_status gdn2_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const void *g,
                                             const void *beta, const void *w, float scale,
                                             const void *initial_state, const void *cu_seqlens, void *out,
                                             void *final_state, const gdn2_dims *dims, void *stream) {
    if (!dims) return GDN2_ERR_NULL;
    if (gdn2_workspace_bytes(dims) > static_cast<size_t>(GDN2_NOALLOC_SCRATCH_BYTES))
        return GDN2_ERR_NOALLOC_LIMIT;
    void *ws = nullptr;
    const gdn2_status st = current_scratch(&ws);
    if (st != GDN2_OK) return st;
    return gdn2_chunk_fwd(q, k, v, g, beta, w, scale, initial_state, cu_seqlens, out, final_state, dims, ws,
                          static_cast<size_t>(GDN2_NOALLOC_SCRATCH_BYTES), stream);
}

extern "C" gdn2_status gdn2_noalloc_device_status(void *stream, int32_t *status) {
    if (!status) return GDN2_ERR_NULL;
    void *ws = nullptr;
    const gdn2_status st = current_scratch(&ws);
    if (st != GDN2_OK) return st;
    return gdn2_device_status(ws, stream, status);
}
