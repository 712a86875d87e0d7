// noalloc.cu -- the layer-by-layer evaluation (first convolution, then the 1x1 convolution)
// with its intermediate held in a fixed device array compiled into the library, for callers
// that must not allocate device memory while they run (see fcm_run_unfused_static in fcm.h).
#include <cuda_runtime.h>

#include <mutex>

#include "fcm_internal.h"

namespace {

// Largest intermediate (N * Ho * Wo * Cm elements of the storage dtype) the entry point takes.
constexpr size_t kStaticScratchBytes = (size_t)16 << 20;   // 16 MiB

// One copy per device that loads the library, kept until the process exits.  Host code must
// not pass this name to a kernel: on the host it only stands in for the symbol.  The device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_addr[kMaxDevices];             // device address of g_static_scratch, per device
unsigned long long g_scratch_ctx[kMaxDevices];  // the context that address belongs to

}  // namespace

extern "C" FCM_API fcm_status fcm_run_unfused_static(fcm_handle *h, const void *in, void *out,
                                                     void *stream) {
    FcmNvtxRange nvtx("fcm_run_unfused_static");
    if (!h) return fcm_fail(FCM_ERR_INVALID_ARG, "handle is NULL");
    const size_t need = h->m_elems * (size_t)h->esize;
    if (need > kStaticScratchBytes)
        return fcm_fail(FCM_ERR_UNSUPPORTED,
                        "intermediate of %zu bytes exceeds the %zu-byte static scratch of "
                        "fcm_run_unfused_static; use fcm_run with FCM_MODE_UNFUSED",
                        need, kStaticScratchBytes);
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fcm_fail(FCM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev != h->device)
        return fcm_fail(FCM_ERR_INVALID_ARG, "current device %d is not the handle's device %d", dev,
                        h->device);
    if (dev < 0 || dev >= kMaxDevices)
        return fcm_fail(FCM_ERR_UNSUPPORTED, "device ordinal %d above %d", dev, kMaxDevices - 1);
    void *scratch = nullptr;
    {
        // set-up with the device current: once per device, and again whenever the device's
        // context has changed since (a device reset loads the library's module anew, at a
        // possibly different address); a context the driver cannot identify looks it up every
        // time
        std::lock_guard<std::mutex> lock(g_mutex);
        const unsigned long long ctx = fcm_current_ctx_id();
        if (!g_scratch_addr[dev] || ctx == 0 || g_scratch_ctx[dev] != ctx) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_static_scratch);
            if (e != cudaSuccess || !p)
                return fcm_fail(FCM_ERR_CUDA, "cudaGetSymbolAddress(static scratch): %s",
                                cudaGetErrorString(e));
            g_scratch_addr[dev] = p;
            g_scratch_ctx[dev] = fcm_current_ctx_id();   // the runtime's context is current now
        }
        scratch = g_scratch_addr[dev];
    }
    // The first kernel writes every element of the intermediate, so nothing needs clearing.
    fcm_status st = fcm_run(h, FCM_MODE_CONV1_ONLY, in, scratch, stream);
    if (st != FCM_OK) return st;
    return fcm_run(h, FCM_MODE_PW_ONLY, scratch, out, stream);
}
