// lora_linear_fwd_static_ws: the LoRA-augmented linear for callers that cannot give the library
// a workspace.
//
// Some hosts cannot allocate device memory when they call into this library.  One example is
// an operator plugin that runs inside someone else's engine: the engine hands it its inputs
// and outputs and owns every allocation, so the plugin has no allocator of its own.  Another
// is a host that runs under a fixed device-memory budget set at start-up and may not grow it.
// For them cudaMalloc is not an option (besides, it synchronises the device).
//
// For them, the shrink output that lora_linear_fwd keeps in the caller's workspace lives here
// in a fixed device array that belongs to the library (g_static_ws, kStaticWsBytes).  Every GPU
// that loads the library holds it until the process exits.  Batches that need more are refused
// with LORA_ENOSPACE.
//
// In host code g_static_ws names a host-side stand-in, not the device array, so the kernels get
// its device address: the first call on a device looks it up with cudaGetSymbolAddress while
// that device is current, checks the result, and caches it per device.  Make that first call
// before any stream capture.  The pool's device must be the current device.
//
// All calls share the one array, which keeps whatever the last call wrote: calls that may run
// at the same time on the GPU (different streams, or graphs replayed concurrently) overwrite
// each other's data.  Nothing in it has to start at zero -- every value a call reads was
// written earlier in the same call (the shrink writes every element of s that the GEMM or the
// expand reads).
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace lora {
namespace {

constexpr size_t kStaticWsBytes = size_t(4) << 20;  // 4 MiB of float32 shrink output
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

std::mutex g_static_ws_mu;
void* g_static_ws_ptr[kMaxDevices] = {};

// Device address of g_static_ws on the pool's device, which must be the current device
// (looked up once per device, with that device current).
int static_ws_address(int pool_device, void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_error(LORA_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (pool_device >= 0 && dev != pool_device)
        return set_error(LORA_EINVAL, "the pool lives on device %d but device %d is current: make the pool's device "
                                      "current before the call", pool_device, dev);
    if (dev < 0 || dev >= kMaxDevices) return set_error(LORA_EUNSUP, "device ordinal %d >= %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_static_ws_mu);
    if (!g_static_ws_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_ws);
        if (e != cudaSuccess || !p)
            return set_error(LORA_ECUDA, "cudaGetSymbolAddress(static workspace): %s", cudaGetErrorString(e));
        g_static_ws_ptr[dev] = p;
    }
    *out = g_static_ws_ptr[dev];
    return LORA_OK;
}

}  // namespace
}  // namespace lora

using namespace lora;

extern "C" int lora_linear_fwd_static_ws(lora_pool_t pool, const void* W_dev, const void* x_dev, void* y_dev,
                                         const lora_segments* seg, int variant, void* stream) {
    if (!pool || !seg) return set_error(LORA_EINVAL, "pool/seg is NULL");
    const PoolView pv = pool_view(pool);
    const int n = seg->n_tokens;
    if (seg->n_slots != pv.S)
        return set_error(LORA_EINVAL, "segments were built for %d slots, pool has %d", seg->n_slots, pv.S);
    if (variant < LORA_VARIANT_AUTO || variant > LORA_VARIANT_CUDA_CORE)
        return set_error(LORA_EINVAL, "bad variant %d", variant);
    if (n == 0) return LORA_OK;
    if (!W_dev || !x_dev || !y_dev) return set_error(LORA_EINVAL, "W/x/y is NULL");
    const size_t align = pv.dtype != LORA_F32 ? 16 : 4;
    if ((reinterpret_cast<uintptr_t>(W_dev) | reinterpret_cast<uintptr_t>(x_dev) | reinterpret_cast<uintptr_t>(y_dev)) %
        align)
        return set_error(LORA_EINVAL, "W/x/y must be %zu-byte aligned", align);
    const size_t need = sizeof(float) * (size_t)n * pv.R * (size_t)shrink_parts(pv, n, false);
    if (need > kStaticWsBytes)
        return set_error(LORA_ENOSPACE,
                         "static workspace holds %zu bytes, this call needs %zu (n=%d, r_max=%d): use lora_linear_fwd "
                         "with a caller workspace",
                         kStaticWsBytes, need, n, pv.R);
    void* ws = nullptr;
    int rc = static_ws_address(pool->device, &ws);
    if (rc) return rc;
    // the same launch sequence as lora_linear_fwd, with the library's array as the workspace
    return linear_fwd_impl(pool, W_dev, x_dev, y_dev, seg, variant, static_cast<float*>(ws), nullptr, 0,
                           static_cast<cudaStream_t>(stream));
}
