// Fixed device scratch for lora_fused_noalloc: the partial V of the tensor-core
// tile path and the dense adapter rows live in file-scope __device__ arrays (the
// tile list travels in the launch parameters), so a call needs no allocation.
// The arrays belong to this file's module, which the CUDA runtime loads on a device
// the first time anything in it is used; lora_ctx_create does that (through
// noalloc_scratch with refresh), so the 12 MB are taken when a context is created,
// not by a lora_fused_noalloc call, and stay until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace lora {

namespace {

// 64 slots of one tile-part each: 64 x 64 KB = 4 MB of partial V, and 8 MB for
// the dense adapter rows of a call whose adapters need copying.
static __device__ __align__(256) float g_noalloc_vparts[kNoAllocSlots * (kVPartBytes / 4)];
static __device__ __align__(256) uint16_t g_noalloc_dense[kNoAllocDenseBytes / 2];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
bool g_ready[kMaxDevices];
NoAllocScratch g_scratch[kMaxDevices];

}  // namespace

cudaError_t noalloc_scratch(int device, bool refresh, NoAllocScratch *out)
{
    if (device < 0 || device >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_ready[device] || refresh) {
        // Host code only ever holds a stand-in for the arrays' names: their device
        // addresses come from the runtime, once per device, with it current.
        // The addresses belong to the device's primary context: a context created
        // after a cudaDeviceReset looks them up again (refresh).
        g_ready[device] = false;
        int prev = 0;
        cudaError_t e = cudaGetDevice(&prev);
        if (e != cudaSuccess)
            return e;
        if (prev != device && (e = cudaSetDevice(device)) != cudaSuccess)
            return e;
        void *v = nullptr, *dn = nullptr;
        cudaError_t e1 = cudaGetSymbolAddress(&v, g_noalloc_vparts);
        const cudaError_t e3 = cudaGetSymbolAddress(&dn, g_noalloc_dense);
        if (prev != device)
            cudaSetDevice(prev);
        if (e1 == cudaSuccess)
            e1 = e3;
        if (e1 != cudaSuccess)
            return e1;
        if (!v || !dn)
            return cudaErrorInvalidSymbol;
        g_scratch[device].vparts = static_cast<float *>(v);
        g_scratch[device].dense = static_cast<uint16_t *>(dn);
        g_ready[device] = true;
    }
    if (out)
        *out = g_scratch[device];
    return cudaSuccess;
}

}  // namespace lora
