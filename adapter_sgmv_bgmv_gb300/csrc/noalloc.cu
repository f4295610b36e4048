// Fixed device scratch for lora_fused_noalloc: the partial V of the tensor-core
// tile path and the dense adapter rows live in file-scope __device__ arrays (the
// tile list travels in the launch parameters), so a call needs no allocation.  Every GPU that loads the library holds these arrays until
// the process exits.
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

int noalloc_scratch(int device, NoAllocScratch *out)
{
    if (device < 0 || device >= kMaxDevices)
        return -1;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_ready[device]) {
        // Host code only ever holds a stand-in for the arrays' names: their device
        // addresses come from the runtime, once per device, with it current.
        int prev = 0;
        if (cudaGetDevice(&prev) != cudaSuccess)
            return -1;
        if (prev != device && cudaSetDevice(device) != cudaSuccess)
            return -1;
        void *v = nullptr, *dn = nullptr;
        const cudaError_t e1 = cudaGetSymbolAddress(&v, g_noalloc_vparts);
        const cudaError_t e3 = cudaGetSymbolAddress(&dn, g_noalloc_dense);
        if (prev != device)
            cudaSetDevice(prev);
        if (e1 != cudaSuccess || e3 != cudaSuccess || !v || !dn)
            return -1;
        g_scratch[device].vparts = static_cast<float *>(v);
        g_scratch[device].dense = static_cast<uint16_t *>(dn);
        g_ready[device] = true;
    }
    *out = g_scratch[device];
    return 0;
}

}  // namespace lora
