// Fixed device scratch for lora_fused_noalloc: the partial V of the tensor-core
// tile path and the tile list live in file-scope __device__ arrays, so a call
// needs no allocation.  Every GPU that loads the library holds these arrays until
// the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace lora {

namespace {

// 64 slots of one tile-part each: 64 x 64 KB = 4 MB of partial V, the list, and
// 8 MB for the dense adapter rows of a call whose adapters need copying.
static __device__ __align__(256) float g_noalloc_vparts[kNoAllocSlots * (kVPartBytes / 4)];
static __device__ __align__(256) TileItem g_noalloc_items[kNoAllocSlots];
static __device__ __align__(256) uint16_t g_noalloc_dense[kNoAllocDenseBytes / 2];

struct ItemsArg {
    TileItem items[kNoAllocSlots];
    int n;
};

// Copies the tile list from the launch's parameter block into the fixed array
// (device code names the array directly).
__global__ void k_put_items(const __grid_constant__ ItemsArg a)
{
    if (int(threadIdx.x) < a.n)
        g_noalloc_items[threadIdx.x] = a.items[threadIdx.x];
}

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
        void *v = nullptr, *it = nullptr, *dn = nullptr;
        const cudaError_t e1 = cudaGetSymbolAddress(&v, g_noalloc_vparts);
        const cudaError_t e2 = cudaGetSymbolAddress(&it, g_noalloc_items);
        const cudaError_t e3 = cudaGetSymbolAddress(&dn, g_noalloc_dense);
        if (prev != device)
            cudaSetDevice(prev);
        if (e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess || !v || !it || !dn)
            return -1;
        g_scratch[device].vparts = static_cast<float *>(v);
        g_scratch[device].items = static_cast<TileItem *>(it);
        g_scratch[device].dense = static_cast<uint16_t *>(dn);
        g_ready[device] = true;
    }
    *out = g_scratch[device];
    return 0;
}

cudaError_t noalloc_put_items(const TileItem *items, int n, cudaStream_t stream)
{
    if (n < 0 || n > kNoAllocSlots)
        return cudaErrorInvalidValue;
    ItemsArg a;
    for (int i = 0; i < n; ++i)
        a.items[i] = items[i];
    a.n = n;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kNoAllocSlots);
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, k_put_items, a);
}

}  // namespace lora
