// Adapter page-in: an adapter's A and B rows copied from page-locked host memory into
// its pages of the pools (S-LoRA: adapters live in host memory and are brought into
// the unified pool on demand, overlapped with compute; VaLoRA: only A and B move).
//
// One CTA per page and side.  The CTA reads its row straight from host memory over
// the CPU-GPU link (the buffer is mapped into the device's address space) with
// 16-byte loads, all of a pass in flight before its first store, and writes the
// pool page.  No staging copy in device memory and one launch per adapter.  The
// launch is an ordinary stream launch (not a programmatic dependent): it starts only
// after every earlier kernel of the stream, some of which may still read the pages
// it overwrites.
#include <cuda_runtime.h>

#include "internal.h"

namespace lora {

namespace {

constexpr int kPageInThreads = 128;
constexpr int kPerThread = 8;                 // 16-byte vectors per thread per pass

__global__ void __launch_bounds__(kPageInThreads) k_page_in(const __grid_constant__ PageInArgs a)
{
    const PageInSide &sd = a.side[blockIdx.y];
    const int j = int(blockIdx.x);            // page j of the adapter
    if (j >= a.rank)
        return;
    const int nv = sd.width / 8;
    const uint4 *src = reinterpret_cast<const uint4 *>(sd.host + int64_t(j) * sd.width);
    uint4 *dst = reinterpret_cast<uint4 *>(sd.pool + int64_t(sd.page[j]) * sd.pw);
    for (int q0 = 0; q0 < nv; q0 += kPerThread * kPageInThreads) {
        uint4 v[kPerThread];
#pragma unroll
        for (int e = 0; e < kPerThread; ++e) {
            const int q = q0 + e * kPageInThreads + int(threadIdx.x);
            if (q < nv)
                v[e] = src[q];
        }
#pragma unroll
        for (int e = 0; e < kPerThread; ++e) {
            const int q = q0 + e * kPageInThreads + int(threadIdx.x);
            if (q < nv)
                dst[q] = v[e];
        }
    }
}

}  // namespace

cudaError_t launch_page_in(const PageInArgs &a, cudaStream_t stream)
{
    if (a.rank <= 0 || a.rank > kPageInMaxRank)
        return cudaErrorInvalidValue;
    k_page_in<<<dim3(unsigned(a.rank), 2u), kPageInThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace lora
