// Self-test of the failure detection every kernel relies on: one thread waits, with
// a short limit, on an mbarrier that nothing ever arrives on -- the same bounded
// wait the pipelines use -- so the limit runs out, the status word records it and
// the kernel returns normally, leaving the context usable.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace lora {

namespace {

__global__ void k_wait_selftest(unsigned *status, uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    // No arrive and no copy will ever complete phase 0.
    mbar_wait_bounded(b, 0, status, kDevTimeoutPipe, limit_ns);
}

}  // namespace

cudaError_t launch_wait_selftest(unsigned *status, uint64_t limit_ns, cudaStream_t stream)
{
    k_wait_selftest<<<1, 1, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace lora
