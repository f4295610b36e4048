// Dense adapter rows for the tensor-core kernels.
//
// The tile shrink, the streaming expand and the merge read an adapter block per K
// block / column chunk.  From a row matrix in which the adapter's pages are
// consecutive rows, that block is one TMA box (or three: 64 + 32 + 16 rows); page
// by page it would be one gather per four pages, and the TMA unit issues those
// too slowly to keep up with the x / y streams.  When every adapter of a call has
// consecutive pages of a rank that is a multiple of 16, the pools are used as they
// are.  Otherwise this kernel copies adapters (S-LoRA's unified pool holds them in
// arbitrary pages) into dense rows, one slot of rp rows per adapter: its rank's
// rows, then zeros up to the rank rounded up to 16 (the rows the tensor-core
// kernels read); the slot's rows beyond those are left unwritten.  The slots are
// the table's cache of dense rows (each adapter copied once, until its pages
// change) or, where that cannot serve, a per-call scratch.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace lora {

namespace {

constexpr int kStageThreads = 128;
constexpr int kPerThread = 8;                 // 16-byte vectors per thread per pass

// Row j of entry blockIdx.x / rp, side blockIdx.y: destination row
// dst_slot[entry] * rp + j, of dst_ld elements.
__device__ __forceinline__ void stage_row(const StageArgs &a)
{
    const StageSide &sd = a.side[blockIdx.y];
    if (!sd.dst)
        return;
    const int row = int(blockIdx.x);
    const int slot = row / a.rp, j = row - slot * a.rp;
    const int rank = a.rank[slot];
    if (j >= ((rank + 15) & ~15))   // the kernels read a slot's rank rounded up to 16 rows
        return;
    const int nv = sd.width / 8;
    uint4 *dst = reinterpret_cast<uint4 *>(sd.dst + (int64_t(a.dst_slot[slot]) * a.rp + j) * sd.dst_ld);
    if (j < rank) {
        const int32_t page = sd.pages[int64_t(a.adapter[slot]) * a.max_rank + j];
        const uint4 *src = reinterpret_cast<const uint4 *>(sd.pool + int64_t(page) * sd.pw);
        // All of a pass's loads are in flight before its first store (a row of up to
        // 8192 elements is one pass), so a row costs one round trip, not one per vector.
        for (int q0 = 0; q0 < nv; q0 += kPerThread * kStageThreads) {
            uint4 v[kPerThread];
#pragma unroll
            for (int e = 0; e < kPerThread; ++e) {
                const int q = q0 + e * kStageThreads + int(threadIdx.x);
                if (q < nv)
                    v[e] = __ldg(src + q);
            }
#pragma unroll
            for (int e = 0; e < kPerThread; ++e) {
                const int q = q0 + e * kStageThreads + int(threadIdx.x);
                if (q < nv)
                    dst[q] = v[e];
            }
        }
    } else {
        // Rank padding: zero, since the expand and the merge multiply these rows.
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        for (int q = threadIdx.x; q < nv; q += kStageThreads)
            dst[q] = z;
    }
}

// One CTA per destination row.  Launched as a programmatic dependent of the kernel
// before it: by default it waits for that kernel first (the pools may be its to
// write).  Early (the caller's guarantee that the kernel just before writes no pool
// or page table; the scratch half is not the one the previous call reads), it copies
// first and waits after -- still before it ends, so that the kernels after it keep
// the stream's order.
__global__ void __launch_bounds__(kStageThreads) k_stage_rows(const __grid_constant__ StageArgs a)
{
    if (!a.early)
        grid_dep_wait();
    stage_row(a);
    if (a.early)
        grid_dep_wait();
}

}  // namespace

cudaError_t launch_stage_rows(const StageArgs &a, cudaStream_t stream)
{
    if (a.n_slots <= 0 || a.n_slots > kStageSlots || a.rp <= 0)
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(a.n_slots * a.rp), 2u);
    cfg.blockDim = dim3(kStageThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_stage_rows, a);
}

}  // namespace lora
