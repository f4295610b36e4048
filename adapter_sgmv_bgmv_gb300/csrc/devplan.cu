// Device-side plan of a row-gather call whose adapter ids live in device memory
// (LoRazor: the operator's launch follows the rows still active; here the active
// rows are found on the device, so a decode step needs no host round trip and can
// be captured in a CUDA graph).
//
// One CTA of 1024 threads, for batches of decode size:
//   1. count the rows of every adapter (ids of -1 are released rows and skipped; an
//      id outside the table or an adapter the table cannot serve leaves its row as
//      it is and raises kDevBadId in the status word);
//   2. exclusive scans over the adapters of the row counts and of the item counts
//      (ceil(count / R) items of at most R rows each);
//   3. write the items {adapter, first perm slot, rows, rank, scale};
//   4. place every active row in its adapter's range of the permutation (an atomic
//      cursor per adapter: the order inside a range is not fixed, and need not be,
//      since every row's result is computed by itself);
//   5. the item count, which the row-gather kernel reads to let surplus CTAs go.
// The counts and offsets live in shared memory, three ints per adapter.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace lora {

namespace {

constexpr int kPlanThreads = 1024;

__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_sums, int &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d)
            x += y;
    }
    if (lane == 31)
        warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, d);
            if (lane >= d)
                w += y;
        }
        warp_sums[lane] = w;   // inclusive over warps
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
    total = warp_sums[31];
    __syncthreads();           // warp_sums is reused by the next scan
    return before;
}

__global__ void __launch_bounds__(kPlanThreads) k_plan_dev(const __grid_constant__ DevPlanArgs a)
{
    extern __shared__ int32_t sm[];
    const int na = a.n_adapters;
    int32_t *cnt = sm;                  // rows per adapter
    int32_t *cur = sm + na;             // row offset, then the placement cursor
    int32_t *ioff = sm + 2 * na;        // item offset
    int *warp_sums = sm + 3 * na;       // 32
    const int tid = threadIdx.x;

    // The ids may be the previous kernel's output, and the previous call's row
    // kernel may still read the permutation and items rewritten here.
    grid_dep_wait();
    grid_dep_launch();                  // the row kernel waits for this grid's end anyway

    for (int k = tid; k < na; k += kPlanThreads)
        cnt[k] = 0;
    __syncthreads();
    bool bad = false;
    for (int i = tid; i < a.n; i += kPlanThreads) {
        const int k = a.ids[i];
        if (k == -1)
            continue;
        if (k < -1 || k >= na || !a.ok[k]) {
            bad = true;
            continue;
        }
        atomicAdd(&cnt[k], 1);
    }
    if (bad)
        raise_status(a.status, kDevBadId);
    __syncthreads();

    // Each thread owns a contiguous chunk of adapters for the scans.
    const int chunk = (na + kPlanThreads - 1) / kPlanThreads;
    const int k0 = min(na, tid * chunk), k1 = min(na, k0 + chunk);
    const int R = a.rows_per_item;
    int rows = 0, items = 0;
    for (int k = k0; k < k1; ++k) {
        rows += cnt[k];
        items += (cnt[k] + R - 1) / R;
    }
    int rows_total = 0, items_total = 0;
    int roff = block_exclusive_scan(rows, warp_sums, rows_total);
    int io = block_exclusive_scan(items, warp_sums, items_total);
    for (int k = k0; k < k1; ++k) {
        const int c = cnt[k];
        cur[k] = roff;
        ioff[k] = io;
        for (int t = 0; t * R < c; ++t) {
            RowItem it;
            it.adapter = k;
            it.p0 = roff + t * R;
            it.nrows = int16_t(min(R, c - t * R));
            it.rank = int16_t(a.rank[k]);
            it.scale = a.scale[k];
            a.items[io + t] = it;
        }
        roff += c;
        io += (c + R - 1) / R;
    }
    __syncthreads();
    for (int i = tid; i < a.n; i += kPlanThreads) {
        const int k = a.ids[i];
        if (k < 0 || k >= na || !a.ok[k])
            continue;
        a.perm[atomicAdd(&cur[k], 1)] = i;
    }
    if (tid == 0)
        *a.n_items = items_total;
}

}  // namespace

size_t dev_plan_smem_bytes(int n_adapters) { return size_t(3 * n_adapters + 32) * sizeof(int32_t); }

cudaError_t launch_plan_dev(const DevPlanArgs &a, cudaStream_t stream)
{
    if (a.n_adapters <= 0 || a.n_adapters > kDevPlanMaxAdapters || a.n < 0 || a.rows_per_item < 1)
        return cudaErrorInvalidValue;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_plan_dev, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(dev_plan_smem_bytes(kDevPlanMaxAdapters)));
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kPlanThreads);
    cfg.dynamicSmemBytes = dev_plan_smem_bytes(a.n_adapters);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_plan_dev, a);
}

}  // namespace lora
