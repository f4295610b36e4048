// Merge / unmerge on the 5th-generation tensor cores:
//     W[c, o] = bf16(W[c, o] + s * sum_j A[c, j] B[j, o])       (s < 0: unmerge)
// (VaLoRA blog, section 4.4.1: Delta W is computed at run time from the stored A
// and B with the batching operator and added to / subtracted from the base weight
// in one pass; here the product never exists in memory, it lives in TMEM).
//
// One CTA per 128 x 128 tile of W, 4 warps:
//   - thread 0 starts the TMA load of the W tile (two 64-column boxes, 128-byte
//     swizzle) and, once the operands are staged, issues the K = rank MMAs
//     (M = 128, N = 128, bf16 in, fp32 accumulate in TMEM) and commits them;
//   - all threads stage A's 128 x r block (column j of A = page j, so the operand is
//     M-major) and B's r x 128 block (row j of B = page j, N-major) from the pages
//     in the 128-byte-swizzled layout the MMA reads, ranks padded to 16 with zeros;
//   - epilogue: thread t owns row t = TMEM lane t, reads its accumulator 32 columns
//     at a time, adds it to the W row in shared memory, and the tile leaves with a
//     TMA store.
// The kernel streams W once in and once out; A and B come from L2 (every tile of a
// row block shares A, every tile of a column block shares B).
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "tc.cuh"
#include "tmap.h"

namespace lora {

namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kThreads = 128;
constexpr uint32_t kTmemCols = 128;

struct MergeTcArgs {
    CUtensorMap tmW;   // 64-byte aligned by its own declaration
    MergeParams p;
};

__host__ __device__ inline int rank_pad(int r) { return (r + 15) & ~15; }

__host__ __device__ inline uint32_t merge_smem_bytes(int r)
{
    const uint32_t rp = uint32_t(rank_pad(r));
    const uint32_t used = 1024u /* alignment slack */ + uint32_t(kBM) * kBN * 2u /* W */ +
                          rp * kBM * 2u /* A */ + rp * kBN * 2u /* B */ + 64u /* barriers */;
    // Keep every address the operand descriptors could form inside the allocation
    // even if the two descriptor strides were read the other way round.
    const uint32_t b_off = 1024u + uint32_t(kBM) * kBN * 2u + rp * kBM * 2u;
    const uint32_t reach = b_off + 2048u + (rp / 8u - 1u) * (rp / 8u) * 1024u + 64u;
    return used > reach ? used : reach;
}

__global__ void __launch_bounds__(kThreads) k_merge_tc(const __grid_constant__ MergeTcArgs args)
{
    const MergeParams &p = args.p;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);

    const int r = p.rank;
    const int rp = rank_pad(r);
    const uint32_t sW = base;                                // 2 boxes x 16 KB
    const uint32_t sA = sW + kBM * kBN * 2;                   // rp * 256 B
    const uint32_t sB = sA + uint32_t(rp) * kBM * 2;          // rp * 256 B
    const uint32_t sBar = sB + uint32_t(rp) * kBN * 2;
    const uint32_t bar_w = sBar, bar_mma = sBar + 8, tmem_slot = sBar + 16;
    uint8_t *gW = gbase;
    uint8_t *gA = gbase + (sA - base);
    uint8_t *gB = gbase + (sB - base);
    const uint32_t *g_tmem = reinterpret_cast<const uint32_t *>(gbase + (tmem_slot - base));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int o0 = blockIdx.x * kBN;
    const int c0 = blockIdx.y * kBM;
    const uint32_t lbo = uint32_t(rp / 8) * 1024u;   // stride between 64-wide M/N atoms
    const uint32_t sbo = 1024u;                       // stride between 8-deep K groups

    if (tid == 0) {
        mbar_init(bar_w, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0)
        tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *g_tmem;

    if (tid == 0) {
        mbar_arrive_expect_tx(bar_w, uint32_t(kBM) * kBN * 2u);
        tc::tma_load_2d(sW, &args.tmW, o0, c0, bar_w);
        tc::tma_load_2d(sW + kBM * 128, &args.tmW, o0 + 64, c0, bar_w);
    }

    // Stage A (M-major) and B (N-major) in the swizzled canonical layout.
    for (int q = tid; q < rp * 16; q += kThreads) {
        const int j = q >> 4, c16 = q & 15;
        uint4 va = make_uint4(0, 0, 0, 0), vb = make_uint4(0, 0, 0, 0);
        if (j < r) {
            const int cA = c0 + 8 * c16;
            if (cA + 8 <= p.d_in)
                va = *reinterpret_cast<const uint4 *>(p.a_pool + int64_t(p.a_pages[j]) * p.a_pw + cA);
            const int oB = o0 + 8 * c16;
            if (oB + 8 <= p.d_out)
                vb = *reinterpret_cast<const uint4 *>(p.b_pool + int64_t(p.b_pages[j]) * p.b_pw + oB);
        }
        const uint32_t off = uint32_t(c16 >> 3) * lbo + uint32_t(j >> 3) * 1024u +
                             tc::sw128(uint32_t(j & 7), uint32_t(c16 & 7));
        *reinterpret_cast<uint4 *>(gA + off) = va;
        *reinterpret_cast<uint4 *>(gB + off) = vb;
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    if (tid == 0) {
        constexpr uint32_t idesc = tc::idesc_bf16(kBM, kBN, 1, 1);
        for (int kk = 0; kk < rp / 16; ++kk) {
            const uint64_t da = tc::smem_desc_sw128(sA + uint32_t(kk) * 2u * sbo, lbo, sbo);
            const uint64_t db = tc::smem_desc_sw128(sB + uint32_t(kk) * 2u * sbo, lbo, sbo);
            tc::mma_bf16(tmem, da, db, idesc, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(bar_mma);
    }

    bool ok = mbar_wait_bounded(bar_mma, 0, p.status, kDevTimeoutMma);
    tc::fence_after_sync();
    ok = mbar_wait_bounded(bar_w, 0, p.status, kDevTimeoutLoad) && ok;
    ok = __syncthreads_and(ok);         // converged, one decision for the whole CTA

    if (ok) {
        const int row = warp * 32 + lane;   // TMEM lane == tile row
#pragma unroll 1
        for (int cc = 0; cc < kBN / 32; ++cc) {
            float acc[32];
            tc::tmem_ld32(tmem + (uint32_t(warp * 32) << 16) + uint32_t(cc * 32), acc);
            uint8_t *box = gW + (cc >> 1) * (kBM * 128);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 *ptr = reinterpret_cast<uint4 *>(
                    box + tc::sw128(uint32_t(row), uint32_t((cc & 1) * 4 + q)));
                float w[8];
                unpack8(*ptr, w);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    w[e] = fmaf(p.scale, acc[q * 8 + e], w[e]);
                *ptr = pack8(w);
            }
        }
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0 && ok) {
        tc::tma_store_2d(&args.tmW, o0, c0, sW);
        if (o0 + 64 < p.d_out)   // a box wholly right of d_out is not stored
            tc::tma_store_2d(&args.tmW, o0 + 64, c0, sW + kBM * 128);
        tc::bulk_commit();
        tc::bulk_wait_read0();
    }
    if (!ok) {
        // Do not release TMEM or leave while an MMA or a load may still be running.
        mbar_wait_bounded(bar_mma, 0, nullptr, 0);
        mbar_wait_bounded(bar_w, 0, nullptr, 0);
    }
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

bool merge_tc_supported(int d_in, int d_out, int rank)
{
    return rank >= 8 && rank <= 64 && d_in > 0 && d_out > 0 && merge_smem_bytes(rank) <= 227u * 1024u;
}

cudaError_t launch_merge_tc(const MergeParams &p, int /*n_split*/, cudaStream_t stream)
{
    MergeTcArgs args;
    args.p = p;
    if (!encode_bf16_2d(&args.tmW, p.W, uint64_t(p.d_out), uint64_t(p.d_in),
                        uint64_t(p.ldw) * 2u, 64, kBM, true))
        return cudaErrorInvalidValue;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_merge_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(merge_smem_bytes(64)));
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.d_out + kBN - 1) / kBN, (p.d_in + kBM - 1) / kBM);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = merge_smem_bytes(p.rank);
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, k_merge_tc, args);
}

}  // namespace lora
