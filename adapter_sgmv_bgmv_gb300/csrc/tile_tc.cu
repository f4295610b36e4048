// Tensor-core multi-LoRA tiles (prefill / SGMV-like case).
//
// Work unit: a tile of up to 128 consecutive rows of x / y that share adapter k
// (Punica groups the requests of a batch by adapter; long prompts give long runs).
//
// k_shrink_tc, ksplit CTAs per tile, CTA s covering the s-th share of the K blocks:
//   V[128 x r] (+)= X_tile[128 x K_s] . A_k[K_s x r]
//   warp 0   fills a ring of stages by TMA alone: per K block the X block (128 rows
//            x 64, 128-byte swizzle) and the matching A_k block -- row j of the
//            MMA's K-major B operand is a 64-element slice of page j of A_k, and in
//            the A row matrix (dense.cu) the pages are consecutive rows, so the
//            block is one to three boxes of 64 / 32 / 16 rows -- all counted on one
//            barrier;
//   warp 1   issues the tcgen05 MMAs (M = 128, N = r, K = 64 per stage) into a TMEM
//            accumulator and frees each stage with tcgen05.commit;
//   warps 2-5 read V from TMEM (row t = lane t) and write it as fp32: into the
//            CTA's partial slot (fused call; the expand sums the slots in order;
//            rank-padding columns written as zeros) or into the caller's v rows
//            (shrink-only call, one CTA per tile).
// A grid of at most one CTA per SM (the host picks the K-split so, where the tiles
// allow) takes a 200 KB ring; a larger grid is sized for two CTAs per SM (100 KB).  The kernel is launched as
// a programmatic dependent of the one before it: barrier set-up and the TMEM
// allocation overlap that kernel's tail, and the expand is released to start its
// own set-up once every CTA has issued its last MMA.
//
// The expand side is the streaming kernel in stream_tc.cu.
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "tc.cuh"
#include "tmap.h"

namespace lora {

namespace {

constexpr int kTM = 128;                       // rows per tile
constexpr int kKB = 64;                        // K elements per box (one 128-byte row)
constexpr int kSub = 2;                        // boxes per stage: 256 bytes of each x row
constexpr int kMaxStages = 8;
constexpr uint32_t kXBox = kTM * 128;          // 16 KB
constexpr uint32_t kXStage = kSub * kXBox;
constexpr uint32_t kRingBudget = 100u * 1024u; // two CTAs per SM
constexpr uint32_t kRingBudgetWide = 200u * 1024u;   // one CTA per SM (a grid of at most one per SM)

// Stage ring of the launch, sized by its largest padded rank: X block + A block.
struct ShrinkRing {
    uint32_t a_box, stage;
    int stages;
};
__host__ __device__ inline ShrinkRing shrink_ring(int max_rank, bool wide)
{
    ShrinkRing g;
    const int rpm = (max_rank + 15) & ~15;
    g.a_box = uint32_t(rpm) * 128u;
    g.stage = (kXStage + kSub * g.a_box + 1023u) & ~1023u;
    g.stages = int((wide ? kRingBudgetWide : kRingBudget) / g.stage);
    if (g.stages > kMaxStages)
        g.stages = kMaxStages;
    return g;
}
constexpr int kShrinkThreads = 192;

struct TileArgs {
    CUtensorMap map;                           // x, 64 x 128 boxes
    CUtensorMap amap[3];                       // the A row matrix, 64 x 16 / 32 / 64 boxes
    TileParams p;
};

__host__ __device__ inline int rank_pad16(int r) { return (r + 15) & ~15; }

__host__ __device__ inline uint32_t shrink_smem_bytes(int max_rank, bool wide)
{
    const ShrinkRing g = shrink_ring(max_rank, wide);
    return 1024u + uint32_t(g.stages) * g.stage + 2u * kMaxStages * 8u + 64u;
}

// ---------------------------------------------------------------------- shrink

__global__ void __launch_bounds__(kShrinkThreads, 2) k_shrink_tc(const __grid_constant__ TileArgs args)
{
    const TileParams &p = args.p;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const ShrinkRing ring = shrink_ring(p.max_tile_rank, p.wide_ring != 0);
    const int kStages = ring.stages;
    const uint32_t kStage = ring.stage;
    const uint32_t full0 = base + uint32_t(kStages) * kStage;
    const uint32_t empty0 = full0 + kMaxStages * 8;
    const uint32_t done = empty0 + kMaxStages * 8;
    const uint32_t tmem_slot = done + 8;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int KS = p.vmode == 0 ? p.ksplit : 1;
    const int tile = blockIdx.x / KS, ks = blockIdx.x - (blockIdx.x / KS) * KS;
    const TileItem it = tile_item(p, tile);
    const int r = it.rank, rp = rank_pad16(r);
    const int nkb_all = (p.d_in + kSub * kKB - 1) / (kSub * kKB);   // stages of kSub boxes
    const int per = (nkb_all + KS - 1) / KS;
    const int kb0 = ks * per;
    const int nkb = max(0, min(nkb_all, kb0 + per) - kb0);
    const uint32_t ncols = rp <= 32 ? 32u : rp <= 64 ? 64u : 128u;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);       // producer's expect-tx; X + A bytes
            mbar_init(empty0 + 8 * s, 1);      // MMA commit
        }
        mbar_init(done, 1);
        fence_mbar_init();
    }
    if (warp == 1)
        tc::tmem_alloc(tmem_slot, ncols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<const uint32_t *>(gbase + (tmem_slot - base));
    // Launched as a programmatic dependent: everything above overlapped the previous
    // kernel; x, the row matrix and the partial slots may be its to write or read.
    // With early_x the caller guarantees that it writes neither x nor the row matrix:
    // the loads and the MMAs (shared memory and TMEM only) then go ahead, and only
    // the epilogue, which writes global memory, waits.
    if (!p.early_x)
        grid_dep_wait();

    bool ok = true;
    if (warp == 0) {
        if (lane == 0) {
            for (int kb = 0; kb < nkb && ok; ++kb) {
                const int s = kb % kStages, u = kb / kStages;
                if (u > 0)
                    ok = mbar_wait_bounded(empty0 + 8 * s, (u - 1) & 1, p.status, kDevTimeoutPipe);
                if (!ok)
                    break;
                const uint32_t xs = base + uint32_t(s) * kStage, as = xs + kXStage;
                const int k0 = (kb0 + kb) * kSub * kKB;
                mbar_arrive_expect_tx(full0 + 8 * s, kXStage + kSub * uint32_t(rp) * 128u);
                for (int h = 0; h < kSub; ++h) {
                    tc::tma_load_2d(xs + h * kXBox, &args.map, k0 + h * kKB, it.row0, full0 + 8 * s);
                    tc::for_row_boxes(rp, [&](int off, int m) {
                        tc::tma_load_2d(as + uint32_t(h * rp + off) * 128u, &args.amap[m], k0 + h * kKB,
                                        it.a_row + off, full0 + 8 * s);
                    });
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16(kTM, rp, 0, 0);
            for (int kb = 0; kb < nkb && ok; ++kb) {
                const int s = kb % kStages, u = kb / kStages;
                ok = mbar_wait_bounded(full0 + 8 * s, u & 1, p.status, kDevTimeoutLoad);
                if (!ok)
                    break;
                tc::fence_after_sync();
                const uint32_t xs = base + uint32_t(s) * kStage, as = xs + kXStage;
#pragma unroll
                for (int h = 0; h < kSub; ++h)
#pragma unroll
                    for (int k4 = 0; k4 < kKB / 16; ++k4) {
                        const uint64_t da = tc::smem_desc_sw128(xs + h * kXBox + 32u * k4, 16u, 1024u);
                        const uint64_t db =
                            tc::smem_desc_sw128(as + uint32_t(h * rp) * 128u + 32u * k4, 16u, 1024u);
                        tc::mma_bf16(tmem, da, db, idesc, (kb > 0 || h > 0 || k4 > 0) ? 1u : 0u);
                    }
                tc::mma_commit(empty0 + 8 * s);
            }
            tc::mma_commit(done);
        }
        __syncwarp();
    } else {
        // Epilogue: this warp reads TMEM lanes 32*(warp%4) .. +31.
        ok = mbar_wait_bounded(done, 0, p.status, kDevTimeoutMma);
        if (p.early_x)
            grid_dep_wait();
        // The expand may start on freed SMs (and load y ahead of its own wait): the
        // kernel before this one has completed by now.
        if (tid == 64)
            grid_dep_launch();
        ok = __all_sync(0xffffffffu, ok);   // warp converged and agreed before tcgen05.ld
        tc::fence_after_sync();
        const int row = 32 * (warp & 3) + lane;
        float v[16];
        for (int c16 = 0; c16 < rp / 16; ++c16) {
            tc::tmem_ld16(tmem + (uint32_t(32 * (warp & 3)) << 16) + uint32_t(16 * c16), v);
            if (!ok)
                continue;
#pragma unroll
            for (int e = 0; e < 16; ++e)   // an empty K share, or a padded rank column
                if (nkb == 0 || 16 * c16 + e >= r)
                    v[e] = 0.f;
            if (p.vmode == 0) {
                // fp32 partial, row-major with row stride rp, in this CTA's slot
                float *dst = p.vparts + size_t(blockIdx.x) * (kVPartBytes / 4) + size_t(row) * rp +
                             16 * c16;
#pragma unroll
                for (int e = 0; e < 16; e += 4)
                    *reinterpret_cast<float4 *>(dst + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
            } else if (row < it.nrows) {
                float *dst = p.v + int64_t(it.row0 + row) * p.ldv + 16 * c16;
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (16 * c16 + e < r)
                        dst[e] = v[e];
            }
        }
    }
    if (!ok)
        mbar_wait_bounded(done, 0, nullptr, 0);   // no dealloc under a running MMA
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, ncols);
    }
}

}  // namespace

bool tile_tc_supported(int d_in, int d_out, int rank)
{
    return rank >= 8 && rank <= 128 && d_in >= 8 && d_out >= 8;
}

cudaError_t launch_shrink_tc(const TileParams &p, cudaStream_t stream)
{
    TileArgs args;
    args.p = p;
    if (!encode_bf16_2d(&args.map, p.x, uint64_t(p.d_in), uint64_t(p.n_rows), uint64_t(p.ldx) * 2u,
                        kKB, kTM, true) ||
        !encode_row_maps(args.amap, p.a_rows, uint64_t(p.d_in), p.a_nrows, p.a_ld))
        return cudaErrorInvalidValue;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_shrink_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             227 * 1024);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(p.n_items) * unsigned(p.vmode == 0 ? p.ksplit : 1));
    cfg.blockDim = dim3(kShrinkThreads);
    cfg.dynamicSmemBytes = shrink_smem_bytes(p.max_tile_rank, p.wide_ring != 0);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_shrink_tc, args);
}

}  // namespace lora
