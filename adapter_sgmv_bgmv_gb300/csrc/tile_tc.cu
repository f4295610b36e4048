// Tensor-core multi-LoRA tiles (prefill / SGMV-like case).
//
// Work unit: a tile of up to 128 consecutive rows of x / y that share adapter k
// (Punica groups the requests of a batch by adapter; long prompts give long runs).
//
// k_shrink_tc, one CTA per tile:   V[128 x r] = X_tile[128 x d_in] . A_k[d_in x r]
//   warp 0   TMA-loads X K-blocks (128 rows x 64, 128-byte swizzle) into a ring of
//            stages;
//   warps 2-5 stage the matching A_k block from the pages (row j of the MMA's
//            K-major B operand = page j of A_k) with 16-byte cp.async, ranks padded
//            to 16 with zeros;
//   warp 1   issues the tcgen05 MMAs (M = 128, N = r, K = 64 per stage) into a TMEM
//            accumulator and frees each stage with tcgen05.commit;
//   warps 2-5 finally read V from TMEM (row t = lane t) and write it either as a
//            pair of bf16 tiles hi = bf16(v), lo = bf16(v - hi) already in the expand
//            MMA's operand layout, or as fp32 rows.
//
// k_expand_tc, one CTA per (tile, 128-column chunk of d_out):
//   y[rows, n0:n0+128] = bf16(y + s_k * V . B_k[:, n0:n0+128])
//   one bulk copy brings the V tiles, TMA brings the y tile, all threads stage B_k's
//   r x 128 block (N-major, from the pages), one thread issues the MMAs
//   acc = V_hi . B + V_lo . B (K = r each) into TMEM, so v enters with about 16
//   significant bits; the epilogue adds s * acc to the y tile in shared memory and
//   stores it with TMA when all 128 rows belong to the tile, else row by row.
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "tc.cuh"
#include "tmap.h"

namespace lora {

namespace {

constexpr int kTM = 128;                       // rows per tile
constexpr int kKB = 64;                        // K elements per stage (one 128-byte row)
constexpr int kStages = 5;
constexpr uint32_t kXStage = kTM * 128;        // 16 KB
constexpr uint32_t kAStage = 128 * 128;        // up to 128 ranks x 128 B
constexpr uint32_t kStage = kXStage + kAStage;
constexpr int kShrinkThreads = 192;
constexpr int kProducers = 128;                // warps 2..5
constexpr int kExpandThreads = 128;
constexpr int kBN = 128;                       // expand columns per CTA

struct TileArgs {
    CUtensorMap map;                           // x (shrink) or y (expand)
    TileParams p;
};

__host__ __device__ inline int rank_pad16(int r) { return (r + 15) & ~15; }

constexpr uint32_t shrink_smem_bytes()
{
    return 1024u + kStages * kStage + 2u * kStages * 8u + 64u + 4u * 128u;
}

// 64-rank atom columns of one V half (hi or lo) for a padded rank.
__host__ __device__ inline int v_atoms(int rp) { return (rp + 63) / 64; }

__host__ __device__ inline uint32_t expand_smem_bytes(int rp)
{
    return 1024u + 2u * uint32_t(v_atoms(rp)) * (kTM * 128u) /* V hi + lo */ +
           uint32_t(rp) * kBN * 2u /* B */ + uint32_t(kTM) * kBN * 2u /* y */ + 64u;
}

// ---------------------------------------------------------------------- shrink

__global__ void __launch_bounds__(kShrinkThreads, 1) k_shrink_tc(const __grid_constant__ TileArgs args)
{
    const TileParams &p = args.p;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t full0 = base + kStages * kStage;
    const uint32_t empty0 = full0 + kStages * 8;
    const uint32_t done = empty0 + kStages * 8;
    const uint32_t tmem_slot = done + 8;
    int32_t *s_pages = reinterpret_cast<int32_t *>(gbase + (tmem_slot + 64 - base));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const TileItem it = p.items[blockIdx.x];
    const int r = it.rank, rp = rank_pad16(r);
    const int nkb = (p.d_in + kKB - 1) / kKB;
    const uint32_t ncols = rp <= 32 ? 32u : rp <= 64 ? 64u : 128u;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, kProducers + 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(done, 1);
        fence_mbar_init();
    }
    if (tid < r)
        s_pages[tid] = p.a_pages[size_t(it.adapter) * p.max_rank + tid];
    if (warp == 1)
        tc::tmem_alloc(tmem_slot, ncols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<const uint32_t *>(gbase + (tmem_slot - base));

    bool ok = true;
    if (warp == 0) {
        if (lane == 0) {
            for (int kb = 0; kb < nkb && ok; ++kb) {
                const int s = kb % kStages, u = kb / kStages;
                if (u > 0)
                    ok = mbar_wait_bounded(empty0 + 8 * s, (u - 1) & 1, p.status, kDevTimeoutPipe);
                if (!ok)
                    break;
                mbar_arrive_expect_tx(full0 + 8 * s, kXStage);
                tc::tma_load_2d(base + s * kStage, &args.map, kb * kKB, it.row0, full0 + 8 * s);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16(kTM, rp, 0, 0);
            for (int kb = 0; kb < nkb && ok; ++kb) {
                const int s = kb % kStages, u = kb / kStages;
                ok = mbar_wait_bounded(full0 + 8 * s, u & 1, p.status, kDevTimeoutLoad);
                if (!ok)
                    break;
                tc::fence_after_sync();
                const uint32_t xs = base + s * kStage, as = xs + kXStage;
#pragma unroll
                for (int k4 = 0; k4 < kKB / 16; ++k4) {
                    const uint64_t da = tc::smem_desc_sw128(xs + 32u * k4, 16u, 1024u);
                    const uint64_t db = tc::smem_desc_sw128(as + 32u * k4, 16u, 1024u);
                    tc::mma_bf16(tmem, da, db, idesc, (kb > 0 || k4 > 0) ? 1u : 0u);
                }
                tc::mma_commit(empty0 + 8 * s);
            }
            tc::mma_commit(done);
        }
    } else {
        // A producers: 16-byte chunks of the r_pad x 64 block of A_k^T for each stage.
        const int t = tid - 64;
        const int nchunks = rp * 8;
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % kStages, u = kb / kStages;
            if (u > 0 && ok)
                ok = mbar_wait_bounded(empty0 + 8 * s, (u - 1) & 1, p.status, kDevTimeoutPipe);
            if (ok) {
                const uint32_t as = base + s * kStage + kXStage;
                for (int q = t; q < nchunks; q += kProducers) {
                    const int j = q >> 3, c = q & 7;
                    const int col = kb * kKB + c * 8;
                    const bool valid = j < r && col + 8 <= p.d_in;
                    const uint16_t *src = valid ? p.a_pool + int64_t(s_pages[j]) * p.a_pw + col
                                                : p.a_pool;
                    tc::cp_async16(as + tc::sw128(uint32_t(j), uint32_t(c)), src, valid ? 16u : 0u);
                }
            }
            tc::cp_async_commit();
            if (kb >= 2) {
                tc::cp_async_wait<2>();
                tc::fence_proxy_async_smem();
                mbar_arrive(full0 + 8 * ((kb - 2) % kStages));
            }
        }
        tc::cp_async_wait<0>();
        tc::fence_proxy_async_smem();
        for (int kb = nkb - 2 < 0 ? 0 : nkb - 2; kb < nkb; ++kb)
            mbar_arrive(full0 + 8 * (kb % kStages));

        // Epilogue: this warp reads TMEM lanes 32*(warp%4) .. +31.
        ok = mbar_wait_bounded(done, 0, p.status, kDevTimeoutMma) && ok;
        ok = __all_sync(0xffffffffu, ok);   // warp converged and agreed before tcgen05.ld
        tc::fence_after_sync();
        const int row = 32 * (warp & 3) + lane;
        float v[16];
        for (int c16 = 0; c16 < rp / 16; ++c16) {
            tc::tmem_ld16(tmem + (uint32_t(32 * (warp & 3)) << 16) + uint32_t(16 * c16), v);
            if (!ok)
                continue;
            if (p.vmode == 0) {
                // bf16 hi and lo, K-major 128-byte-swizzled: 64 ranks per 16 KB atom
                uint8_t *tile = reinterpret_cast<uint8_t *>(p.vtiles) +
                                size_t(blockIdx.x) * kVTileBytes;
                uint8_t *hi = tile + (c16 >> 2) * (kTM * 128);
                uint8_t *lo = tile + (v_atoms(rp) + (c16 >> 2)) * (kTM * 128);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t off = tc::sw128(uint32_t(row), uint32_t((c16 & 3) * 2 + h));
                    float rem[8];
                    const uint4 hv = pack8(v + 8 * h);
                    float back[8];
                    unpack8(hv, back);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        rem[e] = v[8 * h + e] - back[e];
                    *reinterpret_cast<uint4 *>(hi + off) = hv;
                    *reinterpret_cast<uint4 *>(lo + off) = pack8(rem);
                }
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

// ---------------------------------------------------------------------- expand

__global__ void __launch_bounds__(kExpandThreads) k_expand_tc(const __grid_constant__ TileArgs args)
{
    const TileParams &p = args.p;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_chunks = (p.d_out + kBN - 1) / kBN;
    const int item = blockIdx.x / n_chunks;
    const int n0 = (blockIdx.x - item * n_chunks) * kBN;
    const TileItem it = p.items[item];
    const int r = it.rank, rp = rank_pad16(r);
    const uint32_t lbo = uint32_t(rp / 8) * 1024u;     // N-atom stride of the B operand
    const int atoms = v_atoms(rp);
    const uint32_t sV = base;                          // hi atoms, then lo atoms
    const uint32_t sB = sV + 2u * atoms * (kTM * 128); // rp * 256 B
    const uint32_t sY = sB + uint32_t(rp) * kBN * 2u;  // 2 boxes x 16 KB
    const uint32_t bar_in = sY + kTM * kBN * 2u;
    const uint32_t bar_mma = bar_in + 8;
    const uint32_t tmem_slot = bar_in + 16;

    if (tid == 0) {
        mbar_init(bar_in, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0)
        tc::tmem_alloc(tmem_slot, kBN);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<const uint32_t *>(gbase + (tmem_slot - base));

    const uint32_t v_bytes = 2u * atoms * (kTM * 128);
    if (tid == 0) {
        mbar_arrive_expect_tx(bar_in, uint32_t(kTM) * kBN * 2u + (p.vmode == 0 ? v_bytes : 0u));
        tc::tma_load_2d(sY, &args.map, n0, it.row0, bar_in);
        tc::tma_load_2d(sY + kTM * 128, &args.map, n0 + 64, it.row0, bar_in);
        if (p.vmode == 0)
            bulk_g2s(sV, reinterpret_cast<const uint8_t *>(p.vtiles) + size_t(item) * kVTileBytes,
                     v_bytes, bar_in);
    }
    // B_k block: r x 128 columns, N-major, 64-column atoms.
    for (int q = tid; q < rp * 16; q += kExpandThreads) {
        const int j = q >> 4, c16 = q & 15;
        uint4 vb = make_uint4(0, 0, 0, 0);
        const int col = n0 + 8 * c16;
        if (j < r && col + 8 <= p.d_out)
            vb = *reinterpret_cast<const uint4 *>(
                p.b_pool + int64_t(p.b_pages[size_t(it.adapter) * p.max_rank + j]) * p.b_pw + col);
        const uint32_t off = uint32_t(c16 >> 3) * lbo + uint32_t(j >> 3) * 1024u +
                             tc::sw128(uint32_t(j & 7), uint32_t(c16 & 7));
        *reinterpret_cast<uint4 *>(gbase + (sB - base) + off) = vb;
    }
    if (p.vmode == 1) {
        // V from fp32 rows: row t of the tile, split into bf16 hi + lo.
        const int row = tid;
        for (int c = 0; c < rp / 8; ++c) {
            float f[8], back[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int j = 8 * c + e;
                f[e] = (row < it.nrows && j < r) ? p.v[int64_t(it.row0 + row) * p.ldv + j] : 0.f;
            }
            const uint4 hv = pack8(f);
            unpack8(hv, back);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                f[e] -= back[e];
            const uint32_t off = tc::sw128(uint32_t(row), uint32_t(c & 7));
            *reinterpret_cast<uint4 *>(gbase + (sV - base) + (c >> 3) * (kTM * 128) + off) = hv;
            *reinterpret_cast<uint4 *>(gbase + (sV - base) + (atoms + (c >> 3)) * (kTM * 128) +
                                       off) = pack8(f);
        }
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    bool ok = true;
    if (tid == 0) {
        ok = mbar_wait_bounded(bar_in, 0, p.status, kDevTimeoutLoad);
        if (ok) {
            const uint32_t idesc = tc::idesc_bf16(kTM, kBN, 0, 1);
            for (int part = 0; part < 2; ++part) {       // V_hi . B, then + V_lo . B
                const uint32_t vp = sV + uint32_t(part * atoms) * (kTM * 128);
                for (int kk = 0; kk < rp / 16; ++kk) {
                    const uint64_t dv = tc::smem_desc_sw128(
                        vp + uint32_t(kk >> 2) * (kTM * 128) + uint32_t(kk & 3) * 32u, 16u, 1024u);
                    const uint64_t db = tc::smem_desc_sw128(sB + uint32_t(kk) * 2048u, lbo, 1024u);
                    tc::mma_bf16(tmem, dv, db, idesc, (part > 0 || kk > 0) ? 1u : 0u);
                }
            }
        }
        tc::mma_commit(bar_mma);
    }
    ok = mbar_wait_bounded(bar_mma, 0, p.status, kDevTimeoutMma) && ok;
    tc::fence_after_sync();
    ok = mbar_wait_bounded(bar_in, 0, p.status, kDevTimeoutLoad) && ok;
    ok = __all_sync(0xffffffffu, ok);
    ok = __syncthreads_and(ok);         // one decision for the whole CTA

    if (ok) {
        const int row = warp * 32 + lane;
#pragma unroll 1
        for (int cc = 0; cc < kBN / 32; ++cc) {
            float acc[32];
            tc::tmem_ld32(tmem + (uint32_t(warp * 32) << 16) + uint32_t(cc * 32), acc);
            uint8_t *box = gbase + (sY - base) + (cc >> 1) * (kTM * 128);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 *ptr = reinterpret_cast<uint4 *>(
                    box + tc::sw128(uint32_t(row), uint32_t((cc & 1) * 4 + q)));
                float yv[8];
                unpack8(*ptr, yv);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    yv[e] = fmaf(it.scale, acc[q * 8 + e], yv[e]);
                *ptr = pack8(yv);
            }
        }
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (ok) {
        if (it.nrows == kTM) {
            if (tid == 0) {
                tc::tma_store_2d(&args.map, n0, it.row0, sY);
                if (n0 + 64 < p.d_out)   // a box wholly right of d_out is not stored
                    tc::tma_store_2d(&args.map, n0 + 64, it.row0, sY + kTM * 128);
                tc::bulk_commit();
                tc::bulk_wait_read0();
            }
        } else {
            // Only the rows of this tile: two rows per warp pass, 16 lanes x 16 B each.
            const int c16 = lane & 15;
            const int col = n0 + 8 * c16;
            for (int rr = warp * 2 + (lane >> 4); rr < it.nrows; rr += 8) {
                if (col + 8 <= p.d_out) {
                    const uint4 val = *reinterpret_cast<const uint4 *>(
                        gbase + (sY - base) + (c16 >> 3) * (kTM * 128) +
                        tc::sw128(uint32_t(rr), uint32_t(c16 & 7)));
                    *reinterpret_cast<uint4 *>(p.y + int64_t(it.row0 + rr) * p.ldy + col) = val;
                }
            }
        }
    } else {
        mbar_wait_bounded(bar_mma, 0, nullptr, 0);
        mbar_wait_bounded(bar_in, 0, nullptr, 0);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kBN);
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
                        kKB, kTM, true))
        return cudaErrorInvalidValue;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_shrink_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(shrink_smem_bytes()));
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(p.n_items));
    cfg.blockDim = dim3(kShrinkThreads);
    cfg.dynamicSmemBytes = shrink_smem_bytes();
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, k_shrink_tc, args);
}

cudaError_t launch_expand_tc(const TileParams &p, cudaStream_t stream)
{
    TileArgs args;
    args.p = p;
    if (!encode_bf16_2d(&args.map, p.y, uint64_t(p.d_out), uint64_t(p.n_rows), uint64_t(p.ldy) * 2u,
                        64, kTM, true))
        return cudaErrorInvalidValue;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_expand_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(expand_smem_bytes(128)));
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    const int n_chunks = (p.d_out + kBN - 1) / kBN;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(p.n_items) * unsigned(n_chunks));
    cfg.blockDim = dim3(kExpandThreads);
    cfg.dynamicSmemBytes = expand_smem_bytes(rank_pad16(p.max_tile_rank));
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, k_expand_tc, args);
}

}  // namespace lora
