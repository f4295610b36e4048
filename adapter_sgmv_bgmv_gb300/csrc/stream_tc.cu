// Streaming rank-r update of a 128-row block on the tensor cores, shared by the
// expand of the tile path and by the merge / unmerge mode switch:
//
//   expand:  y[rows, :] = bf16(y + s_k * V . B_k)       V = 128 x r   (per tile)
//   merge:   W[c0:c0+128, :] = bf16(W +/- s_k * A_k[c0:c0+128, :] . B_k)
//
// (BEE-30060, Background: the per-request term x_i A_i B_i; VaLoRA blog, section
// 4.4.1: Delta W = A B computed at run time and added to / subtracted from the
// base weight in one pass -- it never exists in memory, only one 128 x 128 block
// of it at a time in TMEM.)
//
// One CTA owns one 128-row block and a group of consecutive 128-column chunks:
//   - the left operand is staged once: V as the in-order sum of the shrink's fp32
//     partials or from the caller's fp32 rows, split into bf16 hi = bf16(v) and
//     lo = bf16(v - hi) (about 16 significant bits; the MMAs run on both), or A_k's
//     128 x r block from the pages (M-major, cp.async);
//   - a ring of NS stages holds, per chunk, B_k's r x 128 block (N-major, cp.async
//     from the pages) and the 128 x 128 y / W tile (two TMA boxes, 128-byte
//     swizzle); chunk i + NS - 1 is fetched while chunk i is computed;
//   - thread 0 issues the MMAs of a chunk (M = 128, N = 128, K = r per part) into
//     TMEM and commits them; all 128 threads (thread t = TMEM lane t = row t) read
//     the accumulator, add s * acc to the tile in shared memory, and the tile leaves
//     by TMA store (or row by row when only part of the block belongs to it).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"
#include "tc.cuh"
#include "tmap.h"

namespace lora {

namespace {

constexpr int kTM = 128;
constexpr int kBN = 128;
constexpr int kThreads = 320;          // producer, MMA, 8 epilogue warps
constexpr int kEpi = 256;
constexpr uint32_t kBox = kTM * 128;          // one 64-column TMA box of 128 rows
constexpr uint32_t kTile = 2 * kBox;          // 128 x 128 bf16
constexpr int kPrefetch = 8;                  // chunks pulled into L2 ahead of their load

enum Left : int { kLeftVParts = 0, kLeftVRows = 1, kLeftAPages = 2 };

struct StreamArgs {
    CUtensorMap map;                          // y (expand) or W (merge)
    TileParams p;                             // expand: items; merge: unused fields
    MergeParams m;                            // merge only
    int left;
    int chunks_per_cta;
    int n_chunks;
    int groups;                               // CTAs per 128-row block
    int stages;
};

__host__ __device__ inline int rank_pad16(int r) { return (r + 15) & ~15; }
__host__ __device__ inline int v_atoms(int rp) { return (rp + 63) / 64; }

// Shared memory: [left operand][stage 0: B | tile] ... [barriers]
__host__ __device__ inline uint32_t left_bytes(int left, int rp)
{
    return left == kLeftAPages ? uint32_t(rp) * kTM * 2u               // A: rp x 128, M-major
                               : 2u * uint32_t(v_atoms(rp)) * kBox;    // V hi + lo, K-major
}

__host__ __device__ inline uint32_t stage_bytes(int rp) { return uint32_t(rp) * kBN * 2u + kTile; }

__host__ __device__ inline uint32_t stream_smem_bytes(int left, int rp, int stages)
{
    return 1024u + left_bytes(left, rp) + uint32_t(stages) * stage_bytes(rp) + 128u;   // + barriers
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Warp roles: warp 0 producer (B chunks by cp.async, y / W tiles by TMA) running up
// to NS chunks ahead; warp 1 MMA issuer (two TMEM accumulators, so the MMAs of
// chunk i + 1 overlap the epilogue of chunk i); warps 2-9 stage the left operand,
// then run the epilogue (warp w reads TMEM lanes 32*(w%4).. and one 64-column half
// of the chunk, both TMEM loads in flight before one wait) and the stores; a stage
// is released one chunk later, once its store has read shared memory, so that wait
// stays off the critical path.
__global__ void __launch_bounds__(kThreads) k_stream_tc(const __grid_constant__ StreamArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- which block, which chunks
    const int blk = blockIdx.x / a.groups;
    const int grp = blockIdx.x - blk * a.groups;
    const int ch0 = grp * a.chunks_per_cta;
    const int nch = min(a.chunks_per_cta, a.n_chunks - ch0);
    int r, row0, nrows, d_out;
    float scale;
    const uint16_t *b_pool;
    int64_t b_pw;
    const int32_t *b_pages;
    unsigned *status;
    if (a.left == kLeftAPages) {
        r = a.m.rank;
        row0 = blk * kTM;
        nrows = min(kTM, a.m.d_in - row0);
        scale = a.m.scale;
        d_out = a.m.d_out;
        b_pool = a.m.b_pool;
        b_pw = a.m.b_pw;
        b_pages = a.m.b_pages;
        status = a.m.status;
    } else {
        const TileItem it = a.p.items[blk];
        r = it.rank;
        row0 = it.row0;
        nrows = it.nrows;
        scale = it.scale;
        d_out = a.p.d_out;
        b_pool = a.p.b_pool;
        b_pw = a.p.b_pw;
        b_pages = a.p.b_pages + size_t(it.adapter) * a.p.max_rank;
        status = a.p.status;
    }
    const int rp = rank_pad16(r);
    const int NS = a.stages;
    const uint32_t sL = base;
    const uint32_t sStage0 = sL + left_bytes(a.left, rp);
    const uint32_t sBar = sStage0 + uint32_t(NS) * stage_bytes(rp);
    // barriers: left, full[4], empty[4], tfull[2], tempty[2]
    const uint32_t bar_left = sBar;
    const uint32_t full0 = sBar + 8, empty0 = sBar + 40;
    const uint32_t tfull0 = sBar + 72, tempty0 = sBar + 88;
    const uint32_t tmem_slot = sBar + 104;
    const uint32_t lbo_b = uint32_t(rp / 8) * 1024u;   // N-atom stride of B (and M-atom of A)
    auto stage_b = [&](int c) { return sStage0 + uint32_t(c % NS) * stage_bytes(rp); };
    auto stage_t = [&](int c) { return stage_b(c) + uint32_t(rp) * kBN * 2u; };
    const bool full_rows = (a.left == kLeftAPages) || nrows == kTM;

    if (tid == 0) {
        mbar_init(bar_left, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(full0 + 8 * s, 2);       // producer lane 0 (B done) + TMA tx
            mbar_init(empty0 + 8 * s, 1);      // epilogue store has read the stage
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);      // MMA commit
            mbar_init(tempty0 + 8 * b, kEpi / 32);   // one arrive per epilogue warp
        }
        fence_mbar_init();
    }
    if (warp == 1)
        tc::tmem_alloc(tmem_slot, 2 * kBN);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<const uint32_t *>(gbase + (tmem_slot - base));
    const int atoms = v_atoms(rp);
    bool ok = true;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // The y / W tile of chunk i goes out by TMA at once; B of chunk i by
        // cp.async, and chunk i's "full" arrival is made one chunk later, once that
        // B group has landed, so the warp never waits on its own copies.  Tiles
        // kPrefetch chunks ahead are pulled into L2 first: the loads into shared
        // memory then see L2 latency, and DRAM sees many more requests in flight
        // than the stage ring could hold.
        auto prefetch_l2 = [&](int c) {
            const int n0 = (ch0 + c) * kBN;
            tc::tma_prefetch_2d(&a.map, n0, row0);
            if (n0 + 64 < d_out)
                tc::tma_prefetch_2d(&a.map, n0 + 64, row0);
        };
        if (lane == 0)
            for (int c = 0; c < kPrefetch && c < nch; ++c)
                prefetch_l2(c);
        for (int i = 0; i <= nch; ++i) {
            if (i < nch) {
                const int s = i % NS, u = i / NS;
                if (u > 0)
                    ok = mbar_wait_bounded(empty0 + 8 * s, uint32_t((u - 1) & 1), status,
                                           kDevTimeoutPipe) && ok;
                ok = __all_sync(0xffffffffu, ok);
                if (!ok)
                    break;
                const int n0 = (ch0 + i) * kBN;
                if (lane == 0) {
                    if (i + kPrefetch < nch)
                        prefetch_l2(i + kPrefetch);
                    mbar_arrive_expect_tx(full0 + 8 * s, kTile);
                    tc::tma_load_2d(stage_t(i), &a.map, n0, row0, full0 + 8 * s);
                    tc::tma_load_2d(stage_t(i) + kBox, &a.map, n0 + 64, row0, full0 + 8 * s);
                }
                const uint32_t sb = stage_b(i);
                for (int q = lane; q < rp * 16; q += 32) {
                    const int j = q >> 4, c16 = q & 15;
                    const int col = n0 + 8 * c16;
                    const bool valid = j < r && col + 8 <= d_out;
                    const uint32_t off = uint32_t(c16 >> 3) * lbo_b + uint32_t(j >> 3) * 1024u +
                                         tc::sw128(uint32_t(j & 7), uint32_t(c16 & 7));
                    tc::cp_async16(sb + off,
                                   valid ? b_pool + int64_t(b_pages[j]) * b_pw + col : b_pool,
                                   valid ? 16u : 0u);
                }
                tc::cp_async_commit();
            }
            if (i > 0) {
                if (i < nch)
                    tc::cp_async_wait<1>();     // B of chunk i - 1 has landed
                else
                    tc::cp_async_wait<0>();
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(full0 + 8 * ((i - 1) % NS));
            }
        }
        tc::cp_async_wait<0>();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            ok = mbar_wait_bounded(bar_left, 0, status, kDevTimeoutLoad);
            const uint32_t idesc = tc::idesc_bf16(kTM, kBN, a.left == kLeftAPages ? 1 : 0, 1);
            const int parts = a.left == kLeftAPages ? 1 : 2;
            for (int i = 0; i < nch && ok; ++i) {
                const int s = i % NS, b = i & 1;
                ok = mbar_wait_bounded(full0 + 8 * s, uint32_t((i / NS) & 1), status, kDevTimeoutLoad);
                if (ok && i >= 2)
                    ok = mbar_wait_bounded(tempty0 + 8 * b, uint32_t(((i >> 1) - 1) & 1), status,
                                           kDevTimeoutPipe);
                if (!ok)
                    break;
                tc::fence_after_sync();
                const uint32_t sb = stage_b(i);
                const uint32_t d = tmem + uint32_t(b * kBN);
                for (int part = 0; part < parts; ++part) {
                    for (int kk = 0; kk < rp / 16; ++kk) {
                        uint64_t dl;
                        if (a.left == kLeftAPages)
                            dl = tc::smem_desc_sw128(sL + uint32_t(kk) * 2048u, lbo_b, 1024u);
                        else
                            dl = tc::smem_desc_sw128(sL + uint32_t(part * atoms + (kk >> 2)) * kBox +
                                                         uint32_t(kk & 3) * 32u,
                                                     16u, 1024u);
                        const uint64_t db = tc::smem_desc_sw128(sb + uint32_t(kk) * 2048u, lbo_b, 1024u);
                        tc::mma_bf16(d, dl, db, idesc, (part > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                tc::mma_commit(tfull0 + 8 * b);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ left operand
        const int et = tid - 64;                 // 0..255
        if (a.left != kLeftAPages && et < kTM) {
            const int row = et;
            const int KS = a.left == kLeftVParts ? a.p.ksplit : 1;
            for (int c = 0; c < rp / 8; ++c) {
                float f[8], back[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    f[e] = 0.f;
                if (a.left == kLeftVParts) {
                    for (int ks = 0; ks < KS; ++ks) {
                        const float *src = a.p.vparts + (size_t(blk) * KS + ks) * (kVPartBytes / 4) +
                                           size_t(row) * rp + 8 * c;
                        const float4 lo4 = *reinterpret_cast<const float4 *>(src);
                        const float4 hi4 = *reinterpret_cast<const float4 *>(src + 4);
                        f[0] += lo4.x; f[1] += lo4.y; f[2] += lo4.z; f[3] += lo4.w;
                        f[4] += hi4.x; f[5] += hi4.y; f[6] += hi4.z; f[7] += hi4.w;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = 8 * c + e;
                        f[e] = (row < nrows && j < r) ? a.p.v[int64_t(row0 + row) * a.p.ldv + j] : 0.f;
                    }
                }
                const uint4 hv = pack8(f);
                unpack8(hv, back);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    f[e] -= back[e];
                const uint32_t off = tc::sw128(uint32_t(row), uint32_t(c & 7));
                *reinterpret_cast<uint4 *>(gbase + (sL - base) + (c >> 3) * kBox + off) = hv;
                *reinterpret_cast<uint4 *>(gbase + (sL - base) + (atoms + (c >> 3)) * kBox + off) =
                    pack8(f);
            }
            tc::fence_proxy_async_smem();
        } else if (a.left == kLeftAPages) {
            // A_k rows row0..row0+127, column j = page j: M-major, 64-row atoms.
            for (int q = et; q < rp * 16; q += kEpi) {
                const int j = q >> 4, c16 = q & 15;
                const int c = row0 + 8 * c16;
                const bool valid = j < r && c + 8 <= a.m.d_in;
                const uint32_t off = uint32_t(c16 >> 3) * lbo_b + uint32_t(j >> 3) * 1024u +
                                     tc::sw128(uint32_t(j & 7), uint32_t(c16 & 7));
                tc::cp_async16(sL + off,
                               valid ? a.m.a_pool + int64_t(a.m.a_pages[j]) * a.m.a_pw + c : a.m.a_pool,
                               valid ? 16u : 0u);
            }
            tc::cp_async_commit();
            tc::cp_async_wait<0>();
            tc::fence_proxy_async_smem();
        }
        named_bar_sync(1, kEpi);
        if (et == 0)
            mbar_arrive(bar_left);

        // ------------------------------------------------------------ epilogue
        const int q4 = warp & 3;                  // TMEM lanes 32*q4 .. 32*q4+31
        const int half = (warp - 2) >> 2;         // columns 64*half .. 64*half+63
        const int row = 32 * q4 + lane;
        for (int i = 0; i < nch; ++i) {
            const int s = i % NS, b = i & 1;
            ok = mbar_wait_bounded(tfull0 + 8 * b, uint32_t((i >> 1) & 1), status, kDevTimeoutMma) && ok;
            ok = mbar_wait_bounded(full0 + 8 * s, uint32_t((i / NS) & 1), status, kDevTimeoutLoad) && ok;
            ok = __all_sync(0xffffffffu, ok);
            if (!ok)
                break;
            tc::fence_after_sync();
            const uint32_t st = stage_t(i);
            uint32_t acc[2][32];
            const uint32_t ta = tmem + (uint32_t(32 * q4) << 16) + uint32_t(b * kBN + 64 * half);
            tc::tmem_ld32_nowait(ta, acc[0]);
            tc::tmem_ld32_nowait(ta + 32, acc[1]);
            tc::tmem_wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(tempty0 + 8 * b);      // accumulator b is free for chunk i + 2
            uint8_t *box = gbase + (st - base) + half * kBox;   // the 64-column TMA box
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 *ptr = reinterpret_cast<uint4 *>(
                        box + tc::sw128(uint32_t(row), uint32_t(cc * 4 + q)));
                    float t[8];
                    unpack8(*ptr, t);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        t[e] = fmaf(scale, __uint_as_float(acc[cc][q * 8 + e]), t[e]);
                    *ptr = pack8(t);
                }
            }
            tc::fence_proxy_async_smem();
            named_bar_sync(1, kEpi);
            const int n0 = (ch0 + i) * kBN;
            if (full_rows) {
                if (et == 0) {
                    tc::tma_store_2d(&a.map, n0, row0, st);
                    if (n0 + 64 < d_out)   // a box wholly right of the matrix is not stored
                        tc::tma_store_2d(&a.map, n0 + 64, row0, st + kBox);
                    tc::bulk_commit();
                    // the previous chunk's store has read its stage by now, usually
                    tc::bulk_wait_read1();
                    if (i > 0)
                        mbar_arrive(empty0 + 8 * ((i - 1) % NS));
                }
            } else {
                const int c16 = lane & 15;
                const int col = n0 + 8 * c16;
                for (int rr = (warp - 2) * 2 + (lane >> 4); rr < nrows; rr += kEpi / 16) {
                    if (col + 8 <= d_out) {
                        const uint4 val = *reinterpret_cast<const uint4 *>(
                            gbase + (st - base) + (c16 >> 3) * kBox +
                            tc::sw128(uint32_t(rr), uint32_t(c16 & 7)));
                        *reinterpret_cast<uint4 *>(a.p.y + int64_t(row0 + rr) * a.p.ldy + col) = val;
                    }
                }
                named_bar_sync(1, kEpi);
                if (et == 0)
                    mbar_arrive(empty0 + 8 * s);
            }
        }
        if (et == 0)
            tc::bulk_wait0();
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 2 * kBN);
    }
}

int pick_stages(int left, int rp)
{
    for (int ns = 4; ns >= 2; --ns)
        if (stream_smem_bytes(left, rp, ns) <= 227u * 1024u)
            return ns;
    return 0;
}

cudaError_t launch_stream(StreamArgs &a, int rp, int blocks, cudaStream_t stream, int sms)
{
    a.stages = pick_stages(a.left, rp);
    if (a.stages == 0)
        return cudaErrorInvalidValue;
    // Chunks per CTA: minimise (waves of CTAs) x (chunks per CTA + one chunk of
    // start-up), with as many CTAs per SM as shared memory allows.
    const uint32_t smem = stream_smem_bytes(a.left, rp, a.stages);
    const int64_t slots = int64_t(sms) * std::max<int64_t>(1, (228 * 1024) / (smem + 1024));
    int cpc = 1;
    int64_t best = -1;
    for (int c = 1; c <= a.n_chunks; ++c) {
        const int64_t ctas = int64_t(blocks) * ((a.n_chunks + c - 1) / c);
        const int64_t cost = ((ctas + slots - 1) / slots) * (c + 1);
        if (best < 0 || cost < best) {
            best = cost;
            cpc = c;
        }
    }
    a.chunks_per_cta = cpc;
    a.groups = (a.n_chunks + cpc - 1) / cpc;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_stream_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             227 * 1024);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks) * unsigned(a.groups));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = stream_smem_bytes(a.left, rp, a.stages);
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, k_stream_tc, a);
}

int device_sms()
{
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0)
            sms = 148;
    }
    return sms;
}

}  // namespace

cudaError_t launch_expand_tc(const TileParams &p, cudaStream_t stream)
{
    StreamArgs a{};
    a.p = p;
    a.left = p.vmode == 0 ? kLeftVParts : kLeftVRows;
    a.n_chunks = (p.d_out + kBN - 1) / kBN;
    if (!encode_bf16_2d(&a.map, p.y, uint64_t(p.d_out), uint64_t(p.n_rows), uint64_t(p.ldy) * 2u,
                        64, kTM, true))
        return cudaErrorInvalidValue;
    return launch_stream(a, rank_pad16(p.max_tile_rank), p.n_items, stream, device_sms());
}

bool merge_tc_supported(int d_in, int d_out, int rank)
{
    return rank >= 8 && rank <= 128 && d_in > 0 && d_out > 0 &&
           pick_stages(kLeftAPages, rank_pad16(rank)) > 0;
}

cudaError_t launch_merge_tc(const MergeParams &p, int /*n_split*/, cudaStream_t stream)
{
    StreamArgs a{};
    a.m = p;
    a.left = kLeftAPages;
    a.n_chunks = (p.d_out + kBN - 1) / kBN;
    if (!encode_bf16_2d(&a.map, p.W, uint64_t(p.d_out), uint64_t(p.d_in), uint64_t(p.ldw) * 2u,
                        64, kTM, true))
        return cudaErrorInvalidValue;
    return launch_stream(a, rank_pad16(p.rank), (p.d_in + kTM - 1) / kTM, stream, device_sms());
}

}  // namespace lora
